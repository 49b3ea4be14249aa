// attn_bwd.cuh -- attention backward on sm_103a (included at the end of
// attn_fwd.cu, whose device helpers, waits and host set-up it shares).
//
// Gradients of O = softmax(scale Q K^T + mask) V (tang, section 3
// "Gradients are comprehensions": the backward is again contractions over
// the same scores; section 6: the flash backward identity
// D_i = sum_j P_ij dP_ij = dO_i . O_i):
//
//   P  = exp(scale S - LSE)           recomputed from the forward's LSE
//   dV = P^T dO      dP = dO V^T      dS = P o (dP - D)
//   dQ = scale dS K  dK = scale dS^T Q
//
// Three kernels: a row pass computes D = rowsum(dO o O) and LSE log2(e) into
// padded per-(batch, head) rows; the dK/dV kernel owns one 128-key block of
// one kv head and walks the query blocks (of every query head of its group),
// with S^T, dP^T, dV, dK in tensor memory; the dQ kernel owns one 128-row
// query block and walks the key blocks, with S, dP, dQ in tensor memory.
// Both recompute the scores, so no partial sums cross CTAs.  Per step the
// softmax warps turn the fp32 tiles into bf16 P^T / dS^T (dS) written over
// the scores they came from; the MMAs that follow read them from tensor
// memory.  The softmax works in two phases (P, then dS), and the next step's
// score product is issued between them, so it runs while dS is formed.
// Fixed and packed batches, d = 64 or 128.

namespace attn {
namespace bwd {

// producer, MMA issuer, 8 softmax warps (two per TMEM lane quarter, one per
// half of the 128 columns of a score tile)
constexpr int BWD_THREADS = 320;
constexpr int BWD_SM_WARPS = 8;

// Sequences: fixed batch (cu == nullptr) sequence b holds token rows
// b N .. b N + N - 1; packed, rows cu[b] .. cu[b+1] - 1.  In the padded row
// space each sequence starts at pstart[b] (whole 128-row blocks); per-row
// values live in [H, rows_pad] arrays with rows_pad = nb_max * 128.
struct BwdParams {
  __nv_bfloat16 *dq, *dk, *dv;
  const __nv_bfloat16 *o, *dout;
  const float *lse;      // the forward's LSE: fixed [B, Hq, N], packed [Hq, T]
  const int *cu;         // packed: cu_seqlens[B+1]; fixed: nullptr
  int *pstart;           // [B+1] padded start of each sequence (set-up pass)
  float *lse2;           // [Hq, rows_pad]: LSE log2(e); +inf on padding rows
  float *dsum;           // [Hq, rows_pad]: D = rowsum(dO o O); 0 on padding rows
                         // (the single pass stores both negated)
  float *dq_acc;         // single pass, d = 64: [Hq, rows_pad, 64] fp32 dS K sums
  int B, Hq, Hkv, N, T, nb_max, group, causal;
  float scale, scale_log2;
  unsigned long long timeout_ns;
  __device__ int rows_pad() const { return nb_max * BM; }
  __device__ int seq_start(int b) const { return cu ? __ldg(cu + b) : b * N; }
  __device__ int seq_len(int b) const { return cu ? __ldg(cu + b + 1) - __ldg(cu + b) : N; }
  __device__ long long lse_index(int b, int h, int i) const {
    return cu ? (long long)h * T + __ldg(cu + b) + i : ((long long)b * Hq + h) * N + i;
  }
};

// Set-up (one thread): padded sequence starts; inconsistent cu_seqlens are
// reported and then no sequence has rows (every unit exits).
__global__ void bwd_setup_kernel(const BwdParams p) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  bool good = !p.cu || (__ldg(p.cu) == 0 && __ldg(p.cu + p.B) == p.T);
  int acc = 0;
  for (int b = 0; b < p.B; ++b) {
    p.pstart[b] = acc;
    const int L = p.seq_len(b);
    if (L < 0) good = false;
    acc += good ? (L + BM - 1) / BM * BM : 0;
  }
  p.pstart[p.B] = acc;
  if (!good || acc > p.nb_max * BM) {
    record_status(ATTN_ERR_BAD_SEQLENS);
    for (int b = 0; b <= p.B; ++b) p.pstart[b] = 0;
  }
}

// The sequence holding padded row r (r < pstart[B]): the last b with
// pstart[b] <= r, by binary search.
__device__ __forceinline__ int seq_of_padded_row(const BwdParams &p, int r) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.pstart[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// A work unit of the dK/dV kernel (kv head, key block) or of the dQ kernel
// (query head, query block).  Heads run fastest, and the blocks come longest
// first so that the last CTAs the hardware schedules are the short ones:
// causal key blocks of the dK/dV kernel see fewer query blocks the later they
// sit in their sequence (ascending block order), query blocks of the dQ
// kernel see more (desc: descending).  Fixed batches order blocks by their
// index within the sequence across all sequences; packed batches by their
// place in the padded row space.  Blocks past the last sequence do nothing.
struct BUnit {
  bool valid;
  int head, seq, blk, start, len, nblk;
};
__device__ __forceinline__ BUnit bwd_unit(const BwdParams &p, int u, int heads, bool desc) {
  BUnit t{};
  t.head = u % heads;
  const int v = u / heads;   // the block's rank in the order above
  int r;                     // padded row of the block's first row
  if (!p.cu) {
    const int nb = (p.N + BM - 1) / BM;
    if (v >= nb * p.B) return t;
    const int blk = v / p.B;
    r = p.pstart[v % p.B] + (desc ? nb - 1 - blk : blk) * BM;
  } else {
    if (v >= p.nb_max) return t;
    r = (desc ? p.nb_max - 1 - v : v) * BM;
  }
  if (r >= p.pstart[p.B]) return t;
  t.seq = seq_of_padded_row(p, r);
  t.blk = (r - p.pstart[t.seq]) / BM;
  t.start = p.seq_start(t.seq);
  t.len = p.seq_len(t.seq);
  t.nblk = (t.len + BM - 1) / BM;
  t.valid = t.blk < t.nblk;
  return t;
}

template <int D>
struct BCfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr uint32_t TILE = CHUNKS * CHUNK_BYTES;   // one 128 x d bf16 tile
  static constexpr int STAGES = 2;
  // dK/dV kernel: K, V, then STAGES x {Q, dO, lse2 row, dsum row}
  static constexpr uint32_t A_SLOT = 2 * TILE + 1024;
  static constexpr uint32_t A_OFF_RING = 2 * TILE;
  static constexpr uint32_t A_OFF_CTL = A_OFF_RING + STAGES * A_SLOT;
  // dQ kernel: Q, dO, then a ring of K_STAGES K tiles and one of V_STAGES V
  // tiles (K is held from S to the dQ product, V only for dP, so K gets the
  // deeper ring: its load for a step starts two steps ahead)
  static constexpr int K_STAGES = 3, V_STAGES = 2;
  static constexpr uint32_t B_OFF_K = 2 * TILE;
  static constexpr uint32_t B_OFF_V = B_OFF_K + K_STAGES * TILE;
  static constexpr uint32_t B_OFF_CTL = B_OFF_V + V_STAGES * TILE;
  static constexpr uint32_t CTL_BYTES = 256;
  // at least 116 KB so that one CTA holds an SM (and all of its tensor memory)
  static constexpr uint32_t MIN_SMEM = 116u << 10;
  static constexpr uint32_t A_SMEM =
      A_OFF_CTL + CTL_BYTES + 1024 > MIN_SMEM ? A_OFF_CTL + CTL_BYTES + 1024 : MIN_SMEM;
  static constexpr uint32_t B_SMEM =
      B_OFF_CTL + CTL_BYTES + 1024 > MIN_SMEM ? B_OFF_CTL + CTL_BYTES + 1024 : MIN_SMEM;
  static_assert(A_SMEM <= 232448 && B_SMEM <= 232448, "shared memory");
  static_assert(256 + 2 * D <= (int)TMEM_COLS, "tensor memory");
};

// barriers of the control block
enum : int {
  B_STATIC_FULL = 0,   // K, V (dK/dV kernel) or Q, dO (dQ kernel) loaded
  B_FULL0,             // ring slot s loaded, s < 2
  B_FULL1,
  B_EMPTY0,            // ring slot s consumed (MMA commit)
  B_EMPTY1,
  B_DONE,              // the accumulators are final
  B_DRAIN,             // abort drain of the MMA issuer
  B_ST_FULL,           // the step's S^T (dK/dV kernel) or S (dQ kernel) in TMEM
  B_DPT_FULL,          // the step's dP^T or dP in TMEM
  B_PT_FULL,           // all softmax warps: P^T written over S^T (dK/dV), or S read (dQ)
  B_DST_FULL,          // all softmax warps: dS^T (dS) written over dP^T (dP)
  B_KFULL0,            // dQ kernel: K ring slot s loaded, s < 3 (B_FULL0/1 and
  B_KEMPTY0 = B_KFULL0 + 3,   // B_EMPTY0/1 serve its V ring); K slot s consumed
  B_DP1 = B_KEMPTY0 + 3,      // dQ kernel: dP in TMEM buffer 1 (B_DPT_FULL: buffer 0)
  B_DS1,                      // dQ kernel: dS written over buffer 1 (B_DST_FULL: 0)
  B_COUNT
};

// ------------------------------------------------------------------ row pass
// Eight lanes per (head, padded row), 16-byte loads: D = sum_c dO o O and
// LSE log2(e); padding rows of a sequence get D = 0 and +inf, which zeroes
// their P in the kernels.  SINGLE (single pass, d = 64): both values are
// stored negated (the kernel then adds them with packed fp32 instructions,
// which take no negated operands), and the row of the fp32 dQ buffer is
// zeroed as well.
template <int D, bool SINGLE = false>
__global__ void __launch_bounds__(256) bwd_rows_kernel(const BwdParams p) {
  const int lane = threadIdx.x & 31, seg = lane & 7;
  const long long row = (long long)blockIdx.x * 32 + (threadIdx.x >> 3);   // h rows_pad + r
  bool live = row < (long long)p.Hq * p.rows_pad();
  const int h = live ? (int)(row / p.rows_pad()) : 0;
  const int r = live ? (int)(row % p.rows_pad()) : 0;
  live = live && r < p.pstart[p.B];
  const int b = live ? seq_of_padded_row(p, r) : 0;
  const int i = r - p.pstart[b];
  const bool pad = live && i >= p.seq_len(b);
  if (SINGLE && live) {
    float4 *z = reinterpret_cast<float4 *>(p.dq_acc + row * 64 + seg * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  live = live && !pad;
  constexpr int PER = D / 8;   // elements per lane: PER / 8 loads of 16 bytes
  float acc = 0.f;
  if (live) {
    const long long off = ((long long)(p.seq_start(b) + i) * p.Hq + h) * D + seg * PER;
    const uint4 *po = reinterpret_cast<const uint4 *>(p.o + off);
    const uint4 *pd = reinterpret_cast<const uint4 *>(p.dout + off);
#pragma unroll
    for (int x = 0; x < PER / 8; ++x) {
      const uint4 a = __ldg(po + x), c = __ldg(pd + x);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        acc += __uint_as_float(wa[y] << 16) * __uint_as_float(wc[y] << 16);
        acc += __uint_as_float(wa[y] & 0xFFFF0000u) * __uint_as_float(wc[y] & 0xFFFF0000u);
      }
    }
  }
  for (int o = 4; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (seg == 0) {
    const float sg = SINGLE ? -1.f : 1.f;
    if (pad) {
      p.lse2[row] = sg * INFINITY;
      p.dsum[row] = 0.f;
    } else if (live) {
      p.dsum[row] = sg * acc;
      p.lse2[row] = sg * (p.lse[p.lse_index(b, h, i)] * 1.4426950408889634f);
    }
  }
}

// ------------------------------------------------------------------ shared pieces
struct BCtl {
  uint32_t bar0;
  uint32_t *words;   // [0] TMEM base, [1] abort flag
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

__device__ __forceinline__ void bwd_init_barriers(const BCtl &c) {
  mbar_init(c.bar(B_STATIC_FULL), 1);
  for (int s = 0; s < 2; ++s) {
    mbar_init(c.bar(B_FULL0 + s), 1);
    mbar_init(c.bar(B_EMPTY0 + s), 1);
  }
  mbar_init(c.bar(B_DONE), 1);
  mbar_init(c.bar(B_DRAIN), 1);
  mbar_init(c.bar(B_ST_FULL), 1);
  mbar_init(c.bar(B_DPT_FULL), 1);
  mbar_init(c.bar(B_PT_FULL), BWD_SM_WARPS);
  mbar_init(c.bar(B_DST_FULL), BWD_SM_WARPS);
  mbar_init(c.bar(B_DP1), 1);
  mbar_init(c.bar(B_DS1), BWD_SM_WARPS);
  for (int s = 0; s < 3; ++s) {
    mbar_init(c.bar(B_KFULL0 + s), 1);
    mbar_init(c.bar(B_KEMPTY0 + s), 1);
  }
  c.words[1] = 0u;
  mbar_init_fence();
}

// K-half h of A (bf16 pairs in TMEM at a_tmem + 64 h: each softmax warp
// writes its half over the first columns of the scores it read itself)
// times rows 64 h .. 64 h + 63 of B (N-major shared-memory tile), N = D,
// accumulated into d_tmem (overwritten by half 0 unless accumulate).
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              int h, bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(D, 1);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(d_tmem, a_tmem + 64u * (uint32_t)h + 8u * (uint32_t)kk,
           desc_add(bdesc, (4 * h + kk) * 2048), IDESC,
           (accumulate || h > 0 || kk > 0) ? 1u : 0u);
}

// issue_pv_half for an issuing warp (every lane, one elected lane issues).
template <int D>
__device__ __forceinline__ void issue_pv_half_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                   uint64_t bdesc, int h, bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(D, 1);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts_warp(d_tmem, a_tmem + 64u * (uint32_t)h + 8u * (uint32_t)kk,
                bdesc + (uint64_t)(((4 * h + kk) * 2048) >> 4), IDESC,
                (accumulate || h > 0 || kk > 0) ? 1u : 0u);
}

// Epilogue of one accumulator row: NCOLS fp32 columns * mul -> bf16, 16-byte
// stores (if live).
template <int NCOLS>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, float mul, __nv_bfloat16 *dst,
                                               bool live) {
#pragma unroll 1
  for (int cc = 0; cc < NCOLS; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
    uint32_t w[16];
#pragma unroll
    for (int x = 0; x < 16; ++x)
      w[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * mul, __uint_as_float(o[2 * x + 1]) * mul);
    if (live) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
      for (int x = 0; x < 4; ++x) d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
    }
  }
}

// ------------------------------------------------------------------ dK, dV
// Unit = (b, kv head, key block jb); steps = (query head of the group, query
// block ib), ib >= jb when causal.  TMEM: S^T [0,128) (P^T bf16 written over
// its first 64 columns), dP^T [128,256) (dS^T over its first 64), dV
// [256, 256+D), dK [256+D, 256+2D).
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl ctl;
  ctl.bar0 = base + C::A_OFF_CTL;
  ctl.words = reinterpret_cast<uint32_t *>(smem + C::A_OFF_CTL + 8 * B_COUNT);
  volatile uint32_t *abort_flag = ctl.words + 1;

  const BUnit un = bwd_unit(p, blockIdx.x, p.Hkv, false);
  if (!un.valid) return;   // uniform over the CTA, before any set-up
  const int jb = un.blk, kvh = un.head, b = un.seq;
  const int nblk = un.nblk, row0 = un.start, len = un.len;
  const int i0 = p.causal ? jb : 0;
  const int steps = p.group * (nblk - i0);
  const uint32_t k_s = base, v_s = base + C::TILE;

  if (warp == 1) {
    if (lane == 0) bwd_init_barriers(ctl);
    __syncwarp();
    tmem_alloc(smem_u32(ctl.words), TMEM_COLS);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_do);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.words[0];
  constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 256 + D;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(B_STATIC_FULL), 2 * C::TILE);
      for (int c = 0; c < C::CHUNKS; ++c) {
        tma_load_3d(k_s + c * CHUNK_BYTES, &tm_k, ctl.bar(B_STATIC_FULL), c * 64, kvh,
                    row0 + jb * BM);
        tma_load_3d(v_s + c * CHUNK_BYTES, &tm_v, ctl.bar(B_STATIC_FULL), c * 64, kvh,
                    row0 + jb * BM);
      }
      for (int s = 0; ok && s < steps; ++s) {
        const int slot = s & 1;
        if (s >= 2 && !(ok = wait_bounded(ctl.bar(B_EMPTY0 + slot), (uint32_t)((s - 2) >> 1) & 1u,
                                          abort_flag, p.timeout_ns)))
          break;
        const int h = kvh * p.group + s / (nblk - i0);
        const int ib = i0 + s % (nblk - i0);
        const uint32_t dst = base + C::A_OFF_RING + slot * C::A_SLOT;
        mbar_arrive_expect_tx(ctl.bar(B_FULL0 + slot), 2 * C::TILE + 1024);
        for (int c = 0; c < C::CHUNKS; ++c) {
          tma_load_3d(dst + c * CHUNK_BYTES, &tm_q, ctl.bar(B_FULL0 + slot), c * 64, h,
                      row0 + ib * BM);
          tma_load_3d(dst + C::TILE + c * CHUNK_BYTES, &tm_do, ctl.bar(B_FULL0 + slot), c * 64, h,
                      row0 + ib * BM);
        }
        const long long prow =
            (long long)h * p.rows_pad() + p.pstart[b] + (long long)ib * BM;   // 512-B aligned
        bulk_load(dst + 2 * C::TILE, p.lse2 + prow, 512, ctl.bar(B_FULL0 + slot));
        bulk_load(dst + 2 * C::TILE + 512, p.dsum + prow, 512, ctl.bar(B_FULL0 + slot));
        ++issued;
      }
      if (*abort_flag) {   // drain: bounded waits for the copies issued
        wait_drain(ctl.bar(B_STATIC_FULL), 0, p.timeout_ns);
        for (int s = 0; s < 2 && s < issued; ++s) {
          const int last = s + 2 * ((issued - 1 - s) / 2);
          wait_drain(ctl.bar(B_FULL0 + s), (uint32_t)(last >> 1) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer: the whole warp runs the loop, one elected lane issues each
    // tcgen05 instruction (a lone lane sharing its sub-partition with two
    // softmax warps issues far more slowly)
    {
      const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
      const uint64_t vdesc = smem_desc_sw128(v_s, 16, 1024);
      bool ok = wait_warp(ctl.bar(B_STATIC_FULL), 0, abort_flag, p.timeout_ns);
      // Per step s: S^T(s) and dP^T(s) in full; dV += P^T(s) dO once the
      // softmax warps have written P^T; then S^T(s+1) (S^T's columns are
      // free once dV(s) has read P^T: one thread's MMAs run in issue order)
      // while the softmax warps form dS^T(s); dK += dS^T(s) Q; then
      // dP^T(s+1).  So the next scores are computed while dS is formed.
      const uint32_t ring = base + C::A_OFF_RING;
      if (ok && steps > 0 &&
          (ok = wait_warp(ctl.bar(B_FULL0), 0, abort_flag, p.timeout_ns))) {
        tc_fence_after();
        issue_qk_warp<D>(tmem + COL_ST, kdesc, smem_desc_sw128(ring, 16, 1024));
        tc_commit_warp(ctl.bar(B_ST_FULL));
        issue_qk_warp<D>(tmem + COL_DPT, vdesc, smem_desc_sw128(ring + C::TILE, 16, 1024));
        tc_commit_warp(ctl.bar(B_DPT_FULL));
      }
      for (int s = 0; ok && s < steps; ++s) {
        const int slot = s & 1;
        const uint32_t q_s = ring + slot * C::A_SLOT;
        const uint32_t q_n = ring + (slot ^ 1) * C::A_SLOT;   // the next step's slot
        const uint64_t do_mn = smem_desc_sw128(q_s + C::TILE, CHUNK_BYTES, 1024);
        const uint64_t q_mn = smem_desc_sw128(q_s, CHUNK_BYTES, 1024);
        if (!(ok = wait_warp(ctl.bar(B_PT_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 0, s > 0);
        issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 1, s > 0);
        const bool more = s + 1 < steps;
        if (more) {
          if (!(ok = wait_warp(ctl.bar(B_FULL0 + (slot ^ 1)), (uint32_t)((s + 1) >> 1) & 1u,
                                  abort_flag, p.timeout_ns)))
            break;
          tc_fence_after();
          issue_qk_warp<D>(tmem + COL_ST, kdesc, smem_desc_sw128(q_n, 16, 1024));
          tc_commit_warp(ctl.bar(B_ST_FULL));
        }
        if (!(ok = wait_warp(ctl.bar(B_DST_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 0, s > 0);
        issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 1, s > 0);
        tc_commit_warp(ctl.bar(B_EMPTY0 + slot));   // Q(s), dO(s) and their rows are read
        if (more) {
          issue_qk_warp<D>(tmem + COL_DPT, vdesc, smem_desc_sw128(q_n + C::TILE, 16, 1024));
          tc_commit_warp(ctl.bar(B_DPT_FULL));
        }
      }
      if (ok) tc_commit_warp(ctl.bar(B_DONE));
      tc_commit_warp(ctl.bar(B_DRAIN));
      wait_drain(ctl.bar(B_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // softmax warps: thread = key row jb*128 + row of TMEM lane quarter warp%4,
    // query columns 64 hf .. 64 hf + 63
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    bool ok = true;
    for (int s = 0; ok && s < steps; ++s) {
      const int slot = s & 1;
      // the slot's rows (loaded long before) first, so that the wait on
      // S^T, which is on the step's critical path, is the last one
      if (!(ok = wait_warp(ctl.bar(B_FULL0 + slot), (uint32_t)(s >> 1) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(ctl.bar(B_ST_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = i0 + s % (nblk - i0);
      const float *lse2 =
          reinterpret_cast<const float *>(smem + C::A_OFF_RING + slot * C::A_SLOT + 2 * C::TILE);
      const float *dsum = lse2 + 128;
      const bool diag = p.causal && ib == jb;
      // phase 1: P^T = 2^(S^T c - LSE2) for this warp's 64 query columns,
      // bf16 over the first 32 of them; the bf16 P stays in registers for
      // phase 2 (dS uses P as the dV product does)
      uint32_t pw[2][16];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * hf + 32 * ch;
        uint32_t us[32];
        tmem_ld32(tmem + lane_off + COL_ST + c0, us);
        tmem_wait_ld();
        reg_fence32(us);
        // the mask test is taken out of the loop (only the diagonal block
        // needs it; inside the loop it cost more than the exponentials)
        if (!diag) {
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + c0 + x);
            pw[ch][x >> 1] = pack_bf16x2(ex2_approx(__uint_as_float(us[x]) * c - l4.x),
                                         ex2_approx(__uint_as_float(us[x + 1]) * c - l4.y));
            pw[ch][(x >> 1) + 1] = pack_bf16x2(ex2_approx(__uint_as_float(us[x + 2]) * c - l4.z),
                                               ex2_approx(__uint_as_float(us[x + 3]) * c - l4.w));
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            const int qc = c0 + x;
            float p0 = ex2_approx(__uint_as_float(us[x]) * c - lse2[qc]);
            float p1 = ex2_approx(__uint_as_float(us[x + 1]) * c - lse2[qc + 1]);
            // query ib*128 + qc sees key iff query >= key
            if (ib * BM + qc < key) p0 = 0.f;
            if (ib * BM + qc + 1 < key) p1 = 0.f;
            pw[ch][x >> 1] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(tmem + lane_off + COL_ST + 64 * hf + 16 * ch, pw[ch]);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(B_PT_FULL));
      // phase 2: dS^T = P^T o (dP^T - D), bf16 over the first 32 columns
      if (!(ok = wait_warp(ctl.bar(B_DPT_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * hf + 32 * ch;
        uint32_t ud[32];
        tmem_ld32(tmem + lane_off + COL_DPT + c0, ud);
        tmem_wait_ld();
        reg_fence32(ud);
        uint32_t dw[16];
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dsum + c0 + x);
          const uint32_t w0 = pw[ch][x >> 1], w1 = pw[ch][(x >> 1) + 1];
          float a0, a1, a2, a3;
          f2_unpack(f2_mul(bf16x2_widen(w0),
                           f2_add(f2_pack(__uint_as_float(ud[x]), __uint_as_float(ud[x + 1])),
                                  f2_pack(-d4.x, -d4.y))), a0, a1);
          f2_unpack(f2_mul(bf16x2_widen(w1),
                           f2_add(f2_pack(__uint_as_float(ud[x + 2]), __uint_as_float(ud[x + 3])),
                                  f2_pack(-d4.z, -d4.w))), a2, a3);
          dw[x >> 1] = pack_bf16x2(a0, a1);
          dw[(x >> 1) + 1] = pack_bf16x2(a2, a3);
        }
        tmem_st16(tmem + lane_off + COL_DPT + 64 * hf + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(B_DST_FULL));
    }
    if (ok && (ok = wait_warp(ctl.bar(B_DONE), 0, abort_flag, p.timeout_ns))) {
      tc_fence_after();
      const bool live = key < len;
      const long long off = ((long long)(row0 + key) * p.Hkv + kvh) * D + hf * (D / 2);
      store_row_bf16<D / 2>(tmem + lane_off + COL_DV + hf * (D / 2), 1.f, p.dv + off, live);
      store_row_bf16<D / 2>(tmem + lane_off + COL_DK + hf * (D / 2), p.scale, p.dk + off, live);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dQ
// Unit = (b, head h, query block ib); steps = key blocks jb (<= ib when
// causal).  TMEM: S [0,128), dP [128,256) (dS bf16 over its first 64
// columns), dQ [256, 256+D).
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl ctl;
  ctl.bar0 = base + C::B_OFF_CTL;
  ctl.words = reinterpret_cast<uint32_t *>(smem + C::B_OFF_CTL + 8 * B_COUNT);
  volatile uint32_t *abort_flag = ctl.words + 1;

  const BUnit un = bwd_unit(p, blockIdx.x, p.Hq, p.causal != 0);
  if (!un.valid) return;   // uniform over the CTA, before any set-up
  const int ib = un.blk, h = un.head, b = un.seq;
  const int row0 = un.start, len = un.len;
  const int kvh = h / p.group;
  const int steps = p.causal ? ib + 1 : un.nblk;
  const uint32_t q_s = base, do_s = base + C::TILE;

  if (warp == 1) {
    if (lane == 0) bwd_init_barriers(ctl);
    __syncwarp();
    tmem_alloc(smem_u32(ctl.words), TMEM_COLS);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_do);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.words[0];
  // S, two dP buffers (step s in buffer s & 1), dQ
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 384;
  static_assert(COL_DQ + D <= TMEM_COLS, "tensor memory");

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(B_STATIC_FULL), 2 * C::TILE);
      for (int c = 0; c < C::CHUNKS; ++c) {
        tma_load_3d(q_s + c * CHUNK_BYTES, &tm_q, ctl.bar(B_STATIC_FULL), c * 64, h,
                    row0 + ib * BM);
        tma_load_3d(do_s + c * CHUNK_BYTES, &tm_do, ctl.bar(B_STATIC_FULL), c * 64, h,
                    row0 + ib * BM);
      }
      int issued_v = 0;
      for (int s = 0; ok && s < steps; ++s) {
        const int ks = s % C::K_STAGES, vs = s % C::V_STAGES;
        if (s >= C::K_STAGES &&
            !(ok = wait_bounded(ctl.bar(B_KEMPTY0 + ks), (uint32_t)(s / C::K_STAGES - 1) & 1u,
                                abort_flag, p.timeout_ns)))
          break;
        const uint32_t kdst = base + C::B_OFF_K + ks * C::TILE;
        mbar_arrive_expect_tx(ctl.bar(B_KFULL0 + ks), C::TILE);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(kdst + c * CHUNK_BYTES, &tm_k, ctl.bar(B_KFULL0 + ks), c * 64, kvh,
                      row0 + s * BM);
        ++issued;
        // V slot vs held V(s - 2), read by dP(s - 2), whose buffer (s - 2) & 1 = vs
        // completes its barrier: that completion frees the slot (no commit of
        // its own; the barrier cannot run ahead, dP(s) needing V(s))
        static_assert(C::V_STAGES == 2, "V slots pair with the two dP buffers");
        if (s >= C::V_STAGES &&
            !(ok = wait_bounded(ctl.bar(vs ? B_DP1 : B_DPT_FULL),
                                (uint32_t)(s / C::V_STAGES - 1) & 1u, abort_flag, p.timeout_ns)))
          break;
        const uint32_t vdst = base + C::B_OFF_V + vs * C::TILE;
        mbar_arrive_expect_tx(ctl.bar(B_FULL0 + vs), C::TILE);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(vdst + c * CHUNK_BYTES, &tm_v, ctl.bar(B_FULL0 + vs), c * 64, kvh,
                      row0 + s * BM);
        ++issued_v;
      }
      if (*abort_flag) {
        wait_drain(ctl.bar(B_STATIC_FULL), 0, p.timeout_ns);
        for (int s = 0; s < C::K_STAGES && s < issued; ++s) {
          const int last = s + C::K_STAGES * ((issued - 1 - s) / C::K_STAGES);
          wait_drain(ctl.bar(B_KFULL0 + s), (uint32_t)(last / C::K_STAGES) & 1u, p.timeout_ns);
        }
        for (int s = 0; s < C::V_STAGES && s < issued_v; ++s) {
          const int last = s + C::V_STAGES * ((issued_v - 1 - s) / C::V_STAGES);
          wait_drain(ctl.bar(B_FULL0 + s), (uint32_t)(last / C::V_STAGES) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer: the whole warp, one elected lane issues (as in the dK/dV kernel)
    {
      const uint64_t qdesc = smem_desc_sw128(q_s, 16, 1024);
      const uint64_t dodesc = smem_desc_sw128(do_s, 16, 1024);
      bool ok = wait_warp(ctl.bar(B_STATIC_FULL), 0, abort_flag, p.timeout_ns);
      // Per step s: S(s+1) and dP(s+1) as soon as the softmax warps have read
      // S(s) (P is no operand here; dP(s+1) goes to the other dP buffer,
      // whose dS(s-1) the dQ product issued before has read: one thread's
      // MMAs run in issue order), then dQ += dS(s) K once they have written
      // dS over dP(s).  So the softmax warps never wait for a product of
      // their own step's chain.  A V slot is released when its dP product is
      // done, a K slot after dQ.
      const uint32_t kring = base + C::B_OFF_K, vring = base + C::B_OFF_V;
      if (ok && steps > 0 &&
          (ok = wait_warp(ctl.bar(B_KFULL0), 0, abort_flag, p.timeout_ns))) {
        tc_fence_after();
        issue_qk_warp<D>(tmem + COL_S, qdesc, smem_desc_sw128(kring, 16, 1024));
        tc_commit_warp(ctl.bar(B_ST_FULL));
        if ((ok = wait_warp(ctl.bar(B_FULL0), 0, abort_flag, p.timeout_ns))) {
          tc_fence_after();
          issue_qk_warp<D>(tmem + COL_DP, dodesc, smem_desc_sw128(vring, 16, 1024));
          tc_commit_warp(ctl.bar(B_DPT_FULL));
        }
      }
      for (int s = 0; ok && s < steps; ++s) {
        const int ks = s % C::K_STAGES, kn = (s + 1) % C::K_STAGES, vn = (s + 1) % C::V_STAGES;
        const uint32_t bn = (uint32_t)(s + 1) & 1u, bs = (uint32_t)s & 1u;
        const bool more = s + 1 < steps;
        if (!(ok = wait_warp(ctl.bar(B_PT_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
          break;
        if (more) {
          if (!(ok = wait_warp(ctl.bar(B_KFULL0 + kn), (uint32_t)((s + 1) / C::K_STAGES) & 1u,
                               abort_flag, p.timeout_ns)))
            break;
          tc_fence_after();
          issue_qk_warp<D>(tmem + COL_S, qdesc, smem_desc_sw128(kring + kn * C::TILE, 16, 1024));
          tc_commit_warp(ctl.bar(B_ST_FULL));
          if (!(ok = wait_warp(ctl.bar(B_FULL0 + vn), (uint32_t)((s + 1) / C::V_STAGES) & 1u,
                               abort_flag, p.timeout_ns)))
            break;
          tc_fence_after();
          issue_qk_warp<D>(tmem + COL_DP + 128u * bn, dodesc,
                           smem_desc_sw128(vring + vn * C::TILE, 16, 1024));
          tc_commit_warp(ctl.bar(bn ? B_DP1 : B_DPT_FULL));
        }
        // dS(s) over buffer s & 1 (one barrier per buffer: the softmax warps
        // may finish step s + 1 before this wait returns)
        if (!(ok = wait_warp(ctl.bar(bs ? B_DS1 : B_DST_FULL), (uint32_t)(s >> 1) & 1u,
                             abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        const uint64_t k_mn = smem_desc_sw128(kring + ks * C::TILE, CHUNK_BYTES, 1024);
        issue_pv_half_warp<D>(tmem + COL_DQ, tmem + COL_DP + 128u * bs, k_mn, 0, s > 0);
        issue_pv_half_warp<D>(tmem + COL_DQ, tmem + COL_DP + 128u * bs, k_mn, 1, s > 0);
        tc_commit_warp(ctl.bar(B_KEMPTY0 + ks));   // K(s) is read
      }
      if (ok) tc_commit_warp(ctl.bar(B_DONE));
      tc_commit_warp(ctl.bar(B_DRAIN));
      wait_drain(ctl.bar(B_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // softmax warps: thread = query row ib*128 + row, key columns 64 hf .. +63
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int qrow = ib * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    const long long prow = (long long)h * p.rows_pad() + p.pstart[b] + qrow;
    const float lse2 = p.lse2[prow];   // +inf on padding rows: P = 0
    const float dsum = p.dsum[prow];
    bool ok = true;
    for (int s = 0; ok && s < steps; ++s) {
      if (!(ok = wait_warp(ctl.bar(B_ST_FULL), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const bool edge = (s * BM + BM > len) || (p.causal && s == ib);
      // phase 1: this warp's 64 scores into registers, S released at once
      // (the next S is computed while P and dS are formed), then P
      float pv[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + lane_off + COL_S + 64 * hf, u0);
        tmem_ld32(tmem + lane_off + COL_S + 64 * hf + 32, u1);
        tmem_wait_ld();
        reg_fence32(u0);
        reg_fence32(u1);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          pv[x] = __uint_as_float(u0[x]);
          pv[32 + x] = __uint_as_float(u1[x]);
        }
      }
      tc_fence_before();
      warp_arrive(ctl.bar(B_PT_FULL));
      // the mask test is taken out of the loop (only the last block of a
      // sequence and the causal diagonal need it)
      if (!edge) {
        const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(-lse2, -lse2);
#pragma unroll
        for (int x = 0; x < 64; x += 2) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(pv[x], pv[x + 1]), c2, nl2), a0, a1);
          pv[x] = ex2_approx(a0);
          pv[x + 1] = ex2_approx(a1);
        }
      } else {
#pragma unroll
        for (int x = 0; x < 64; ++x) {
          const int k0 = s * BM + 64 * hf + x;
          float pe = ex2_approx(pv[x] * c - lse2);
          if (k0 >= len || (p.causal && k0 > qrow)) pe = 0.f;   // past the sequence, or causal
          pv[x] = pe;
        }
      }
      // phase 2: dS = P o (dP - D), bf16 over the first 32 of the 64 columns
      // of dP buffer s & 1
      const uint32_t bs = (uint32_t)s & 1u, col_dp = COL_DP + 128u * bs;
      if (!(ok = wait_warp(ctl.bar(bs ? B_DP1 : B_DPT_FULL), (uint32_t)(s >> 1) & 1u, abort_flag,
                           p.timeout_ns)))
        break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * hf + 32 * ch;
        uint32_t ud[32];
        tmem_ld32(tmem + lane_off + col_dp + c0, ud);
        tmem_wait_ld();
        reg_fence32(ud);
        uint32_t dw[16];
        const uint64_t nd2 = f2_pack(-dsum, -dsum);
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float a0, a1;
          f2_unpack(f2_mul(f2_pack(pv[32 * ch + x], pv[32 * ch + x + 1]),
                           f2_add(f2_pack(__uint_as_float(ud[x]), __uint_as_float(ud[x + 1])), nd2)),
                    a0, a1);
          dw[x >> 1] = pack_bf16x2(a0, a1);
        }
        tmem_st16(tmem + lane_off + col_dp + 64 * hf + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(bs ? B_DS1 : B_DST_FULL));
    }
    if (ok && (ok = wait_warp(ctl.bar(B_DONE), 0, abort_flag, p.timeout_ns))) {
      tc_fence_after();
      store_row_bf16<D / 2>(tmem + lane_off + COL_DQ + hf * (D / 2), p.scale,
                            p.dq + ((long long)(row0 + qrow) * p.Hq + h) * D + hf * (D / 2),
                            qrow < len);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace bwd
}  // namespace attn

#include "attn_bwd256.cuh"
#include "attn_bwd_fused.cuh"

// ------------------------------------------------------------------ host
namespace attn {
namespace bwd {
// Padded 128-row blocks of all sequences: B ceil(N / 128) for a fixed batch
// is at most ceil(rows / 128) + B, which also bounds a packed batch.
static long long bwd_nb_max(int B, long long rows) { return (rows + BM - 1) / BM + B; }

// Bytes of the fp32 dQ buffer of the single pass (d = 64), 0 otherwise.
static size_t bwd_acc_bytes(int B, int Hq, int N, int packed) {
  const long long rows = packed ? (long long)N : (long long)B * N;
  return (size_t)Hq * (size_t)bwd_nb_max(B, rows) * BM * 64 * sizeof(float);
}

// fp32 [rows, 64] buffer seen as boxes of 32 rows x 16 columns, 64-byte
// swizzle: the target of the single pass's reduce-adds.
static bool make_acc_map(EncodeTiledFn enc, CUtensorMap *m, float *base, long long rows) {
  cuuint64_t dims[2] = {64, (cuuint64_t)rows};
  cuuint64_t strides[1] = {64 * sizeof(float)};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Argument checks, the per-device shared-memory opt-in, the tensor maps of
// Q, dO, K, V and the parameters, shared by both backward entry points.
// single: the single pass (d = 64, the fp32 dQ buffer at the workspace's
// start).  Returns ATTN_OK with *empty set when there is nothing to do.
static attn_status bwd_prepare(const void *q, const void *k, const void *v, const void *o,
                               const void *dout, const float *lse, void *dq, void *dk,
                               void *dv, int B, int Hq, int Hkv, int N, int d, float scale,
                               int causal, const int *cu_seqlens, void *workspace,
                               size_t workspace_bytes, bool single, CUtensorMap (&maps)[5],
                               BwdParams &p, bool *empty) {
  *empty = false;
  if (B < 0 || N < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (single ? d != 64 : (d != 64 && d != 128 && d != 256)) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(dout, 16) || misaligned(dq, 16) || misaligned(dk, 16) || misaligned(dv, 16) ||
      misaligned(lse, 4) || misaligned(workspace, 16) || misaligned(cu_seqlens, 4))
    return ATTN_ERR_ALIGNMENT;
  const long long rows = cu_seqlens ? (long long)N : (long long)B * N;
  if (rows > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
  const long long nb_max = bwd_nb_max(B, rows);
  if (nb_max * BM * (long long)Hq > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
  const int packed = cu_seqlens ? 1 : 0;
  const size_t acc = single ? bwd_acc_bytes(B, Hq, N, packed) : 0;
  const size_t need = acc + attn_bwd_workspace_bytes(B, Hq, N, packed);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status st = prepare_device(dev);
  if (st != ATTN_OK) return st;
  {
    static std::mutex mu;
    static bool ready[MAX_DEVICES];
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      if (!opt_in_smem(attn_bwd_dkdv_kernel<64>, BCfg<64>::A_SMEM) ||
          !opt_in_smem(attn_bwd_dkdv_kernel<128>, BCfg<128>::A_SMEM) ||
          !opt_in_smem(attn_bwd_dq_kernel<64>, BCfg<64>::B_SMEM) ||
          !opt_in_smem(attn_bwd_dq_kernel<128>, BCfg<128>::B_SMEM) ||
          !opt_in_smem(attn_bwd_dv256_kernel, B256::V_SMEM) ||
          !opt_in_smem(attn_bwd_dk256_kernel, B256::K_SMEM) ||
          !opt_in_smem(attn_bwd_dq256_kernel, B256::Q_SMEM) ||
          !opt_in_smem(attn_bwd_fused_kernel, FCfg::SMEM))
        return ATTN_ERR_CUDA;
      ready[dev] = true;
    }
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  if (!make_map(enc, &maps[0], q, Hq, rows, d) || !make_map(enc, &maps[1], dout, Hq, rows, d) ||
      !make_map(enc, &maps[2], k, Hkv, rows, d) || !make_map(enc, &maps[3], v, Hkv, rows, d))
    return ATTN_ERR_INVALID_ARG;

  p = BwdParams{};
  p.dq = reinterpret_cast<__nv_bfloat16 *>(dq);
  p.dk = reinterpret_cast<__nv_bfloat16 *>(dk);
  p.dv = reinterpret_cast<__nv_bfloat16 *>(dv);
  p.o = reinterpret_cast<const __nv_bfloat16 *>(o);
  p.dout = reinterpret_cast<const __nv_bfloat16 *>(dout);
  p.lse = lse;
  p.cu = cu_seqlens;
  p.nb_max = (int)nb_max;
  p.dq_acc = single ? reinterpret_cast<float *>(workspace) : nullptr;
  p.lse2 = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + acc);
  p.dsum = p.lse2 + (size_t)Hq * nb_max * BM;
  p.pstart = reinterpret_cast<int *>(p.dsum + (size_t)Hq * nb_max * BM);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = cu_seqlens ? 0 : N;
  p.T = (int)rows;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  if (single && !make_acc_map(enc, &maps[4], p.dq_acc, (long long)Hq * nb_max * BM))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}
}  // namespace bwd
}  // namespace attn

extern "C" size_t attn_bwd_workspace_bytes(int B, int Hq, int N, int packed) {
  if (B < 1 || Hq < 1 || N < 1) return 0;
  const long long rows = packed ? (long long)N : (long long)B * N;
  const size_t rows_pad = (size_t)attn::bwd::bwd_nb_max(B, rows) * attn::BM;
  return 2 * (size_t)Hq * rows_pad * sizeof(float) + ((size_t)B + 1) * sizeof(int);
}

extern "C" attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, void *dq, void *dk,
                                void *dv, int B, int Hq, int Hkv, int N, int d, float scale,
                                int causal, const int *cu_seqlens, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  using namespace attn;
  using namespace attn::bwd;
  CUtensorMap maps[5];
  BwdParams p;
  bool empty = false;
  const attn_status st = bwd_prepare(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale,
                                     causal, cu_seqlens, workspace, workspace_bytes, false, maps,
                                     p, &empty);
  if (st != ATTN_OK || empty) return st;
  const CUtensorMap &mq = maps[0], &mdo = maps[1], &mk = maps[2], &mv = maps[3];
  const unsigned row_blocks = (unsigned)(((long long)Hq * p.nb_max * BM + 31) / 32);
  const unsigned kv_units = (unsigned)((long long)Hkv * p.nb_max);
  const unsigned q_units = (unsigned)((long long)Hq * p.nb_max);
  bwd_setup_kernel<<<1, 32, 0, stream>>>(p);
  if (d == 64) {
    bwd_rows_kernel<64><<<row_blocks, 256, 0, stream>>>(p);
    attn_bwd_dkdv_kernel<64><<<kv_units, BWD_THREADS, BCfg<64>::A_SMEM, stream>>>(mq, mdo, mk, mv, p);
    attn_bwd_dq_kernel<64><<<q_units, BWD_THREADS, BCfg<64>::B_SMEM, stream>>>(mq, mdo, mk, mv, p);
  } else if (d == 128) {
    bwd_rows_kernel<128><<<row_blocks, 256, 0, stream>>>(p);
    attn_bwd_dkdv_kernel<128><<<kv_units, BWD_THREADS, BCfg<128>::A_SMEM, stream>>>(mq, mdo, mk, mv, p);
    attn_bwd_dq_kernel<128><<<q_units, BWD_THREADS, BCfg<128>::B_SMEM, stream>>>(mq, mdo, mk, mv, p);
  } else {   // d = 256: dV, dK and dQ in three kernels (attn_bwd256.cuh)
    bwd_rows_kernel<256><<<row_blocks, 256, 0, stream>>>(p);
    // two-CTA clusters: a unit's steps split over the pair
    attn_bwd_dv256_kernel<<<2 * kv_units, BWD_THREADS, B256::V_SMEM, stream>>>(mq, mdo, mk, p);
    attn_bwd_dk256_kernel<<<2 * kv_units, BWD_THREADS, B256::K_SMEM, stream>>>(mq, mdo, mk, mv, p);
    attn_bwd_dq256_kernel<<<q_units, BWD_THREADS, B256::Q_SMEM, stream>>>(mq, mdo, mk, mv, p);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" size_t attn_bwd_single_pass_workspace_bytes(int B, int Hq, int N, int packed) {
  if (B < 1 || Hq < 1 || N < 1) return 0;
  return attn::bwd::bwd_acc_bytes(B, Hq, N, packed) + attn_bwd_workspace_bytes(B, Hq, N, packed);
}

extern "C" attn_status attn_bwd_single_pass(const void *q, const void *k, const void *v,
                                            const void *o, const void *dout, const float *lse,
                                            void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                                            int N, int d, float scale, int causal,
                                            const int *cu_seqlens, void *workspace,
                                            size_t workspace_bytes, cudaStream_t stream) {
  using namespace attn;
  using namespace attn::bwd;
  CUtensorMap maps[5];
  BwdParams p;
  bool empty = false;
  const attn_status st = bwd_prepare(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale,
                                     causal, cu_seqlens, workspace, workspace_bytes, true, maps,
                                     p, &empty);
  if (st != ATTN_OK || empty) return st;
  const unsigned row_blocks = (unsigned)(((long long)Hq * p.nb_max * BM + 31) / 32);
  const unsigned kv_units = (unsigned)((long long)Hkv * p.nb_max);
  bwd_setup_kernel<<<1, 32, 0, stream>>>(p);
  bwd_rows_kernel<64, true><<<row_blocks, 256, 0, stream>>>(p);
  attn_bwd_fused_kernel<<<kv_units, F_THREADS, FCfg::SMEM, stream>>>(maps[0], maps[1], maps[2],
                                                                      maps[3], maps[4], p);
  bwd_dq_convert_kernel<<<row_blocks, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
