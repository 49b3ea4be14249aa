// attn_bwd256.cuh -- attention backward at head dim 256 (included by
// attn_bwd.cuh, whose parameters, units, row pass and epilogue it shares).
//
// The gradients are those of attn_bwd.cuh (tang, section 3 "Gradients are
// comprehensions"; section 6, the flash backward identity D_i = dO_i . O_i).
// At d = 256 one 128 x 128 step of the d <= 128 dK/dV kernel would need K, V,
// Q and dO tiles of 64 KB each in shared memory (227 KB exist) and S^T, dP^T,
// dV and dK in 768 tensor-memory columns (512 exist), and its dQ kernel Q,
// dO, K and V.  So three kernels share the work, each within both budgets:
//
//   dV kernel: per 128-key block, S^T = K Q^T, P^T, dV += P^T dO
//              (K resident; Q, dO one slot each; TMEM S^T 128 + dV 256)
//   dK kernel: per 128-key block, S^T = K Q^T, dP^T = V dO^T, dS^T,
//              dK += dS^T Q (K, V resident; Q one slot; dO streamed in
//              64-column chunks through a two-slot ring, since only dP^T
//              reads it; TMEM S^T 128 + dP^T 128 + dK 256)
//   dQ kernel: per 128-row query block, S = Q K^T, dP = dO V^T, dS,
//              dQ += dS K (Q, dO resident; K one slot; V streamed in
//              64-column chunks, since only dP reads it; TMEM S 128 +
//              dP 128 + dQ 256)
//
// Per key/query block pair that is 16 products of 128^3 against the 10 of
// a single pass (the scores are formed three times, dP twice).  Warp roles as
// in attn_bwd.cuh: warp 0 producer, warp 1 MMA issue loop (one elected lane
// issues), warps 2-9 softmax (two per TMEM lane quarter, 64 columns each).
//
// A dV or dK unit (one kv head's 128-key block) walks group x blocks steps,
// up to 8 x 128 at 16k rows with 8 query heads per kv head -- longer than a
// whole SM's fair share when there are few kv heads.  So each unit runs on
// a two-CTA cluster: rank 0 takes the first half of the steps, rank 1 the
// second, and at the end rank 1 adds its fp32 partial accumulator into rank
// 0's shared memory (distributed shared memory), which rank 0 sums into its
// own before the bf16 store.

namespace attn {
namespace bwd {

struct B256 {
  static constexpr int D = 256;
  static constexpr uint32_t TILE = 4 * CHUNK_BYTES;   // 128 x 256 bf16
  static constexpr uint32_t CTL = 256;
  // dV kernel: K | Q | dO | two lse2 rows
  static constexpr uint32_t V_OFF_K = 0, V_OFF_Q = TILE, V_OFF_DO = 2 * TILE;
  static constexpr uint32_t V_OFF_ROWS = 3 * TILE, V_OFF_CTL = V_OFF_ROWS + 1024;
  // dK kernel: K | V | Q | dO chunk ring | lse2 and dsum rows
  static constexpr uint32_t K_OFF_K = 0, K_OFF_V = TILE, K_OFF_Q = 2 * TILE;
  static constexpr uint32_t K_OFF_RING = 3 * TILE, K_OFF_ROWS = K_OFF_RING + 2 * CHUNK_BYTES;
  static constexpr uint32_t K_OFF_CTL = K_OFF_ROWS + 1024;
  // dQ kernel: Q | dO | K | V chunk ring
  static constexpr uint32_t Q_OFF_Q = 0, Q_OFF_DO = TILE, Q_OFF_K = 2 * TILE;
  static constexpr uint32_t Q_OFF_RING = 3 * TILE, Q_OFF_CTL = Q_OFF_RING + 2 * CHUNK_BYTES;
  // + 1024 for the alignment of the dynamic shared memory
  static constexpr uint32_t V_SMEM = V_OFF_CTL + CTL + 1024;
  static constexpr uint32_t K_SMEM = K_OFF_CTL + CTL + 1024;
  static constexpr uint32_t Q_SMEM = Q_OFF_CTL + CTL + 1024;
  static_assert(V_SMEM <= 232448 && K_SMEM <= 232448 && Q_SMEM <= 232448, "shared memory");
};

enum : int {
  X_STATIC = 0,   // the unit's resident tiles loaded
  X_A_FULL,       // dV/dK: Q(s) and the step's rows loaded; dQ: K(s) loaded
  X_A_EMPTY,      // ... read by every product that needs it (commit)
  X_DO_FULL,      // dV kernel: dO(s) loaded
  X_DO_EMPTY,
  X_C_FULL0,      // chunk ring slot c loaded, c < 2
  X_C_FULL1,
  X_C_EMPTY0,     // chunk ring slot c read (commit)
  X_C_EMPTY1,
  X_ST_FULL,      // S^T (S) in TMEM (commit)
  X_DPT_FULL,     // dP^T (dP) in TMEM (commit)
  X_PT_FULL,      // all softmax warps: dV kernel P^T written; dQ kernel S read
  X_DST_FULL,     // all softmax warps: dS^T (dS) written over dP^T (dP)
  X_DONE,         // the accumulator is final (commit)
  X_DRAIN,        // teardown drain of the MMA warp
  X_R_FULL0,      // dV kernel: lse2 row slot r loaded, r < 2 (the softmax warps
  X_R_FULL1,      // wait on these, not on X_A_FULL, which may run a phase ahead)
  X_COUNT
};

__device__ __forceinline__ void x_init_barriers(const BCtl &c) {
  for (int i = 0; i < X_COUNT; ++i)
    mbar_init(c.bar(i), (i == X_PT_FULL || i == X_DST_FULL) ? BWD_SM_WARPS : 1);
  c.words[1] = 0u;
  mbar_init_fence();
}

// 64 contraction columns (one chunk) of a 128 x 128 score product into TMEM:
// A and B are K-major 128-row chunks (128-byte swizzle); `first`: overwrite.
__device__ __forceinline__ void issue_chunk_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 bool first) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BN, 0);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ss_warp(d_tmem, adesc + (uint64_t)(kk * 32 >> 4), bdesc + (uint64_t)(kk * 32 >> 4), IDESC,
                (first && kk == 0) ? 0u : 1u);
}

// Phase 1 of a key-row softmax warp (dV and dK kernels): P^T = 2^(S^T c -
// LSE2) for the warp's 64 query columns of step block ib, bf16 pairs into pw
// (diagonal blocks masked: query ib*128 + q sees key iff query >= key).
__device__ __forceinline__ void keyrow_p(const uint32_t (&us0)[32], const uint32_t (&us1)[32],
                                         const float *lse2, float c, bool diag, int ib, int hf,
                                         int key, uint32_t (&pw)[2][16]) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    const uint32_t *us = ch ? us1 : us0;
    const int c0 = 64 * hf + 32 * ch;
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
        if (ib * BM + qc < key) p0 = 0.f;
        if (ib * BM + qc + 1 < key) p1 = 0.f;
        pw[ch][x >> 1] = pack_bf16x2(p0, p1);
      }
    }
  }
}

// This warp's 64 columns of a 128-column fp32 TMEM tile at taddr.
__device__ __forceinline__ void load64(uint32_t taddr, uint32_t (&u0)[32], uint32_t (&u1)[32]) {
  tmem_ld32(taddr, u0);
  tmem_ld32(taddr + 32, u1);
  tmem_wait_ld();
  reg_fence32(u0);
  reg_fence32(u1);
}

// Pair exchange area: 128 rows x 256 fp32 (1 KB a row), the 16-byte pieces
// of a row XOR-swizzled by row % 8 so that a warp's 32 rows spread over
// every bank.
__device__ __forceinline__ uint32_t xch_addr(uint32_t area, int row, int piece) {
  return area + (uint32_t)row * 1024u + ((uint32_t)(piece ^ (row & 7)) << 4);
}

// Rank 1: this thread's 128 accumulator columns (half hf of the row) into
// the peer's exchange area.
__device__ __forceinline__ void pair_send(uint32_t taddr, uint32_t peer_area, int row, int hf) {
#pragma unroll 1
  for (int cc = 0; cc < 128; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
#pragma unroll
    for (int x = 0; x < 8; ++x)
      st_cluster_v4(xch_addr(peer_area, row, (hf * 128 + cc) / 4 + x),
                    make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]));
  }
}

// Rank 0: (own accumulator + the peer's partial, if it has one) * mul as
// bf16, 16-byte stores (if live).
__device__ __forceinline__ void pair_store(uint32_t taddr, uint32_t area, bool peer, int row,
                                           int hf, float mul, __nv_bfloat16 *dst, bool live) {
#pragma unroll 1
  for (int cc = 0; cc < 128; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
    float f[32];
#pragma unroll
    for (int x = 0; x < 32; ++x) f[x] = __uint_as_float(o[x]);
    if (peer) {
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint4 w = ld_shared_v4(xch_addr(area, row, (hf * 128 + cc) / 4 + x));
        f[4 * x] += __uint_as_float(w.x);
        f[4 * x + 1] += __uint_as_float(w.y);
        f[4 * x + 2] += __uint_as_float(w.z);
        f[4 * x + 3] += __uint_as_float(w.w);
      }
    }
    uint32_t w[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) w[x] = pack_bf16x2(f[2 * x] * mul, f[2 * x + 1] * mul);
    if (live) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
    }
  }
}

// The pair's share of a unit's steps: rank 0 [0, half), rank 1 [half, n).
struct PairSteps {
  int s0, n, peer_n;
};
__device__ __forceinline__ PairSteps pair_steps(int total, uint32_t rank) {
  const int half = (total + 1) >> 1;
  return rank ? PairSteps{half, total - half, half} : PairSteps{0, half, total - half};
}

// ------------------------------------------------------------------ dV
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dv256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl ctl;
  ctl.bar0 = base + C::V_OFF_CTL;
  ctl.words = reinterpret_cast<uint32_t *>(smem + C::V_OFF_CTL + 8 * X_COUNT);
  volatile uint32_t *abort_flag = ctl.words + 1;

  const uint32_t rank = cluster_ctarank();
  const BUnit un = bwd_unit(p, blockIdx.x >> 1, p.Hkv, false);
  if (!un.valid) return;   // uniform over the cluster, before any set-up
  const int jb = un.blk, kvh = un.head, b = un.seq;
  const int nblk = un.nblk, row0 = un.start, len = un.len;
  const int i0 = p.causal ? jb : 0;
  const PairSteps ps = pair_steps(p.group * (nblk - i0), rank);
  const int steps = ps.n;   // this CTA's steps t = 0 .. steps-1 are unit steps s0 + t
  const uint32_t k_s = base + C::V_OFF_K, q_s = base + C::V_OFF_Q, do_s = base + C::V_OFF_DO;
  bool have = false;   // softmax threads: this CTA's accumulator row is final
  constexpr uint32_t COL_ST = 0, COL_DV = 256;

  if (warp == 1) {
    if (lane == 0) x_init_barriers(ctl);
    __syncwarp();
    tmem_alloc(smem_u32(ctl.words), TMEM_COLS);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_do);
    tma_prefetch_map(&tm_k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.words[0];

  if (warp == 0) {
    // producer: K once; per step Q(s) with its lse2 row (row slot s & 1) once
    // S^T(s-1) has read Q(s-1), and dO(s) once dV(s-1) has read dO(s-1)
    if (lane == 0 && steps > 0) {
      int issued_a = 0, issued_do = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), C::TILE);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(k_s + c * CHUNK_BYTES, &tm_k, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
      for (int s = 0; ok && s < steps; ++s) {
        const int h = kvh * p.group + (ps.s0 + s) / (nblk - i0);
        const int ib = i0 + (ps.s0 + s) % (nblk - i0);
        if (s > 0 && !(ok = wait_bounded(ctl.bar(X_A_EMPTY), (uint32_t)(s - 1) & 1u, abort_flag,
                                         p.timeout_ns)))
          break;
        mbar_arrive_expect_tx(ctl.bar(X_A_FULL), C::TILE);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(q_s + c * CHUNK_BYTES, &tm_q, ctl.bar(X_A_FULL), c * 64, h, row0 + ib * BM);
        const long long prow = (long long)h * p.rows_pad() + p.pstart[b] + (long long)ib * BM;
        mbar_arrive_expect_tx(ctl.bar(X_R_FULL0 + (s & 1)), 512);
        bulk_load(base + C::V_OFF_ROWS + (s & 1) * 512, p.lse2 + prow, 512,
                  ctl.bar(X_R_FULL0 + (s & 1)));
        ++issued_a;
        if (s > 0 && !(ok = wait_bounded(ctl.bar(X_DO_EMPTY), (uint32_t)(s - 1) & 1u, abort_flag,
                                         p.timeout_ns)))
          break;
        mbar_arrive_expect_tx(ctl.bar(X_DO_FULL), C::TILE);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(do_s + c * CHUNK_BYTES, &tm_do, ctl.bar(X_DO_FULL), c * 64, h,
                      row0 + ib * BM);
        ++issued_do;
      }
      if (*abort_flag) {   // drain: bounded waits for the copies issued
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        if (issued_a > 0) wait_drain(ctl.bar(X_A_FULL), (uint32_t)(issued_a - 1) & 1u, p.timeout_ns);
        if (issued_do > 0)
          wait_drain(ctl.bar(X_DO_FULL), (uint32_t)(issued_do - 1) & 1u, p.timeout_ns);
        for (int sl = 0; sl < 2 && sl < issued_a; ++sl) {
          const int last = sl + 2 * ((issued_a - 1 - sl) / 2);
          wait_drain(ctl.bar(X_R_FULL0 + sl), (uint32_t)(last >> 1) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp: per step S^T(s) (it overwrites P^T(s-1), which dV(s-1),
    // issued before, has read), then dV += P^T(s) dO(s) once P^T is written
    const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
    const uint64_t qdesc = smem_desc_sw128(q_s, 16, 1024);
    const uint64_t do_mn = smem_desc_sw128(do_s, CHUNK_BYTES, 1024);
    if (steps > 0) {
      bool ok = wait_warp(ctl.bar(X_STATIC), 0, abort_flag, p.timeout_ns);
      for (int s = 0; ok && s < steps; ++s) {
        const uint32_t par = (uint32_t)s & 1u;
        if (!(ok = wait_warp(ctl.bar(X_A_FULL), par, abort_flag, p.timeout_ns))) break;
        tc_fence_after();
        issue_qk_warp<D>(tmem + COL_ST, kdesc, qdesc);
        tc_commit_warp(ctl.bar(X_ST_FULL));
        tc_commit_warp(ctl.bar(X_A_EMPTY));   // Q(s) is read
        if (!(ok = wait_warp(ctl.bar(X_PT_FULL), par, abort_flag, p.timeout_ns)) ||
            !(ok = wait_warp(ctl.bar(X_DO_FULL), par, abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 0, s > 0);
        issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 1, s > 0);
        tc_commit_warp(ctl.bar(X_DO_EMPTY));   // dO(s) and P^T(s) are read
      }
      if (ok) tc_commit_warp(ctl.bar(X_DONE));
      tc_commit_warp(ctl.bar(X_DRAIN));
      wait_drain(ctl.bar(X_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // softmax warps: thread = key row jb*128 + row, query columns 64 hf .. +63
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    bool ok = steps > 0;
    for (int s = 0; ok && s < steps; ++s) {
      const uint32_t par = (uint32_t)s & 1u;
      // the step's lse2 row (slot s & 1), then S^T(s)
      if (!(ok = wait_warp(ctl.bar(X_R_FULL0 + (s & 1)), (uint32_t)(s >> 1) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(ctl.bar(X_ST_FULL), par, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = i0 + (ps.s0 + s) % (nblk - i0);
      const float *lse2 = reinterpret_cast<const float *>(smem + C::V_OFF_ROWS + (s & 1) * 512);
      uint32_t us0[32], us1[32], pw[2][16];
      load64(tmem + lane_off + COL_ST + 64 * hf, us0, us1);
      keyrow_p(us0, us1, lse2, c, p.causal && ib == jb, ib, hf, key, pw);
      // P^T bf16 over the first 32 of this warp's 64 score columns
      tmem_st16(tmem + lane_off + COL_ST + 64 * hf, pw[0]);
      tmem_st16(tmem + lane_off + COL_ST + 64 * hf + 16, pw[1]);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(X_PT_FULL));
    }
    if (ok && wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns)) {
      tc_fence_after();
      have = true;
    }
  }
  // every product of both CTAs is complete: rank 0's Q and dO tiles are free
  cluster_sync_all();
  if (warp >= 2) {
    const int row = (warp & 3) * 32 + lane, hf = (warp - 2) >> 2;
    const uint32_t acc = tmem + ((uint32_t)((warp & 3) * 32) << 16) + COL_DV + hf * (D / 2);
    if (rank == 1 && have) pair_send(acc, mapa_shared(q_s, 0), row, hf);
    cluster_sync_all();   // rank 1's partial is in rank 0's exchange area
    if (rank == 0 && have) {
      const long long off = ((long long)(row0 + jb * BM + row) * p.Hkv + kvh) * D + hf * (D / 2);
      pair_store(acc, q_s, ps.peer_n > 0, row, hf, 1.f, p.dv + off, jb * BM + row < len);
    }
  } else {
    cluster_sync_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dK
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dk256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl ctl;
  ctl.bar0 = base + C::K_OFF_CTL;
  ctl.words = reinterpret_cast<uint32_t *>(smem + C::K_OFF_CTL + 8 * X_COUNT);
  volatile uint32_t *abort_flag = ctl.words + 1;

  const uint32_t rank = cluster_ctarank();
  const BUnit un = bwd_unit(p, blockIdx.x >> 1, p.Hkv, false);
  if (!un.valid) return;   // uniform over the cluster
  const int jb = un.blk, kvh = un.head, b = un.seq;
  const int nblk = un.nblk, row0 = un.start, len = un.len;
  const int i0 = p.causal ? jb : 0;
  const PairSteps ps = pair_steps(p.group * (nblk - i0), rank);
  const int steps = ps.n;
  const uint32_t k_s = base + C::K_OFF_K, v_s = base + C::K_OFF_V, q_s = base + C::K_OFF_Q;
  bool have = false;
  const uint32_t ring = base + C::K_OFF_RING;
  constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DK = 256;

  if (warp == 1) {
    if (lane == 0) x_init_barriers(ctl);
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

  if (warp == 0) {
    // producer: K, V once; per step the first two dO(s) chunks, Q(s) with its
    // rows once dK(s-1) has read Q(s-1), then the last two dO chunks (dO
    // chunk position 4 s + c goes to ring slot (4 s + c) % 2)
    if (lane == 0 && steps > 0) {
      int issued = 0, cpos = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), 2 * C::TILE);
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(k_s + c * CHUNK_BYTES, &tm_k, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
        tma_load_3d(v_s + c * CHUNK_BYTES, &tm_v, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
      }
      for (int s = 0; ok && s < steps; ++s) {
        const int h = kvh * p.group + (ps.s0 + s) / (nblk - i0);
        const int ib = i0 + (ps.s0 + s) % (nblk - i0);
        for (int c = 0; ok && c < 4; ++c, ++cpos) {
          if (c == 2) {   // Q(s) and the step's rows
            if (s > 0 && !(ok = wait_bounded(ctl.bar(X_A_EMPTY), (uint32_t)(s - 1) & 1u,
                                             abort_flag, p.timeout_ns)))
              break;
            mbar_arrive_expect_tx(ctl.bar(X_A_FULL), C::TILE + 1024);
            for (int cc = 0; cc < 4; ++cc)
              tma_load_3d(q_s + cc * CHUNK_BYTES, &tm_q, ctl.bar(X_A_FULL), cc * 64, h,
                          row0 + ib * BM);
            const long long prow =
                (long long)h * p.rows_pad() + p.pstart[b] + (long long)ib * BM;
            bulk_load(base + C::K_OFF_ROWS, p.lse2 + prow, 512, ctl.bar(X_A_FULL));
            bulk_load(base + C::K_OFF_ROWS + 512, p.dsum + prow, 512, ctl.bar(X_A_FULL));
            ++issued;
          }
          const int slot = cpos & 1;
          if (cpos >= 2 && !(ok = wait_bounded(ctl.bar(X_C_EMPTY0 + slot),
                                               (uint32_t)((cpos >> 1) - 1) & 1u, abort_flag,
                                               p.timeout_ns)))
            break;
          mbar_arrive_expect_tx(ctl.bar(X_C_FULL0 + slot), CHUNK_BYTES);
          tma_load_3d(ring + slot * CHUNK_BYTES, &tm_do, ctl.bar(X_C_FULL0 + slot), c * 64, h,
                      row0 + ib * BM);
        }
      }
      if (*abort_flag) {
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        if (issued > 0) wait_drain(ctl.bar(X_A_FULL), (uint32_t)(issued - 1) & 1u, p.timeout_ns);
        for (int sl = 0; sl < 2 && sl < cpos; ++sl) {
          const int last = sl + 2 * ((cpos - 1 - sl) / 2);
          wait_drain(ctl.bar(X_C_FULL0 + sl), (uint32_t)(last >> 1) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp, per step: dP^T(s) = V dO(s)^T chunk by chunk (its columns
    // are free: dK(s-1), issued before, has read dS^T(s-1)), S^T(s) = K Q^T
    // once Q(s) landed (the softmax warps loaded S^T(s-1) before they wrote
    // dS^T(s-1)), dK += dS^T(s) Q(s) once dS^T is written
    const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
    const uint64_t qdesc = smem_desc_sw128(q_s, 16, 1024);
    const uint64_t q_mn = smem_desc_sw128(q_s, CHUNK_BYTES, 1024);
    bool ok = steps > 0 && wait_warp(ctl.bar(X_STATIC), 0, abort_flag, p.timeout_ns);
    int cpos = 0;
    for (int s = 0; ok && s < steps; ++s) {
      const uint32_t par = (uint32_t)s & 1u;
      for (int c = 0; ok && c < 4; ++c, ++cpos) {
        const int slot = cpos & 1;
        if (!(ok = wait_warp(ctl.bar(X_C_FULL0 + slot), (uint32_t)(cpos >> 1) & 1u, abort_flag,
                             p.timeout_ns)))
          break;
        tc_fence_after();
        issue_chunk_warp(tmem + COL_DPT, smem_desc_sw128(v_s + c * CHUNK_BYTES, 16, 1024),
                         smem_desc_sw128(ring + slot * CHUNK_BYTES, 16, 1024), c == 0);
        tc_commit_warp(ctl.bar(X_C_EMPTY0 + slot));
      }
      if (!ok) break;
      tc_commit_warp(ctl.bar(X_DPT_FULL));
      if (!(ok = wait_warp(ctl.bar(X_A_FULL), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_qk_warp<D>(tmem + COL_ST, kdesc, qdesc);
      tc_commit_warp(ctl.bar(X_ST_FULL));
      if (!(ok = wait_warp(ctl.bar(X_DST_FULL), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 0, s > 0);
      issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 1, s > 0);
      tc_commit_warp(ctl.bar(X_A_EMPTY));   // Q(s) and the rows are read
    }
    if (steps > 0) {
      if (ok) tc_commit_warp(ctl.bar(X_DONE));
      tc_commit_warp(ctl.bar(X_DRAIN));
      wait_drain(ctl.bar(X_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    const float *lse2 = reinterpret_cast<const float *>(smem + C::K_OFF_ROWS);
    const float *dsum = lse2 + 128;
    bool ok = steps > 0;
    for (int s = 0; ok && s < steps; ++s) {
      const uint32_t par = (uint32_t)s & 1u;
      if (!(ok = wait_warp(ctl.bar(X_A_FULL), par, abort_flag, p.timeout_ns)) ||
          !(ok = wait_warp(ctl.bar(X_ST_FULL), par, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = i0 + (ps.s0 + s) % (nblk - i0);
      // phase 1: P^T in registers (no product reads it here)
      uint32_t us0[32], us1[32], pw[2][16];
      load64(tmem + lane_off + COL_ST + 64 * hf, us0, us1);
      keyrow_p(us0, us1, lse2, c, p.causal && ib == jb, ib, hf, key, pw);
      // phase 2: dS^T = P^T o (dP^T - D), bf16 over the first 32 columns
      if (!(ok = wait_warp(ctl.bar(X_DPT_FULL), par, abort_flag, p.timeout_ns))) break;
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
                                  f2_pack(-d4.x, -d4.y))),
                    a0, a1);
          f2_unpack(f2_mul(bf16x2_widen(w1),
                           f2_add(f2_pack(__uint_as_float(ud[x + 2]), __uint_as_float(ud[x + 3])),
                                  f2_pack(-d4.z, -d4.w))),
                    a2, a3);
          dw[x >> 1] = pack_bf16x2(a0, a1);
          dw[(x >> 1) + 1] = pack_bf16x2(a2, a3);
        }
        tmem_st16(tmem + lane_off + COL_DPT + 64 * hf + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(X_DST_FULL));
    }
    if (ok && wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns)) {
      tc_fence_after();
      have = true;
    }
  }
  // every product of both CTAs is complete: rank 0's V and Q tiles are free
  cluster_sync_all();
  if (warp >= 2) {
    const int row = (warp & 3) * 32 + lane, hf = (warp - 2) >> 2;
    const uint32_t acc = tmem + ((uint32_t)((warp & 3) * 32) << 16) + COL_DK + hf * (D / 2);
    if (rank == 1 && have) pair_send(acc, mapa_shared(v_s, 0), row, hf);
    cluster_sync_all();   // rank 1's partial is in rank 0's exchange area
    if (rank == 0 && have) {
      const long long off = ((long long)(row0 + jb * BM + row) * p.Hkv + kvh) * D + hf * (D / 2);
      pair_store(acc, v_s, ps.peer_n > 0, row, hf, p.scale, p.dk + off, jb * BM + row < len);
    }
  } else {
    cluster_sync_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dQ
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BCtl ctl;
  ctl.bar0 = base + C::Q_OFF_CTL;
  ctl.words = reinterpret_cast<uint32_t *>(smem + C::Q_OFF_CTL + 8 * X_COUNT);
  volatile uint32_t *abort_flag = ctl.words + 1;

  const BUnit un = bwd_unit(p, blockIdx.x, p.Hq, p.causal != 0);
  if (!un.valid) return;
  const int ib = un.blk, h = un.head, b = un.seq;
  const int row0 = un.start, len = un.len;
  const int kvh = h / p.group;
  const int steps = p.causal ? ib + 1 : un.nblk;
  const uint32_t q_s = base + C::Q_OFF_Q, do_s = base + C::Q_OFF_DO, k_s = base + C::Q_OFF_K;
  const uint32_t ring = base + C::Q_OFF_RING;
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256;

  if (warp == 1) {
    if (lane == 0) x_init_barriers(ctl);
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

  if (warp == 0) {
    // producer: Q, dO once; per key block the first two V(s) chunks, K(s)
    // once dQ(s-1) has read K(s-1), then the last two V chunks
    if (lane == 0) {
      int issued = 0, cpos = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), 2 * C::TILE);
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(q_s + c * CHUNK_BYTES, &tm_q, ctl.bar(X_STATIC), c * 64, h, row0 + ib * BM);
        tma_load_3d(do_s + c * CHUNK_BYTES, &tm_do, ctl.bar(X_STATIC), c * 64, h,
                    row0 + ib * BM);
      }
      for (int s = 0; ok && s < steps; ++s) {
        for (int c = 0; ok && c < 4; ++c, ++cpos) {
          if (c == 2) {   // K(s)
            if (s > 0 && !(ok = wait_bounded(ctl.bar(X_A_EMPTY), (uint32_t)(s - 1) & 1u,
                                             abort_flag, p.timeout_ns)))
              break;
            mbar_arrive_expect_tx(ctl.bar(X_A_FULL), C::TILE);
            for (int cc = 0; cc < 4; ++cc)
              tma_load_3d(k_s + cc * CHUNK_BYTES, &tm_k, ctl.bar(X_A_FULL), cc * 64, kvh,
                          row0 + s * BM);
            ++issued;
          }
          const int slot = cpos & 1;
          if (cpos >= 2 && !(ok = wait_bounded(ctl.bar(X_C_EMPTY0 + slot),
                                               (uint32_t)((cpos >> 1) - 1) & 1u, abort_flag,
                                               p.timeout_ns)))
            break;
          mbar_arrive_expect_tx(ctl.bar(X_C_FULL0 + slot), CHUNK_BYTES);
          tma_load_3d(ring + slot * CHUNK_BYTES, &tm_v, ctl.bar(X_C_FULL0 + slot), c * 64, kvh,
                      row0 + s * BM);
        }
      }
      if (*abort_flag) {
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        if (issued > 0) wait_drain(ctl.bar(X_A_FULL), (uint32_t)(issued - 1) & 1u, p.timeout_ns);
        for (int sl = 0; sl < 2 && sl < cpos; ++sl) {
          const int last = sl + 2 * ((cpos - 1 - sl) / 2);
          wait_drain(ctl.bar(X_C_FULL0 + sl), (uint32_t)(last >> 1) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp, per key block s: dP(s) = dO V(s)^T chunk by chunk (dQ(s-1),
    // issued before, has read dS(s-1) from these columns); S(s) = Q K(s)^T
    // once the softmax warps have read S(s-1) and K(s) landed; dQ += dS(s)
    // K(s) once dS is written
    const uint64_t qdesc = smem_desc_sw128(q_s, 16, 1024);
    const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(k_s, CHUNK_BYTES, 1024);
    bool ok = wait_warp(ctl.bar(X_STATIC), 0, abort_flag, p.timeout_ns);
    int cpos = 0;
    for (int s = 0; ok && s < steps; ++s) {
      const uint32_t par = (uint32_t)s & 1u;
      for (int c = 0; ok && c < 4; ++c, ++cpos) {
        const int slot = cpos & 1;
        if (!(ok = wait_warp(ctl.bar(X_C_FULL0 + slot), (uint32_t)(cpos >> 1) & 1u, abort_flag,
                             p.timeout_ns)))
          break;
        tc_fence_after();
        issue_chunk_warp(tmem + COL_DP, smem_desc_sw128(do_s + c * CHUNK_BYTES, 16, 1024),
                         smem_desc_sw128(ring + slot * CHUNK_BYTES, 16, 1024), c == 0);
        tc_commit_warp(ctl.bar(X_C_EMPTY0 + slot));
      }
      if (!ok) break;
      tc_commit_warp(ctl.bar(X_DPT_FULL));
      if ((s > 0 && !(ok = wait_warp(ctl.bar(X_PT_FULL), (uint32_t)(s - 1) & 1u, abort_flag,
                                     p.timeout_ns))) ||
          !(ok = wait_warp(ctl.bar(X_A_FULL), par, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      issue_qk_warp<D>(tmem + COL_S, qdesc, kdesc);
      tc_commit_warp(ctl.bar(X_ST_FULL));
      if (!(ok = wait_warp(ctl.bar(X_DST_FULL), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_pv_half_warp<D>(tmem + COL_DQ, tmem + COL_DP, k_mn, 0, s > 0);
      issue_pv_half_warp<D>(tmem + COL_DQ, tmem + COL_DP, k_mn, 1, s > 0);
      tc_commit_warp(ctl.bar(X_A_EMPTY));   // K(s) is read
    }
    if (ok) tc_commit_warp(ctl.bar(X_DONE));
    tc_commit_warp(ctl.bar(X_DRAIN));
    wait_drain(ctl.bar(X_DRAIN), 0, p.timeout_ns);
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
      const uint32_t par = (uint32_t)s & 1u;
      if (!(ok = wait_warp(ctl.bar(X_ST_FULL), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      const bool edge = (s * BM + BM > len) || (p.causal && s == ib);
      float pv[64];
      {
        uint32_t u0[32], u1[32];
        load64(tmem + lane_off + COL_S + 64 * hf, u0, u1);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          pv[x] = __uint_as_float(u0[x]);
          pv[32 + x] = __uint_as_float(u1[x]);
        }
      }
      tc_fence_before();
      warp_arrive(ctl.bar(X_PT_FULL));   // S(s) is read: S(s+1) may overwrite it
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
          if (k0 >= len || (p.causal && k0 > qrow)) pe = 0.f;
          pv[x] = pe;
        }
      }
      if (!(ok = wait_warp(ctl.bar(X_DPT_FULL), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * hf + 32 * ch;
        uint32_t ud[32];
        tmem_ld32(tmem + lane_off + COL_DP + c0, ud);
        tmem_wait_ld();
        reg_fence32(ud);
        uint32_t dw[16];
        const uint64_t nd2 = f2_pack(-dsum, -dsum);
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float a0, a1;
          f2_unpack(f2_mul(f2_pack(pv[32 * ch + x], pv[32 * ch + x + 1]),
                           f2_add(f2_pack(__uint_as_float(ud[x]), __uint_as_float(ud[x + 1])),
                                  nd2)),
                    a0, a1);
          dw[x >> 1] = pack_bf16x2(a0, a1);
        }
        tmem_st16(tmem + lane_off + COL_DP + 64 * hf + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(X_DST_FULL));
    }
    if (ok && (ok = wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns))) {
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
