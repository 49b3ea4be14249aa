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
//   dV kernel: per 128-key block (K resident), per step S^T = K Q^T into
//              one of two TMEM buffers, P^T over it, dV += P^T dO
//              (TMEM: 2 x 128 score columns + 256 for dV)
//   dK kernel: per 128-key block (K, V resident), S^T = K Q^T,
//              dP^T = V dO^T, dS^T, dK += dS^T Q (TMEM 128 + 128 + 256)
//   dQ kernel: per 128-row query block (Q, dO resident), S = Q K^T,
//              dP = dO V^T, dS, dQ += dS K (TMEM 128 + 128 + 256)
//
// Per key/query block pair that is 16 products of 128^3 against the 10 of
// a single pass (the scores are formed three times, dP twice).  Warp roles as
// in attn_bwd.cuh: warp 0 producer, warp 1 MMA issue loop (one elected lane
// issues), warps 2-9 softmax (two per TMEM lane quarter, 64 columns each).
//
// The per-step operands stream through a ring of 32 KB slots, one d-half
// (128 rows x 128 columns, two 64-column swizzle chunks) per slot, in the
// order the products read them: a score product reads two slots as its
// K-major B operand, an accumulation product two slots as N-major B with
// N = 128 each.  The accumulation operand of a step is streamed a second
// time rather than held, so that the score product of the next step never
// waits for the accumulation of this one: in the dK and dQ kernels the next
// scores are issued as soon as the softmax warps have read this step's
// scores, and run while they form dS.
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
  static constexpr uint32_t SLOT = 2 * CHUNK_BYTES;   // 128 x 128 bf16: one d-half
  static constexpr uint32_t CTL = 256;
  static constexpr uint32_t SMEM_MAX = 232448;
  // dV kernel: K | ring | four lse2 rows
  static constexpr int V_NS = 5;
  static constexpr uint32_t V_OFF_K = 0, V_OFF_RING = TILE;
  static constexpr uint32_t V_OFF_ROWS = V_OFF_RING + V_NS * SLOT;
  static constexpr uint32_t V_OFF_CTL = V_OFF_ROWS + 4 * 512;
  // dK kernel: K | V | ring | two {lse2, dsum} row pairs
  static constexpr int K_NS = 3;
  static constexpr uint32_t K_OFF_K = 0, K_OFF_V = TILE, K_OFF_RING = 2 * TILE;
  static constexpr uint32_t K_OFF_ROWS = K_OFF_RING + K_NS * SLOT;
  static constexpr uint32_t K_OFF_CTL = K_OFF_ROWS + 2 * 1024;
  // dQ kernel: Q | dO | ring
  static constexpr int Q_NS = 3;
  static constexpr uint32_t Q_OFF_Q = 0, Q_OFF_DO = TILE, Q_OFF_RING = 2 * TILE;
  static constexpr uint32_t Q_OFF_CTL = Q_OFF_RING + Q_NS * SLOT;
  // The allocation: the layout plus up to 1024 bytes for aligning the
  // dynamic shared memory, capped at the opt-in maximum (the kernels check
  // that the alignment they meet fits in what is left).
#define B256_ALLOC(need) ((need) + 1024 > SMEM_MAX ? SMEM_MAX : (need) + 1024)
  static constexpr uint32_t V_SMEM = B256_ALLOC(V_OFF_CTL + CTL);
  static constexpr uint32_t K_SMEM = B256_ALLOC(K_OFF_CTL + CTL);
  static constexpr uint32_t Q_SMEM = B256_ALLOC(Q_OFF_CTL + CTL);
#undef B256_ALLOC
  static_assert(V_OFF_CTL + CTL <= SMEM_MAX && K_OFF_CTL + CTL <= SMEM_MAX &&
                    Q_OFF_CTL + CTL <= SMEM_MAX,
                "shared memory");
};

enum : int {
  X_STATIC = 0,       // the unit's resident tiles loaded
  X_FULL0 = 1,        // ring slot i loaded, i < 5
  X_EMPTY0 = 6,       // ring slot i read by its product (commit)
  X_ST0 = 11,         // scores in TMEM buffer b (commit); dK and dQ use buffer 0
  X_ST1 = 12,
  X_DP = 13,          // dP^T (dP) in TMEM (commit)
  X_P0 = 14,          // softmax warps: dV kernel P^T written over buffer b;
  X_P1 = 15,          //   dK and dQ kernels the scores read (buffer 0)
  X_DS = 16,          // softmax warps: dS^T (dS) written over dP^T (dP)
  X_ROWF0 = 17,       // row slot r loaded, r < 4
  X_ROWE0 = 21,       // softmax warps: row slot r read
  X_DONE = 25,        // the accumulator is final (commit)
  X_DRAIN = 26,       // teardown drain of the MMA warp
  X_COUNT = 27
};
static_assert(8 * X_COUNT + 8 <= (int)B256::CTL, "control block");

__device__ __forceinline__ void x_init_barriers(const BCtl &c) {
  for (int i = 0; i < X_COUNT; ++i) {
    const bool warps = i == X_P0 || i == X_P1 || i == X_DS || (i >= X_ROWE0 && i < X_ROWE0 + 4);
    mbar_init(c.bar(i), warps ? BWD_SM_WARPS : 1);
  }
  c.words[1] = 0u;
  mbar_init_fence();
}

// The 1024-byte-aligned start of the dynamic shared memory; false if the
// layout (need bytes) does not fit behind it in the allocation.
__device__ __forceinline__ bool smem_fits(const uint8_t *raw, uint32_t need, uint32_t alloc,
                                          uint32_t &pad) {
  pad = (1024u - (smem_u32(raw) & 1023u)) & 1023u;
  return pad + need <= alloc;
}

// ------------------------------------------------------------------ ring
// Producer: ring item pos (slot pos % ns) = d-half h of the 128-row tile of
// `map` at (head, row).  False if the wait for the slot gave up.
__device__ __forceinline__ bool ring_load(const BCtl &ctl, uint32_t ring, int ns, int pos,
                                          const CUtensorMap *map, int h, int head, int row,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns) {
  const int slot = pos % ns;
  if (pos >= ns && !wait_bounded(ctl.bar(X_EMPTY0 + slot), (uint32_t)(pos / ns - 1) & 1u,
                                 abort_flag, timeout_ns))
    return false;
  const uint32_t dst = ring + (uint32_t)slot * B256::SLOT, bar = ctl.bar(X_FULL0 + slot);
  mbar_arrive_expect_tx(bar, B256::SLOT);
  tma_load_3d(dst, map, bar, 128 * h, head, row);
  tma_load_3d(dst + CHUNK_BYTES, map, bar, 128 * h + 64, head, row);
  return true;
}

// Producer teardown after an abort: bounded waits for the copies issued
// into each slot of a ring of ns slots that received `count` items.
__device__ __forceinline__ void drain_slots(const BCtl &ctl, int bar0, int ns, int count,
                                            unsigned long long timeout_ns) {
  for (int sl = 0; sl < ns && sl < count; ++sl) {
    const int last = sl + ns * ((count - 1 - sl) / ns);
    wait_drain(ctl.bar(bar0 + sl), (uint32_t)(last / ns) & 1u, timeout_ns);
  }
}

// MMA warp: wait for ring item pos, return its slot's address (0: gave up).
__device__ __forceinline__ uint32_t ring_wait(const BCtl &ctl, uint32_t ring, int ns, int pos,
                                              volatile uint32_t *abort_flag,
                                              unsigned long long timeout_ns) {
  const int slot = pos % ns;
  if (!wait_warp(ctl.bar(X_FULL0 + slot), (uint32_t)(pos / ns) & 1u, abort_flag, timeout_ns))
    return 0u;
  tc_fence_after();
  return ring + (uint32_t)slot * B256::SLOT;
}

// Scores over d-half h (128 contraction columns): d_tmem (+)= A_h B_h^T with
// A the resident 128 x 256 tile (a_desc at its base) and B_h a ring slot,
// both K-major; h = 0 overwrites.
__device__ __forceinline__ void issue_score_half_warp(uint32_t d_tmem, uint64_t a_desc,
                                                      uint32_t b_slot, int h) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BN, 0);
  const uint64_t b_desc = smem_desc_sw128(b_slot, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t c = (uint32_t)kk >> 2, k4 = (uint32_t)kk & 3u;
    mma_ss_warp(d_tmem, a_desc + (uint64_t)(((2u * h + c) * CHUNK_BYTES + k4 * 32u) >> 4),
                b_desc + (uint64_t)((c * CHUNK_BYTES + k4 * 32u) >> 4), IDESC,
                (h == 0 && kk == 0) ? 0u : 1u);
  }
}

// Accumulation into d-half h: acc[:, 128 h .. 128 h + 127] (+)= A B_h with A
// bf16 pairs in TMEM over 128 contraction rows (each softmax warp packs its
// 64 columns into the first 32 of them) and B_h a ring slot holding d-half
// h of a 128-row tile, N-major.
__device__ __forceinline__ void issue_acc_half_warp(uint32_t acc, uint32_t a_tmem,
                                                    uint32_t b_slot, int h, bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(128, 1);
  const uint64_t b_desc = smem_desc_sw128(b_slot, CHUNK_BYTES, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(acc + 128u * (uint32_t)h, a_tmem + 64u * ((uint32_t)kk >> 2) + 8u * ((uint32_t)kk & 3u),
                b_desc + (uint64_t)((kk * 2048) >> 4), IDESC, (accumulate || kk > 0) ? 1u : 0u);
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
// Step t of this CTA: query head and block of unit step s0 + t.
struct StepMap {
  int kvh, group, i0, nq, s0;
  __device__ int head(int t) const { return kvh * group + (s0 + t) / nq; }
  __device__ int blk(int t) const { return i0 + (s0 + t) % nq; }
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dv256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D, NS = C::V_NS;
  extern __shared__ uint8_t smem_raw[];
  uint32_t pad;
  if (!smem_fits(smem_raw, C::V_OFF_CTL + C::CTL, C::V_SMEM, pad)) {   // uniform
    if (threadIdx.x == 0) record_status(ATTN_ERR_UNSUPPORTED_DEVICE);
    return;
  }
  uint8_t *smem = smem_raw + pad;
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
  const int n = ps.n;   // this CTA's steps
  const StepMap sm{kvh, p.group, i0, nblk - i0, ps.s0};
  const uint32_t k_s = base + C::V_OFF_K, ring = base + C::V_OFF_RING;
  constexpr uint32_t COL_DV = 256;   // score buffers at columns 0 and 128
  bool have = false;                 // softmax threads: this CTA's dV row is final

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
    // producer.  Ring: Q(0), Q(1), then per step t dO(t) and Q(t+2), two
    // d-halves each.  lse2 rows: row t in slot t % 4; row t + 3 (t >= 1)
    // once the softmax warps are done with row t - 1.
    if (lane == 0 && n > 0) {
      int pos = 0, nrows = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), C::TILE);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(k_s + c * CHUNK_BYTES, &tm_k, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
      auto load_row = [&](int r) {
        const uint32_t bar = ctl.bar(X_ROWF0 + (r & 3));
        const long long prow =
            (long long)sm.head(r) * p.rows_pad() + p.pstart[b] + (long long)sm.blk(r) * BM;
        mbar_arrive_expect_tx(bar, 512);
        bulk_load(base + C::V_OFF_ROWS + (r & 3) * 512, p.lse2 + prow, 512, bar);
      };
      auto load_tile = [&](const CUtensorMap *map, int t) {
        for (int h = 0; ok && h < 2; ++h) {
          ok = ring_load(ctl, ring, NS, pos, map, h, sm.head(t), row0 + sm.blk(t) * BM,
                         abort_flag, p.timeout_ns);
          if (ok) ++pos;
        }
      };
      for (; nrows < 4 && nrows < n; ++nrows) load_row(nrows);
      load_tile(&tm_q, 0);
      if (n > 1) load_tile(&tm_q, 1);
      for (int t = 0; ok && t < n; ++t) {
        load_tile(&tm_do, t);
        if (t + 2 < n) load_tile(&tm_q, t + 2);
        if (ok && t >= 1 && t + 3 < n) {
          if (!(ok = wait_bounded(ctl.bar(X_ROWE0 + ((t - 1) & 3)), (uint32_t)((t - 1) >> 2) & 1u,
                                  abort_flag, p.timeout_ns)))
            break;
          load_row(t + 3);
          ++nrows;
        }
      }
      if (*abort_flag) {   // drain: bounded waits for the copies issued
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        drain_slots(ctl, X_FULL0, NS, pos, p.timeout_ns);
        drain_slots(ctl, X_ROWF0, 4, nrows, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp: S^T(0) and S^T(1) into buffers 0 and 1; per step t, once
    // P^T(t) is written, dV += P^T(t) dO(t), then S^T(t + 2) into the same
    // buffer (dV(t), issued before, has read P^T(t) by then: one thread's
    // products run in issue order)
    const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
    if (n > 0) {
      int pos = 0;
      bool ok = wait_warp(ctl.bar(X_STATIC), 0, abort_flag, p.timeout_ns);
      auto scores = [&](uint32_t buf) {
        for (int h = 0; ok && h < 2; ++h, ++pos) {
          const uint32_t slot = ring_wait(ctl, ring, NS, pos, abort_flag, p.timeout_ns);
          if (!(ok = slot != 0u)) break;
          issue_score_half_warp(tmem + 128u * buf, kdesc, slot, h);
          tc_commit_warp(ctl.bar(X_EMPTY0 + pos % NS));
        }
        if (ok) tc_commit_warp(ctl.bar(X_ST0 + (int)buf));
      };
      if (ok) scores(0);
      if (ok && n > 1) scores(1);
      for (int t = 0; ok && t < n; ++t) {
        const uint32_t buf = (uint32_t)t & 1u;
        if (!(ok = wait_warp(ctl.bar(X_P0 + (int)buf), (uint32_t)(t >> 1) & 1u, abort_flag,
                             p.timeout_ns)))
          break;
        tc_fence_after();
        for (int h = 0; ok && h < 2; ++h, ++pos) {
          const uint32_t slot = ring_wait(ctl, ring, NS, pos, abort_flag, p.timeout_ns);
          if (!(ok = slot != 0u)) break;
          issue_acc_half_warp(tmem + COL_DV, tmem + 128u * buf, slot, h, t > 0);
          tc_commit_warp(ctl.bar(X_EMPTY0 + pos % NS));
        }
        if (ok && t + 2 < n) scores(buf);
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
    bool ok = n > 0;
    for (int t = 0; ok && t < n; ++t) {
      const uint32_t buf = (uint32_t)t & 1u;
      if (!(ok = wait_warp(ctl.bar(X_ROWF0 + (t & 3)), (uint32_t)(t >> 2) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(ctl.bar(X_ST0 + (int)buf), (uint32_t)(t >> 1) & 1u, abort_flag,
                           p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = sm.blk(t);
      const float *lse2 = reinterpret_cast<const float *>(smem + C::V_OFF_ROWS + (t & 3) * 512);
      const uint32_t sc = tmem + lane_off + 128u * buf + 64 * hf;
      uint32_t us0[32], us1[32], pw[2][16];
      load64(sc, us0, us1);
      keyrow_p(us0, us1, lse2, c, p.causal && ib == jb, ib, hf, key, pw);
      // P^T bf16 over the first 32 of this warp's 64 score columns
      tmem_st16(sc, pw[0]);
      tmem_st16(sc + 16, pw[1]);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ctl.bar(X_P0 + (int)buf));
      warp_arrive(ctl.bar(X_ROWE0 + (t & 3)));
    }
    if (ok && wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns)) {
      tc_fence_after();
      have = true;
    }
  }
  // every product of both CTAs is complete: rank 0's ring is free
  cluster_sync_all();
  if (warp >= 2) {
    const int row = (warp & 3) * 32 + lane, hf = (warp - 2) >> 2;
    const uint32_t acc = tmem + ((uint32_t)((warp & 3) * 32) << 16) + COL_DV + hf * (D / 2);
    if (rank == 1 && have) pair_send(acc, mapa_shared(ring, 0), row, hf);
    cluster_sync_all();   // rank 1's partial is in rank 0's exchange area
    if (rank == 0 && have) {
      const long long off = ((long long)(row0 + jb * BM + row) * p.Hkv + kvh) * D + hf * (D / 2);
      pair_store(acc, ring, ps.peer_n > 0, row, hf, 1.f, p.dv + off, jb * BM + row < len);
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

// ------------------------------------------------------------------ dK, dQ
// The MMA issue order shared by the dK and dQ kernels (A_S / A_DP: the
// resident score and dP operands; the ring carries, in this order, the
// score operand and the dP operand of step 0, then per step t the score
// operand of step t + 1, the accumulation operand of step t and the dP
// operand of step t + 1):
//   scores(0), dP(0); per step t: scores(t + 1) once the softmax warps have
//   read scores(t); acc += dS(t) B(t) once dS(t) is written; dP(t + 1)
//   (its columns hold dS(t), which the accumulation, issued before, reads).
__device__ __forceinline__ void mma_loop_sdp(const BCtl &ctl, uint32_t ring, uint32_t tmem,
                                             uint64_t a_s, uint64_t a_dp, int n,
                                             volatile uint32_t *abort_flag,
                                             unsigned long long timeout_ns) {
  constexpr int NS = 3;
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_ACC = 256;
  int pos = 0;
  bool ok = wait_warp(ctl.bar(X_STATIC), 0, abort_flag, timeout_ns);
  auto product = [&](uint32_t d, uint64_t a, int bar) {
    for (int h = 0; ok && h < 2; ++h, ++pos) {
      const uint32_t slot = ring_wait(ctl, ring, NS, pos, abort_flag, timeout_ns);
      if (!(ok = slot != 0u)) break;
      issue_score_half_warp(d, a, slot, h);
      tc_commit_warp(ctl.bar(X_EMPTY0 + pos % NS));
    }
    if (ok) tc_commit_warp(ctl.bar(bar));
  };
  if (ok) product(tmem + COL_S, a_s, X_ST0);
  if (ok) product(tmem + COL_DP, a_dp, X_DP);
  for (int t = 0; ok && t < n; ++t) {
    const uint32_t par = (uint32_t)t & 1u;
    if (t + 1 < n) {
      if (!(ok = wait_warp(ctl.bar(X_P0), par, abort_flag, timeout_ns))) break;
      tc_fence_after();
      product(tmem + COL_S, a_s, X_ST0);
      if (!ok) break;
    }
    if (!(ok = wait_warp(ctl.bar(X_DS), par, abort_flag, timeout_ns))) break;
    tc_fence_after();
    for (int h = 0; ok && h < 2; ++h, ++pos) {
      const uint32_t slot = ring_wait(ctl, ring, NS, pos, abort_flag, timeout_ns);
      if (!(ok = slot != 0u)) break;
      issue_acc_half_warp(tmem + COL_ACC, tmem + COL_DP, slot, h, t > 0);
      tc_commit_warp(ctl.bar(X_EMPTY0 + pos % NS));
    }
    if (ok && t + 1 < n) product(tmem + COL_DP, a_dp, X_DP);
  }
  if (ok) tc_commit_warp(ctl.bar(X_DONE));
  tc_commit_warp(ctl.bar(X_DRAIN));
  wait_drain(ctl.bar(X_DRAIN), 0, timeout_ns);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dk256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D, NS = C::K_NS;
  static_assert(NS == 3, "mma_loop_sdp");
  extern __shared__ uint8_t smem_raw[];
  uint32_t pad;
  if (!smem_fits(smem_raw, C::K_OFF_CTL + C::CTL, C::K_SMEM, pad)) {   // uniform
    if (threadIdx.x == 0) record_status(ATTN_ERR_UNSUPPORTED_DEVICE);
    return;
  }
  uint8_t *smem = smem_raw + pad;
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
  const int n = ps.n;
  const StepMap sm{kvh, p.group, i0, nblk - i0, ps.s0};
  const uint32_t k_s = base + C::K_OFF_K, v_s = base + C::K_OFF_V, ring = base + C::K_OFF_RING;
  constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DK = 256;
  bool have = false;

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
    // producer.  Ring: Q(0), dO(0), then per step t Q(t+1) (scores),
    // Q(t) (dK), dO(t+1).  Rows {lse2, dsum}: row t in slot t % 2; row t + 2
    // once the softmax warps are done with row t.
    if (lane == 0 && n > 0) {
      int pos = 0, nrows = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), 2 * C::TILE);
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(k_s + c * CHUNK_BYTES, &tm_k, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
        tma_load_3d(v_s + c * CHUNK_BYTES, &tm_v, ctl.bar(X_STATIC), c * 64, kvh, row0 + jb * BM);
      }
      auto load_row = [&](int r) {
        const uint32_t bar = ctl.bar(X_ROWF0 + (r & 1));
        const long long prow =
            (long long)sm.head(r) * p.rows_pad() + p.pstart[b] + (long long)sm.blk(r) * BM;
        const uint32_t dst = base + C::K_OFF_ROWS + (r & 1) * 1024;
        mbar_arrive_expect_tx(bar, 1024);
        bulk_load(dst, p.lse2 + prow, 512, bar);
        bulk_load(dst + 512, p.dsum + prow, 512, bar);
      };
      auto load_tile = [&](const CUtensorMap *map, int t) {
        for (int h = 0; ok && h < 2; ++h) {
          ok = ring_load(ctl, ring, NS, pos, map, h, sm.head(t), row0 + sm.blk(t) * BM,
                         abort_flag, p.timeout_ns);
          if (ok) ++pos;
        }
      };
      for (; nrows < 2 && nrows < n; ++nrows) load_row(nrows);
      load_tile(&tm_q, 0);
      load_tile(&tm_do, 0);
      for (int t = 0; ok && t < n; ++t) {
        if (t + 1 < n) load_tile(&tm_q, t + 1);
        load_tile(&tm_q, t);
        if (t + 1 < n) load_tile(&tm_do, t + 1);
        if (ok && t + 2 < n) {
          if (!(ok = wait_bounded(ctl.bar(X_ROWE0 + (t & 1)), (uint32_t)(t >> 1) & 1u, abort_flag,
                                  p.timeout_ns)))
            break;
          load_row(t + 2);
          ++nrows;
        }
      }
      if (*abort_flag) {
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        drain_slots(ctl, X_FULL0, NS, pos, p.timeout_ns);
        drain_slots(ctl, X_ROWF0, 2, nrows, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp: scores S^T = K Q^T, dP^T = V dO^T, dK += dS^T Q
    if (n > 0)
      mma_loop_sdp(ctl, ring, tmem, smem_desc_sw128(k_s, 16, 1024),
                   smem_desc_sw128(v_s, 16, 1024), n, abort_flag, p.timeout_ns);
    __syncwarp();
  } else {
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    bool ok = n > 0;
    for (int t = 0; ok && t < n; ++t) {
      const uint32_t par = (uint32_t)t & 1u;
      if (!(ok = wait_warp(ctl.bar(X_ROWF0 + (t & 1)), (uint32_t)(t >> 1) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(ctl.bar(X_ST0), par, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = sm.blk(t);
      const float *lse2 = reinterpret_cast<const float *>(smem + C::K_OFF_ROWS + (t & 1) * 1024);
      const float *dsum = lse2 + 128;
      // phase 1: P^T in registers (no product reads it here); then the
      // scores' columns are free for the next step's
      uint32_t us0[32], us1[32], pw[2][16];
      load64(tmem + lane_off + COL_ST + 64 * hf, us0, us1);
      tc_fence_before();
      warp_arrive(ctl.bar(X_P0));
      keyrow_p(us0, us1, lse2, c, p.causal && ib == jb, ib, hf, key, pw);
      // phase 2: dS^T = P^T o (dP^T - D), bf16 over the first 32 columns
      if (!(ok = wait_warp(ctl.bar(X_DP), par, abort_flag, p.timeout_ns))) break;
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
      warp_arrive(ctl.bar(X_DS));
      warp_arrive(ctl.bar(X_ROWE0 + (t & 1)));
    }
    if (ok && wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns)) {
      tc_fence_after();
      have = true;
    }
  }
  // every product of both CTAs is complete: rank 0's V tile and ring are free
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

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq256_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = B256;
  constexpr int D = C::D, NS = C::Q_NS;
  static_assert(NS == 3, "mma_loop_sdp");
  extern __shared__ uint8_t smem_raw[];
  uint32_t pad;
  if (!smem_fits(smem_raw, C::Q_OFF_CTL + C::CTL, C::Q_SMEM, pad)) {   // uniform
    if (threadIdx.x == 0) record_status(ATTN_ERR_UNSUPPORTED_DEVICE);
    return;
  }
  uint8_t *smem = smem_raw + pad;
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
  const int n = p.causal ? ib + 1 : un.nblk;   // key blocks
  const uint32_t q_s = base + C::Q_OFF_Q, do_s = base + C::Q_OFF_DO, ring = base + C::Q_OFF_RING;
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
    // producer.  Ring: K(0), V(0), then per key block t K(t+1) (scores),
    // K(t) (dQ), V(t+1).
    if (lane == 0) {
      int pos = 0;
      bool ok = true;
      mbar_arrive_expect_tx(ctl.bar(X_STATIC), 2 * C::TILE);
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(q_s + c * CHUNK_BYTES, &tm_q, ctl.bar(X_STATIC), c * 64, h, row0 + ib * BM);
        tma_load_3d(do_s + c * CHUNK_BYTES, &tm_do, ctl.bar(X_STATIC), c * 64, h,
                    row0 + ib * BM);
      }
      auto load_tile = [&](const CUtensorMap *map, int t) {
        for (int hh = 0; ok && hh < 2; ++hh) {
          ok = ring_load(ctl, ring, NS, pos, map, hh, kvh, row0 + t * BM, abort_flag,
                         p.timeout_ns);
          if (ok) ++pos;
        }
      };
      load_tile(&tm_k, 0);
      load_tile(&tm_v, 0);
      for (int t = 0; ok && t < n; ++t) {
        if (t + 1 < n) load_tile(&tm_k, t + 1);
        load_tile(&tm_k, t);
        if (t + 1 < n) load_tile(&tm_v, t + 1);
      }
      if (*abort_flag) {
        wait_drain(ctl.bar(X_STATIC), 0, p.timeout_ns);
        drain_slots(ctl, X_FULL0, NS, pos, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA warp: scores S = Q K^T, dP = dO V^T, dQ += dS K
    mma_loop_sdp(ctl, ring, tmem, smem_desc_sw128(q_s, 16, 1024),
                 smem_desc_sw128(do_s, 16, 1024), n, abort_flag, p.timeout_ns);
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
    for (int t = 0; ok && t < n; ++t) {
      const uint32_t par = (uint32_t)t & 1u;
      if (!(ok = wait_warp(ctl.bar(X_ST0), par, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      const bool edge = (t * BM + BM > len) || (p.causal && t == ib);
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
      warp_arrive(ctl.bar(X_P0));   // S(t) is read: S(t+1) may overwrite it
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
          const int k0 = t * BM + 64 * hf + x;
          float pe = ex2_approx(pv[x] * c - lse2);
          if (k0 >= len || (p.causal && k0 > qrow)) pe = 0.f;
          pv[x] = pe;
        }
      }
      if (!(ok = wait_warp(ctl.bar(X_DP), par, abort_flag, p.timeout_ns))) break;
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
      warp_arrive(ctl.bar(X_DS));
    }
    if (ok && wait_warp(ctl.bar(X_DONE), 0, abort_flag, p.timeout_ns)) {
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
