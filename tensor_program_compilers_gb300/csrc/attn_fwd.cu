// attn_fwd.cu -- fused attention forward for sm_103a (GB300) and its C ABI.
//
// One CTA computes one 128-row query tile of one (sequence, query head):
//
//   for each 128-key tile j (causal: only j <= the diagonal tile)
//     S    = Q K_j^T                       tcgen05.mma, bf16 -> fp32 in TMEM
//     m'   = max(m, rowmax S)              online-softmax monoid state (m, l)
//     P    = 2^(S*c - m'*c), c = scale*log2(e), rounded to bf16 into TMEM
//     l    = l * 2^((m - m')*c) + rowsum P
//     O    = O * 2^((m - m')*c) + P V_j    tcgen05.mma, P read from TMEM
//   O / l -> bf16, LSE = m*scale + ln(l)
//
// This is the online-softmax reduction tang derives with stabilize_softmax
// (tang, muni.works/research/tang, section 2.3 and Table 1 rows "online
// softmax" and "FlashAttention forward"), in the block order of the TileLang
// explainer's loop (ai.thesatyajit.com/articles/tilelang, "FlashAttention,
// in tiles").  Two liberties, both exact in real arithmetic:
//  * the running max m is only moved when the tile max exceeds it by more
//    than 8 (base-2 units): softmax is shift invariant (tang, section 6), so
//    any reference value works as long as O and l share it and the
//    exponentials stay in range (they are <= 2^8 here);
//  * masked keys read -inf, the identity of max (tang, section 2.1, guarded
//    views), so fully masked tiles are skipped rather than computed.
//
// Warp roles (192 threads):
//   warp 0     TMA producer: Q tile once, then K_0, K_1, V_0, K_2, V_1, ...
//              into a ring of shared-memory slots (128-byte swizzle)
//   warp 1     TMEM allocator and MMA issuer (one thread)
//   warps 2-5  softmax warpgroup: thread t owns query row t (TMEM lane t)
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)   S  (fp32 scores of the current tile)
//   [128,192) P0 and [192,256) P1  (bf16 probabilities, two per column)
//   [256,256+d) O (fp32 accumulator)
//
// Every pipeline wait is bounded: past a time limit it records
// ATTN_ERR_TIMEOUT in a device status word and every role stops issuing,
// waits (bounded) for its copies and MMAs in flight, and the CTA releases
// its tensor memory and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <cstdlib>
#include <mutex>

#include "../../include/attn.h"
#include "ptx.cuh"

namespace attn {

constexpr int BM = 128;            // query rows per tile
constexpr int BN = 128;            // keys per tile
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_P0 = 128;   // P buffer b at COL_P0 + 64*b
constexpr uint32_t COL_O = 256;
constexpr uint32_t CHUNK_BYTES = 128 * 128;   // 128 rows x 64 bf16
constexpr float RESCALE_THRESHOLD = 8.0f;     // log2 units

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr uint32_t TILE_BYTES = CHUNKS * CHUNK_BYTES;   // one Q, K or V tile
  static constexpr int STAGES = D == 64 ? 8 : (D == 128 ? 5 : 2);
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = TILE_BYTES;
  static constexpr uint32_t OFF_CTL = TILE_BYTES * (1 + STAGES);
  static constexpr uint32_t CTL_BYTES = 512;
  static constexpr uint32_t SMEM_BYTES = OFF_CTL + CTL_BYTES + 1024;   // + alignment slack
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory");
};

// Barrier slots in the control block.
enum : int {
  BAR_Q_FULL = 0,
  BAR_S_FULL,
  BAR_S_FREE,
  BAR_P_FULL0,
  BAR_P_FULL1,
  BAR_PV_DONE0,
  BAR_PV_DONE1,
  BAR_DRAIN,
  BAR_RING   // full[0..STAGES), then empty[0..STAGES)
};

struct Params {
  __nv_bfloat16 *o;
  float *lse;
  const int *cu_seqlens;
  int B, Hq, Hkv, N, group;
  int causal;
  int num_qt;           // fixed batch: ceil(N / BM)
  float scale;          // score multiplier
  float scale_log2;     // scale * log2(e)
  unsigned long long timeout_ns;
};

__device__ int g_status;   // first device-side error since the last read

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_status, 0, code); }

// Bounded wait on a barrier phase.  Returns false if the CTA is aborting or
// the time limit passed (then it starts the abort).
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns || it > (1u << 30)) {
        *abort_flag = 1u;
        record_status(ATTN_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait for the softmax warps: the tcgen05.ld/st that
// follow are warp-collective, so all lanes must take the same branch.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag, timeout_ns));
}

// Bounded wait that ignores the abort flag: used while draining after an
// abort, for work this thread itself started.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                        unsigned long long timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > timeout_ns) return;
  }
}

struct Tile {
  int valid;
  int seq_start;   // token row of the sequence's first token
  int len;         // sequence length
  int qt;          // query tile index within the sequence
  int h;           // query head
  long long lse_base;   // LSE index of the sequence's row 0 for head h
};

// Packed batches: number of 128-row tiles of sequence s.
__device__ __forceinline__ int seq_tiles(const int *cu, int s) {
  int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  return b > a ? (b - a + BM - 1) / BM : 0;
}

// Number of (sequence, query tile) pairs whose tile index is >= x.
__device__ int pairs_at_or_above(const int *cu, int B, int x) {
  int c = 0;
  for (int s = threadIdx.x & 31; s < B; s += 32) c += max(0, seq_tiles(cu, s) - x);
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Map this CTA to its tile (all 32 lanes of one warp).  Tiles are ordered
// longest first -- descending query-tile index, the number of causal key
// tiles -- with heads fastest so that the query heads of one key/value head
// run side by side.
__device__ Tile decode_tile(const Params &p) {
  Tile t{};
  const int lane = threadIdx.x & 31;
  const long long idx = blockIdx.x;
  if (p.cu_seqlens == nullptr) {
    const long long per = (long long)p.B * p.Hq;
    const int lvl = (int)(idx / per);
    const int rem = (int)(idx % per);
    const int b = rem / p.Hq;
    t.h = rem % p.Hq;
    t.qt = p.num_qt - 1 - lvl;
    t.seq_start = b * p.N;
    t.len = p.N;
    t.lse_base = ((long long)b * p.Hq + t.h) * p.N;
    t.valid = t.qt >= 0;
    return t;
  }
  const int *cu = p.cu_seqlens;
  // validate the offsets and find the total and largest tile counts
  int bad = 0, nmax = 0, ntot = 0;
  for (int s = lane; s < p.B; s += 32) {
    int a = __ldg(cu + s), b = __ldg(cu + s + 1);
    bad |= (b < a);
    int n = b > a ? (b - a + BM - 1) / BM : 0;
    nmax = max(nmax, n);
    ntot += n;
  }
  if (lane == 0) bad |= (__ldg(cu) != 0) | (__ldg(cu + p.B) != p.N);
  for (int o = 16; o > 0; o >>= 1) {
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
    ntot += __shfl_xor_sync(0xffffffffu, ntot, o);
  }
  if (bad) {
    if (lane == 0 && blockIdx.x == 0) record_status(ATTN_ERR_BAD_SEQLENS);
    t.valid = 0;
    return t;
  }
  const int u = (int)(idx / p.Hq);   // pair index
  t.h = (int)(idx % p.Hq);
  if (u >= ntot) {
    t.valid = 0;
    return t;
  }
  // largest x with pairs_at_or_above(x) > u: pair u sits at tile level x
  int lo = 0, hi = nmax;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (pairs_at_or_above(cu, p.B, mid) > u) lo = mid; else hi = mid;
  }
  const int x = lo;
  int r = u - pairs_at_or_above(cu, p.B, x + 1);   // rank among sequences with > x tiles
  int seq = -1;
  for (int base = 0; base < p.B; base += 32) {
    const int s = base + lane;
    const bool has = s < p.B && seq_tiles(cu, s) > x;
    const unsigned m = __ballot_sync(0xffffffffu, has);
    const int cnt = __popc(m);
    if (r < cnt) {
      seq = base + (int)__fns(m, 0, r + 1);
      break;
    }
    r -= cnt;
  }
  if (seq < 0) {   // cannot happen with consistent offsets
    t.valid = 0;
    return t;
  }
  t.seq_start = __ldg(cu + seq);
  t.len = __ldg(cu + seq + 1) - t.seq_start;
  t.qt = x;
  t.lse_base = (long long)t.h * p.N + t.seq_start;
  t.valid = 1;
  return t;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t base_s = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_CTL);
  uint32_t *ctl = reinterpret_cast<uint32_t *>(bars + BAR_RING + 2 * C::STAGES);
  volatile uint32_t *abort_flag = ctl + 1;
  int *tile_info = reinterpret_cast<int *>(ctl + 2);
  auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };
  auto bar_full = [&](int s) -> uint32_t { return bar(BAR_RING + s); };
  auto bar_empty = [&](int s) -> uint32_t { return bar(BAR_RING + C::STAGES + s); };

  // ---- set-up: tile decode (warp 0), barriers (warp 1) ----
  if (warp == 0) {
    Tile t = decode_tile(p);
    if (lane == 0) {
      tile_info[0] = t.valid;
      tile_info[1] = t.seq_start;
      tile_info[2] = t.len;
      tile_info[3] = t.qt;
      tile_info[4] = t.h;
      *reinterpret_cast<long long *>(tile_info + 6) = t.lse_base;
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
  } else if (warp == 1 && lane == 0) {
    mbar_init(bar(BAR_Q_FULL), 1);
    mbar_init(bar(BAR_S_FULL), 1);
    mbar_init(bar(BAR_S_FREE), 4 * 32);
    mbar_init(bar(BAR_P_FULL0), 4 * 32);
    mbar_init(bar(BAR_P_FULL1), 4 * 32);
    mbar_init(bar(BAR_PV_DONE0), 1);
    mbar_init(bar(BAR_PV_DONE1), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    *abort_flag = 0u;
    mbar_init_fence();
  }
  __syncthreads();
  if (!tile_info[0]) return;   // no tile for this CTA (uniform)

  const int seq_start = tile_info[1];
  const int len = tile_info[2];
  const int qt = tile_info[3];
  const int h = tile_info[4];
  const long long lse_base = *reinterpret_cast<long long *>(tile_info + 6);
  const int kvh = h / p.group;
  const int kv_tiles_total = (len + BN - 1) / BN;
  const int n_kv = p.causal ? min(qt + 1, kv_tiles_total) : kv_tiles_total;

  if (warp == 1) {
    tmem_alloc(smem_u32(ctl), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl[0];

  const uint32_t q_s = base_s + C::OFF_Q;
  const uint32_t kv_s = base_s + C::OFF_KV;

  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      const int row0 = seq_start + qt * BM;
      mbar_arrive_expect_tx(bar(BAR_Q_FULL), C::TILE_BYTES);
      for (int c = 0; c < C::CHUNKS; ++c)
        tma_load_3d(q_s + c * CHUNK_BYTES, &tm_q, bar(BAR_Q_FULL), c * 64, h, row0);
      int it = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap *tm, int j) -> bool {
        const int slot = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        if (!wait_bounded(bar_empty(slot), ph ^ 1u, abort_flag, p.timeout_ns)) return false;
        mbar_arrive_expect_tx(bar_full(slot), C::TILE_BYTES);
        const uint32_t dst = kv_s + slot * C::TILE_BYTES;
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(dst + c * CHUNK_BYTES, tm, bar_full(slot), c * 64, kvh, seq_start + j * BN);
        ++it;
        return true;
      };
      // consumption order of the MMA issuer: K0, K1, V0, K2, V1, ..., V_{n-1}
      for (int j = 0; ok && j < n_kv; ++j) {
        ok = load(&tm_k, j);
        if (ok && j >= 1) ok = load(&tm_v, j - 1);
      }
      if (ok) ok = load(&tm_v, n_kv - 1);
      if (!ok) {
        // drain: wait for the copies this thread issued
        wait_drain(bar(BAR_Q_FULL), 0, p.timeout_ns);
        for (int s = 0; s < C::STAGES && s < it; ++s) {
          const int last = s + C::STAGES * ((it - 1 - s) / C::STAGES);
          wait_drain(bar_full(s), (uint32_t)(last / C::STAGES) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // =========================== MMA issuer =============================
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BN, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(D, 1);
      int it = 0;
      bool ok = wait_bounded(bar(BAR_Q_FULL), 0, abort_flag, p.timeout_ns);
      auto pv = [&](int i) -> bool {
        if (!wait_bounded(bar(BAR_P_FULL0 + (i & 1)), (uint32_t)(i >> 1) & 1u, abort_flag,
                          p.timeout_ns))
          return false;
        const int slot = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        if (!wait_bounded(bar_full(slot), ph, abort_flag, p.timeout_ns)) return false;
        tc_fence_after();
        const uint32_t v_s = kv_s + slot * C::TILE_BYTES;
        const uint32_t p_t = tmem + COL_P0 + 64u * (uint32_t)(i & 1);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // V tile: keys are K (16 per step = 2048 bytes), d is N (64-wide
          // swizzle atoms CHUNK_BYTES apart), 8-key groups 1024 bytes apart.
          const uint64_t bdesc = smem_desc_sw128(v_s + kk * 2048, CHUNK_BYTES, 1024);
          mma_ts(tmem + COL_O, p_t + kk * 8, bdesc, IDESC_PV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(BAR_PV_DONE0 + (i & 1)));
        tc_commit(bar_empty(slot));
        ++it;
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j > 0) ok = wait_bounded(bar(BAR_S_FREE), (uint32_t)(j - 1) & 1u, abort_flag,
                                     p.timeout_ns);
        if (!ok) break;
        const int slot = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        ok = wait_bounded(bar_full(slot), ph, abort_flag, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t k_s = kv_s + slot * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // Q and K tiles: rows are M / N, head dim is K (16 per step = 32
          // bytes inside a 128-byte swizzle row; 64-wide chunks apart).
          const uint32_t koff = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
          const uint64_t adesc = smem_desc_sw128(q_s + koff, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(k_s + koff, 16, 1024);
          mma_ss(tmem + COL_S, adesc, bdesc, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(BAR_S_FULL));
        tc_commit(bar_empty(slot));
        ++it;
        if (j > 0) ok = pv(j - 1);
      }
      if (ok) ok = pv(n_kv - 1);
      // no MMA may be in flight when the tensor memory is released
      tc_commit(bar(BAR_DRAIN));
      wait_drain(bar(BAR_DRAIN), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // =========================== softmax warpgroup ======================
    const int wq = warp & 3;                      // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int q_idx = qt * BM + row;              // row within the sequence
    const float c = p.scale_log2;
    float m_ref = -INFINITY;                      // running max, raw score units
    float l = 0.f;                                // running sum (relative to m_ref)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = wait_warp(bar(BAR_S_FULL), (uint32_t)j & 1u, abort_flag, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tmem_ld32(tmem + lane_off + COL_S + 0, s0);
      tmem_ld32(tmem + lane_off + COL_S + 32, s1);
      tmem_ld32(tmem + lane_off + COL_S + 64, s2);
      tmem_ld32(tmem + lane_off + COL_S + 96, s3);
      tmem_wait_ld();
      reg_fence32(s0);
      reg_fence32(s1);
      reg_fence32(s2);
      reg_fence32(s3);
      tc_fence_before();
      mbar_arrive(bar(BAR_S_FREE));   // S may now be overwritten by the next QK^T

      float s[BN];
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        s[x] = __uint_as_float(s0[x]);
        s[32 + x] = __uint_as_float(s1[x]);
        s[64 + x] = __uint_as_float(s2[x]);
        s[96 + x] = __uint_as_float(s3[x]);
      }
      // masking: causal diagonal tile and the sequence tail only
      const int kv0 = j * BN;
      const bool need_mask = (kv0 + BN > len) || (p.causal && kv0 + BN - 1 > qt * BM);
      if (need_mask) {
        const int lim = p.causal ? min(len, q_idx + 1) : len;   // keys < lim are visible
#pragma unroll
        for (int x = 0; x < BN; ++x)
          if (kv0 + x >= lim) s[x] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int x = 1; x < BN; ++x) mx = fmaxf(mx, s[x]);
      // move the reference max only when the tile max passes it by > threshold
      const float m_new = fmaxf(m_ref, mx);
      const bool rescale = (m_ref == -INFINITY) ? (m_new != -INFINITY)
                                                : ((m_new - m_ref) * c > RESCALE_THRESHOLD);
      float alpha = 1.f;
      if (rescale) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx((m_ref - m_new) * c);
        m_ref = m_new;
        l *= alpha;
      }
      const float neg_mc = (m_ref == -INFINITY) ? 0.f : -m_ref * c;
      uint32_t pk[BN / 2];
      float rs = 0.f;
#pragma unroll
      for (int x = 0; x < BN; x += 2) {
        const float e0 = ex2_approx(fmaf(s[x], c, neg_mc));
        const float e1 = ex2_approx(fmaf(s[x + 1], c, neg_mc));
        rs += e0 + e1;
        pk[x / 2] = pack_bf16x2(e0, e1);
      }
      l += rs;

      // P buffer j&1 was last read by PV_{j-2}
      if (j >= 2) {
        ok = wait_warp(bar(BAR_PV_DONE0 + (j & 1)), (uint32_t)((j - 2) >> 1) & 1u,
                          abort_flag, p.timeout_ns);
        if (!ok) break;
      }
      // rescale the O rows of this warp (after PV_{j-1} has landed)
      if (__any_sync(0xffffffffu, rescale && j > 0)) {
        ok = wait_warp(bar(BAR_PV_DONE0 + ((j - 1) & 1)), (uint32_t)((j - 1) >> 1) & 1u,
                          abort_flag, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + COL_O + cc, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(tmem + lane_off + COL_O + cc, o);
        }
      }
      const uint32_t p_col = COL_P0 + 64u * (uint32_t)(j & 1);
      {
        uint32_t a[32], b[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          a[x] = pk[x];
          b[x] = pk[32 + x];
        }
        tmem_st32(tmem + lane_off + p_col, a);
        tmem_st32(tmem + lane_off + p_col + 32, b);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(BAR_P_FULL0 + (j & 1)));
    }

    // ---- epilogue: O / l -> bf16, LSE ----
    if (ok)
      ok = wait_warp(bar(BAR_PV_DONE0 + ((n_kv - 1) & 1)), (uint32_t)((n_kv - 1) >> 1) & 1u,
                        abort_flag, p.timeout_ns);
    if (ok) {
      tc_fence_after();
      const bool live = q_idx < len;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *orow =
          p.o + ((long long)(seq_start + q_idx) * p.Hq + h) * (long long)D;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + COL_O + cc, o);
        tmem_wait_ld();
        reg_fence32(o);
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * inv_l,
                             __uint_as_float(o[2 * x + 1]) * inv_l);
        if (live) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + cc);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        }
      }
      if (live) {
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        p.lse[lse_base + q_idx] = l > 0.f ? m_use * p.scale + logf(l) : -INFINITY;
      }
    }
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// One block waits on a barrier that nobody signals, with a short limit: the
// wait runs out and records ATTN_ERR_TIMEOUT.  Used to test that path.
__global__ void selftest_timeout_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t barrier_word;
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&barrier_word), 1);
    abort_word = 0u;
    mbar_init_fence();
  }
  __syncthreads();
  wait_bounded(smem_u32(&barrier_word), 0, &abort_word, timeout_ns);
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [rows, heads, d] bf16, boxes of 128 rows x 64 columns of one head.
static bool make_map(EncodeTiledFn enc, CUtensorMap *m, const void *base, int heads,
                     long long rows, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)BM};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

constexpr int MAX_DEVICES = 64;

// Per device: compute capability check and the shared-memory opt-in of the
// three kernel instantiations, done once.
static attn_status prepare_device(int dev) {
  static std::mutex mu;
  static signed char state[MAX_DEVICES];   // 0 unknown, 1 ready, -1 unsupported
  if (dev < 0 || dev >= MAX_DEVICES) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (state[dev] == 1) return ATTN_OK;
  if (state[dev] == -1) return ATTN_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) {
    state[dev] = -1;
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  if (cudaFuncSetAttribute(attn_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<64>::SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<128>::SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(attn_fwd_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<256>::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  state[dev] = 1;
  return ATTN_OK;
}

static unsigned long long wait_timeout_ns() {
  static unsigned long long t = [] {
    const char *e = std::getenv("ATTN_WAIT_TIMEOUT_MS");
    long long ms = e ? std::atoll(e) : 0;
    if (ms <= 0 || ms > 600000) ms = 2000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return t;
}

template <int D>
static attn_status launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const Params &p, long long grid, cudaStream_t stream) {
  attn_fwd_kernel<D><<<(unsigned)grid, NUM_THREADS, Cfg<D>::SMEM_BYTES, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

extern "C" attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                const int *cu_seqlens, cudaStream_t stream) {
  using namespace attn;
  if (B < 0 || N < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 4))
    return ATTN_ERR_ALIGNMENT;
  const long long rows = cu_seqlens ? (long long)N : (long long)B * N;
  if (rows > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;   // TMA coordinates are int32

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status st = prepare_device(dev);
  if (st != ATTN_OK) return st;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return ATTN_ERR_CUDA;

  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, q, Hq, rows, d) || !make_map(enc, &mk, k, Hkv, rows, d) ||
      !make_map(enc, &mv, v, Hkv, rows, d))
    return ATTN_ERR_INVALID_ARG;

  Params p{};
  p.o = reinterpret_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.num_qt = (N + BM - 1) / BM;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();

  // fixed batch: exactly the tiles; packed: an upper bound on them
  // (sum_s ceil(L_s/128) <= T/128 + B), surplus CTAs exit at once.
  const long long pairs = cu_seqlens ? (long long)(N + BM - 1) / BM + B : (long long)p.num_qt * B;
  const long long grid = pairs * Hq;
  if (grid > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;

  switch (d) {
    case 64: return launch<64>(mq, mk, mv, p, grid, stream);
    case 128: return launch<128>(mq, mk, mv, p, grid, stream);
    default: return launch<256>(mq, mk, mv, p, grid, stream);
  }
}

extern "C" attn_status attn_get_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int value = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&value, attn::g_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (value != 0 && cudaMemcpyToSymbol(attn::g_status, &zero, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return static_cast<attn_status>(value);
}

extern "C" const char *attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "ATTN_ERR_UNSUPPORTED_DEVICE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_BAD_SEQLENS: return "ATTN_ERR_BAD_SEQLENS";
  }
  return "ATTN_UNKNOWN_STATUS";
}

extern "C" attn_status attn_selftest_timeout(int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status st = attn::prepare_device(dev);
  if (st != ATTN_OK) return st;
  attn::selftest_timeout_kernel<<<1, 32, 0, stream>>>((unsigned long long)timeout_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  return attn_get_status(stream);
}
