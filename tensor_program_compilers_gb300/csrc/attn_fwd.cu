// attn_fwd.cu -- fused attention forward for sm_103a (GB300) and its C ABI.
//
// A CTA works on 128-row query tiles of one (sequence, query head) at a time
// (one tile, or two in the two-tile kernel) and walks the key tiles of that
// sequence:
//
//   for each 128-key tile j (causal: only j <= the diagonal tile)
//     S    = Q K_j^T                       tcgen05.mma, bf16 -> fp32 in TMEM
//     m'   = max(m, rowmax S)              online-softmax monoid state (m, l)
//     P    = 2^(S*c - m'*c), c = scale*log2(e), rounded to bf16 into TMEM
//     l    = l * 2^((m - m')*c) + rowsum P      (two sums: of the fp32 P for
//                                               the LSE, of the rounded P for O)
//     O    = O * 2^((m - m')*c) + P V_j    tcgen05.mma, P read from TMEM
//   O / l -> bf16, LSE = m*scale + ln(l)
//
// This is the online-softmax reduction tang derives with stabilize_softmax
// (tang, muni.works/research/tang, section 2.3 and Table 1 rows "online
// softmax" and "FlashAttention forward"), in the block order of the TileLang
// explainer's loop (ai.thesatyajit.com/articles/tilelang, "FlashAttention,
// in tiles").  Two liberties, both exact in real arithmetic:
//  * the running max m is only moved when the exponentials against it would
//    leave range (a half-row sum above 2^16): softmax is shift invariant
//    (tang, section 6), so any reference value works as long as O and l share
//    it and the exponentials stay in range (each P <= 2^16 here);
//  * masked keys read -inf, the identity of max (tang, section 2.1, guarded
//    views), so fully masked tiles are skipped rather than computed.
//
// Two kernels share this file's pieces.  attn_fwd2.cuh holds the one used
// for head dims 64 and 128 without a key window or score modifier: two
// 128-row query tiles per CTA, one softmax thread per row.  The kernel below
// serves everything else (d = 256, windows, soft cap, ALiBi, decode, paged
// caches): one 128-row query tile per CTA.  Its warp roles (352 threads):
//   warp 0     TMA producer: Q, then K_0, K_1, V_0, K_2, V_1, ... into a ring
//              of shared-memory slots (128-byte swizzle)
//   warp 1     TMEM allocator and QK^T issuer (one thread); at d = 256 also
//              the PV issuer, keeping the order QK_{j+1}, PV_j
//   warps 2-9  softmax: warp w handles the rows of TMEM lane quarter w % 4
//              and keys 64 h .. 64 h + 63 of each key tile, h = (w - 2) / 4;
//              the two warps of a lane quarter share one reference maximum
//   warp 10    PV issuer (one thread), d <= 128
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S     [0, 128)          fp32 scores of the current key tile
//   P_b   [128 + 64 b, +64) bf16 probabilities (two per column), b < 2
//   O     [256, 256 + d)    fp32 accumulator
//   L     [256 + d, +16)    row sums of the rounded P (tensor core), d <= 128
// QK_{j+1} is issued as soon as the softmax warps have read S_j into
// registers, so it runs while they compute P_j.

// Every pipeline wait is bounded: past a time limit it records
// ATTN_ERR_TIMEOUT in a device status word and every role stops issuing,
// waits (bounded) for its copies and MMAs in flight, and the CTA releases
// its tensor memory and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "../../include/attn.h"
#include "ptx.cuh"

namespace attn {

// Diagnostic timeline (compiled in only with -DATTN_TRACE): clock() stamps of
// pipeline events of up to four chosen CTAs, read back with
// attn_trace_read().  Without the macro the hooks compile to nothing.
#ifdef ATTN_TRACE
constexpr int TRACE_CTAS = 4, TRACE_ROLES = 11, TRACE_STEPS = 64, TRACE_EVENTS = 12;
__device__ unsigned g_trace[TRACE_CTAS][TRACE_ROLES][TRACE_STEPS][TRACE_EVENTS];
__device__ int g_trace_cta[TRACE_CTAS] = {-1, -1, -1, -1};
__device__ __forceinline__ int trace_slot() {
  for (int i = 0; i < TRACE_CTAS; ++i)
    if ((int)blockIdx.x == g_trace_cta[i]) return i;
  return -1;
}
__device__ __forceinline__ void trace_ev(int slot, int role, long long step, int ev) {
  if (slot >= 0 && step >= 0 && step < TRACE_STEPS) {
    unsigned c;
    asm volatile("mov.u32 %0, %%clock;" : "=r"(c));
    g_trace[slot][role][step][ev] = c;
  }
}
__device__ __forceinline__ unsigned trace_clock() {
  unsigned c;
  asm volatile("mov.u32 %0, %%clock;" : "=r"(c));
  return c;
}
__device__ __forceinline__ void trace_put(int slot, int role, long long step, int ev, unsigned c) {
  if (slot >= 0 && step >= 0 && step < TRACE_STEPS) g_trace[slot][role][step][ev] = c;
}
#define ATTN_TRACE_SLOT() trace_slot()
#define ATTN_TRACE_EV(role, step, ev) trace_ev(tslot, role, step, ev)
// stamp now, store later (so that the store does not precede a release)
#define ATTN_TRACE_CLK(v) ((v) = trace_clock())
#define ATTN_TRACE_PUT(role, step, ev, v) trace_put(tslot, role, step, ev, v)
// stamps kept in shared memory (events 0..7 of steps 0..15), copied out at the end
#define ATTN_TRACE_SM(buf, step, ev) \
  do { if ((step) < 16) (buf)[(step) * 8 + (ev)] = trace_clock(); } while (0)
#define ATTN_TRACE_SM_FLUSH(buf, role)                                           \
  do {                                                                           \
    for (int s_ = 0; s_ < 16; ++s_)                                              \
      for (int e_ = 0; e_ < 8; ++e_) trace_put(tslot, role, s_, e_, (buf)[s_ * 8 + e_]); \
  } while (0)
#else
#define ATTN_TRACE_SLOT() (-1)
#define ATTN_TRACE_EV(role, step, ev) ((void)tslot)
#define ATTN_TRACE_CLK(v) ((void)(v))
#define ATTN_TRACE_PUT(role, step, ev, v) ((void)tslot)
#define ATTN_TRACE_SM(buf, step, ev) ((void)(buf))
#define ATTN_TRACE_SM_FLUSH(buf, role) ((void)(buf))
#endif

constexpr int BM = 128;            // query rows per tile (one per TMEM lane)
constexpr int BN = 128;            // keys per tile
constexpr int THREADS = 352;   // 11 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t CHUNK_BYTES = 128 * 128;   // 128 rows x 64 bf16, one swizzle column
// The reference max of a row moves only when a half-row's sum of P exceeds
// this (so every stored P is <= 2^16) or is not finite.
constexpr float P_SUM_LIMIT = 65536.0f;

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr uint32_t TILE_BYTES = CHUNKS * CHUNK_BYTES;   // one Q, K or V tile
  static constexpr int QB = D == 256 ? 1 : 2;                       // Q buffers
  static constexpr int STAGES = D == 64 ? 10 : (D == 128 ? 5 : 2);  // K/V ring slots
  // Separate QK^T and PV issuing threads when the ring is deep enough; with
  // two slots (d = 256) one thread keeps the order QK_{j+1}, PV_j so that the
  // load of V_j overlaps QK_{j+1}.
  static constexpr bool SPLIT_ISSUE = STAGES >= 4;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = TILE_BYTES * QB;
  static constexpr uint32_t OFF_CTL = OFF_KV + TILE_BYTES * STAGES;
  // Rounded row sums of P by the tensor core (P times a block of ones into
  // tensor-memory columns COL_L..+15) where tensor memory has room for them.
  static constexpr bool MMA_SUM = D <= 128;
  static constexpr uint32_t CTL_BYTES = D == 64 ? 3072 : 2048;
  static constexpr uint32_t ONES_BYTES = 512;   // 16 x 16 bf16 ones, no swizzle
  static constexpr uint32_t OFF_ONES = OFF_CTL + CTL_BYTES - ONES_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_CTL + CTL_BYTES + 1024;   // + alignment
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_P0 = 128;
  static constexpr uint32_t COL_O = 256;
  static constexpr uint32_t COL_L = COL_O + D;
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(!MMA_SUM || COL_L + 32 <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory");
};

// Barrier slots of the control block, then the K/V ring (full[0..STAGES),
// empty[0..STAGES)).
enum : int {
  BAR_Q_FULL0 = 0,   // Q buffer b loaded (TMA), b < 2
  BAR_Q_FULL1,
  BAR_Q_EMPTY0,      // Q buffer b no longer read (QK issuer commit)
  BAR_Q_EMPTY1,
  BAR_S_FULL,        // S written (QK issuer commit)
  BAR_S_FREE,        // S read into registers (softmax warps)
  BAR_P_FULL0,       // P_b written (softmax warps), b < 2
  BAR_P_FULL1,
  BAR_PV_DONE0,      // the PV reading P_b completed (PV issuer commit)
  BAR_PV_DONE1,
  BAR_O_FREE,        // O read by the epilogue (softmax warps)
  BAR_INFO_FULL0,    // tile-info entry e written (producer), e < INFO_SLOTS
  BAR_INFO_EMPTY0 = BAR_INFO_FULL0 + 4,   // tile-info entry e consumed
  BAR_DRAIN_QK = BAR_INFO_EMPTY0 + 4,     // abort drain of each issuer
  BAR_DRAIN_PV,
  BAR_PAIR0,         // softmax pair of TMEM lane quarter q, q < 4
  BAR_PAIR_END = BAR_PAIR0 + 4,
  BAR_RING = BAR_PAIR_END   // K/V ring: full[0..STAGES), then empty[0..STAGES)
};
constexpr int INFO_SLOTS = 4;
constexpr int INFO_INTS = 8;
constexpr int SOFTMAX_WARP0 = 2, SOFTMAX_WARPS = 8;
constexpr int WARP_PV = SOFTMAX_WARP0 + SOFTMAX_WARPS;   // 10

struct Params {
  const __nv_bfloat16 *q;
  __nv_bfloat16 *o;
  float *lse;
  const int *cu_seqlens;
  int B, Hq, Hkv, N, group;
  int causal;
  // key window: row i sees keys i - wl .. i + wr (clamped to the sequence;
  // causal makes wr 0; an unbounded side is the largest sequence length)
  int wl, wr;
  // score modifiers (kernels with MOD): soft cap s -> cap_k1 tanh(s cap_k2)
  // in raw score units (cap_k1 = cap / scale, cap_k2 = scale / cap), then
  // minus alibi[h] / scale * |i - j|
  int has_cap;
  float cap_k1, cap_k2;
  const float *alibi;
  // decode (split keys): q [B, dq_n, Hq, d] are the last dq_n positions of
  // sequences with keys k, v [B, dk_n, Hkv, d] rows 0 .. seqlens_k[b] - 1;
  // a work unit is (b, kv head, split) over keys split * chunk .. + chunk,
  // rows = the group's query heads x dq_n positions (head fastest).
  int dq_n, dk_n, splits, chunk;
  const int *seqlens_k;
  // paged caches (KIND 3): k, v [num_pages, page_size, Hkv, d]; key j of
  // sequence b is row j % page_size of page block_table[b * max_blocks +
  // j / page_size]; dk_n = max_blocks * page_size
  const int *block_table;
  int max_blocks, page_size, num_pages;
  int page_shift;   // log2(page_size) for a power of two, else -1
  // decode on the CUDA cores: the caches' rows, read with plain loads
  const __nv_bfloat16 *kc, *vc;
  float *ws_o;          // splits > 1: partial O / l [B, Hq, dq_n, splits, d]
  float *ws_lse;        // and partial LSE [B, Hq, dq_n, splits]
  int unit_rows;        // query rows per CTA work unit (one tile)
  int num_units;        // fixed batch: ceil(N / unit_rows)
  float scale;          // score multiplier
  float scale_log2;     // scale * log2(e)
  unsigned long long timeout_ns;
};

__device__ int g_status;   // first device-side error since the last read

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_status, 0, code); }

// ---------------------------------------------------------------- bounded waits
// Bounded wait on a barrier phase, slow path (kept out of line: a call costs
// a couple of hundred cycles, so the common already-complete case is tested
// inline by wait_bounded below).  Returns false if the CTA is aborting or the
// time limit passed (then it starts the abort).
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity,
                                       volatile uint32_t *abort_flag,
                                       unsigned long long timeout_ns) {
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

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t *abort_flag,
                                             unsigned long long timeout_ns) {
  return mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag, timeout_ns);
}

// Bounded wait by polling (mbarrier.test_wait in a loop), for barriers that
// other threads complete with plain arrivals: a thread suspended in try_wait
// on such a barrier was measured to resume several hundred cycles after the
// phase completed; a polling thread sees it within one shared-memory round
// trip.
__device__ __forceinline__ bool wait_poll_slow(uint32_t bar, uint32_t parity,
                                            volatile uint32_t *abort_flag,
                                            unsigned long long timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns || it > (1u << 30)) {
        *abort_flag = 1u;
        record_status(ATTN_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_poll(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns) {
  return mbar_test_wait(bar, parity) || wait_poll_slow(bar, parity, abort_flag, timeout_ns);
}

// One arrival per warp (count barriers in warps): after every lane's prior
// work (each lane fenced its tcgen05 operations before this point).
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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

// ---------------------------------------------------------------- tile schedule
struct Tile {
  int valid;
  int seq_start;   // token row of the sequence's first token
  int len;         // sequence length
  int unit;        // work-unit index within the sequence (unit_rows query rows)
  int h;           // query head
  long long lse_base;   // LSE index of the sequence's row 0 for head h
};

// Packed batches: number of work units of sequence s.
__device__ __forceinline__ int seq_units(const int *cu, int s, int unit_rows) {
  int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  return b > a ? (b - a + unit_rows - 1) / unit_rows : 0;
}

// Per-lane cache of the unit counts of sequences lane, lane+32, ... (up to
// SEQ_CACHE per lane); larger batches read cu_seqlens again each time.
constexpr int SEQ_CACHE = 4;

struct SeqUnits {
  int n[SEQ_CACHE];
  bool cached;
};

// Number of (sequence, unit) pairs whose unit index is >= x (warp-wide).
__device__ int units_at_or_above(const SeqUnits &su, const int *cu, int B, int x,
                                 int unit_rows) {
  int c = 0;
  if (su.cached) {
#pragma unroll
    for (int i = 0; i < SEQ_CACHE; ++i) c += max(0, su.n[i] - x);
  } else {
    for (int s = threadIdx.x & 31; s < B; s += 32) c += max(0, seq_units(cu, s, unit_rows) - x);
  }
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Map this CTA to its work unit (all 32 lanes of one warp).  Units are
// ordered longest first -- descending unit index, i.e. descending number of
// causal key tiles -- with heads fastest so that the query heads of one
// key/value head run side by side.
__device__ Tile decode_tile(const Params &p, long long idx, bool dec) {
  Tile t{};
  const int lane = threadIdx.x & 31;
  const int U = p.unit_rows;
  if (dec) {   // (b, kv head, split), split fastest
    const long long units = (long long)p.B * p.Hkv * p.splits;
    if (idx >= units) return t;
    const int s = (int)(idx % p.splits);
    const long long r = idx / p.splits;
    t.h = (int)(r % p.Hkv);
    t.seq_start = (int)(r / p.Hkv);   // the sequence index b
    const int L = p.seqlens_k ? __ldg(p.seqlens_k + t.seq_start) : p.dk_n;
    t.valid = 1;
    if (L < p.dq_n || L > p.dk_n) {   // an impossible length: report; no keys (skipped)
      if (lane == 0) record_status(ATTN_ERR_BAD_SEQLENS);
      t.len = 0;
      return t;
    }
    t.len = L;
    t.unit = s;
    t.valid = 1;
    return t;
  }
  if (p.cu_seqlens == nullptr) {
    const long long per = (long long)p.B * p.Hq;
    const int lvl = (int)(idx / per);
    const int rem = (int)(idx % per);
    const int b = rem / p.Hq;
    t.h = rem % p.Hq;
    t.unit = p.num_units - 1 - lvl;
    t.seq_start = b * p.N;
    t.len = p.N;
    t.lse_base = ((long long)b * p.Hq + t.h) * p.N;
    t.valid = t.unit >= 0 && idx < (long long)p.num_units * per;
    return t;
  }
  const int *cu = p.cu_seqlens;
  // validate the offsets and find the total and largest unit counts
  SeqUnits su;
  su.cached = p.B <= 32 * SEQ_CACHE;
#pragma unroll
  for (int i = 0; i < SEQ_CACHE; ++i) su.n[i] = 0;
  int bad = 0, nmax = 0, ntot = 0;
  for (int s = lane, i = 0; s < p.B; s += 32, ++i) {
    int a = __ldg(cu + s), b = __ldg(cu + s + 1);
    bad |= (b < a);
    int n = b > a ? (b - a + U - 1) / U : 0;
    if (su.cached) {
#pragma unroll
      for (int k = 0; k < SEQ_CACHE; ++k)
        if (k == i) su.n[k] = n;
    }
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
  const int u = (int)(idx / p.Hq);   // (sequence, unit) pair index
  t.h = (int)(idx % p.Hq);
  if (u >= ntot) {
    t.valid = 0;
    return t;
  }
  // largest x with units_at_or_above(x) > u: pair u sits at unit level x
  int lo = 0, hi = nmax;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (units_at_or_above(su, cu, p.B, mid, U) > u) lo = mid; else hi = mid;
  }
  const int x = lo;
  int r = u - units_at_or_above(su, cu, p.B, x + 1, U);   // rank among sequences with > x units
  int seq = -1;
  for (int base = 0, i = 0; base < p.B; base += 32, ++i) {
    const int s = base + lane;
    int n = 0;
    if (su.cached) {
#pragma unroll
      for (int k = 0; k < SEQ_CACHE; ++k)
        if (k == i) n = su.n[k];
    } else if (s < p.B) {
      n = seq_units(cu, s, U);
    }
    const bool has = s < p.B && n > x;
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
  t.unit = x;
  t.lse_base = (long long)t.h * p.N + t.seq_start;
  t.valid = 1;
  return t;
}

// ---------------------------------------------------------------- softmax pieces
// Two softmax warps share each TMEM lane quarter: for a query row, the thread
// of the first warp handles keys 0..63 of the key tile and the thread of the
// second keys 64..127 ("halves").  They keep one reference max per row.
constexpr int HB = BN / 2;   // keys per softmax thread

// This thread's 64 scores (TMEM columns col..col+63 of its lane).
__device__ __forceinline__ void load_half(uint32_t taddr, float (&h)[HB]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
  reg_fence32(a);
  reg_fence32(b);
#pragma unroll
  for (int x = 0; x < 32; ++x) {
    h[x] = __uint_as_float(a[x]);
    h[32 + x] = __uint_as_float(b[x]);
  }
}

// Keys key0 + x outside [lo, lim) are invisible: they read -inf, the
// identity of max.
__device__ __forceinline__ void mask_half(float (&h)[HB], int key0, int lo, int lim) {
#pragma unroll
  for (int x = 0; x < HB; ++x)
    if (key0 + x < lo || key0 + x >= lim) h[x] = -INFINITY;
}

// Score modifiers, in raw score units (the softmax multiplies by scale
// later): soft cap k1 tanh(s k2), then the ALiBi term -ak |i - j|.
__device__ __forceinline__ void modify_half(float (&h)[HB], int key0, int row, bool cap,
                                            float k1, float k2, float ak) {
#pragma unroll
  for (int x = 0; x < HB; ++x) {
    float v = h[x];
    if (cap) v = k1 * tanhf(v * k2);
    v -= ak * fabsf((float)(row - (key0 + x)));
    h[x] = v;
  }
}

// Key tiles a query tile visits: first tile j_lo and count n (keys any of
// rows r0 .. r0 + BM - 1 sees through the window, within the sequence).
__device__ __forceinline__ void kv_range(const Params &p, int qt, int len, int &j_lo, int &n,
                                         bool dec) {
  if (dec) {   // the split's keys qt * chunk .. min(len, (qt + 1) * chunk) - 1
    const int k0 = qt * p.chunk;
    const int k1 = min(len, k0 + p.chunk);
    j_lo = k0 / BN;
    n = k1 > k0 ? (k1 - k0 + BN - 1) / BN : 0;
    return;
  }
  const long long r0 = (long long)qt * BM;
  const long long lo_key = r0 - p.wl > 0 ? r0 - p.wl : 0;
  long long hi_key = r0 + BM - 1 + p.wr;
  if (hi_key > len - 1) hi_key = len - 1;
  j_lo = (int)(lo_key / BN);
  n = hi_key >= lo_key ? (int)(hi_key / BN) - j_lo + 1 : 0;
}

// Maximum of 64 scores: four independent chains of 3-input max.
__device__ __forceinline__ float max_half(const float (&h)[HB]) {
  float mk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m = max3f(h[k], h[k + 4], h[k + 8]);
#pragma unroll
    for (int i = 3; i + 1 < 16; i += 2) m = max3f(m, h[k + 4 * i], h[k + 4 * (i + 1)]);
    mk[k] = fmaxf(m, h[k + 4 * 15]);
  }
  return fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3]));
}

// p = 2^(h*c - m*c) for 64 scores: bf16 pairs into pk; sums of the fp32
// values into acc and, with RSUM, of the bf16-rounded values into accr (four
// packed accumulators each).
template <bool RSUM>
__device__ __forceinline__ void exp_half(const float (&h)[HB], uint64_t c2, uint64_t nm2,
                                         uint32_t (&pk)[HB / 2], uint64_t (&acc)[4],
                                         uint64_t (&accr)[4]) {
#pragma unroll
  for (int x = 0; x < HB; x += 2) {
    const uint64_t a = f2_fma(f2_pack(h[x], h[x + 1]), c2, nm2);
    float a0, a1;
    f2_unpack(a, a0, a1);
    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
    const uint32_t w = pack_bf16x2(e0, e1);
    pk[x >> 1] = w;
    acc[(x >> 1) & 3] = f2_add(acc[(x >> 1) & 3], f2_pack(e0, e1));
    // the rounded values too: the P.V product sees exactly these weights
    if (RSUM) accr[(x >> 1) & 3] = f2_add(accr[(x >> 1) & 3], bf16x2_widen(w));
  }
}

__device__ __forceinline__ float sum_acc(const uint64_t (&acc)[4]) {
  float a, b;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a, b);
  return a + b;
}

// Online-softmax state of one half-row: the row's reference max (raw score
// units, shared by both halves), the running sum of 2^((s - m) * c) over this
// half's keys (for the LSE) and the running sum of the same weights rounded
// to bf16 as the P.V product uses them (for O / l: a row dominated by one key
// then returns that key's value exactly).  Where the tensor core forms the
// rounded sums (next to O in tensor memory), lr stays unused.
struct RowState {
  float m;
  float l;
  float lr;
};

// The pair of softmax warps that share a TMEM lane quarter synchronise on an
// mbarrier of their own (one arrival per warp per round, bounded waits) and exchange
// values through shared memory.  Both warps run the same sequence of rounds,
// so `round` counts identically on both sides.
struct Pair {
  int wq, half, lane;
  uint32_t bar;          // this pair's mbarrier
  volatile float *xv;    // [4 quarters][2 halves][32 lanes] row values
  volatile int *xf;      // [2 buffers][4 quarters][2 halves] per-warp flags
  uint32_t round;
  volatile uint32_t *abort_flag;
  unsigned long long timeout_ns;
  __device__ bool sync() {
    warp_arrive(bar);
    const bool ok = wait_bounded(bar, round & 1u, abort_flag, timeout_ns);
    ++round;
    return __all_sync(0xffffffffu, ok);
  }
  // The partner's value of v for this row (two rounds: the slot is reused).
  __device__ bool exchange(float v, float &o) {
    xv[(wq * 2 + half) * 32 + lane] = v;
    if (!sync()) return false;
    o = xv[(wq * 2 + (half ^ 1)) * 32 + lane];
    return sync();
  }
  // OR of a warp-uniform flag over the pair, in one round split in two so
  // that other work can overlap the round trip: post() publishes the flag and
  // arrives, collect() waits and reads the partner's.  Flags are
  // double-buffered by round parity; a buffer is rewritten only after the
  // partner has finished the next round, i.e. has read it.
  __device__ void post(bool f) {
    if (lane == 0) xf[((round & 1u) * 4 + wq) * 2 + half] = f ? 1 : 0;
    warp_arrive(bar);
  }
  __device__ bool collect(bool f, bool &any) {
    const bool ok =
        __all_sync(0xffffffffu, wait_bounded(bar, round & 1u, abort_flag, timeout_ns));
    any = f || xf[((round & 1u) * 4 + wq) * 2 + (half ^ 1)] != 0;
    ++round;
    return ok;
  }
};

template <int NCOLS>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float alpha);

// Barrier addresses and parities one softmax step needs.
struct StepBars {
  uint32_t p_full;       // P_b written (this step)
  uint32_t pbuf_done;    // PV that last read P_b (step g-2) completed
  uint32_t pbuf_parity;
  uint32_t prev_done;    // PV of step g-1 completed (before rescaling O)
  uint32_t prev_parity;
  uint32_t s_full;       // S of the next step written
  uint32_t s_next_parity;
};

// One key tile of this thread's half-row, after its scores h are in
// registers (warp-collective: TMEM stores).  Writes P = 2^(s*c - m*c) as
// bf16 pairs to TMEM columns p_addr .. +31, rescales this half's O columns
// when the reference moves, and publishes P (P_FULL).  Returns false on a
// failed wait.  s_next_ready: a non-blocking early test of the next step's
// scores, to be used by the caller (valid if test_next).
//
// With a reference in place, the exponentials are taken against it straight
// away and stored; the pair moves the reference -- to the row maximum over
// both halves -- and redoes the tile only if some half-row's sum exceeds
// P_SUM_LIMIT (so every stored P is <= 2^16) or is not finite.  The first
// tile of a row takes the maximum first.  Either way P and both running sums
// share one reference, which is all that shift invariance requires.  The
// waits whose conditions usually hold already are tested early and collected
// late, so their shared-memory round trips overlap other work.
template <int OC, bool RSUM>
__device__ __forceinline__ bool softmax_step(const float (&h)[HB], RowState &st, float c,
                                             uint32_t p_addr, uint32_t o_addr, uint32_t l_addr,
                                             Pair &pr,
                                             const StepBars &sb, bool check_pbuf, bool rescale_ok,
                                             bool test_next, bool &s_next_ready,
                                             volatile uint32_t *abort_flag,
                                             unsigned long long timeout_ns, int tslot,
                                             int trole, long long g) {
  const bool pbuf_early = !check_pbuf || mbar_test_wait(sb.pbuf_done, sb.pbuf_parity);
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 8);
  const uint64_t c2 = f2_pack(c, c);
  uint64_t acc[4] = {0, 0, 0, 0}, accr[4] = {0, 0, 0, 0};
  uint32_t pk[HB / 2];
  // identical across the pair (same rows, same reference) and voted warp-wide
  const bool have_ref = __all_sync(0xffffffffu, st.m != -INFINITY);
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 9);
  float sum = 0.f;
  if (have_ref) {
    const float neg_mc = -st.m * c;
    exp_half<RSUM>(h, c2, f2_pack(neg_mc, neg_mc), pk, acc, accr);
    if (trole >= 0) ATTN_TRACE_EV(trole, g, 10);
    sum = sum_acc(acc);
  }
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 11);
  const bool want = __any_sync(0xffffffffu, !have_ref || !(sum <= P_SUM_LIMIT));
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 2);
  pr.post(want);
  // the P buffer must be free (its previous PV done) before it is written
  if (!__all_sync(0xffffffffu, pbuf_early) &&
      !wait_warp(sb.pbuf_done, sb.pbuf_parity, abort_flag, timeout_ns))
    return false;
  tc_fence_after();
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 3);
  if (have_ref) tmem_st32(p_addr, pk);   // optimistic; rewritten on a redo
  s_next_ready = test_next && mbar_test_wait(sb.s_full, sb.s_next_parity);
  bool redo;
  if (!pr.collect(want, redo)) return false;
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 4);
  float alpha = 1.f;
  bool moved = false;
  if (redo) {   // first tile, or the reference must move: take the row maximum
    const float hmax = max_half(h);
    float other;
    if (!pr.exchange(hmax, other)) return false;
    const float m_new = fmaxf(st.m, fmaxf(hmax, other));
    if (m_new != st.m) {
      alpha = (st.m == -INFINITY) ? 0.f : ex2_approx((st.m - m_new) * c);
      st.m = m_new;
      st.l *= alpha;
      st.lr *= alpha;
      moved = true;
    }
    const float neg_mc = (st.m == -INFINITY) ? 0.f : -st.m * c;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = accr[i] = 0;
    exp_half<RSUM>(h, c2, f2_pack(neg_mc, neg_mc), pk, acc, accr);
    tmem_st32(p_addr, pk);
    sum = sum_acc(acc);
  }
  st.l += sum;
  if (RSUM) st.lr += sum_acc(accr);
  if (__any_sync(0xffffffffu, moved && rescale_ok)) {   // rescale O after PV_{g-1} landed
    if (!wait_warp(sb.prev_done, sb.prev_parity, abort_flag, timeout_ns)) return false;
    tc_fence_after();
    rescale_o<OC>(o_addr, alpha);
    if (!RSUM && pr.half == 0)   // the row-sum column (one copy per row)
      tmem_st1(l_addr, __float_as_uint(__uint_as_float(tmem_ld_wait1(l_addr)) * alpha));
  }
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 5);
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(sb.p_full);
  if (trole >= 0) ATTN_TRACE_EV(trole, g, 6);
  return true;
}

// O[cols] *= alpha for NCOLS columns of this lane starting at taddr.  The
// caller issues tcgen05.wait::st before publishing.
template <int NCOLS>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
  for (int cc = 0; cc < NCOLS; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
#pragma unroll
    for (int x = 0; x < 32; x += 2) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[x]), __uint_as_float(o[x + 1])), a2), lo, hi);
      o[x] = __float_as_uint(lo);
      o[x + 1] = __float_as_uint(hi);
    }
    tmem_st32(taddr + cc, o);
  }
}

// Epilogue of NCOLS columns of one row: O / l -> bf16, 16-byte stores to orow
// (if live).
template <int NCOLS>
__device__ __forceinline__ void store_cols(uint32_t taddr, float inv_l, __nv_bfloat16 *orow,
                                           bool live) {
  const uint64_t s2 = f2_pack(inv_l, inv_l);
#pragma unroll 1
  for (int cc = 0; cc < NCOLS; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
    uint32_t w[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * x]), __uint_as_float(o[2 * x + 1])), s2),
                lo, hi);
      w[x] = pack_bf16x2(lo, hi);
    }
    if (live) {
      uint4 *dst = reinterpret_cast<uint4 *>(orow + cc);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        dst[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
    }
  }
}

// As store_cols, in fp32 (partial results of a key split).
template <int NCOLS>
__device__ __forceinline__ void store_cols_f32(uint32_t taddr, float inv_l, float *orow,
                                               bool live) {
#pragma unroll 1
  for (int cc = 0; cc < NCOLS; cc += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + cc, o);
    tmem_wait_ld();
    reg_fence32(o);
    if (live) {
      uint4 *dst = reinterpret_cast<uint4 *>(orow + cc);
#pragma unroll
      for (int x = 0; x < 8; ++x)
        dst[x] = make_uint4(__float_as_uint(__uint_as_float(o[4 * x]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * x + 1]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * x + 2]) * inv_l),
                            __float_as_uint(__uint_as_float(o[4 * x + 3]) * inv_l));
    }
  }
}

// Decode: the producer warp copies the query rows of work unit (b, kv head
// kvh) -- row r = query head kvh * group + r % group at position r / group --
// into a Q buffer in the layout a 128-byte-swizzled tile load would give
// (row r at byte 128 r of each 64-column chunk, 16-byte pieces XOR r % 8).
// The other rows of the buffer stay zero.
template <int D>
__device__ __forceinline__ void gather_q(const Params &p, int b, int kvh, uint32_t dst) {
  const int lane = threadIdx.x & 31;
  const int G = p.group, rows = G * p.dq_n;
  constexpr int PIECES = D / 8;   // 16-byte pieces per row
  for (int idx = lane; idx < rows * PIECES; idx += 32) {
    const int r = idx / PIECES, piece = idx % PIECES;
    const long long src_row = ((long long)b * p.dq_n + r / G) * p.Hq + (long long)kvh * G + r % G;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.q + src_row * D) + piece);
    st_shared_v4(dst + (uint32_t)(piece >> 3) * CHUNK_BYTES + (uint32_t)r * 128u +
                     ((uint32_t)((piece & 7) ^ (r & 7)) << 4),
                 v);
  }
}

// One 128x128xd QK^T into TMEM: A = Q tile (qdesc), B = K tile (kdesc), both
// K-major in 64-column swizzle chunks.  Per step of 16 head-dim columns the
// operands advance 32 bytes inside a 128-byte swizzle row, and CHUNK_BYTES
// from one 64-column chunk to the next.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BN, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t koff = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
    mma_ss(d_tmem, desc_add(qdesc, koff), desc_add(kdesc, koff), IDESC, kk > 0 ? 1u : 0u);
  }
}

// issue_qk for an issuing warp: every lane runs it with the same operands and
// one elected lane issues each MMA (descriptor offsets as plain integer
// additions: the 14-bit address field cannot carry, shared addresses stay
// below 256 KB).
template <int D>
__device__ __forceinline__ void issue_qk_warp(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BN, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t koff = ((kk >> 2) * CHUNK_BYTES + (kk & 3) * 32) >> 4;
    mma_ss_warp(d_tmem, qdesc + koff, kdesc + koff, IDESC, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V_j: A = P from TMEM (bf16 pairs), B = V tile (vdesc) with keys as
// K and the head dim as N (N contiguous: 64-wide swizzle atoms CHUNK_BYTES
// apart, 8-key groups 1024 bytes apart, 16 keys = 2048 bytes per step).
//
// With SUM, each step also adds P times a 16x16 block of ones into the
// 16 columns at l_tmem: every such column then holds the row sums of P as
// the product used them (bf16-rounded weights, fp32 accumulation).
template <int D, bool SUM>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                         uint32_t l_tmem, uint64_t ones_desc, bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(D, 1);
  constexpr uint32_t IDESC_SUM = idesc_bf16_f32(16, 0);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ts(d_tmem, p_tmem + kk * 8, desc_add(vdesc, kk * 2048), IDESC,
           (accumulate || kk > 0) ? 1u : 0u);
    if (SUM) mma_ts(l_tmem, p_tmem + kk * 8, ones_desc, IDESC_SUM, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// ---------------------------------------------------------------- control block
struct Ctl {
  uint32_t bar0;       // shared address of barrier 0 (barriers are 8 bytes apart)
  uint32_t *words;     // [0] TMEM base, [1] abort flag
  int *info;           // INFO_SLOTS entries of INFO_INTS ints
  float *xv;           // softmax pair exchange: 4 x 2 x 32 floats
  int *xf;             // softmax pair flags: 2 x 4 x 2 ints
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

template <int STAGES>
__device__ __forceinline__ void init_barriers(const Ctl &c, uint32_t info_consumers) {
  for (int b = 0; b < 2; ++b) {
    mbar_init(c.bar(BAR_Q_FULL0 + b), 1);
    mbar_init(c.bar(BAR_Q_EMPTY0 + b), 1);
    mbar_init(c.bar(BAR_P_FULL0 + b), SOFTMAX_WARPS);
    mbar_init(c.bar(BAR_PV_DONE0 + b), 1);
  }
  mbar_init(c.bar(BAR_S_FULL), 1);
  mbar_init(c.bar(BAR_S_FREE), SOFTMAX_WARPS);
  mbar_init(c.bar(BAR_O_FREE), SOFTMAX_WARPS);
  for (int e = 0; e < INFO_SLOTS; ++e) {
    mbar_init(c.bar(BAR_INFO_FULL0 + e), 1);
    mbar_init(c.bar(BAR_INFO_EMPTY0 + e), info_consumers);
  }
  mbar_init(c.bar(BAR_DRAIN_QK), 1);
  mbar_init(c.bar(BAR_DRAIN_PV), 1);
  for (int q = 0; q < 4; ++q) mbar_init(c.bar(BAR_PAIR0 + q), 2);
  for (int s = 0; s < STAGES; ++s) {
    mbar_init(c.bar(BAR_RING + s), 1);
    mbar_init(c.bar(BAR_RING + STAGES + s), 1);
  }
  c.words[1] = 0u;
  mbar_init_fence();
}

// A decoded work tile as the roles use it.
struct TileInfo {
  int valid, seq_start, len, qt, h;
  long long lse_base;
  int n_kv;   // key tiles to visit
};

// Consumer side of the tile-info ring: entry k % INFO_SLOTS (warp-uniform).
__device__ __forceinline__ bool read_tile(const Ctl &c, int k, TileInfo &t,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns, bool arrive) {
  const int e = k % INFO_SLOTS;
  if (!wait_bounded(c.bar(BAR_INFO_FULL0 + e), (uint32_t)(k / INFO_SLOTS) & 1u, abort_flag,
                    timeout_ns))
    return false;
  const volatile int *src = c.info + e * INFO_INTS;
  t.valid = src[0];
  t.seq_start = src[1];
  t.len = src[2];
  t.qt = src[3];
  t.h = src[4];
  t.n_kv = src[5];
  t.lse_base = (long long)(unsigned)src[6] | ((long long)src[7] << 32);
  if (arrive) mbar_arrive(c.bar(BAR_INFO_EMPTY0 + e));
  return true;
}

// O (+)= P_g V_i for global key step g (local step i of the tile): waits for
// P_g (softmax warps) and V_i at ring position pos, issues the MMAs, commits
// PV_DONE and the slot release.  The first step of a tile overwrites O.
template <int D>
__device__ __forceinline__ bool pv_step(const Ctl &ctl, uint32_t tmem, uint32_t kv_s, long long g,
                                        int i, long long pos, volatile uint32_t *abort_flag,
                                        unsigned long long timeout_ns, int tslot) {
  using C = Cfg<D>;
  const int slot = (int)(pos % C::STAGES);
  const int pb = (int)(g & 1);
  if (!wait_bounded(ctl.bar(BAR_P_FULL0 + pb), (uint32_t)(g >> 1) & 1u, abort_flag, timeout_ns))
    return false;
  ATTN_TRACE_EV(1, g, 0);
  if (!wait_bounded(ctl.bar(BAR_RING + slot), (uint32_t)(pos / C::STAGES) & 1u, abort_flag,
                    timeout_ns))
    return false;
  ATTN_TRACE_EV(1, g, 1);
  tc_fence_after();
  issue_pv<D, C::MMA_SUM>(tmem + C::COL_O, tmem + C::COL_P0 + 64u * (uint32_t)pb,
                          desc_add(smem_desc_sw128(kv_s, CHUNK_BYTES, 1024), slot * C::TILE_BYTES),
                          tmem + C::COL_L, smem_desc_plain(kv_s - C::OFF_KV + C::OFF_ONES, 128, 256),
                          i > 0);
  tc_commit(ctl.bar(BAR_PV_DONE0 + pb));
  tc_commit(ctl.bar(BAR_RING + C::STAGES + slot));
  ATTN_TRACE_EV(1, g, 2);
  return true;
}

// Ring positions of a tile's loads, in the producer's order K_0, K_1, V_0,
// K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1} (2n items from `base`).
__device__ __forceinline__ long long pos_k(long long base, int j) {
  return base + (j == 0 ? 0 : 2 * j - 1);
}
__device__ __forceinline__ long long pos_v(long long base, int i, int n) {
  return base + (i == n - 1 ? 2 * n - 1 : 2 * i + 2);
}

// The producer's load order K_0, K_1, V_0, K_2, V_1, ..., V_{n-1}: item 0 is
// K_0, the last item V_{n-1}, odd items K_{(item+1)/2}, even ones V_{item/2-1}.
__device__ __forceinline__ bool item_is_v(int item, int n) {
  return item == 2 * n - 1 || (item > 0 && (item & 1) == 0);
}
__device__ __forceinline__ int item_tile(int item, int n) {
  return item == 2 * n - 1 ? n - 1
                           : (item == 0 ? 0 : ((item & 1) == 0 ? item / 2 - 1 : (item + 1) / 2));
}

// ================================================================ kernel
// Persistent: with G = gridDim.x CTAs, CTA b processes one tile of each
// round of G tiles of the longest-first list -- tile b of even rounds, tile
// G-1-b of odd rounds -- until the producer publishes an invalid tile.
// KIND 0: plain; 1: score modifiers (soft cap, ALiBi); 2: decode (split
// keys); 3: decode from paged caches.
template <int D, int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D>;
  constexpr bool MOD = KIND == 1;
  constexpr bool DEC = KIND >= 2;
  constexpr bool PAGED = KIND == 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base_s = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_CTL);
  Ctl ctl;
  ctl.bar0 = smem_u32(bars);
  ctl.words = reinterpret_cast<uint32_t *>(bars + BAR_RING + 2 * C::STAGES);
  ctl.info = reinterpret_cast<int *>(ctl.words + 4);
  ctl.xv = reinterpret_cast<float *>(ctl.info + INFO_SLOTS * INFO_INTS);
  ctl.xf = reinterpret_cast<int *>(ctl.xv + 4 * 2 * 32);
  static_assert((BAR_RING + 2 * C::STAGES) * 8 + 16 + INFO_SLOTS * INFO_INTS * 4 + 4 * 2 * 32 * 4 +
                        2 * 4 * 2 * 4 <=
                    C::CTL_BYTES - C::ONES_BYTES,
                "control block");
  volatile uint32_t *abort_flag = ctl.words + 1;
  const uint32_t q_s = base_s + C::OFF_Q;
  const uint32_t kv_s = base_s + C::OFF_KV;
  const int tslot = ATTN_TRACE_SLOT();   // -1 unless built for tracing
  // consumers of each tile-info entry: QK issuer, PV issuer, the softmax warps
  constexpr uint32_t INFO_CONSUMERS = (C::SPLIT_ISSUE ? 2 : 1) + SOFTMAX_WARPS;

  if (warp == 1) {
    if (lane == 0) init_barriers<C::STAGES>(ctl, INFO_CONSUMERS);
    __syncwarp();
    tmem_alloc(smem_u32(ctl.words), TMEM_COLS);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  } else if (C::MMA_SUM && warp == SOFTMAX_WARP0) {
    // the block of ones (bf16 1.0 = 0x3F80) that the row-sum products read
    reinterpret_cast<uint4 *>(smem + C::OFF_ONES)[lane] =
        make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.words[0];

  if (warp == 0) {
    // ---------------- producer: decode tiles, publish them, load Q and K/V
    long long pos = 0;   // global ring position
    int q_loads = 0;     // Q tiles loaded so far (buffer q_loads % QB next)
    bool ok = true;
    long long round = 0;
    if (DEC) {   // padding rows of both Q buffers stay zero
      for (uint32_t off = (uint32_t)lane * 16u; off < C::QB * C::TILE_BYTES; off += 512u)
        st_shared_zero16(q_s + off);
    }
    for (int k = 0; ok; ++k) {
      // round r covers units [r G, (r+1) G); odd rounds run backwards so that
      // the CTA given the longest unit of a round gets the shortest next.
      // Decode splits past the end of their sequence hold no keys: skipped.
      const long long G = gridDim.x;
      Tile t;
      int j_lo = 0, n = 0;
      for (;;) {
        t = decode_tile(p, round * G + ((round & 1) ? G - 1 - blockIdx.x : blockIdx.x), DEC);
        ++round;
        if (!t.valid) break;
        kv_range(p, t.unit, t.len, j_lo, n, DEC);
        if (n > 0) break;
      }
      if (lane == 0) {
        const int e = k % INFO_SLOTS;
        ok = wait_bounded(ctl.bar(BAR_INFO_EMPTY0 + e), ((uint32_t)(k / INFO_SLOTS) & 1u) ^ 1u,
                          abort_flag, p.timeout_ns);
        if (ok) {
          int *dst = ctl.info + e * INFO_INTS;
          dst[0] = t.valid;
          dst[1] = t.seq_start;
          dst[2] = t.len;
          dst[3] = t.unit;
          dst[4] = t.h;
          dst[5] = n;
          dst[6] = (int)(unsigned)(t.lse_base & 0xFFFFFFFFll);
          dst[7] = (int)(t.lse_base >> 32);
          mbar_arrive(ctl.bar(BAR_INFO_FULL0 + e));   // release: the entry is visible
        }
      }
      const int qb = k % C::QB;
      if (DEC) {
        // Q buffer qb last served tile k - QB; then the warp gathers the
        // group's query rows (head fastest) into it in the swizzled layout
        if (lane == 0 && ok && t.valid && k >= C::QB)
          ok = wait_bounded(ctl.bar(BAR_Q_EMPTY0 + qb), (uint32_t)(k / C::QB - 1) & 1u,
                            abort_flag, p.timeout_ns);
        if (__shfl_sync(0xffffffffu, (ok && t.valid) ? 1 : 0, 0)) {
          gather_q<D>(p, t.seq_start, t.h, q_s + qb * C::TILE_BYTES);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl.bar(BAR_Q_FULL0 + qb));
        }
      }
      if (lane == 0) {
        if (ok && t.valid) {
          const int kvh = DEC ? t.h : t.h / p.group;
          // first key row of the sequence in the K/V tensors
          const int kv_row0 = DEC ? t.seq_start * p.dk_n : t.seq_start;
          if (!DEC) {
            // Q buffer qb last served tile k - QB
            if (k >= C::QB)
              ok = wait_bounded(ctl.bar(BAR_Q_EMPTY0 + qb), (uint32_t)(k / C::QB - 1) & 1u,
                                abort_flag, p.timeout_ns);
            if (ok) {
              ++q_loads;
              mbar_arrive_expect_tx(ctl.bar(BAR_Q_FULL0 + qb), C::TILE_BYTES);
              for (int c = 0; c < C::CHUNKS; ++c)
                tma_load_3d(q_s + qb * C::TILE_BYTES + c * CHUNK_BYTES, &tm_q,
                            ctl.bar(BAR_Q_FULL0 + qb), c * 64, t.h, t.seq_start + t.unit * BM);
            }
          }
          // K_0, K_1, V_0, K_2, V_1, ..., V_{n-1} (paged caches: below, by the warp)
          for (int item = 0; !PAGED && ok && item < 2 * n; ++item, ++pos) {
            const int slot = (int)(pos % C::STAGES);
            if (!(ok = wait_bounded(ctl.bar(BAR_RING + C::STAGES + slot),
                                    ((uint32_t)(pos / C::STAGES) & 1u) ^ 1u, abort_flag,
                                    p.timeout_ns)))
              break;
            const int kt = item_tile(item, n);
            const bool is_v = item_is_v(item, n);
            mbar_arrive_expect_tx(ctl.bar(BAR_RING + slot), C::TILE_BYTES);
            ATTN_TRACE_EV(10, pos >> 2, (int)(pos & 3));
            const uint32_t dst = kv_s + slot * C::TILE_BYTES;
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_3d(dst + c * CHUNK_BYTES, is_v ? &tm_v : &tm_k, ctl.bar(BAR_RING + slot),
                          c * 64, kvh, kv_row0 + (j_lo + kt) * BN);
          }
        }
      }
      if (PAGED) {
        // The tile's keys come in boxes of min(page, 128) rows, each from its
        // page: lane i issues box i / CHUNKS, column chunk i % CHUNKS (at most
        // 8 boxes x 4 chunks), so the page-number loads and the copies of one
        // tile go out together.  Keys past the sequence (and bad page
        // numbers) read a box wholly outside the tensor, i.e. zeros.
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && t.valid;
        const int rows = min(p.page_size, BN);
        const int boxes = BN / rows;
        const int *tbl = p.block_table + (long long)t.seq_start * p.max_blocks;
        for (int item = 0; ok && item < 2 * n; ++item, ++pos) {
          const int slot = (int)(pos % C::STAGES);
          if (lane == 0) {
            ok = wait_bounded(ctl.bar(BAR_RING + C::STAGES + slot),
                              ((uint32_t)(pos / C::STAGES) & 1u) ^ 1u, abort_flag, p.timeout_ns);
            if (ok) mbar_arrive_expect_tx(ctl.bar(BAR_RING + slot), C::TILE_BYTES);
          }
          if (!(ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0)) break;
          const int kt = item_tile(item, n);
          const bool is_v = item_is_v(item, n);
          if (lane < boxes * C::CHUNKS) {
            const int i = lane / C::CHUNKS, c = lane % C::CHUNKS;
            const int j = (j_lo + kt) * BN + i * rows;
            int page = -1;
            if (j < t.len) {
              page = __ldg(tbl + j / p.page_size);
              if (page < 0 || page >= p.num_pages) {
                record_status(ATTN_ERR_BAD_PAGE_TABLE);
                page = -1;
              }
            }
            const int row = page < 0 ? -rows : page * p.page_size + j % p.page_size;
            tma_load_3d(kv_s + slot * C::TILE_BYTES + c * CHUNK_BYTES + (uint32_t)(i * rows) * 128u,
                        is_v ? &tm_v : &tm_k, ctl.bar(BAR_RING + slot), c * 64,
                        DEC ? t.h : t.h / p.group, row);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && t.valid;
    }
    if (lane == 0 && *abort_flag) {
      // drain: wait (bounded) for the copies this thread issued
      for (int b = 0; b < C::QB && b < q_loads; ++b) {
        const int last = b + C::QB * ((q_loads - 1 - b) / C::QB);
        wait_drain(ctl.bar(BAR_Q_FULL0 + b), (uint32_t)(last / C::QB) & 1u, p.timeout_ns);
      }
      for (int s = 0; s < C::STAGES && s < pos; ++s) {
        const long long last = s + C::STAGES * ((pos - 1 - s) / C::STAGES);
        wait_drain(ctl.bar(BAR_RING + s), (uint32_t)(last / C::STAGES) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- QK^T issuer: S = Q K_j^T once the softmax warps have
    // read the previous S.  Without a separate PV issuer this thread also
    // issues PV_{j-1} right after QK_j.
    if (lane == 0) {
      const uint64_t kdesc0 = smem_desc_sw128(kv_s, 16, 1024);
      long long g = 0, base = 0;   // global key step, ring position of the tile's first load
      bool ok = true;
      for (int k = 0; ok; ++k) {
        TileInfo t;
        if (!(ok = read_tile(ctl, k, t, abort_flag, p.timeout_ns, true)) || !t.valid) break;
        const int qb = k % C::QB;
        const uint64_t qdesc = smem_desc_sw128(q_s + qb * C::TILE_BYTES, 16, 1024);
        if (!(ok = wait_bounded(ctl.bar(BAR_Q_FULL0 + qb), (uint32_t)(k / C::QB) & 1u,
                                abort_flag, p.timeout_ns)))
          break;
        for (int j = 0; ok && j < t.n_kv; ++j, ++g) {
          const long long pos = pos_k(base, j);
          const int slot = (int)(pos % C::STAGES);
          if (g > 0 && !(ok = wait_bounded(ctl.bar(BAR_S_FREE), (uint32_t)(g - 1) & 1u,
                                           abort_flag, p.timeout_ns)))
            break;
          ATTN_TRACE_EV(0, g, 0);
          if (!(ok = wait_bounded(ctl.bar(BAR_RING + slot), (uint32_t)(pos / C::STAGES) & 1u,
                                  abort_flag, p.timeout_ns)))
            break;
          ATTN_TRACE_EV(0, g, 1);
          tc_fence_after();
          issue_qk<D>(tmem + C::COL_S, qdesc, desc_add(kdesc0, slot * C::TILE_BYTES));
          tc_commit(ctl.bar(BAR_S_FULL));
          ATTN_TRACE_EV(0, g, 2);
          tc_commit(ctl.bar(BAR_RING + C::STAGES + slot));
          if (j == t.n_kv - 1) tc_commit(ctl.bar(BAR_Q_EMPTY0 + qb));   // Q buffer free
          if (!C::SPLIT_ISSUE && j > 0) {
            if (j == 1 && k > 0 &&   // the tile's first PV overwrites O
                !(ok = wait_bounded(ctl.bar(BAR_O_FREE), (uint32_t)(k - 1) & 1u, abort_flag,
                                    p.timeout_ns)))
              break;
            ok = pv_step<D>(ctl, tmem, kv_s, g - 1, j - 1, pos_v(base, j - 1, t.n_kv),
                            abort_flag, p.timeout_ns, tslot);
          }
        }
        if (!C::SPLIT_ISSUE && ok) {
          if (t.n_kv == 1 && k > 0)
            ok = wait_bounded(ctl.bar(BAR_O_FREE), (uint32_t)(k - 1) & 1u, abort_flag,
                              p.timeout_ns);
          if (ok)
            ok = pv_step<D>(ctl, tmem, kv_s, g - 1, t.n_kv - 1, pos_v(base, t.n_kv - 1, t.n_kv),
                            abort_flag, p.timeout_ns, tslot);
        }
        base += 2 * t.n_kv;
      }
      tc_commit(ctl.bar(BAR_DRAIN_QK));   // no MMA may be in flight at teardown
      wait_drain(ctl.bar(BAR_DRAIN_QK), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == WARP_PV) {
    // ---------------- PV issuer: O (+)= P_i V_i once the softmax warps have
    // written P_i; a tile's first PV also waits until the epilogue of the
    // previous tile has read O.
    if (C::SPLIT_ISSUE && lane == 0) {
      long long g = 0, base = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        TileInfo t;
        if (!(ok = read_tile(ctl, k, t, abort_flag, p.timeout_ns, true)) || !t.valid) break;
        for (int i = 0; ok && i < t.n_kv; ++i, ++g) {
          if (i == 0 && k > 0 &&
              !(ok = wait_bounded(ctl.bar(BAR_O_FREE), (uint32_t)(k - 1) & 1u, abort_flag,
                                  p.timeout_ns)))
            break;
          ok = pv_step<D>(ctl, tmem, kv_s, g, i, pos_v(base, i, t.n_kv), abort_flag,
                          p.timeout_ns, tslot);
        }
        base += 2 * t.n_kv;
      }
      tc_commit(ctl.bar(BAR_DRAIN_PV));
      wait_drain(ctl.bar(BAR_DRAIN_PV), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < WARP_PV) {
    // ---------------- softmax warps 2-9: warp w handles the rows of TMEM
    // lane quarter w % 4 and keys 64 * half .. 64 * half + 63 of every tile,
    // half = (w - 2) / 4; O columns are split the same way.
    const int wq = warp & 3;
    const int half = (warp - SOFTMAX_WARP0) >> 2;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    Pair pr{wq, half, lane, ctl.bar(BAR_PAIR0 + wq), ctl.xv, ctl.xf, 0u, abort_flag, p.timeout_ns};
    constexpr int OC = D / 2;   // O columns per half
    const float c = p.scale_log2;
    long long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      TileInfo t;
      ok = __all_sync(0xffffffffu, read_tile(ctl, k, t, abort_flag, p.timeout_ns, false));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(BAR_INFO_EMPTY0 + k % INFO_SLOTS));
      if (!t.valid) break;
      const int q_idx = t.qt * BM + row;            // row within the sequence
      int j_lo, n_unused;
      kv_range(p, t.qt, t.len, j_lo, n_unused, DEC);
      // decode: the row is query head (kv head * group + row % group) at
      // position row / group of the dq_n last positions; the split ends at
      // key k_end, and causal rows see keys up to their own position
      const int dq_pos = DEC ? row / p.group : 0;
      const int k_end = DEC ? min(t.len, (t.qt + 1) * p.chunk) : t.len;
      const int dec_lim =
          (p.causal && dq_pos < p.dq_n) ? min(k_end, t.len - p.dq_n + dq_pos + 1) : k_end;
      // this row's visible keys [lo, lim); a tile needs masking when some
      // row of the query tile does not see all of its keys
      const int lo = DEC ? 0 : q_idx - p.wl;                           // wl <= N
      const int lim = DEC ? dec_lim
                          : (p.wr >= t.len - q_idx ? t.len : q_idx + p.wr + 1);   // no overflow
      const int r0 = t.qt * BM;
      const float ak = (MOD && p.alibi) ? __ldg(p.alibi + t.h) / p.scale : 0.f;
      RowState st{-INFINITY, 0.f, 0.f};
      bool s_ready = false;   // early test of this step's S (from the previous step)
      for (int j = 0; j < t.n_kv; ++j, ++g) {
        if (!__all_sync(0xffffffffu, s_ready) &&
            !(ok = wait_warp(ctl.bar(BAR_S_FULL), (uint32_t)g & 1u, abort_flag, p.timeout_ns)))
          break;
        if (lane == 0) ATTN_TRACE_EV(2 + 2 * wq + half, g, 0);
        tc_fence_after();
        float hs[HB];
        load_half(tmem + lane_off + C::COL_S + HB * half, hs);
        tc_fence_before();
        warp_arrive(ctl.bar(BAR_S_FREE));   // S may now take the next scores
        if (lane == 0) ATTN_TRACE_EV(2 + 2 * wq + half, g, 1);
        const int kb = (j_lo + j) * BN;   // the tile's first key
        const int key0 = kb + HB * half;
        if (MOD) modify_half(hs, key0, q_idx, p.has_cap != 0, p.cap_k1, p.cap_k2, ak);
        // some row of the query tile misses keys of this tile: the sequence
        // ends inside it, or it reaches past the window of row r0 (right) or
        // of row r0 + BM - 1 (left)
        if (DEC ? (kb + BN > k_end || (p.causal && kb + BN - 1 > t.len - p.dq_n))
                : (kb + BN > t.len || kb + BN - 1 - r0 > p.wr || r0 + BM - 1 - kb > p.wl))
          mask_half(hs, key0, lo, lim);
        const int pb = (int)(g & 1);
        StepBars sb;
        sb.p_full = ctl.bar(BAR_P_FULL0 + pb);
        sb.pbuf_done = ctl.bar(BAR_PV_DONE0 + pb);             // P_b last read by PV_{g-2}
        sb.pbuf_parity = (uint32_t)((g - 2) >> 1) & 1u;
        sb.prev_done = ctl.bar(BAR_PV_DONE0 + (pb ^ 1));       // PV_{g-1}
        sb.prev_parity = (uint32_t)((g - 1) >> 1) & 1u;
        sb.s_full = ctl.bar(BAR_S_FULL);
        sb.s_next_parity = (uint32_t)(g + 1) & 1u;
        ok = softmax_step<OC, !C::MMA_SUM>(
            hs, st, c, tmem + lane_off + C::COL_P0 + 64u * (uint32_t)pb + 32u * (uint32_t)half,
            tmem + lane_off + C::COL_O + OC * half, tmem + lane_off + C::COL_L, pr, sb, g >= 2,
            j > 0, j + 1 < t.n_kv,
            s_ready, abort_flag, p.timeout_ns, tslot, lane == 0 ? 2 + 2 * wq + half : -1, g);
        if (!ok) break;
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE; then O is free for the next tile
      const long long gl = g - 1;   // the tile's last key step
      ok = wait_warp(ctl.bar(BAR_PV_DONE0 + (int)(gl & 1)), (uint32_t)(gl >> 1) & 1u, abort_flag,
                     p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      float l_other, lr;   // the partner half's exact sum; the row's rounded sum
      if (!(ok = pr.exchange(st.l, l_other))) break;
      if (C::MMA_SUM) {
        lr = __uint_as_float(tmem_ld_wait1(tmem + lane_off + C::COL_L));
      } else {
        float lr_other;
        if (!(ok = pr.exchange(st.lr, lr_other))) break;
        lr = st.lr + lr_other;
      }
      const float l = st.l + l_other;
      const float m_use = (st.m == -INFINITY) ? 0.f : st.m;
      const float lse_val = l > 0.f ? m_use * p.scale + logf(l) : -INFINITY;
      if (DEC) {
        // row -> (position, query head); o [B, dq_n, Hq, d], lse [B, Hq, dq_n]
        const bool live = row < p.group * p.dq_n;
        const int hq = t.h * p.group + row % p.group;
        const long long lrow = ((long long)t.seq_start * p.Hq + hq) * p.dq_n + dq_pos;
        if (p.splits == 1) {
          store_cols<OC>(tmem + lane_off + C::COL_O + OC * half, lr > 0.f ? 1.f / lr : 0.f,
                         p.o + (((long long)t.seq_start * p.dq_n + dq_pos) * p.Hq + hq) * D +
                             OC * half,
                         live);
          if (live && half == 0) p.lse[lrow] = lse_val;
        } else {   // partial state of this split: O / l and its LSE
          store_cols_f32<OC>(tmem + lane_off + C::COL_O + OC * half, lr > 0.f ? 1.f / lr : 0.f,
                             p.ws_o + (lrow * p.splits + t.qt) * D + OC * half, live);
          if (live && half == 0) p.ws_lse[lrow * p.splits + t.qt] = lse_val;
        }
      } else {
        const bool live = q_idx < t.len;
        store_cols<OC>(tmem + lane_off + C::COL_O + OC * half, lr > 0.f ? 1.f / lr : 0.f,
                       p.o + ((long long)(t.seq_start + q_idx) * p.Hq + t.h) * (long long)D +
                           OC * half,
                       live);
        if (live && half == 0) p.lse[t.lse_base + q_idx] = lse_val;
      }
      tc_fence_before();
      warp_arrive(ctl.bar(BAR_O_FREE));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace attn

#include "attn_fwd2.cuh"

namespace attn {

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

// Decode with several key splits: merge the partial states of each row
// (one warp per row) with the online-softmax combine in (LSE, O) form:
// LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.  Splits past a
// sequence's end hold nothing and are skipped.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.Hq * p.dq_n;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);   // (b Hq + h) dq_n + r
  if (row >= rows) return;
  const int b = (int)(row / ((long long)p.Hq * p.dq_n));
  const int h = (int)((row / p.dq_n) % p.Hq);
  const int r = (int)(row % p.dq_n);
  const int L = p.seqlens_k ? __ldg(p.seqlens_k + b) : p.dk_n;
  if (L < p.dq_n || L > p.dk_n) return;   // reported by the attention kernel
  const int ns = (L + p.chunk - 1) / p.chunk;
  const float *lse_s = p.ws_lse + row * p.splits;
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, lse_s[s]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  constexpr int PER = D / 32;   // columns per lane
  float acc[PER];
#pragma unroll
  for (int x = 0; x < PER; ++x) acc[x] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float w = expf(lse_s[s] - m);
      wsum += w;
      const float *os = p.ws_o + (row * p.splits + s) * D + lane * PER;
#pragma unroll
      for (int x = 0; x < PER; ++x) acc[x] += w * os[x];
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16 *dst = p.o + (((long long)b * p.dq_n + r) * p.Hq + h) * D + lane * PER;
#pragma unroll
  for (int x = 0; x < PER; ++x) dst[x] = __float2bfloat16_rn(acc[x] * inv);
  if (lane == 0) p.lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
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
                     long long rows, int d, int box_rows = BM) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

constexpr int MAX_DEVICES = 64;

template <typename K>
static bool opt_in_smem(K kernel, uint32_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
         cudaSuccess;
}

// Per device: compute capability check and the shared-memory opt-in of the
// kernel instantiations, done once.
static int g_sm_count[MAX_DEVICES];
static bool g_two_tiles_ok[MAX_DEVICES];
// attn_debug_one_tile: run every forward through the one-tile kernel.
static std::atomic<int> g_force_one_tile{0};

// Scratch of attn_fwd_decode_static: a fixed device array (the library
// allocates nothing); its address on each device is looked up once, when
// the device is first prepared.
constexpr size_t DECODE_SCRATCH_BYTES = 8u << 20;
static __device__ __align__(256) float g_decode_scratch[DECODE_SCRATCH_BYTES / sizeof(float)];
static void *g_scratch_ptr[MAX_DEVICES];

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
  if (cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess ||
      g_sm_count[dev] < 1)
    return ATTN_ERR_CUDA;
  if (!opt_in_smem(attn_fwd_kernel<64, 0>, Cfg<64>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<128, 0>, Cfg<128>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<256, 0>, Cfg<256>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<64, 1>, Cfg<64>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<128, 1>, Cfg<128>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<256, 1>, Cfg<256>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<64, 2>, Cfg<64>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<128, 2>, Cfg<128>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<256, 2>, Cfg<256>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<64, 3>, Cfg<64>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<128, 3>, Cfg<128>::SMEM_BYTES) ||
      !opt_in_smem(attn_fwd_kernel<256, 3>, Cfg<256>::SMEM_BYTES) ||
      !opt_in_smem(two::attn_fwd2_kernel<64>, two::Cfg2<64>::SMEM_BYTES) ||
      !opt_in_smem(two::attn_fwd2_kernel<128>, two::Cfg2<128>::SMEM_BYTES))
    return ATTN_ERR_CUDA;
  // the two-tile kernel's register split needs its launch share
  cudaFuncAttributes fa64, fa128;
  if (cudaFuncGetAttributes(&fa64, two::attn_fwd2_kernel<64>) != cudaSuccess ||
      cudaFuncGetAttributes(&fa128, two::attn_fwd2_kernel<128>) != cudaSuccess)
    return ATTN_ERR_CUDA;
  g_two_tiles_ok[dev] = fa64.numRegs >= two::REGS_NEEDED && fa128.numRegs >= two::REGS_NEEDED;
  if (cudaGetSymbolAddress(&g_scratch_ptr[dev], g_decode_scratch) != cudaSuccess)
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

}  // namespace attn

#include "attn_decode_cc.cuh"

extern "C" attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                const int *cu_seqlens, cudaStream_t stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, cu_seqlens, nullptr,
                     stream);
}

extern "C" attn_status attn_fwd_ex(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int Hq, int Hkv, int N, int d, float scale,
                                   int causal, const int *cu_seqlens, const attn_variant *var,
                                   cudaStream_t stream) {
  using namespace attn;
  if (B < 0 || N < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const float cap = var ? var->softcap : 0.f;
  if (!(cap >= 0.f) || !std::isfinite(cap)) return ATTN_ERR_INVALID_ARG;
  const float *slopes = var ? var->alibi_slopes : nullptr;
  if (slopes && (reinterpret_cast<uintptr_t>(slopes) & 3u)) return ATTN_ERR_ALIGNMENT;
  if (B == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
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
  p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
  p.o = reinterpret_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  // window bounds; a bound of N or more never masks anything
  const long long wl_in = var ? var->window_left : -1, wr_in = var ? var->window_right : -1;
  p.wl = (int)((wl_in < 0 || wl_in > N) ? N : wl_in);
  p.wr = causal ? 0 : (int)((wr_in < 0 || wr_in > N) ? N : wr_in);
  p.has_cap = cap > 0.f ? 1 : 0;
  p.cap_k1 = cap > 0.f ? cap / scale : 0.f;
  p.cap_k2 = cap > 0.f ? scale / cap : 0.f;
  p.alibi = slopes;
  const bool mod = cap > 0.f || slopes != nullptr;
  // Two query tiles per CTA (head dims 64, 128) unless a window or a score
  // modifier asks for the one-tile kernel.
  const bool two_tiles = g_two_tiles_ok[dev] && !g_force_one_tile.load() && !mod && d <= 128 &&
                         p.wl >= N && (causal || p.wr >= N);
  p.unit_rows = two_tiles ? two::UNIT_ROWS : BM;
  p.num_units = (N + p.unit_rows - 1) / p.unit_rows;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();

  // Persistent grid: one CTA per SM (at most one per work unit).  Fixed
  // batch: exactly num_units * B * Hq units; packed: an upper bound
  // (sum_s ceil(L_s/U) <= T/U + B, times Hq) -- the tile decoder marks the
  // surplus invalid.
  const long long units =
      (cu_seqlens ? (long long)p.num_units + B : (long long)p.num_units * B) * Hq;
  if (units > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
  // One CTA per tile when there are at most two tiles per SM (the hardware
  // scheduler balances small grids better than fixed rounds).
  const long long grid = units <= 2LL * g_sm_count[dev] ? units : (long long)g_sm_count[dev];

  const unsigned gr = (unsigned)grid;
  if (two_tiles) {
    if (d == 64)
      two::attn_fwd2_kernel<64><<<gr, two::THREADS2, two::Cfg2<64>::SMEM_BYTES, stream>>>(
          mq, mk, mv, p);
    else
      two::attn_fwd2_kernel<128><<<gr, two::THREADS2, two::Cfg2<128>::SMEM_BYTES, stream>>>(
          mq, mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  switch (d * 2 + (mod ? 1 : 0)) {
    case 128: attn_fwd_kernel<64, 0><<<gr, THREADS, Cfg<64>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
    case 129: attn_fwd_kernel<64, 1><<<gr, THREADS, Cfg<64>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
    case 256: attn_fwd_kernel<128, 0><<<gr, THREADS, Cfg<128>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
    case 257: attn_fwd_kernel<128, 1><<<gr, THREADS, Cfg<128>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
    case 512: attn_fwd_kernel<256, 0><<<gr, THREADS, Cfg<256>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
    default: attn_fwd_kernel<256, 1><<<gr, THREADS, Cfg<256>::SMEM_BYTES, stream>>>(mq, mk, mv, p); break;
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace attn {
// Key splits of a decode launch: at most one unit per SM, whole key tiles.
// Few query rows per (sequence, kv head) -- the group's heads x the new
// positions -- go to the CUDA-core decode kernel (dcc), more to the tile path.
static bool decode_on_cores(int Hq, int Hkv, int Nq, int d) {
  return (long long)(Hq / Hkv) * Nq <= 8 && (d == 64 || d == 128 || d == 256);
}

static int decode_cc_rows(int Hq, int Hkv, int Nq) {
  const long long rows = (long long)(Hq / Hkv) * Nq;
  return rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
}

// CUDA-core decode (one CTA of 8-16 warps per SM): whole (sequence, kv head)
// pairs once they fill half of the SMs -- a split costs a merge pass, which
// measured more than the idle SMs (B 16, Hkv 8 on 152 SMs: 0.103 ms with one
// split, 0.117 with two) -- else as many key splits (of at least 128 keys) as
// fit one round.
static void decode_splits_cc(int B, int Hkv, int Nk, int sms, int &splits, int &chunk) {
  const long long per = (long long)B * Hkv;
  long long want = 2 * per >= sms ? 1 : sms / per;
  const long long tiles = ((long long)Nk + BN - 1) / BN;
  if (want > tiles) want = tiles;
  if (want < 1) want = 1;
  chunk = (int)(((tiles + want - 1) / want) * BN);
  splits = (int)(((long long)Nk + chunk - 1) / chunk);
}

static void decode_splits(int B, int Hkv, int Nk, int sms, int &splits, int &chunk) {
  // At most one round of units: as many splits as keep every (sequence, kv
  // head) on whole SMs.  Measured (B 16, Hkv 8, Nk 8192 on 152 SMs): one
  // split 5.33 TB/s, two 4.84, three 4.77 -- the merge pass and the second
  // round's tail cost more than the idle SMs of a single round.
  const long long per = (long long)B * Hkv;
  long long want = sms / per;
  const int tiles = (Nk + BN - 1) / BN;
  if (want > tiles) want = tiles;
  if (want < 1) want = 1;
  chunk = (int)(((tiles + want - 1) / want) * BN);
  splits = (Nk + chunk - 1) / chunk;
}

static size_t decode_ws_bytes(int B, int Hq, int Nq, int d, int splits) {
  if (splits <= 1) return 0;
  return (size_t)B * Hq * Nq * splits * ((size_t)d + 1) * sizeof(float);
}
}  // namespace attn

extern "C" size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  using namespace attn;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || prepare_device(dev) != ATTN_OK) return 0;
  int splits, chunk;
  if (decode_on_cores(Hq, Hkv, Nq, d))
    decode_splits_cc(B, Hkv, Nk, g_sm_count[dev], splits, chunk);
  else
    decode_splits(B, Hkv, Nk, g_sm_count[dev], splits, chunk);
  return decode_ws_bytes(B, Hq, Nq, d, splits);
}

namespace attn {
template <int D, int RP, bool PAGED>
static bool launch_dcc_kernel(unsigned grid, const Params &p, cudaStream_t stream) {
  static std::atomic<bool> opted[MAX_DEVICES];   // its ring exceeds the default 48 KB
  constexpr int bytes = dcc::ring_bytes(RP);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return false;
  if (!opted[dev].load()) {
    if (cudaFuncSetAttribute(dcc::attn_decode_cc_kernel<D, RP, PAGED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return false;
    opted[dev].store(true);
  }
  dcc::attn_decode_cc_kernel<D, RP, PAGED>
      <<<grid, dcc::warps_for(RP) * 32, bytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess;
}
template <int D, int RP>
static bool launch_dcc(bool paged, unsigned grid, const Params &p, cudaStream_t stream) {
  return paged ? launch_dcc_kernel<D, RP, true>(grid, p, stream)
               : launch_dcc_kernel<D, RP, false>(grid, p, stream);
}
template <int D>
static bool launch_dcc_rows(int rp, bool paged, unsigned grid, const Params &p,
                            cudaStream_t stream) {
  switch (rp) {
    case 1: return launch_dcc<D, 1>(paged, grid, p, stream);
    case 2: return launch_dcc<D, 2>(paged, grid, p, stream);
    case 4: return launch_dcc<D, 4>(paged, grid, p, stream);
    default: return launch_dcc<D, 8>(paged, grid, p, stream);
  }
}
static bool launch_decode_cc(int d, int rp, bool paged, unsigned grid, const Params &p,
                             cudaStream_t stream) {
  switch (d) {
    case 64: return launch_dcc_rows<64>(rp, paged, grid, p, stream);
    case 128: return launch_dcc_rows<128>(rp, paged, grid, p, stream);
    default: return launch_dcc_rows<256>(rp, paged, grid, p, stream);
  }
}

// The decode call; with use_static the workspace is the fixed device array.
struct PagedArgs {
  const int *block_table;
  int max_blocks, page_size, num_pages;
};

// The decode call; with use_static the workspace is the fixed device array;
// with pg the caches are paged (Nk = max_blocks * page_size).
static attn_status decode_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                               int causal, const int *seqlens_k, void *workspace,
                               size_t workspace_bytes, bool use_static, const PagedArgs *pg,
                               cudaStream_t stream) {
  if (B < 0 || Nq < 0 || Nk < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((long long)(Hq / Hkv) * Nq > BM || Nq > Nk) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 4) || misaligned(seqlens_k, 4) || misaligned(workspace, 16))
    return ATTN_ERR_ALIGNMENT;
  const long long krows = pg ? (long long)pg->num_pages * pg->page_size : (long long)B * Nk;
  if (krows > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status st = prepare_device(dev);
  if (st != ATTN_OK) return st;
  const bool cores = decode_on_cores(Hq, Hkv, Nq, d);
  int splits, chunk;
  if (cores)
    decode_splits_cc(B, Hkv, Nk, g_sm_count[dev], splits, chunk);
  else
    decode_splits(B, Hkv, Nk, g_sm_count[dev], splits, chunk);
  const size_t need = decode_ws_bytes(B, Hq, Nq, d, splits);
  if (use_static) {
    workspace = g_scratch_ptr[dev];
    workspace_bytes = DECODE_SCRATCH_BYTES;
  }
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_INVALID_ARG;
  CUtensorMap mk, mv;
  if (!cores) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return ATTN_ERR_CUDA;
    const int box_rows = pg ? std::min(pg->page_size, BN) : BM;
    if (!make_map(enc, &mk, k, Hkv, krows, d, box_rows) ||
        !make_map(enc, &mv, v, Hkv, krows, d, box_rows))
      return ATTN_ERR_INVALID_ARG;
  }

  Params p{};
  p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
  p.o = reinterpret_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = Nk;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.dq_n = Nq;
  p.dk_n = Nk;
  p.splits = splits;
  p.chunk = chunk;
  p.seqlens_k = seqlens_k;
  if (pg) {
    p.block_table = pg->block_table;
    p.max_blocks = pg->max_blocks;
    p.page_size = pg->page_size;
    p.num_pages = pg->num_pages;
    p.page_shift = (pg->page_size & (pg->page_size - 1)) == 0 ? __builtin_ctz(pg->page_size) : -1;
  }
  p.ws_o = reinterpret_cast<float *>(workspace);
  p.ws_lse = need > 0 ? p.ws_o + (size_t)B * Hq * Nq * splits * d : nullptr;
  p.unit_rows = BM;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.kc = reinterpret_cast<const __nv_bfloat16 *>(k);
  p.vc = reinterpret_cast<const __nv_bfloat16 *>(v);

  const long long units = (long long)B * Hkv * splits;
  if (cores) {
    if (units > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
    if (!launch_decode_cc(d, decode_cc_rows(Hq, Hkv, Nq), pg != nullptr, (unsigned)units, p,
                          stream))
      return ATTN_ERR_CUDA;
  } else {
    const long long grid = units <= 2LL * g_sm_count[dev] ? units : (long long)g_sm_count[dev];
    const unsigned gr = (unsigned)grid;
    switch (d * 2 + (pg ? 1 : 0)) {   // no Q tensor map: decode gathers its query rows
      case 128: attn_fwd_kernel<64, 2><<<gr, THREADS, Cfg<64>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
      case 129: attn_fwd_kernel<64, 3><<<gr, THREADS, Cfg<64>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
      case 256: attn_fwd_kernel<128, 2><<<gr, THREADS, Cfg<128>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
      case 257: attn_fwd_kernel<128, 3><<<gr, THREADS, Cfg<128>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
      case 512: attn_fwd_kernel<256, 2><<<gr, THREADS, Cfg<256>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
      default: attn_fwd_kernel<256, 3><<<gr, THREADS, Cfg<256>::SMEM_BYTES, stream>>>(mk, mk, mv, p); break;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (splits > 1) {
    const unsigned cg = (unsigned)(((long long)B * Hq * Nq + 7) / 8);
    switch (d) {
      case 64: attn_combine_kernel<64><<<cg, 256, 0, stream>>>(p); break;
      case 128: attn_combine_kernel<128><<<cg, 256, 0, stream>>>(p); break;
      default: attn_combine_kernel<256><<<cg, 256, 0, stream>>>(p); break;
    }
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}
}  // namespace attn

extern "C" attn_status attn_fwd_decode(const void *q, const void *k, const void *v, void *o,
                                       float *lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                       float scale, int causal, const int *seqlens_k,
                                       void *workspace, size_t workspace_bytes,
                                       cudaStream_t stream) {
  return attn::decode_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, seqlens_k,
                           workspace, workspace_bytes, false, nullptr, stream);
}

extern "C" size_t attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int Nq,
                                                     int max_blocks, int page_size, int d) {
  const long long nk = (long long)max_blocks * page_size;
  if (max_blocks < 1 || page_size < 1 || nk > 0x7FFFFFFFLL) return 0;
  return attn_decode_workspace_bytes(B, Hq, Hkv, Nq, (int)nk, d);
}

extern "C" attn_status attn_fwd_decode_paged(const void *q, const void *k_cache,
                                             const void *v_cache, void *o, float *lse, int B,
                                             int Hq, int Hkv, int Nq, int d, float scale,
                                             int causal, const int *seqlens_k,
                                             const int *block_table, int max_blocks,
                                             int page_size, int num_pages, void *workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
  // pages of 16, 32 or 64 rows fill a 128-key tile with several boxes;
  // pages of a multiple of 128 rows hold whole tiles
  constexpr int BN = attn::BN;
  const bool page_ok = page_size >= 16 && ((BN % page_size == 0 && (page_size & 15) == 0) ||
                                           page_size % BN == 0);
  if (!page_ok || max_blocks < 1 || num_pages < 1 || !seqlens_k || !block_table)
    return ATTN_ERR_INVALID_ARG;
  if ((long long)max_blocks * page_size > 0x7FFFFFFFLL) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_table) & 3u) return ATTN_ERR_ALIGNMENT;
  const attn::PagedArgs pg{block_table, max_blocks, page_size, num_pages};
  return attn::decode_impl(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Nq, max_blocks * page_size,
                           d, scale, causal, seqlens_k, workspace, workspace_bytes, false, &pg,
                           stream);
}

extern "C" attn_status attn_fwd_decode_static(const void *q, const void *k, const void *v,
                                              void *o, float *lse, int B, int Hq, int Hkv,
                                              int Nq, int Nk, int d, float scale, int causal,
                                              const int *seqlens_k, cudaStream_t stream) {
  return attn::decode_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, seqlens_k,
                           nullptr, 0, true, nullptr, stream);
}

namespace attn {
// The status word is taken and cleared in one atomic exchange on the device,
// so an error that a kernel on another stream records at any moment is
// either returned by this read or kept for the next one.
__device__ int g_status_taken;
__global__ void take_status_kernel() { g_status_taken = atomicExch(&g_status, 0); }
}  // namespace attn

extern "C" attn_status attn_get_status(cudaStream_t stream) {
  static std::mutex mu;   // one g_status_taken per device, shared by all callers
  std::lock_guard<std::mutex> lock(mu);
  attn::take_status_kernel<<<1, 1, 0, stream>>>();
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  int value = 0;
  if (cudaMemcpyFromSymbolAsync(&value, attn::g_status_taken, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return static_cast<attn_status>(value);
}

#ifdef ATTN_TRACE
// Diagnostic builds only: choose the traced CTAs (and clear the buffer), and
// copy the stamps out (TRACE_CTAS x TRACE_ROLES x TRACE_STEPS x TRACE_EVENTS).
extern "C" int attn_trace_setup(const int *ctas) {
  static unsigned zero[attn::TRACE_CTAS][attn::TRACE_ROLES][attn::TRACE_STEPS]
                      [attn::TRACE_EVENTS];
  if (cudaMemcpyToSymbol(attn::g_trace, zero, sizeof zero) != cudaSuccess) return 1;
  return cudaMemcpyToSymbol(attn::g_trace_cta, ctas, sizeof(int) * attn::TRACE_CTAS) !=
         cudaSuccess;
}
extern "C" int attn_trace_read(unsigned *out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  return cudaMemcpyFromSymbol(out, attn::g_trace, sizeof(attn::g_trace)) != cudaSuccess;
}
#endif

extern "C" int attn_debug_one_tile(int on) { return attn::g_force_one_tile.exchange(on ? 1 : 0); }

extern "C" const char *attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "ATTN_ERR_UNSUPPORTED_DEVICE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_BAD_SEQLENS: return "ATTN_ERR_BAD_SEQLENS";
    case ATTN_ERR_BAD_PAGE_TABLE: return "ATTN_ERR_BAD_PAGE_TABLE";
  }
  return "ATTN_UNKNOWN_STATUS";
}

namespace attn {
// Pointer chase for the latency term of the time floor: entry i holds the
// index of the entry `stride` further on (mod n).
__global__ void probe_init_kernel(unsigned long long *buf, unsigned long long n,
                                  unsigned long long stride) {
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x)
    buf[i] = (i + stride) % n;
}
__global__ void probe_chase_kernel(const unsigned long long *buf, int hops,
                                   unsigned long long *result) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  unsigned long long idx = 0;
  const uint64_t t0 = globaltimer_ns();
  for (int h = 0; h < hops; ++h) {
    unsigned long long nxt;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(nxt) : "l"(buf + idx) : "memory");
    idx = nxt;
  }
  const uint64_t t1 = globaltimer_ns();
  result[0] = t1 - t0;
  result[1] = idx;
}
}  // namespace attn

extern "C" attn_status attn_probe_dram_latency(void *scratch, size_t bytes, int hops,
                                               unsigned long long *result, cudaStream_t stream) {
  if (!scratch || !result || hops < 1 || hops > 1000000 || bytes < (64ull << 20))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scratch) & 15u) || (reinterpret_cast<uintptr_t>(result) & 7u))
    return ATTN_ERR_ALIGNMENT;
  const unsigned long long n = bytes / 8, stride = 4160 / 8;
  attn::probe_init_kernel<<<1024, 256, 0, stream>>>(static_cast<unsigned long long *>(scratch), n,
                                                    stride);
  attn::probe_chase_kernel<<<1, 32, 0, stream>>>(
      static_cast<const unsigned long long *>(scratch), hops, result);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
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

#include "attn_bwd.cuh"
