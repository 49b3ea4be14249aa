// attn_fwd2.cuh -- the attention forward with two query tiles per CTA, for
// head dims 64 and 128 without a key window or score modifier.  Included by
// attn_fwd.cu, whose helpers (waits, tile decoding, softmax pieces, MMA
// issue) it uses.
//
// A work unit is 256 query rows of one (sequence, query head): tile A is rows
// 0..127 of the unit, tile B rows 128..255.  Both tiles walk the same key
// tiles, so each K_j and V_j is loaded once for 256 rows.  Every softmax
// thread owns one whole query row (all 128 keys of a key tile), so no two
// warps share a row; while the softmax warps of one tile work on P, the
// tensor core runs the other tile's products.  The computation per row is the
// one attn_fwd.cu describes (online softmax with a lazily moved reference
// maximum; tang, section 2.3, Table 1 "FlashAttention forward").  O is
// divided by the sum of the bf16-rounded weights exactly as P.V uses them
// (so a row whose weight sits on one key returns that key's value), the LSE
// taken from the sum of the fp32 weights.  The rounded sum is formed after P
// is handed to the MMA issuer, off the path to it.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax of tile A: lane t of warp w owns query row 32 w + t
//              (TMEM lane 32 w + t)
//   warps 4-7  softmax of tile B (TMEM lane quarter w % 4)
//   warp 8     TMA producer: Q_A, Q_B of the unit, then K_0, V_0, K_1, V_1, ...
//   warp 9     TMEM allocator and MMA issuer: the whole warp runs the issue
//              loop and one elected lane issues each tcgen05 instruction
//   warp 10    K/V watcher: adds one arrival to P_FULL_X(j) once V_j (and
//              K_{j+1}, if tile X computes S(j+1)) have landed, so that the
//              MMA warp waits on nothing but P_FULL between its batches
//   warp 11    idle (completes the third warpgroup, which hands part of its
//              registers to the softmax warpgroups)
//
// Tensor memory (512 columns): S_A [0, 128), S_B [128, 256),
// O_A [256, 256 + d), O_B [256 + d, 256 + 2d).  P_X (bf16 pairs, keys 2c and
// 2c + 1 in column c) is written over columns [0, 64) of S_X.
//
// MMA order (one warp; the tensor core runs its MMAs in issue order):
// QK_A(0), QK_B(0), then for each key step j
//   PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1).
// QK_X(j+1) overwrites S_X only after PV_X(j) has read P_X(j) from it, and
// the commit that signals S_X(j+1) also covers PV_X(j): a softmax warp that
// sees S_X(j+1) may rescale O_X at once.
//
// Measured on this GPU, a tcgen05.mma costs the issuing warp ~45 cycles
// against the 64 the tensor core takes to run a 128 x 128 x 16 product, so the
// issue loop holds only ~16 cycles of slack per MMA: one wait per batch (P),
// the commits the consumers need, and a warp-uniform (elected-lane) issue,
// which kept its rate beside the busy softmax warps of its sub-partition
// where a single diverged lane fell far behind.

namespace attn {
namespace two {

constexpr int THREADS2 = 384;   // three warpgroups
// Warpgroups 0 and 1: the softmax of tiles A and B; warpgroup 2: producer
// and MMA issuer (warps 10, 11 only complete it).
constexpr int SM_WARP0 = 0, WARP_PROD = 8, WARP_MMA = 9, WARP_WATCH = 10;
// Register split (setmaxnreg): the kernel is built for 168 registers a thread
// (384 threads; three warps share each SM sub-partition); the third
// warpgroup gives part of its share to the softmax warpgroups:
// 2 x 128 x 208 + 128 x 88 = 64,512 = 384 x 168.  The host checks
// the built register count against this before it uses the kernel.
constexpr int REGS_SOFTMAX = 208, REGS_OTHER = 88;
constexpr int REGS_NEEDED = (2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER + THREADS2 - 1) / THREADS2;
constexpr int UNIT_ROWS = 2 * BM;
constexpr int UNIT_INTS = 10;   // valid, seq_start, len, unit, h, nA, nB, lse lo/hi

template <int D>
struct Cfg2 {
  static constexpr int CHUNKS = D / 64;
  static constexpr uint32_t TILE_BYTES = CHUNKS * CHUNK_BYTES;   // one 128-row Q, K or V tile
  // Q buffers (two tiles each) and K/V ring slots.  At d = 128 one Q buffer
  // pair and five ring slots: a K/V tile's load then starts about two key
  // steps before its first reader (with two Q buffer pairs and three slots,
  // about one, and the MMAs waited for their operands), at the cost of
  // loading the next unit's Q only after this unit's last QK.
  static constexpr int QB = D == 64 ? 2 : 1;
  static constexpr int STAGES = D == 64 ? 8 : 5;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = 2 * TILE_BYTES * QB;
  static constexpr uint32_t OFF_CTL = OFF_KV + TILE_BYTES * STAGES;
  static constexpr uint32_t CTL_BYTES = 1024;
  static constexpr uint32_t SMEM_BYTES = OFF_CTL + CTL_BYTES + 1024;   // + alignment
  static constexpr uint32_t COL_O = 256;                               // O_X at COL_O + D X
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(COL_O + 2 * D <= TMEM_COLS, "tensor memory");
};

enum : int {
  T_Q_FULL0 = 0,   // Q buffer b (both tiles) loaded, b < 2
  T_Q_FULL1,
  T_Q_EMPTY0,      // Q buffer b no longer read (MMA issuer commit)
  T_Q_EMPTY1,
  T_S_FULL0,       // S_X written (commit; also covers PV_X of the previous step), X < 2
  T_S_FULL1,
  T_P_FULL0,       // P_X written over S_X (the tile's four softmax warps) and V_j, K_{j+1} landed (watcher)
  T_P_FULL1,
  T_PV_DONE0,      // PV_X completed (commit)
  T_PV_DONE1,
  T_O_FREE0,       // O_X read by the epilogue (four warps)
  T_O_FREE1,
  T_INFO_FULL0,                            // unit-info entry e written (producer)
  T_INFO_EMPTY0 = T_INFO_FULL0 + INFO_SLOTS,   // entry e consumed
  T_DRAIN = T_INFO_EMPTY0 + INFO_SLOTS,    // teardown drain of the MMA issuer
  T_RING                                   // K/V ring: full[0..STAGES), empty[0..STAGES)
};

struct Ctl2 {
  uint32_t bar0;     // shared address of barrier 0 (8 bytes apart)
  uint32_t *words;   // [0] TMEM base, [1] abort flag
  int *info;         // INFO_SLOTS entries of UNIT_INTS ints
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

struct UnitInfo {
  int valid, seq_start, len, unit, h, n[2];
  long long lse_base;
};

// Key tiles of the two tiles of unit u of a sequence of len rows: causal
// rows see keys up to their own position (tile A's last key tile is 2u, tile
// B's 2u + 1); a tile that starts past the sequence has none.
__device__ __forceinline__ void unit_steps(int causal, int u, int len, int &nA, int &nB) {
  const int r0 = UNIT_ROWS * u;
  const int kt = (len + BN - 1) / BN;
  nA = r0 < len ? (causal ? min(kt, 2 * u + 1) : kt) : 0;
  nB = r0 + BM < len ? (causal ? min(kt, 2 * u + 2) : kt) : 0;
}

__device__ __forceinline__ bool read_unit(const Ctl2 &c, int k, UnitInfo &t,
                                          volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns) {
  const int e = k % INFO_SLOTS;
  if (!wait_bounded(c.bar(T_INFO_FULL0 + e), (uint32_t)(k / INFO_SLOTS) & 1u, abort_flag,
                    timeout_ns))
    return false;
  const volatile int *src = c.info + e * UNIT_INTS;
  t.valid = src[0];
  t.seq_start = src[1];
  t.len = src[2];
  t.unit = src[3];
  t.h = src[4];
  t.n[0] = src[5];
  t.n[1] = src[6];
  t.lse_base = (long long)(unsigned)src[7] | ((long long)src[8] << 32);
  return true;
}

// p = 2^(h c - m c) for the row's 128 scores (two halves) into pk0, pk1
// (bf16 pairs); returns the sum of the fp32 values.
__device__ __forceinline__ float exp_row(const float (&h0)[HB], const float (&h1)[HB], float c,
                                         float m, uint32_t (&pk0)[HB / 2],
                                         uint32_t (&pk1)[HB / 2]) {
  const uint64_t c2 = f2_pack(c, c);
  const float nmc = (m == -INFINITY) ? 0.f : -m * c;
  const uint64_t nm2 = f2_pack(nmc, nmc);
  uint64_t acc[4] = {0, 0, 0, 0}, unused[4] = {0, 0, 0, 0};
  exp_half<false>(h0, c2, nm2, pk0, acc, unused);
  exp_half<false>(h1, c2, nm2, pk1, acc, unused);
  return sum_acc(acc);
}

// The row's 128 scores (TMEM columns col..col+127 of this thread's lane):
// four loads, one wait.
__device__ __forceinline__ void load_row(uint32_t taddr, float (&h0)[HB], float (&h1)[HB]) {
  uint32_t a[32], b[32], c[32], d[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_ld32(taddr + 64, c);
  tmem_ld32(taddr + 96, d);
  tmem_wait_ld();
  reg_fence32(a);
  reg_fence32(b);
  reg_fence32(c);
  reg_fence32(d);
#pragma unroll
  for (int x = 0; x < 32; ++x) {
    h0[x] = __uint_as_float(a[x]);
    h0[32 + x] = __uint_as_float(b[x]);
    h1[x] = __uint_as_float(c[x]);
    h1[32 + x] = __uint_as_float(d[x]);
  }
}

// Sum of the row's 128 bf16 weights exactly as P.V uses them.
__device__ __forceinline__ float sum_rounded(const uint32_t (&pk0)[HB / 2],
                                             const uint32_t (&pk1)[HB / 2]) {
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int x = 0; x < HB / 2; x += 2) {
    add_bf16x2_f32(a[0], a[1], pk0[x]);
    add_bf16x2_f32(a[2], a[3], pk0[x + 1]);
    add_bf16x2_f32(a[4], a[5], pk1[x]);
    add_bf16x2_f32(a[6], a[7], pk1[x + 1]);
  }
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// K/V ring slot of position ps: its full and empty barriers and the parity of
// the fill that position ps belongs to.
template <int STAGES>
__device__ __forceinline__ uint32_t ring_full(const Ctl2 &ctl, long long ps) {
  return ctl.bar(T_RING + (int)(ps % STAGES));
}
template <int STAGES>
__device__ __forceinline__ uint32_t ring_empty(const Ctl2 &ctl, long long ps) {
  return ctl.bar(T_RING + STAGES + (int)(ps % STAGES));
}
template <int STAGES>
__device__ __forceinline__ uint32_t ring_parity(long long ps) {
  return (uint32_t)(ps / STAGES) & 1u;
}

struct IssueState {
  long long npv;   // PV_X issued so far (P_FULL_X phases)
  int nunits;      // units in which tile X had work (O_FREE_X and PV_DONE_X phases)
};

// Tile X's share of key step j of a unit: PV_X(j) (O_X (+)= P_X(j) V_j; the
// unit's first overwrites O_X, after the previous epilogue has read it), then
// QK_X(j+1).  K_j sits at ring position base + 2j, V_j at base + 2j + 1.
// Executed by every lane of the MMA warp; each tcgen05 instruction is issued
// by one elected lane.  One tcgen05.mma costs the issuing warp about 45
// cycles against the 64 the tensor core takes to run it at N = 128, and the
// warp runs only a few instructions ahead of the tensor core, so whatever it
// does between batches beyond ~16 cycles per MMA leaves the tensor core
// idle.  The warp therefore waits only for P_X(j) (the watcher's arrival in
// P_FULL_X(j) says that V_j and K_{j+1} have landed), and its commits are
// S_FULL_X after QK_X(j+1), the release of each ring slot after its last
// reader, and PV_DONE_X after the tile's last PV (for the epilogue).
// Descriptor offsets are plain integer additions (the address field cannot
// carry: shared addresses stay below 256 KB).
template <int D, int X>
__device__ __forceinline__ bool tile_step(const Ctl2 &ctl, volatile uint32_t *abort_flag,
                                          unsigned long long timeout_ns, uint32_t tmem,
                                          uint64_t kdesc0, uint64_t vdesc0, uint64_t qdesc,
                                          int v_slot, int k_slot, int j, int nA, int nB,
                                          IssueState &st, volatile unsigned *trb) {
  using C = Cfg2<D>;
  constexpr uint32_t IDESC_PV = idesc_bf16_f32(D, 1);
  (void)trb;
  const int nx = X ? nB : nA;
  if (j >= nx) return true;
  const bool has_qk = j + 1 < nx;
  const bool last_user = X == 1 || j >= nB;   // B's MMAs come last in a step
  if (j == 0 && st.nunits > 0 &&
      !wait_warp(ctl.bar(T_O_FREE0 + X), (uint32_t)(st.nunits - 1) & 1u, abort_flag, timeout_ns))
    return false;
  ATTN_TRACE_SM(trb, st.npv, 6 + X);
  if (!wait_warp(ctl.bar(T_P_FULL0 + X), (uint32_t)st.npv & 1u, abort_flag, timeout_ns))
    return false;
  ATTN_TRACE_SM(trb, st.npv, 3 * X);
  tc_fence_after();
  const uint64_t vdesc = vdesc0 + (((uint32_t)v_slot * C::TILE_BYTES) >> 4);
  const uint32_t s_x = tmem + 128u * X;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    mma_ts_warp(tmem + C::COL_O + (uint32_t)(D * X), s_x + kk * 8, vdesc + (kk * 2048 >> 4),
                IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
  if (!has_qk) tc_commit_warp(ctl.bar(T_PV_DONE0 + X));   // the tile's last PV: O_X is final
  if (last_user) tc_commit_warp(ctl.bar(T_RING + C::STAGES + v_slot));   // V_j's last use
  ATTN_TRACE_SM(trb, st.npv, 3 * X + 1);
  ++st.npv;
  if (has_qk) {   // QK_X(j+1)
    issue_qk_warp<D>(s_x, qdesc, kdesc0 + (((uint32_t)k_slot * C::TILE_BYTES) >> 4));
    tc_commit_warp(ctl.bar(T_S_FULL0 + X));
    if (last_user) tc_commit_warp(ctl.bar(T_RING + C::STAGES + k_slot));   // K_{j+1}'s last use
    ATTN_TRACE_SM(trb, st.npv, 3 * X + 2);
  }
  return true;
}

// ================================================================ kernel
template <int D>
__global__ void __launch_bounds__(THREADS2, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg2<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base_s = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_CTL);
  Ctl2 ctl;
  ctl.bar0 = smem_u32(bars);
  ctl.words = reinterpret_cast<uint32_t *>(bars + T_RING + 2 * C::STAGES);
  ctl.info = reinterpret_cast<int *>(ctl.words + 4);
  static_assert((T_RING + 2 * C::STAGES) * 8 + 16 + INFO_SLOTS * UNIT_INTS * 4 <= 512 &&
                    512 + 16 * 8 * 4 <= C::CTL_BYTES,
                "control block (the last 512 bytes hold trace stamps in trace builds)");
  volatile uint32_t *abort_flag = ctl.words + 1;
  const uint32_t q_s = base_s + C::OFF_Q;
  const uint32_t kv_s = base_s + C::OFF_KV;
  constexpr uint32_t INFO_CONSUMERS = 1 + 8 + 1;   // the MMA issuer, the softmax warps, the watcher
  const int tslot = ATTN_TRACE_SLOT();          // -1 unless built for tracing

  // The producer sets up the barriers and sends its first unit's loads before
  // the set-up barrier, so that their DRAM latency overlaps the TMEM
  // allocation and the barrier (in a short launch after the L2 was flushed,
  // the parameters, tensor maps and inputs all come from DRAM).
  int primed = 0;           // producer lane 0: ring items of its first unit already issued
  bool q_primed = false;    // producer lane 0: the first unit's Q already issued
  if (warp == WARP_PROD) {
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      for (int b = 0; b < 2; ++b) {
        mbar_init(ctl.bar(T_Q_FULL0 + b), 1);
        mbar_init(ctl.bar(T_Q_EMPTY0 + b), 1);
        mbar_init(ctl.bar(T_S_FULL0 + b), 1);
        mbar_init(ctl.bar(T_P_FULL0 + b), 4 + 1);   // the tile's softmax warps, the watcher
        mbar_init(ctl.bar(T_PV_DONE0 + b), 1);
        mbar_init(ctl.bar(T_O_FREE0 + b), 4);
      }
      for (int e = 0; e < INFO_SLOTS; ++e) {
        mbar_init(ctl.bar(T_INFO_FULL0 + e), 1);
        mbar_init(ctl.bar(T_INFO_EMPTY0 + e), INFO_CONSUMERS);
      }
      mbar_init(ctl.bar(T_DRAIN), 1);
      for (int s = 0; s < C::STAGES; ++s) {
        mbar_init(ctl.bar(T_RING + s), 1);
        mbar_init(ctl.bar(T_RING + C::STAGES + s), 1);
      }
      ctl.words[1] = 0u;
      mbar_init_fence();
    }
    __syncwarp();
    const Tile t = decode_tile(p, blockIdx.x, false);   // the first unit (round 0)
    if (t.valid && lane == 0) {
      int nA = 0, nB = 0;
      unit_steps(p.causal, t.unit, t.len, nA, nB);
      const int kvh = t.h / p.group;
      const int row0 = t.seq_start + UNIT_ROWS * t.unit;
      const int tiles = nB > 0 ? 2 : 1;
      mbar_arrive_expect_tx(ctl.bar(T_Q_FULL0), C::TILE_BYTES * tiles);
      for (int x = 0; x < tiles; ++x)
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(q_s + x * C::TILE_BYTES + c * CHUNK_BYTES, &tm_q, ctl.bar(T_Q_FULL0), c * 64,
                      t.h, row0 + BM * x);
      q_primed = true;
      primed = min(2 * max(nA, nB), C::STAGES);   // ring slots start empty
      for (int item = 0; item < primed; ++item) {
        mbar_arrive_expect_tx(ctl.bar(T_RING + item), C::TILE_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(kv_s + item * C::TILE_BYTES + c * CHUNK_BYTES, (item & 1) ? &tm_v : &tm_k,
                      ctl.bar(T_RING + item), c * 64, kvh, t.seq_start + (item >> 1) * BN);
      }
    }
  } else if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(ctl.words), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.words[0];

  if (warp < SM_WARP0 || warp >= SM_WARP0 + 8) {
   setmaxnreg_dec<REGS_OTHER>();
   if (warp == WARP_PROD) {
    // ---------------- producer: decode units, publish them, load Q and K/V
    long long pos = primed;        // global ring position (the primed items are issued)
    int q_loads = q_primed ? 1 : 0;
    bool ok = true;
    long long round = 0;
    for (int k = 0; ok; ++k) {
      // round r covers units [r G, (r+1) G), odd rounds backwards (longest
      // units first overall, so each CTA's total evens out)
      const long long G = gridDim.x;
      const Tile t =
          decode_tile(p, round * G + ((round & 1) ? G - 1 - blockIdx.x : blockIdx.x), false);
      ++round;
      int nA = 0, nB = 0;
      if (t.valid) unit_steps(p.causal, t.unit, t.len, nA, nB);
      if (lane == 0) {
        const int e = k % INFO_SLOTS;
        ok = wait_bounded(ctl.bar(T_INFO_EMPTY0 + e), ((uint32_t)(k / INFO_SLOTS) & 1u) ^ 1u,
                          abort_flag, p.timeout_ns);
        if (ok) {
          int *dst = ctl.info + e * UNIT_INTS;
          dst[0] = t.valid;
          dst[1] = t.seq_start;
          dst[2] = t.len;
          dst[3] = t.unit;
          dst[4] = t.h;
          dst[5] = nA;
          dst[6] = nB;
          dst[7] = (int)(unsigned)(t.lse_base & 0xFFFFFFFFll);
          dst[8] = (int)(t.lse_base >> 32);
          mbar_arrive(ctl.bar(T_INFO_FULL0 + e));   // release: the entry is visible
        }
        if (ok && t.valid) {
          const int qb = k % C::QB;
          const int kvh = t.h / p.group;
          const int row0 = t.seq_start + UNIT_ROWS * t.unit;
          if (k >= C::QB)
            ok = wait_bounded(ctl.bar(T_Q_EMPTY0 + qb), (uint32_t)(k / C::QB - 1) & 1u,
                              abort_flag, p.timeout_ns);
          if (ok && !(k == 0 && q_primed)) {
            const int tiles = nB > 0 ? 2 : 1;
            ++q_loads;
            mbar_arrive_expect_tx(ctl.bar(T_Q_FULL0 + qb), C::TILE_BYTES * tiles);
            for (int x = 0; x < tiles; ++x)
              for (int c = 0; c < C::CHUNKS; ++c)
                tma_load_3d(q_s + (2 * qb + x) * C::TILE_BYTES + c * CHUNK_BYTES, &tm_q,
                            ctl.bar(T_Q_FULL0 + qb), c * 64, t.h, row0 + BM * x);
          }
          // K_0, V_0, K_1, V_1, ...
          const int n = max(nA, nB);
          for (int item = k == 0 ? primed : 0; ok && item < 2 * n; ++item, ++pos) {
            const int slot = (int)(pos % C::STAGES);
            if (!(ok = wait_bounded(ctl.bar(T_RING + C::STAGES + slot),
                                    ((uint32_t)(pos / C::STAGES) & 1u) ^ 1u, abort_flag,
                                    p.timeout_ns)))
              break;
            mbar_arrive_expect_tx(ctl.bar(T_RING + slot), C::TILE_BYTES);
            const uint32_t dst = kv_s + slot * C::TILE_BYTES;
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_3d(dst + c * CHUNK_BYTES, (item & 1) ? &tm_v : &tm_k,
                          ctl.bar(T_RING + slot), c * 64, kvh, t.seq_start + (item >> 1) * BN);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && t.valid;
    }
    if (lane == 0 && *abort_flag) {
      // drain: wait (bounded) for the copies this thread issued
      for (int b = 0; b < C::QB && b < q_loads; ++b) {
        const int last = b + C::QB * ((q_loads - 1 - b) / C::QB);
        wait_drain(ctl.bar(T_Q_FULL0 + b), (uint32_t)(last / C::QB) & 1u, p.timeout_ns);
      }
      for (int s = 0; s < C::STAGES && s < pos; ++s) {
        const long long last = s + C::STAGES * ((pos - 1 - s) / C::STAGES);
        wait_drain(ctl.bar(T_RING + s), (uint32_t)(last / C::STAGES) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
   } else if (warp == WARP_MMA) {
    // ---------------- MMA issuer (the whole warp; one elected lane issues)
    {
      const uint64_t kdesc0 = smem_desc_sw128(kv_s, 16, 1024);
      const uint64_t vdesc0 = smem_desc_sw128(kv_s, CHUNK_BYTES, 1024);
      // trace builds: issuer stamps in the spare end of the control block
      volatile unsigned *trb = reinterpret_cast<volatile unsigned *>(smem + C::OFF_CTL + 512);
      (void)trb;
      long long base = 0;            // ring position of the unit's first load (K_0)
      IssueState st0{0, 0}, st1{0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        UnitInfo t;
        if (!(ok = __all_sync(0xffffffffu, read_unit(ctl, k, t, abort_flag, p.timeout_ns))))
          break;
        __syncwarp();
        if (lane == 0) mbar_arrive(ctl.bar(T_INFO_EMPTY0 + k % INFO_SLOTS));
        if (!t.valid) break;
        const int qb = k % C::QB;
        if (!(ok = wait_warp(ctl.bar(T_Q_FULL0 + qb), (uint32_t)(k / C::QB) & 1u, abort_flag,
                             p.timeout_ns)))
          break;
        const uint64_t qd0 = smem_desc_sw128(q_s + 2 * qb * C::TILE_BYTES, 16, 1024);
        const uint64_t qd1 = smem_desc_sw128(q_s + (2 * qb + 1) * C::TILE_BYTES, 16, 1024);
        const int nA = t.n[0], nB = t.n[1];
        const int n = max(nA, nB);
        if (!(ok = wait_warp(ring_full<C::STAGES>(ctl, base), ring_parity<C::STAGES>(base),
                             abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        const uint64_t kd = kdesc0 + (((uint32_t)(base % C::STAGES) * C::TILE_BYTES) >> 4);
        if (nA > 0) {
          issue_qk_warp<D>(tmem, qd0, kd);
          tc_commit_warp(ctl.bar(T_S_FULL0));
        }
        if (nB > 0) {
          issue_qk_warp<D>(tmem + 128u, qd1, kd);
          tc_commit_warp(ctl.bar(T_S_FULL1));
        }
        tc_commit_warp(ring_empty<C::STAGES>(ctl, base));   // K_0 read by both prologue QKs
        // The Q buffer is free once the unit's last QK has run (the prologue's
        // when it has one step, else those of step n - 2).
        if (n == 1) tc_commit_warp(ctl.bar(T_Q_EMPTY0 + qb));
        // ring slots of V_j and K_{j+1} (positions base + 2j + 1, + 2), kept
        // as 32-bit counters rather than recomputed from 64-bit positions
        int v_slot = (int)((base + 1) % C::STAGES);
        for (int j = 0; ok && j < n; ++j) {
          const int k_slot = v_slot + 1 == C::STAGES ? 0 : v_slot + 1;
          ok = tile_step<D, 0>(ctl, abort_flag, p.timeout_ns, tmem, kdesc0, vdesc0, qd0, v_slot,
                               k_slot, j, nA, nB, st0, trb) &&
               tile_step<D, 1>(ctl, abort_flag, p.timeout_ns, tmem, kdesc0, vdesc0, qd1, v_slot,
                               k_slot, j, nA, nB, st1, trb);
          if (ok && j == n - 2) tc_commit_warp(ctl.bar(T_Q_EMPTY0 + qb));
          v_slot = k_slot + 1 == C::STAGES ? 0 : k_slot + 1;
        }
        if (!ok) break;
        if (nA > 0) ++st0.nunits;
        if (nB > 0) ++st1.nunits;
        base += 2 * n;
      }
      tc_commit_warp(ctl.bar(T_DRAIN));   // no MMA may be in flight at teardown
      wait_drain(ctl.bar(T_DRAIN), 0, p.timeout_ns);
      if (lane == 0) ATTN_TRACE_SM_FLUSH(trb, 0);
    }
    __syncwarp();
   } else if (warp == WARP_WATCH) {
    // ---------------- K/V watcher (one thread): adds one arrival to P_FULL_X(j)
    // once V_j and, if tile X computes S(j+1), K_{j+1} have landed, so that
    // the MMA issuer waits for P_FULL alone.  It arrives for step j only after
    // the phase of step j - 1 has completed, so that an early arrival never
    // counts towards the previous phase.
    if (lane == 0) {
      // ring position of the next load as (slot, fill parity), advanced one
      // position at a time
      int slot = 0;
      uint32_t par = 0;
      const auto advance = [&]() {
        if (++slot == C::STAGES) {
          slot = 0;
          par ^= 1u;
        }
      };
      uint32_t gx[2] = {0, 0};   // P_FULL_X phases arrived at so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        UnitInfo t;
        if (!(ok = read_unit(ctl, k, t, abort_flag, p.timeout_ns))) break;
        mbar_arrive(ctl.bar(T_INFO_EMPTY0 + k % INFO_SLOTS));
        if (!t.valid) break;
        const int n = max(t.n[0], t.n[1]);
        advance();   // K_0
        for (int j = 0; ok && j < n; ++j) {
          // V_j at (slot, par); K_{j+1} at the next position
          const int v_slot = slot, k_slot = slot + 1 == C::STAGES ? 0 : slot + 1;
          const uint32_t v_par = par, k_par = k_slot == 0 ? par ^ 1u : par;
          ok = wait_bounded(ctl.bar(T_RING + v_slot), v_par, abort_flag, p.timeout_ns);
          for (int x = 0; ok && x < 2; ++x) {
            if (j >= t.n[x]) continue;
            if (j + 1 < t.n[x])
              ok = wait_bounded(ctl.bar(T_RING + k_slot), k_par, abort_flag, p.timeout_ns);
            if (ok && gx[x] > 0)
              ok = wait_bounded(ctl.bar(T_P_FULL0 + x), (gx[x] - 1u) & 1u, abort_flag,
                                p.timeout_ns);
            if (ok) {
              mbar_arrive(ctl.bar(T_P_FULL0 + x));
              ++gx[x];
            }
          }
          advance();   // V_j
          if (j + 1 < n) advance();   // K_{j+1}
        }
      }
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<REGS_SOFTMAX>();
    // ---------------- softmax warps: tile x = warp / 4, lane quarter warp % 4
    const int x = (warp - SM_WARP0) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t s_t = tmem + lane_off + 128u * (uint32_t)x;
    const uint32_t o_t = tmem + lane_off + C::COL_O + (uint32_t)(D * x);
    const float c = p.scale_log2;
    long long g = 0;   // key steps of tile x so far (S_FULL and P_FULL phases)
    int units_x = 0;   // units in which tile x had work (PV_DONE phases)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      UnitInfo t;
      ok = __all_sync(0xffffffffu, read_unit(ctl, k, t, abort_flag, p.timeout_ns));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(ctl.bar(T_INFO_EMPTY0 + k % INFO_SLOTS));
      if (!t.valid) break;
      const int nx = x ? t.n[1] : t.n[0];
      if (nx == 0) continue;
      const int r0 = UNIT_ROWS * t.unit + BM * x;   // the tile's first row
      const int q_idx = r0 + row;
      const int lim = p.causal ? min(t.len, q_idx + 1) : t.len;   // visible keys [0, lim)
      // reference max (raw score units); row sums of the fp32 weights (for the
      // LSE) and of the bf16-rounded ones (for O)
      float m = -INFINITY, l = 0.f, lr = 0.f;
      bool s_ready = false;   // early test of this step's S
      for (int j = 0; j < nx; ++j, ++g) {
        if (!__all_sync(0xffffffffu, s_ready) &&
            !(ok = wait_warp(ctl.bar(T_S_FULL0 + x), (uint32_t)g & 1u, abort_flag,
                             p.timeout_ns)))
          break;
        unsigned tr_s = 0, tr_e = 0, tr_w = 0;   // trace stamps, stored after the arrival
        ATTN_TRACE_CLK(tr_s);
        tc_fence_after();
        const int kb = j * BN;
        const bool masked = kb + BN > t.len || (p.causal && kb + BN - 1 > r0);
        float h0[HB], h1[HB];
        load_row(s_t, h0, h1);
        if (masked) {
          mask_half(h0, kb, 0, lim);
          mask_half(h1, kb + HB, 0, lim);
        }
        uint32_t pk0[HB / 2], pk1[HB / 2];
        float alpha = 1.f, sum;
        bool moved = false;
        // A row without a reference yet (its first visible keys) takes the
        // tile's maximum first; the others exponentiate against their
        // reference, and only if some row's sum leaves range do the scores
        // come again (S_x is intact until P is stored) for a second pass with
        // the maximum.  One copy of the exponential loop serves both passes.
        bool want = m == -INFINITY, again = false;
        for (;;) {
          if (want) {
            const float m_new = fmaxf(m, fmaxf(max_half(h0), max_half(h1)));
            if (m_new != m) {
              alpha = (m == -INFINITY) ? 0.f : ex2_approx((m - m_new) * c);
              m = m_new;
              l *= alpha;
              lr *= alpha;
              moved = true;
            }
          }
          sum = exp_row(h0, h1, c, m, pk0, pk1);
          const bool need = !(sum <= P_SUM_LIMIT);
          if (again || !__any_sync(0xffffffffu, need)) break;
          again = true;
          want = need;
          load_row(s_t, h0, h1);
          if (masked) {
            mask_half(h0, kb, 0, lim);
            mask_half(h1, kb + HB, 0, lim);
          }
        }
        ATTN_TRACE_CLK(tr_e);
        // O_x holds P_x(j-1) V_{j-1} (the commit of S_x(j) covers that PV)
        if (j > 0 && __any_sync(0xffffffffu, moved)) rescale_o<D>(o_t, alpha);
        tmem_st32(s_t, pk0);
        tmem_st32(s_t + HB / 2, pk1);
        l += sum;
        s_ready = j + 1 < nx && mbar_test_wait(ctl.bar(T_S_FULL0 + x), (uint32_t)(g + 1) & 1u);
        tmem_wait_st();
        ATTN_TRACE_CLK(tr_w);
        tc_fence_before();
        warp_arrive(ctl.bar(T_P_FULL0 + x));
        // the rounded sum, off the path to P: the warp would wait for S now
        lr += sum_rounded(pk0, pk1);
        if (lane == 0) {
          ATTN_TRACE_EV(2 + warp - SM_WARP0, g, 2);
          ATTN_TRACE_PUT(2 + warp - SM_WARP0, g, 0, tr_s);
          ATTN_TRACE_PUT(2 + warp - SM_WARP0, g, 1, tr_e);
          ATTN_TRACE_PUT(2 + warp - SM_WARP0, g, 3, tr_w);
        }
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE; then O_x is free for the next unit
      ok = wait_warp(ctl.bar(T_PV_DONE0 + x), (uint32_t)units_x & 1u, abort_flag, p.timeout_ns);
      if (!ok) break;
      ++units_x;
      tc_fence_after();
      const bool live = q_idx < t.len;
      const float m_use = (m == -INFINITY) ? 0.f : m;
      store_cols<D>(o_t, lr > 0.f ? 1.f / lr : 0.f,
                    p.o + ((long long)(t.seq_start + q_idx) * p.Hq + t.h) * (long long)D, live);
      if (live) p.lse[t.lse_base + q_idx] = l > 0.f ? m_use * p.scale + logf(l) : -INFINITY;
      tc_fence_before();
      warp_arrive(ctl.bar(T_O_FREE0 + x));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace two
}  // namespace attn
