// attn_bwd_fused.cuh -- single-pass attention backward, head dim 64
// (included from attn_bwd.cuh, whose parameters, unit order, row pass and
// helpers it shares).
//
// One CTA per (kv head, 128-key block), as in the dK/dV kernel, walking the
// query blocks of every query head of the group.  Per step it forms the same
// S^T, dP^T, dV += P^T dO and dK += dS^T Q, and also the key block's share
// of the query gradient, dS K, which is added into an fp32 buffer with bulk
// tensor reduce-adds (tang, section 8.3 "Attention backward on Hopper": one
// kernel per key block, dK and dV held on chip, dQ added by bulk
// asynchronous reductions).  That is five 128 x 128 x 64 products per (key
// block, query block) pair where the two-kernel path, which recomputes S and
// dP in its dQ kernel, takes seven, and the exponentials of P are taken once
// instead of twice.  The row pass zeroes the buffer; a last pass scales it
// into bf16 dq.  The reduce-adds land in whatever order the key blocks reach
// them, so dq's fp32 rounding (not its value within the tolerance) varies
// from run to run.
//
// Tensor memory: S^T [0,128) (P^T bf16 over the first 16 of each 32
// columns), dP^T [128,256), dV [256,320), dK [320,384), the dQ share
// [384,448), dS^T in bf16 [448,512) (the A operand of dK).  The dQ product
// takes dS from shared memory: the softmax warps also write their dS^T rows
// there (one 128-byte swizzled line per key, the query index contiguous: an
// M-major A operand), and K serves both as the K-major A of S^T and as the
// N-major B of dS K.

namespace attn {
namespace bwd {

// producer, MMA issuer, 16 softmax warps (four per TMEM lane quarter, one per
// 32 of the 128 columns of a score tile: four warps per sub-partition hide
// one another's TMEM and shared-memory latencies), and four dQ warps (one
// per lane quarter) that move the dQ share out, off the softmax warps' path
constexpr int F_SM_WARPS = 16, F_DQ_WARPS = 4;
constexpr int F_THREADS = 64 + 32 * (F_SM_WARPS + F_DQ_WARPS);

struct FCfg {
  static constexpr int D = 64;
  // ring slots: a step's Q and dO take about a step to arrive, so they are
  // requested two steps ahead
  static constexpr int STAGES = 3;
  static constexpr uint32_t TILE = CHUNK_BYTES;                  // 128 x 64 bf16
  static constexpr uint32_t SLOT = 2 * TILE + 1024;              // Q, dO, lse2 row, dsum row
  static constexpr uint32_t OFF_RING = 2 * TILE;                 // after K, V
  static constexpr uint32_t OFF_DS = OFF_RING + STAGES * SLOT;   // dS, 128 queries x 128 keys
  static constexpr uint32_t OFF_STG = OFF_DS + 2 * TILE;         // 4 dQ warps x 32 rows x 64 fp32
  static constexpr uint32_t STG_WARP = 32 * 256;                 // four boxes of 16 columns
  static constexpr uint32_t OFF_CTL = OFF_STG + F_DQ_WARPS * STG_WARP;
  static constexpr uint32_t CTL_BYTES = 256;
  static constexpr uint32_t SMEM = OFF_CTL + CTL_BYTES + 1024;
  static_assert(OFF_DS % 1024 == 0 && OFF_STG % 1024 == 0, "swizzle atoms");
  static_assert(SMEM >= BCfg<64>::MIN_SMEM && SMEM <= 232448, "shared memory");
};

enum : int {
  F_STATIC = 0,   // K, V loaded
  F_FULL0,        // ring slot s loaded, s < 3
  F_EMPTY0 = F_FULL0 + FCfg::STAGES,   // ring slot s consumed
  F_DONE = F_EMPTY0 + FCfg::STAGES,    // dK, dV final
  F_DRAIN,        // abort drain of the MMA issuer
  F_ST,           // S^T of the step in TMEM
  F_DPT,          // dP^T of the step in TMEM
  F_PT,           // softmax warps: P^T written
  F_DST,          // softmax warps: dS^T written (TMEM and shared memory)
  F_DQ,           // the step's dQ share in TMEM
  F_DQ_READ,      // dQ warps: the share loaded (its columns are free)
  F_COUNT
};
static_assert(8 * F_COUNT + 8 <= (int)FCfg::CTL_BYTES, "control block");

// Bulk tensor reduce-add of a shared-memory box into global memory (the
// element type and the add come from the tensor map: fp32), tracked by this
// thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, int c0, int c1,
                                                  uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2}], [%3];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's earlier bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... and their writes to global memory are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// A (K = 128 queries, bf16 pairs in TMEM) times B (N-major shared-memory
// tile, 64 columns), accumulated into d_tmem (overwritten unless
// accumulate).  Each softmax warp packs its 32 query columns into the first
// 16 of the 32 TMEM columns it read itself (so no warp writes columns that
// another still reads): queries 16 kk .. 16 kk + 15 sit at columns
// 32 (kk / 2) + 8 (kk % 2).
__device__ __forceinline__ void issue_pv_quarters_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                       uint64_t bdesc, bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(64, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(d_tmem, a_tmem + 32u * (uint32_t)(kk >> 1) + 8u * (uint32_t)(kk & 1),
                bdesc + (uint64_t)((kk * 2048) >> 4), IDESC, (accumulate || kk > 0) ? 1u : 0u);
}

// dK += dS^T Q: A = dS^T in TMEM (bf16 pairs, queries 16 kk .. 16 kk + 15 at
// column 8 kk), B = Q (queries x head dim, N-major, 16 queries = 2048 bytes
// per step).  (A read from the shared dS tile instead, an N = 64 product
// that fetches 6 KB of operands per 32-cycle MMA, was measured slower.)
__device__ __forceinline__ void issue_dk_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t q_mn,
                                              bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(64, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(d_tmem, a_tmem + 8u * (uint32_t)kk, q_mn + (uint64_t)((kk * 2048) >> 4), IDESC,
                (accumulate || kk > 0) ? 1u : 0u);
}

// Instruction descriptor for dS K: A (dS) and B (K) both stored with the
// M / N index contiguous.
constexpr uint32_t IDESC_DQ = idesc_bf16_f32(64, 1) | (1u << 15);

// A dQ warp's part of the share: rows 32 wq .. 32 wq + 31 of the query block,
// all 64 columns, loaded from TMEM (then released on F_DQ_READ), written to
// the warp's staging area as four boxes of 16 columns (64-byte swizzle: one
// 64-byte line per row, its 16-byte pieces permuted by bits 1-2 of the row)
// and reduce-added into the buffer at buffer row c1.  Lane 0 first waits
// until the warp's previous reduce-adds have read the area.
__device__ __forceinline__ void dq_share_out(uint32_t taddr, uint32_t stg, uint32_t read_bar,
                                             const CUtensorMap *map, int c1) {
  const int lane = threadIdx.x & 31;
  uint32_t u0[32], u1[32];
  tmem_ld32(taddr, u0);
  tmem_ld32(taddr + 32, u1);
  tmem_wait_ld();
  reg_fence32(u0);
  reg_fence32(u1);
  tc_fence_before();
  warp_arrive(read_bar);
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const uint32_t line = stg + (uint32_t)lane * 64u;
  const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    st_shared_v4(line + ((j ^ sw) << 4),
                 make_uint4(u0[4 * j], u0[4 * j + 1], u0[4 * j + 2], u0[4 * j + 3]));
    st_shared_v4(line + 2048 + ((j ^ sw) << 4),
                 make_uint4(u0[16 + 4 * j], u0[17 + 4 * j], u0[18 + 4 * j], u0[19 + 4 * j]));
    st_shared_v4(line + 4096 + ((j ^ sw) << 4),
                 make_uint4(u1[4 * j], u1[4 * j + 1], u1[4 * j + 2], u1[4 * j + 3]));
    st_shared_v4(line + 6144 + ((j ^ sw) << 4),
                 make_uint4(u1[16 + 4 * j], u1[17 + 4 * j], u1[18 + 4 * j], u1[19 + 4 * j]));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) tma_reduce_add_2d(map, 16 * q, c1, stg + 2048u * q);
    bulk_commit_group();
  }
}

__global__ void __launch_bounds__(F_THREADS, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_dqacc, const BwdParams p) {
  using C = FCfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = base + C::OFF_CTL;
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *words = reinterpret_cast<uint32_t *>(smem + C::OFF_CTL + 8 * F_COUNT);
  volatile uint32_t *abort_flag = words + 1;

  const BUnit un = bwd_unit(p, blockIdx.x, p.Hkv, false);
  if (!un.valid) return;   // uniform over the CTA, before any set-up
  const int jb = un.blk, kvh = un.head, b = un.seq;
  const int nblk = un.nblk, row0 = un.start, len = un.len;
  const int i0 = p.causal ? jb : 0;
  const int nq = nblk - i0;   // query blocks per head
  const int steps = p.group * nq;
  const uint32_t k_s = base, v_s = base + C::TILE, ds_s = base + C::OFF_DS;

  if (warp == 1) {
    if (lane == 0) {
      mbar_init(bar(F_STATIC), 1);
      for (int s = 0; s < C::STAGES; ++s) {
        mbar_init(bar(F_FULL0 + s), 1);
        mbar_init(bar(F_EMPTY0 + s), 1);
      }
      mbar_init(bar(F_DONE), 1);
      mbar_init(bar(F_DRAIN), 1);
      mbar_init(bar(F_ST), 1);
      mbar_init(bar(F_DPT), 1);
      mbar_init(bar(F_PT), F_SM_WARPS);
      mbar_init(bar(F_DST), F_SM_WARPS);
      mbar_init(bar(F_DQ), 1);
      mbar_init(bar(F_DQ_READ), F_DQ_WARPS);
      words[1] = 0u;
      mbar_init_fence();
    }
    __syncwarp();
    tmem_alloc(smem_u32(words), TMEM_COLS);
    tmem_relinquish();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_do);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    tma_prefetch_map(&tm_dqacc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = words[0];
  constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 320, COL_DQ = 384,
                     COL_DS = 448;

  if (warp == 0) {
    // producer: K, V once, then Q(s), dO(s) and the two rows of each step
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(F_STATIC), 2 * C::TILE);
      tma_load_3d(k_s, &tm_k, bar(F_STATIC), 0, kvh, row0 + jb * BM);
      tma_load_3d(v_s, &tm_v, bar(F_STATIC), 0, kvh, row0 + jb * BM);
      for (int s = 0; ok && s < steps; ++s) {
        const int slot = s % C::STAGES;
        if (s >= C::STAGES &&
            !(ok = wait_bounded(bar(F_EMPTY0 + slot), (uint32_t)(s / C::STAGES - 1) & 1u,
                                abort_flag, p.timeout_ns)))
          break;
        const int h = kvh * p.group + s / nq;
        const int ib = i0 + s % nq;
        const uint32_t dst = base + C::OFF_RING + slot * C::SLOT;
        mbar_arrive_expect_tx(bar(F_FULL0 + slot), 2 * C::TILE + 1024);
        tma_load_3d(dst, &tm_q, bar(F_FULL0 + slot), 0, h, row0 + ib * BM);
        tma_load_3d(dst + C::TILE, &tm_do, bar(F_FULL0 + slot), 0, h, row0 + ib * BM);
        const long long prow =
            (long long)h * p.rows_pad() + p.pstart[b] + (long long)ib * BM;   // 512-B aligned
        bulk_load(dst + 2 * C::TILE, p.lse2 + prow, 512, bar(F_FULL0 + slot));
        bulk_load(dst + 2 * C::TILE + 512, p.dsum + prow, 512, bar(F_FULL0 + slot));
        ++issued;
      }
      if (*abort_flag) {   // drain: bounded waits for the copies issued
        wait_drain(bar(F_STATIC), 0, p.timeout_ns);
        for (int s = 0; s < C::STAGES && s < issued; ++s) {
          const int last = s + C::STAGES * ((issued - 1 - s) / C::STAGES);
          wait_drain(bar(F_FULL0 + s), (uint32_t)(last / C::STAGES) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer (whole warp, one elected lane issues).  Per step s: dV +=
    // P^T(s) dO(s) once P^T is written; S^T(s+1) (its columns are free once
    // dV(s) has read P^T: one thread's MMAs run in issue order); then, once
    // dS(s) is written, dK += dS^T(s) Q(s), the dQ share dS(s) K, and
    // dP^T(s+1).  dQ(s) overwrites the share once the dQ warps have loaded
    // the previous one; the softmax warps rewrite dS^T (TMEM) and the dS tile
    // only after dP^T(s+1), which follows dQ(s), has completed.  (Issuing
    // dP^T(s+1) before dK(s) and dQ(s), as soon as dP^T(s) is loaded, was
    // measured slower.)
    const uint64_t kdesc = smem_desc_sw128(k_s, 16, 1024);
    const uint64_t vdesc = smem_desc_sw128(v_s, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(k_s, CHUNK_BYTES, 1024);
    const uint64_t ds_mn = smem_desc_sw128(ds_s, CHUNK_BYTES, 1024);
    const uint32_t ring = base + C::OFF_RING;
    bool ok = wait_warp(bar(F_STATIC), 0, abort_flag, p.timeout_ns);
    if (ok && steps > 0 && (ok = wait_warp(bar(F_FULL0), 0, abort_flag, p.timeout_ns))) {
      tc_fence_after();
      issue_qk_warp<D>(tmem + COL_ST, kdesc, smem_desc_sw128(ring, 16, 1024));
      tc_commit_warp(bar(F_ST));
      issue_qk_warp<D>(tmem + COL_DPT, vdesc, smem_desc_sw128(ring + C::TILE, 16, 1024));
      tc_commit_warp(bar(F_DPT));
    }
    for (int s = 0; ok && s < steps; ++s) {
      const int slot = s % C::STAGES, nslot = (s + 1) % C::STAGES;
      const uint32_t q_s = ring + slot * C::SLOT;
      const uint32_t q_n = ring + nslot * C::SLOT;
      const uint64_t do_mn = smem_desc_sw128(q_s + C::TILE, CHUNK_BYTES, 1024);
      const uint64_t q_mn = smem_desc_sw128(q_s, CHUNK_BYTES, 1024);
      if (!(ok = wait_warp(bar(F_PT), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_pv_quarters_warp(tmem + COL_DV, tmem + COL_ST, do_mn, s > 0);
      const bool more = s + 1 < steps;
      if (more) {
        if (!(ok = wait_warp(bar(F_FULL0 + nslot), (uint32_t)((s + 1) / C::STAGES) & 1u,
                             abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        issue_qk_warp<D>(tmem + COL_ST, kdesc, smem_desc_sw128(q_n, 16, 1024));
        tc_commit_warp(bar(F_ST));
      }
      if (!(ok = wait_warp(bar(F_DST), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_dk_warp(tmem + COL_DK, tmem + COL_DS, q_mn, s > 0);
      tc_commit_warp(bar(F_EMPTY0 + slot));   // Q(s), dO(s) and their rows are read
      if (s > 0 && !(ok = wait_warp(bar(F_DQ_READ), (uint32_t)(s - 1) & 1u, abort_flag,
                                    p.timeout_ns)))
        break;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)   // 16 keys per MMA: two 8-row groups of both operands
        mma_ss_warp(tmem + COL_DQ, ds_mn + (uint64_t)((kk * 2048) >> 4),
                    k_mn + (uint64_t)((kk * 2048) >> 4), IDESC_DQ, kk > 0 ? 1u : 0u);
      tc_commit_warp(bar(F_DQ));
      if (more) {
        issue_qk_warp<D>(tmem + COL_DPT, vdesc, smem_desc_sw128(q_n + C::TILE, 16, 1024));
        tc_commit_warp(bar(F_DPT));
      }
    }
    if (ok) tc_commit_warp(bar(F_DONE));
    tc_commit_warp(bar(F_DRAIN));
    wait_drain(bar(F_DRAIN), 0, p.timeout_ns);
    __syncwarp();
  } else if (warp >= 2 + F_SM_WARPS) {
    // dQ warps: query rows 32 (warp%4) .. + 31 of each step's block
    const int wq = warp & 3;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t stg = base + C::OFF_STG + (uint32_t)(warp - 2 - F_SM_WARPS) * C::STG_WARP;
    const long long hrow = (long long)p.pstart[b] + 32 * wq;   // + h rows_pad + ib 128
    bool ok = true;
    for (int s = 0; ok && s < steps; ++s) {
      if (!(ok = wait_warp(bar(F_DQ), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      const int h = kvh * p.group + s / nq;
      dq_share_out(tmem + lane_off + COL_DQ, stg, bar(F_DQ_READ), &tm_dqacc,
                   (int)((long long)h * p.rows_pad() + hrow + (long long)(i0 + s % nq) * BM));
    }
    if (lane == 0) bulk_wait_all();   // the reduce-adds are done with the staging area
    __syncwarp();
  } else {
    // softmax warps: thread = key row jb*128 + row of TMEM lane quarter
    // warp%4, query columns 32 cq .. 32 cq + 31 (cq = 0..3; in the shared dS
    // tile, piece ch = cq % 2 of half hf = cq / 2)
    const int wq = warp & 3;
    const int cq = (warp - 2) >> 2;
    const int hf = cq >> 1, ch = cq & 1;
    const int c0 = 32 * cq;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t ds_line = ds_s + (uint32_t)hf * CHUNK_BYTES + (uint32_t)row * 128u;
    const float c = p.scale_log2;
    const bool kdead = key >= len;
    bool ok = true;
    for (int s = 0; ok && s < steps; ++s) {
      const int slot = s % C::STAGES;
      if (!(ok = wait_warp(bar(F_FULL0 + slot), (uint32_t)(s / C::STAGES) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(bar(F_ST), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = i0 + s % nq;
      // the step's rows, stored negated by the row pass: -LSE log2(e), -D
      const float *nlse2 =
          reinterpret_cast<const float *>(smem + C::OFF_RING + slot * C::SLOT + 2 * C::TILE);
      const float *ndsum = nlse2 + 128;
      const bool diag = p.causal && ib == jb;
      // phase 1: P^T = 2^(S^T c - LSE2), bf16, kept in registers for dS; a
      // key past the end of its sequence gets P = 0 (its dK, dV rows are not
      // stored, but its dS would enter every query's dQ)
      uint32_t pw[16];
      {
        uint32_t us[32];
        tmem_ld32(tmem + lane_off + COL_ST + c0, us);
        tmem_wait_ld();
        reg_fence32(us);
        if (!diag && !kdead) {
          const uint64_t c2 = f2_pack(c, c);
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(nlse2 + c0 + x);
            float a0, a1, a2, a3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(us[x]), __uint_as_float(us[x + 1])), c2,
                             f2_pack(l4.x, l4.y)), a0, a1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(us[x + 2]), __uint_as_float(us[x + 3])), c2,
                             f2_pack(l4.z, l4.w)), a2, a3);
            pw[x >> 1] = pack_bf16x2(ex2_approx(a0), ex2_approx(a1));
            pw[(x >> 1) + 1] = pack_bf16x2(ex2_approx(a2), ex2_approx(a3));
          }
        } else {
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            const int qc = c0 + x;
            float p0 = ex2_approx(fmaf(__uint_as_float(us[x]), c, nlse2[qc]));
            float p1 = ex2_approx(fmaf(__uint_as_float(us[x + 1]), c, nlse2[qc + 1]));
            // query ib*128 + qc sees key iff query >= key
            if (kdead || (diag && ib * BM + qc < key)) p0 = 0.f;
            if (kdead || (diag && ib * BM + qc + 1 < key)) p1 = 0.f;
            pw[x >> 1] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(tmem + lane_off + COL_ST + c0, pw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(F_PT));
      // phase 2: dS^T = P^T o (dP^T - D), bf16, into TMEM (for dK) and into
      // the shared dS tile (for dQ)
      if (!(ok = wait_warp(bar(F_DPT), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      {
        uint32_t ud[32];
        tmem_ld32(tmem + lane_off + COL_DPT + c0, ud);
        tmem_wait_ld();
        reg_fence32(ud);
        uint32_t dw[16];
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
          const float4 d4 = *reinterpret_cast<const float4 *>(ndsum + c0 + x);
          const uint32_t w0 = pw[x >> 1], w1 = pw[(x >> 1) + 1];
          float a0, a1, a2, a3;
          f2_unpack(f2_mul(bf16x2_widen(w0),
                           f2_add(f2_pack(__uint_as_float(ud[x]), __uint_as_float(ud[x + 1])),
                                  f2_pack(d4.x, d4.y))), a0, a1);
          f2_unpack(f2_mul(bf16x2_widen(w1),
                           f2_add(f2_pack(__uint_as_float(ud[x + 2]), __uint_as_float(ud[x + 3])),
                                  f2_pack(d4.z, d4.w))), a2, a3);
          dw[x >> 1] = pack_bf16x2(a0, a1);
          dw[(x >> 1) + 1] = pack_bf16x2(a2, a3);
        }
        tmem_st16(tmem + lane_off + COL_DS + 16 * cq, dw);
        // queries 32 cq .. 32 cq + 31: four 16-byte pieces of the key's
        // 128-byte line in half hf of the tile
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(ds_line + ((uint32_t)((4 * ch + j) ^ (row & 7)) << 4),
                       make_uint4(dw[4 * j], dw[4 * j + 1], dw[4 * j + 2], dw[4 * j + 3]));
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(bar(F_DST));
    }
    if (ok && (ok = wait_warp(bar(F_DONE), 0, abort_flag, p.timeout_ns))) {
      tc_fence_after();
      // column quarters 0, 1: the two halves of dV; 2, 3: those of dK
      const bool live = key < len, is_k = cq >= 2;
      const long long off = ((long long)(row0 + key) * p.Hkv + kvh) * D + ch * (D / 2);
      store_row_bf16<D / 2>(tmem + lane_off + (is_k ? COL_DK : COL_DV) + ch * (D / 2),
                            is_k ? p.scale : 1.f, (is_k ? p.dk : p.dv) + off, live);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// dq = scale x the fp32 buffer, on the rows of real tokens: eight lanes per
// (head, padded row), eight columns each.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const BwdParams p) {
  const int seg = threadIdx.x & 7;
  const long long row = (long long)blockIdx.x * 32 + (threadIdx.x >> 3);   // h rows_pad + r
  if (row >= (long long)p.Hq * p.rows_pad()) return;
  const int h = (int)(row / p.rows_pad());
  const int r = (int)(row % p.rows_pad());
  if (r >= p.pstart[p.B]) return;
  const int b = seq_of_padded_row(p, r);
  const int i = r - p.pstart[b];
  if (i >= p.seq_len(b)) return;
  const float4 *src = reinterpret_cast<const float4 *>(p.dq_acc + row * 64 + seg * 8);
  const float4 a = src[0], e = src[1];
  const float s = p.scale;
  const uint4 w = make_uint4(pack_bf16x2(a.x * s, a.y * s), pack_bf16x2(a.z * s, a.w * s),
                             pack_bf16x2(e.x * s, e.y * s), pack_bf16x2(e.z * s, e.w * s));
  *reinterpret_cast<uint4 *>(p.dq + ((long long)(p.seq_start(b) + i) * p.Hq + h) * 64 + seg * 8) =
      w;
}

}  // namespace bwd
}  // namespace attn
