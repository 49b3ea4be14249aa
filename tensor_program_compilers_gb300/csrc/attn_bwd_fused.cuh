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
// Tensor memory: S^T [0,128) (P^T bf16 over its first 64 columns), dP^T
// [128,256) (dS^T over its first 64), dV [256,320), dK [320,384), the dQ
// share [384,448).  The dQ product takes dS from shared memory: the softmax
// warps write their dS^T rows there as well, in the 128-byte-swizzled
// layout with the query index contiguous (an M-major A operand), and K
// serves both as the K-major A of S^T and as the N-major B of dS K.

namespace attn {
namespace bwd {

struct FCfg {
  static constexpr int D = 64;
  static constexpr uint32_t TILE = CHUNK_BYTES;                  // 128 x 64 bf16
  static constexpr uint32_t SLOT = 2 * TILE + 1024;              // Q, dO, lse2 row, dsum row
  static constexpr uint32_t OFF_RING = 2 * TILE;                 // after K, V
  static constexpr uint32_t OFF_DS = OFF_RING + 2 * SLOT;        // dS, 128 queries x 128 keys
  static constexpr uint32_t OFF_STG = OFF_DS + 2 * TILE;         // 8 warps x 32 rows x 32 fp32
  static constexpr uint32_t STG_WARP = 32 * 128;
  static constexpr uint32_t OFF_CTL = OFF_STG + BWD_SM_WARPS * STG_WARP;
  static constexpr uint32_t CTL_BYTES = 256;
  static constexpr uint32_t SMEM = OFF_CTL + CTL_BYTES + 1024;
  static_assert(OFF_DS % 1024 == 0 && OFF_STG % 1024 == 0, "swizzle atoms");
  static_assert(SMEM >= BCfg<64>::MIN_SMEM && SMEM <= 232448, "shared memory");
};

enum : int {
  F_STATIC = 0,   // K, V loaded
  F_FULL0,        // ring slot s loaded, s < 2
  F_FULL1,
  F_EMPTY0,       // ring slot s consumed
  F_EMPTY1,
  F_DONE,         // dK, dV final
  F_DRAIN,        // abort drain of the MMA issuer
  F_ST,           // S^T of the step in TMEM
  F_DPT,          // dP^T of the step in TMEM
  F_PT,           // softmax warps: P^T written
  F_DST,          // softmax warps: dS^T written (TMEM and shared memory), dQ share read
  F_DQ,           // the step's dQ share in TMEM
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

// Instruction descriptor for dS K: A (dS) and B (K) both stored with the
// M / N index contiguous.
constexpr uint32_t IDESC_DQ = idesc_bf16_f32(64, 1) | (1u << 15);

// One warp's share of the dQ product: rows 32 wq .. 32 wq + 31 of the query
// block, columns 32 hf .. 32 hf + 31, from TMEM into the warp's staging box
// (128-byte swizzle, one 128-byte line per row) and reduce-added into the
// buffer at (column c0, buffer row c1).  Lane 0 first waits until the
// warp's previous reduce-add has read the box (issued a step earlier).
__device__ __forceinline__ void dq_share_out(uint32_t taddr, uint32_t stg,
                                             const CUtensorMap *map, int c0, int c1) {
  const int lane = threadIdx.x & 31;
  uint32_t u[32];
  tmem_ld32(taddr, u);
  tmem_wait_ld();
  reg_fence32(u);
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const uint32_t line = stg + (uint32_t)lane * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(line + ((uint32_t)(j ^ (lane & 7)) << 4),
                 make_uint4(u[4 * j], u[4 * j + 1], u[4 * j + 2], u[4 * j + 3]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_reduce_add_2d(map, c0, c1, stg);
    bulk_commit_group();
  }
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
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
      for (int s = 0; s < 2; ++s) {
        mbar_init(bar(F_FULL0 + s), 1);
        mbar_init(bar(F_EMPTY0 + s), 1);
      }
      mbar_init(bar(F_DONE), 1);
      mbar_init(bar(F_DRAIN), 1);
      mbar_init(bar(F_ST), 1);
      mbar_init(bar(F_DPT), 1);
      mbar_init(bar(F_PT), BWD_SM_WARPS);
      mbar_init(bar(F_DST), BWD_SM_WARPS);
      mbar_init(bar(F_DQ), 1);
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
  constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 320, COL_DQ = 384;

  if (warp == 0) {
    // producer: K, V once, then Q(s), dO(s) and the two rows of each step
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(F_STATIC), 2 * C::TILE);
      tma_load_3d(k_s, &tm_k, bar(F_STATIC), 0, kvh, row0 + jb * BM);
      tma_load_3d(v_s, &tm_v, bar(F_STATIC), 0, kvh, row0 + jb * BM);
      for (int s = 0; ok && s < steps; ++s) {
        const int slot = s & 1;
        if (s >= 2 && !(ok = wait_bounded(bar(F_EMPTY0 + slot), (uint32_t)((s - 2) >> 1) & 1u,
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
        for (int s = 0; s < 2 && s < issued; ++s) {
          const int last = s + 2 * ((issued - 1 - s) / 2);
          wait_drain(bar(F_FULL0 + s), (uint32_t)(last >> 1) & 1u, p.timeout_ns);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer (whole warp, one elected lane issues).  Per step s: dV +=
    // P^T(s) dO(s) once P^T is written; S^T(s+1) (its columns are free once
    // dV(s) has read P^T: one thread's MMAs run in issue order); then, once
    // dS is written, dK += dS^T(s) Q(s), dQ share = dS(s) K, and dP^T(s+1).
    // dQ(s) overwrites the share that the softmax warps read before
    // writing dS(s); the softmax warps rewrite the shared dS tile only after
    // dP^T(s+1), which follows dQ(s), has completed.
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
      const int slot = s & 1;
      const uint32_t q_s = ring + slot * C::SLOT;
      const uint32_t q_n = ring + (slot ^ 1) * C::SLOT;
      const uint64_t do_mn = smem_desc_sw128(q_s + C::TILE, CHUNK_BYTES, 1024);
      const uint64_t q_mn = smem_desc_sw128(q_s, CHUNK_BYTES, 1024);
      if (!(ok = wait_warp(bar(F_PT), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 0, s > 0);
      issue_pv_half_warp<D>(tmem + COL_DV, tmem + COL_ST, do_mn, 1, s > 0);
      const bool more = s + 1 < steps;
      if (more) {
        if (!(ok = wait_warp(bar(F_FULL0 + (slot ^ 1)), (uint32_t)((s + 1) >> 1) & 1u,
                             abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        issue_qk_warp<D>(tmem + COL_ST, kdesc, smem_desc_sw128(q_n, 16, 1024));
        tc_commit_warp(bar(F_ST));
      }
      if (!(ok = wait_warp(bar(F_DST), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
      tc_fence_after();
      issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 0, s > 0);
      issue_pv_half_warp<D>(tmem + COL_DK, tmem + COL_DPT, q_mn, 1, s > 0);
      tc_commit_warp(bar(F_EMPTY0 + slot));   // Q(s), dO(s) and their rows are read
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
  } else {
    // softmax warps: thread = key row jb*128 + row of TMEM lane quarter
    // warp%4, query columns 64 hf .. 64 hf + 63; for the dQ share, query row
    // 32 (warp%4) + lane of the step's block, columns 32 hf .. 32 hf + 31
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int row = wq * 32 + lane;
    const int key = jb * BM + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t stg = base + C::OFF_STG + (uint32_t)(warp - 2) * C::STG_WARP;
    const uint32_t ds_line = ds_s + (uint32_t)hf * CHUNK_BYTES + (uint32_t)row * 128u;
    const float c = p.scale_log2;
    const bool kdead = key >= len;
    const long long hrow = (long long)p.pstart[b] + 32 * wq;   // + h rows_pad + ib 128
    // buffer row of the share of step t: head and query block of t
    auto share_row = [&](int t) {
      const int h = kvh * p.group + t / nq;
      return (int)((long long)h * p.rows_pad() + hrow + (long long)(i0 + t % nq) * BM);
    };
    bool ok = true;
    for (int s = 0; ok && s < steps; ++s) {
      const int slot = s & 1;
      if (!(ok = wait_warp(bar(F_FULL0 + slot), (uint32_t)(s >> 1) & 1u, abort_flag,
                           p.timeout_ns)) ||
          !(ok = wait_warp(bar(F_ST), (uint32_t)s & 1u, abort_flag, p.timeout_ns)))
        break;
      tc_fence_after();
      const int ib = i0 + s % nq;
      const float *lse2 =
          reinterpret_cast<const float *>(smem + C::OFF_RING + slot * C::SLOT + 2 * C::TILE);
      const float *dsum = lse2 + 128;
      const bool diag = p.causal && ib == jb;
      // phase 1: P^T = 2^(S^T c - LSE2), bf16, kept in registers for dS; a
      // key past the end of its sequence gets P = 0 (its dK, dV rows are not
      // stored, but its dS would enter every query's dQ)
      uint32_t pw[2][16];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * hf + 32 * ch;
        uint32_t us[32];
        tmem_ld32(tmem + lane_off + COL_ST + c0, us);
        tmem_wait_ld();
        reg_fence32(us);
        if (!diag && !kdead) {
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
            if (kdead || (diag && ib * BM + qc < key)) p0 = 0.f;
            if (kdead || (diag && ib * BM + qc + 1 < key)) p1 = 0.f;
            pw[ch][x >> 1] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(tmem + lane_off + COL_ST + 64 * hf + 16 * ch, pw[ch]);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(F_PT));
      // the previous step's dQ share, while dP^T(s) is formed
      if (s > 0) {
        if (!(ok = wait_warp(bar(F_DQ), (uint32_t)(s - 1) & 1u, abort_flag, p.timeout_ns)))
          break;
        tc_fence_after();
        dq_share_out(tmem + lane_off + COL_DQ + 32 * hf, stg, &tm_dqacc, 32 * hf,
                     share_row(s - 1));
      }
      // phase 2: dS^T = P^T o (dP^T - D), bf16, into TMEM (for dK) and into
      // the shared dS tile (for dQ)
      if (!(ok = wait_warp(bar(F_DPT), (uint32_t)s & 1u, abort_flag, p.timeout_ns))) break;
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
        // queries 32 ch .. 32 ch + 31 of this half: four 16-byte pieces of
        // the key's 128-byte line
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
    if (ok && steps > 0 &&
        (ok = wait_warp(bar(F_DQ), (uint32_t)(steps - 1) & 1u, abort_flag, p.timeout_ns))) {
      tc_fence_after();
      dq_share_out(tmem + lane_off + COL_DQ + 32 * hf, stg, &tm_dqacc, 32 * hf,
                   share_row(steps - 1));
    }
    if (lane == 0) bulk_wait_all();   // the reduce-adds are done with the staging box
    __syncwarp();
    if (ok && (ok = wait_warp(bar(F_DONE), 0, abort_flag, p.timeout_ns))) {
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
