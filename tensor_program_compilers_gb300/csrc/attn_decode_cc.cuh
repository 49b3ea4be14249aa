// attn_decode_cc.cuh -- split-key decode on the CUDA cores (included by
// attn_fwd.cu, whose Params, status word and combine pass it shares).
//
// Decode reads every key and value row of a sequence once for a handful of
// query rows (the group's query heads x the new positions, R <= 8): per key
// it moves 2 d bf16 and does 4 R d FLOP, so it is bound by HBM, not by the
// tensor cores (tang, section 9.2: the time floor of a memory-bound kernel
// is its bytes over the bandwidth).  Here every warp streams rows with
// 16-byte loads -- eight columns per lane, D / 8 lanes per row -- instead of
// one producer warp issuing TMA boxes, so a paged cache costs the same as a
// contiguous one whatever its page size (a box per 16-row page limited the
// tile path to about half the bandwidth).  Scores, the online softmax
// (TileLang explainer, "FlashAttention, in tiles": running max, rescale,
// exp2 with log2 e folded into the scale) and P V stay in fp32 registers.
//
// A CTA (16 warps; 8 for R > 4, whose registers fill the file at 8) owns
// one (sequence, kv head, split of the keys).  Per step each warp takes U
// key slots of KPW keys (one key per lane group); one lane per key finds its
// row (through the page table) and shares it by shuffle.  The lanes copy
// their 16-byte pieces of the K and V rows with cp.async into a ring of NST
// stages in shared memory -- each lane's own 16 bytes per row and slot,
// which only that lane reads back, so no barrier orders them -- and keep
// NST - 1 steps of copies in flight while they compute on the oldest: the R
// partial dot products of each key in f32 pairs, reduced over the lane group
// by a transposed butterfly that leaves each lane one row's score (so a lane
// exponentiates once per key and keeps one running max and sum), then p V
// for every row.  Warps keep separate (m, l, o) states, merged through
// shared memory at the end; the split's state goes to the output (one
// split) or to the workspace for attn_combine_kernel.

namespace attn {
namespace dcc {

constexpr int U = 4, NST = 3;
// per warp and stage: U slots x (K, V) x 32 lanes x 16 bytes
constexpr int STAGE_BYTES = U * 2 * 32 * 16;
// warps per CTA for RP rows: every warp's rows in registers (RP 8: ~250 a
// thread) and its ring in shared memory (NST x 4 KB)
__host__ __device__ constexpr int warps_for(int rp) { return rp <= 4 ? 16 : 8; }
__host__ __device__ constexpr int ring_bytes(int rp) { return warps_for(rp) * NST * STAGE_BYTES; }

// 16 bytes global -> shared, bypassing L1; src_bytes 0 writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// all but the newest NST - 2 groups of this thread's copies are complete
__device__ __forceinline__ void cp_async_wait_ring() {
  asm volatile("cp.async.wait_group %0;" ::"n"(NST - 2) : "memory");
}

// Transposed reduction of a lane group's partial dot products: v holds
// N row sums of this lane's columns; each level of the butterfly (xor W)
// hands the partner the half of the rows it keeps and adds the half it
// receives, so after log2 N levels the lane holds one row (the top bits of
// its position in the group, most significant first) and the remaining
// levels add plain sums.  N + log2(lanes) shuffles instead of N log2(lanes).
template <int N, int W>
__device__ __forceinline__ float reduce_to_row(float *v, int lane) {
  if constexpr (W == 0) {
    return v[0];
  } else if constexpr (N > 1) {
    const bool hi = (lane & W) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = hi ? v[i] : v[i + N / 2];
      const float keep = hi ? v[i + N / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, W);
    }
    return reduce_to_row<N / 2, W / 2>(v, lane);
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], W);
    return reduce_to_row<1, W / 2>(v, lane);
  }
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// One split of a unit (sequence b, kv head kvh): keys [k_begin, k_end) of
// its L, for every query row of the unit.  With one split the result goes
// to the outputs, else (O / l and the LSE) to the split's workspace rows for
// attn_combine_kernel.
// RP: rows rounded up to a power of two (rows >= R are zero and unwritten).
template <int D, int RP, bool PAGED>
__device__ __forceinline__ void run_split(const Params &p, uint8_t *ring, float (*sh_m)[RP],
                                          float (*sh_l)[RP], int b, int kvh, int L, int split,
                                          int k_begin, int k_end) {
  constexpr int WARPS = warps_for(RP), THREADS = WARPS * 32;
  constexpr int LPR = D / 8;        // lanes per key row
  constexpr int KPW = 32 / LPR;     // keys per warp and slot
  constexpr int NK = U * KPW;       // keys per warp and step
  constexpr int KSTEP = WARPS * NK; // keys per CTA step
  static_assert(RP <= LPR && NK <= 32, "lane layout");
  constexpr int SH = ilog2(LPR) - ilog2(RP);   // my row = my position in the group >> SH
  static_assert(RP * D * 4 <= NST * STAGE_BYTES, "a warp's O fits in its ring");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int myrow = sub >> SH;
  const int G = p.group, R = G * p.dq_n;

  // this lane's eight columns of every query row (scale log2 e folded in),
  // as four f32 pairs; the key limit of this lane's own row
  uint64_t q2[RP][4];
#pragma unroll
  for (int r = 0; r < RP; ++r) {
    const int pos = r / G, hq = kvh * G + r % G;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (r < R)
      w = __ldg(reinterpret_cast<const uint4 *>(
          p.q + (((long long)b * p.dq_n + pos) * p.Hq + hq) * D + sub * 8));
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
    for (int i = 0; i < 4; ++i) q2[r][i] = f2_mul(bf16x2_widen(x[i]), c2);
  }
  const int lim_my =
      myrow < R ? (p.causal ? L - p.dq_n + myrow / G + 1 : L) : 0;   // keys [0, lim_my)

  float m_my = -INFINITY, l_my = 0.f;   // running max and sum of this lane's row
  uint64_t o2[RP][4];                   // P V of every row, this lane's columns
#pragma unroll
  for (int r = 0; r < RP; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) o2[r][i] = 0ull;
  const int *tbl = PAGED ? p.block_table + (long long)b * p.max_blocks : nullptr;
  const uint32_t my_ring = smem_u32(ring) + (uint32_t)(warp * NST * STAGE_BYTES + lane * 16);

  // copies of step `it` into its stage: lane j < NK finds the row of the
  // warp's key j (-1: none, or a bad page, read as zeros), then every lane
  // fetches its slots' rows
  auto issue = [&](int it) {
    const int kb = k_begin + it * KSTEP + warp * NK;
    int rowj = -1;
    if (lane < NK && kb + lane < k_end) {
      const int key = kb + lane;
      if (PAGED) {
        const int blk = p.page_shift >= 0 ? key >> p.page_shift : key / p.page_size;
        const int page = __ldg(tbl + blk);
        if (page >= 0 && page < p.num_pages)
          rowj = page * p.page_size + (key - blk * p.page_size);
        else
          record_status(ATTN_ERR_BAD_PAGE_TABLE);
      } else {
        rowj = b * p.dk_n + key;
      }
    }
    const uint32_t st = my_ring + (uint32_t)((it % NST) * STAGE_BYTES);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = __shfl_sync(0xffffffffu, rowj, u * KPW + grp);
      const long long off = ((long long)max(row, 0) * p.Hkv + kvh) * D + sub * 8;
      const uint32_t n = row >= 0 ? 16u : 0u;
      cp_async16(st + (uint32_t)(u * 2 * 512), p.kc + off, n);
      cp_async16(st + (uint32_t)((u * 2 + 1) * 512), p.vc + off, n);
    }
  };
  const int steps = (k_end - k_begin + KSTEP - 1) / KSTEP;
#pragma unroll
  for (int it = 0; it < NST - 1; ++it) {
    if (it < steps) issue(it);
    cp_async_commit();
  }

  for (int it = 0; it < steps; ++it) {
    cp_async_wait_ring();   // this lane's copies of step it have landed
    const uint32_t st = my_ring + (uint32_t)((it % NST) * STAGE_BYTES);
    uint4 kw[U], vw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      kw[u] = ld_shared_v4(st + (uint32_t)(u * 2 * 512));
      vw[u] = ld_shared_v4(st + (uint32_t)((u * 2 + 1) * 512));
    }
    // the stage read last step is free: refill it with step it + NST - 1
    if (it + NST - 1 < steps) issue(it + NST - 1);
    cp_async_commit();
    const int kb = k_begin + it * KSTEP + warp * NK + grp;   // + u KPW: slot u's key
    // this lane's row's score for each slot's key (log2 units), -inf if hidden
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t x[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
      uint64_t k2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) k2[i] = bf16x2_widen(x[i]);
      float a[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        uint64_t acc = f2_mul(q2[r][0], k2[0]);
#pragma unroll
        for (int i = 1; i < 4; ++i) acc = f2_fma(q2[r][i], k2[i], acc);
        float lo, hi;
        f2_unpack(acc, lo, hi);
        a[r] = lo + hi;
      }
      const float sc = reduce_to_row<RP, LPR / 2>(a, lane);
      const int key = kb + u * KPW;
      s[u] = key < lim_my && key < k_end ? sc : -INFINITY;
    }
    // the step's max of this lane's row over the warp's keys; rescale on a move
    float mb = s[0];
#pragma unroll
    for (int u = 1; u < U; ++u) mb = fmaxf(mb, s[u]);
#pragma unroll
    for (int w = 16; w >= LPR; w >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, w));
    const bool move = mb > m_my;
    if (__any_sync(0xffffffffu, move)) {
      const float alpha = !move ? 1.f : (m_my == -INFINITY ? 0.f : ex2_approx(m_my - mb));
      if (move) m_my = mb;
      l_my *= alpha;
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const float ar = __shfl_sync(0xffffffffu, alpha, grp * LPR + (r << SH));
        const uint64_t a2 = f2_pack(ar, ar);
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[r][i] = f2_mul(o2[r][i], a2);
      }
    }
    // p of this lane's row, shared with the group; p V for every row
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float pe = s[u] == -INFINITY ? 0.f : ex2_approx(s[u] - m_my);
      l_my += pe;
      const uint32_t x[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
      uint64_t v2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v2[i] = bf16x2_widen(x[i]);
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const float pr = __shfl_sync(0xffffffffu, pe, grp * LPR + (r << SH));
        const uint64_t p2 = f2_pack(pr, pr);
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[r][i] = f2_fma(p2, v2[i], o2[r][i]);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");   // nothing left in flight
  __syncwarp();   // every lane's copies have landed before the ring is reused

  // the lane groups of a warp share its max: add their sums and P V
#pragma unroll
  for (int w = 16; w >= LPR; w >>= 1) {
    l_my += __shfl_xor_sync(0xffffffffu, l_my, w);
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float lo, hi;
        f2_unpack(o2[r][i], lo, hi);
        lo += __shfl_xor_sync(0xffffffffu, lo, w);
        hi += __shfl_xor_sync(0xffffffffu, hi, w);
        o2[r][i] = f2_pack(lo, hi);
      }
  }
  // each warp's O over its own (drained) ring
  auto sh_o = [&](int w, int r) {
    return reinterpret_cast<float *>(ring + w * NST * STAGE_BYTES) + r * D;
  };
  if (grp == 0) {
    if ((sub & ((1 << SH) - 1)) == 0) {   // one lane per row
      sh_m[warp][myrow] = m_my;
      sh_l[warp][myrow] = l_my;
    }
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2_unpack(o2[r][i], f[2 * i], f[2 * i + 1]);
      float *dst = sh_o(warp, r) + sub * 8;
      *reinterpret_cast<float4 *>(dst) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4 *>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  __syncthreads();
  // merge the warps' states, one (row, column) per thread and round
  for (int idx = threadIdx.x; idx < R * D; idx += THREADS) {
    const int r = idx / D, col = idx % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) mm = fmaxf(mm, sh_m[w][r]);
    float lt = 0.f, ot = 0.f;
    if (mm != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float sc = sh_m[w][r] == -INFINITY ? 0.f : ex2_approx(sh_m[w][r] - mm);
        lt += sh_l[w][r] * sc;
        ot += sh_o(w, r)[col] * sc;
      }
    }
    const int pos = r / G, hq = kvh * G + r % G;
    const long long lrow = ((long long)b * p.Hq + hq) * p.dq_n + pos;
    const float lse = lt > 0.f ? (mm + log2f(lt)) * 0.6931471805599453f : -INFINITY;
    const float ov = lt > 0.f ? ot / lt : 0.f;
    if (p.splits == 1) {
      p.o[(((long long)b * p.dq_n + pos) * p.Hq + hq) * D + col] = __float2bfloat16_rn(ov);
      if (col == 0) p.lse[lrow] = lse;
    } else {
      p.ws_o[(lrow * p.splits + split) * D + col] = ov;
      if (col == 0) p.ws_lse[lrow * p.splits + split] = lse;
    }
  }
}

// Decode kernel: CTA = one (sequence, kv head, split of the keys).
template <int D, int RP, bool PAGED>
__global__ void __launch_bounds__(warps_for(RP) * 32, 1) attn_decode_cc_kernel(const Params p) {
  constexpr int WARPS = warps_for(RP);
  __shared__ float sh_m[WARPS][RP], sh_l[WARPS][RP];
  // ring_bytes(RP): each warp's ring of NST stages, and after the loop its O
  extern __shared__ __align__(16) uint8_t ring[];
  const int split = (int)(blockIdx.x % (unsigned)p.splits);
  const long long bk = blockIdx.x / (unsigned)p.splits;
  const int kvh = (int)(bk % p.Hkv), b = (int)(bk / p.Hkv);
  const int L = p.seqlens_k ? __ldg(p.seqlens_k + b) : p.dk_n;
  if (L < p.dq_n || L > p.dk_n) {   // an impossible length: report, write nothing
    if (threadIdx.x == 0) record_status(ATTN_ERR_BAD_SEQLENS);
    return;
  }
  const int k_begin = split * p.chunk;
  const int k_end = min(L, k_begin + p.chunk);
  if (k_begin >= k_end) return;   // past the sequence: the merge skips this split
  run_split<D, RP, PAGED>(p, ring, sh_m, sh_l, b, kvh, L, split, k_begin, k_end);
}

}  // namespace dcc
}  // namespace attn
