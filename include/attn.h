/*
 * attn.h -- C ABI of libattn: fused attention forward for sm_103a (GB300).
 *
 * The operation
 * -------------
 * For every sequence, query head h and query row i:
 *
 *     kv     = h / (Hq / Hkv)                     (contiguous head groups)
 *     s_ij   = scale * <q[i,h,:], k[j,kv,:]>      for visible keys j
 *     o[i,h] = softmax_j(s_ij) . v[:,kv,:]
 *     lse    = ln sum_j exp(s_ij)                 (natural logarithm)
 *
 * visible keys: all keys of the same sequence, or, when causal, keys j <= i.
 * The score matrix is never written to memory: the kernel keeps a running
 * row maximum and a rescaled running sum per row (the online-softmax monoid
 * of tang, muni.works/research/tang, section 2.2 and Table 1 "online
 * softmax" / "FlashAttention forward"; the per-block loop of the TileLang
 * explainer, ai.thesatyajit.com/articles/tilelang, "FlashAttention, in
 * tiles").  The grouped-query head split follows tang section 2.1 "Views";
 * the logsumexp output is tang Table 1 "logsumexp".
 *
 * Arithmetic: bf16 inputs, fp32 accumulation on the tensor cores, fp32
 * softmax with base-2 exponentials, probabilities rounded to bf16 before the
 * P.V product, output rounded to bf16 (nearest even), LSE in fp32.
 *
 * Layouts (all row-major, contiguous, no padding)
 * -----------------------------------------------
 *   fixed batch (cu_seqlens == NULL):
 *     q, o : [B, N, Hq,  d] bf16      k, v : [B, N, Hkv, d] bf16
 *     lse  : [B, Hq, N] fp32
 *   packed variable-length batch (cu_seqlens != NULL):
 *     q, o : [T, Hq,  d] bf16         k, v : [T, Hkv, d] bf16
 *     lse  : [Hq, T] fp32,  T = N = cu_seqlens[B]
 *     sequence s owns token rows cu_seqlens[s] .. cu_seqlens[s+1]-1.
 *
 * Ownership: every pointer is caller-owned DEVICE memory on the current
 * device.  The library allocates no memory and keeps no reference after the
 * call returns.  Calls are asynchronous and ordered on `stream`.
 */
#ifndef LIBATTN_ATTN_H_
#define LIBATTN_ATTN_H_

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,        /* a size, flag or pointer is out of range    */
  ATTN_ERR_ALIGNMENT = 2,          /* q/k/v/o not 16-byte aligned, lse not 4     */
  ATTN_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  ATTN_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed           */
  ATTN_ERR_TIMEOUT = 5,            /* a kernel pipeline wait ran out (device-side) */
  ATTN_ERR_BAD_SEQLENS = 6,        /* cu_seqlens inconsistent (device-side check)  */
  ATTN_ERR_BAD_PAGE_TABLE = 7      /* a page number outside the cache (device-side) */
} attn_status;

/*
 * attn_fwd -- O = softmax(scale * Q K^T + mask) V and the per-row LSE.
 *
 *   q, k, v   : device bf16 inputs in the layouts above (16-byte aligned).
 *   o         : device bf16 output (16-byte aligned).
 *   lse       : device fp32 output (4-byte aligned).
 *   B         : batch size, or number of packed sequences (>= 0).
 *   Hq, Hkv   : query and key/value heads, Hq % Hkv == 0, both >= 1.
 *   N         : fixed batch: tokens per sequence (>= 0);
 *               packed: total tokens T = cu_seqlens[B].
 *   d         : head dimension, one of 64, 128, 256.
 *   scale     : score multiplier, finite and > 0 (usually 1/sqrt(d)).
 *   causal    : nonzero masks keys after the query (j > i, per sequence).
 *   cu_seqlens: NULL for a fixed batch, else device int32[B+1] with
 *               cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = N.
 *               The kernel checks this and reports ATTN_ERR_BAD_SEQLENS
 *               through attn_get_status() (outputs then stay unwritten).
 *   stream    : CUDA stream (0 = legacy default stream).
 *
 * Returns ATTN_OK once the kernel is enqueued (or when there is no work:
 * B == 0 or N == 0).  Host-side argument errors return their code without
 * launching anything.  Device-side errors (a pipeline wait that ran past
 * its time limit, bad cu_seqlens) are recorded in a per-device status word
 * read by attn_get_status().
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     const int *cu_seqlens, cudaStream_t stream);

/*
 * attn_variant -- score and mask variants of attn_fwd_ex.  They change only
 * the scores or the mask, not the online-softmax monoid (tang, section 2.3
 * and section 7.3, "Attention variants against FlexAttention and FA2": soft
 * cap, ALiBi, a sliding window of 128).  The pages print no formulas; these
 * are the common readings.  With s = scale * q_i . k_j:
 *
 *   window_left  : keys j < i - window_left are masked (< 0: unbounded).
 *   window_right : keys j > i + window_right are masked (< 0: unbounded;
 *                  causal forces 0).  Key tiles that no row of a query tile
 *                  sees are skipped, not computed.
 *   softcap      : > 0: s -> softcap * tanh(s / softcap); 0: off.
 *   alibi_slopes : NULL, or device fp32[Hq] (4-byte aligned): after the cap,
 *                  s -> s - alibi_slopes[h] * |i - j|.
 *
 * The LSE is that of the modified, masked scores.  A row that sees no key
 * (possible only for padding rows) gets O = 0 and LSE = -inf.
 */
typedef struct {
  int window_left;
  int window_right;
  float softcap;
  const float *alibi_slopes;
} attn_variant;

/*
 * attn_fwd_ex -- attn_fwd with score and mask variants (var == NULL: none;
 * same as attn_fwd).  Same arguments, layouts, ownership and errors as
 * attn_fwd, plus ATTN_ERR_INVALID_ARG for a softcap that is negative or not
 * finite and ATTN_ERR_ALIGNMENT for misaligned alibi_slopes.
 */
attn_status attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                        const int *cu_seqlens, const attn_variant *var, cudaStream_t stream);

/*
 * attn_fwd_decode -- attention of a few new queries against long key/value
 * caches, split along the keys (the online-softmax merge is associative:
 * tang, section 2.2, "Online softmax is the monoid ..."; section 2.5, "split
 * ... valid for any monoid because combine is associative, including online
 * softmax").  Each (sequence, kv head, key split) computes a partial state
 * of its rows (the group's Hq/Hkv query heads x Nq positions); a second
 * kernel merges the splits: LSE = log sum_s exp(LSE_s),
 * O = sum_s exp(LSE_s - LSE) O_s.
 *
 *   q        : device bf16 [B, Nq, Hq, d] -- the last Nq positions of each
 *              sequence (16-byte aligned).
 *   k, v     : device bf16 [B, Nk, Hkv, d] caches; sequence b uses rows
 *              0 .. seqlens_k[b] - 1.  Rows past a sequence's length must
 *              hold finite values (they are read, weighted by zero).
 *   o        : device bf16 [B, Nq, Hq, d];  lse: device fp32 [B, Hq, Nq].
 *   Nq, Nk   : queries per sequence, cache rows per sequence;
 *              1 <= Nq <= Nk and (Hq / Hkv) * Nq <= 128.
 *   causal   : nonzero: query r of sequence b sees keys
 *              j <= seqlens_k[b] - Nq + r (bottom-right alignment);
 *              zero: all seqlens_k[b] keys.
 *   seqlens_k: NULL (every sequence has Nk keys), or device int32[B] with
 *              Nq <= seqlens_k[b] <= Nk (checked on the device; a bad value
 *              is reported as ATTN_ERR_BAD_SEQLENS by attn_get_status and
 *              that sequence's outputs stay unwritten).
 *   workspace: device memory owned by the caller, 16-byte aligned, at least
 *              attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) bytes
 *              (may be NULL when that is 0).  It holds the partial states
 *              between the two kernels; nothing else is allocated.
 *
 * Other arguments and errors as attn_fwd; too small a workspace is
 * ATTN_ERR_INVALID_ARG.  The split count depends on the device's SM count.
 *
 * attn_decode_workspace_bytes returns 0 both when the problem needs no
 * workspace (one split) and when it cannot size one (invalid arguments, an
 * unsupported or unusable device); rely on the status that attn_fwd_decode
 * (or attn_fwd_decode_static) returns for the actual error.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d);
attn_status attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                            int causal, const int *seqlens_k, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_fwd_decode_paged -- attn_fwd_decode reading paged key/value caches
 * (tang, section 2.1 "Views": a paged KV cache is a gathered read, the page
 * number of a key being data read from an index tensor; Table 1 row "paged
 * KV cache").
 *
 *   k_cache, v_cache: device bf16 [num_pages, page_size, Hkv, d], 16-byte
 *              aligned.  Rows of pages past a sequence's length must hold
 *              finite values (they are read, weighted by zero).
 *   seqlens_k: device int32[B] (required), Nq <= seqlens_k[b] <=
 *              max_blocks * page_size.
 *   block_table: device int32[B * max_blocks] (4-byte aligned): key j of
 *              sequence b is row j % page_size of page
 *              block_table[b * max_blocks + j / page_size].  Entries past
 *              a sequence's last page are not read.  A page number outside
 *              [0, num_pages) is reported as ATTN_ERR_BAD_PAGE_TABLE through
 *              attn_get_status (its keys then read as zeros).
 *   page_size: 16, 32 or 64, or a multiple of 128.
 *   workspace: at least attn_decode_paged_workspace_bytes(B, Hq, Hkv, Nq,
 *              max_blocks, page_size, d) bytes (may be NULL when that is 0).
 *
 * Everything else as attn_fwd_decode.
 */
size_t attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int Nq, int max_blocks,
                                         int page_size, int d);
attn_status attn_fwd_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                                  void *o, float *lse, int B, int Hq, int Hkv, int Nq, int d,
                                  float scale, int causal, const int *seqlens_k,
                                  const int *block_table, int max_blocks, int page_size,
                                  int num_pages, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/*
 * attn_fwd_decode_static -- attn_fwd_decode without a caller workspace and
 * without any allocation: the partial states live in a fixed 8 MiB device
 * array inside the library (one per device).  The pages have no
 * counterpart.  It is for callers that can neither allocate device memory
 * nor hand one over: a plug-in whose host program owns all device memory
 * through its own allocator and lends it none, or a serving loop that
 * allows no allocation once it runs, because cudaMalloc and cudaFree can
 * synchronise the whole device and stall every other stream.
 *
 *   - Problems whose attn_decode_workspace_bytes() exceeds 8 MiB
 *     (8388608 bytes) are rejected with ATTN_ERR_INVALID_ARG.
 *   - The array's address is looked up once per device, on the first call
 *     of any entry point on that device; make that first call outside
 *     stream capture.
 *   - Nothing in the array needs to start at zero: every slot the merge
 *     kernel reads is written earlier in the same call.
 *   - Calls that overlap in time on one device (different streams, or host
 *     threads) race on the array: serialise them, e.g. on one stream.
 *
 * Other arguments, layouts and errors as attn_fwd_decode.
 */
attn_status attn_fwd_decode_static(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                   float scale, int causal, const int *seqlens_k,
                                   cudaStream_t stream);

/*
 * attn_bwd -- gradients of attn_fwd (fixed or packed batches): dq, dk, dv of
 * O = softmax(scale Q K^T + mask) V for the output gradient dout (tang,
 * section 3 "Gradients are comprehensions"; section 6: the flash backward
 * identity D_i = sum_j P_ij dP_ij = dO_i . O_i):
 *   P = exp(scale S - LSE) (recomputed), dV = P^T dO, dP = dO V^T,
 *   dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q
 * (dK, dV summed over the query heads of each kv head).
 *
 *   q, o, dout, dq, k, v, dk, dv: device bf16 in the layouts of attn_fwd
 *              (fixed [B, N, H, d], packed [T, H, d]; 16-byte aligned);
 *   lse      : the forward's fp32 LSE in its layout ([B, Hq, N] or [Hq, T]).
 *   N, cu_seqlens: as attn_fwd (packed: N = T, cu_seqlens device int32[B+1];
 *              bad offsets are reported as ATTN_ERR_BAD_SEQLENS).
 *   d        : 64, 128 or 256 (256: dV, dK and dQ in three kernels, the
 *              scores recomputed in each).
 *   workspace: caller-owned device memory of at least
 *              attn_bwd_workspace_bytes(B, Hq, N, cu_seqlens != NULL) bytes,
 *              16-byte aligned (per-row D and LSE log2(e), sequence
 *              offsets); nothing else is allocated.
 * Other arguments, ownership and errors as attn_fwd; too small a workspace
 * is ATTN_ERR_INVALID_ARG.  dq, dk, dv are overwritten (no accumulation).
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int N, int packed);
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                     int Hq, int Hkv, int N, int d, float scale, int causal,
                     const int *cu_seqlens, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * attn_bwd_single_pass -- the same gradients as attn_bwd, for d = 64, in one
 * kernel per (kv head, 128-key block) (tang, section 8.3 "Attention backward
 * on Hopper": one kernel per key block, dK and dV held on chip, dQ added
 * with bulk asynchronous reductions).  Each key block adds its share of dQ,
 * dS K, into an fp32 buffer in the workspace with bulk tensor reduce-adds;
 * a last pass writes dq = scale x that buffer in bf16.  Five matrix products
 * per (key block, query block) pair instead of attn_bwd's seven.
 *
 * Arguments, layouts, ownership and errors as attn_bwd, except:
 *   d        : 64 only (anything else is ATTN_ERR_INVALID_ARG);
 *   workspace: at least attn_bwd_single_pass_workspace_bytes(B, Hq, N,
 *              cu_seqlens != NULL) bytes, 16-byte aligned: the fp32 dQ
 *              buffer (Hq x padded rows x 64) followed by attn_bwd's.
 * dk and dv are bitwise those of attn_bwd.  dq is not bitwise reproducible:
 * the key blocks' fp32 shares are added in the order they arrive, so its
 * rounding can differ between runs (its accuracy does not).
 */
size_t attn_bwd_single_pass_workspace_bytes(int B, int Hq, int N, int packed);
attn_status attn_bwd_single_pass(const void *q, const void *k, const void *v, const void *o,
                                 const void *dout, const float *lse, void *dq, void *dk,
                                 void *dv, int B, int Hq, int Hkv, int N, int d, float scale,
                                 int causal, const int *cu_seqlens, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_get_status -- takes and clears the current device's status word (the
 * first device-side error recorded since the last read) in one atomic
 * exchange, ordered on `stream` after the work already queued there, then
 * synchronises `stream` and returns the value taken: ATTN_OK,
 * ATTN_ERR_TIMEOUT, ATTN_ERR_BAD_SEQLENS, ATTN_ERR_BAD_PAGE_TABLE, or
 * ATTN_ERR_CUDA if the launch, the copy or the synchronisation failed.
 * The word is one per device, shared by every stream: an error that a
 * kernel on another stream records is returned by whichever read follows
 * it (no error is lost between the read and the clear).  Calls from several
 * host threads are serialised inside the library.
 */
attn_status attn_get_status(cudaStream_t stream);

/*
 * attn_debug_one_tile -- diagnostic switch for tests: nonzero makes every
 * later attn_fwd / attn_fwd_ex call in this process run the one-tile kernel
 * (one 128-row query tile per CTA), which otherwise serves only d = 256,
 * key windows, score modifiers, and devices whose register budget cannot
 * take the two-tile kernel.  Results agree within the stated tolerances;
 * only speed and rounding order differ.  Returns the previous setting.
 */
int attn_debug_one_tile(int on);

/* attn_status_string -- a static, human-readable name for a status code. */
const char *attn_status_string(attn_status s);

/*
 * attn_selftest_timeout -- exercises the kernels' bounded-wait path without
 * faulting the GPU: launches one block that waits on a pipeline barrier no
 * one signals, with a time limit of `timeout_us` microseconds (1..1000000).
 * The wait runs out, the kernel records ATTN_ERR_TIMEOUT in the status word
 * and returns.  This call synchronises `stream` and returns what
 * attn_get_status() then reports (ATTN_ERR_TIMEOUT when the path works).
 */
attn_status attn_selftest_timeout(int timeout_us, cudaStream_t stream);

/*
 * attn_probe_dram_latency -- the DRAM-latency term of the time floor under
 * a short launch (tang, section 9.2 "the time floor": launch overhead plus
 * memory latency plus bytes over bandwidth, latency taken from a one-thread
 * pointer chase).  Writes a chain of 8-byte indices into `scratch` (device,
 * caller-owned, `bytes` long, 16-byte aligned; bytes >= 64 MiB so that the
 * chain's start has left the L2 by the time it is chased) whose successive
 * entries lie 4,160 bytes apart, then follows `hops` (1..1,000,000) of them
 * with one thread, each load cached in L2 only, and writes to
 * `result[0]` (device, caller-owned, two 8-byte words) the nanoseconds the
 * chase took by the GPU's global timer and to result[1] the final index (so
 * the loads cannot be elided).  Asynchronous on `stream`; scratch's contents
 * are overwritten.  Errors: ATTN_ERR_INVALID_ARG for null pointers, bad
 * sizes or hop counts, ATTN_ERR_ALIGNMENT, ATTN_ERR_CUDA for a failed launch.
 */
attn_status attn_probe_dram_latency(void *scratch, size_t bytes, int hops,
                                    unsigned long long *result, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_ATTN_H_ */
