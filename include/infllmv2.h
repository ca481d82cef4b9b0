/*
 * infllmv2.h -- C ABI of the InfLLM v2 block-sparse attention library (sm_103a).
 *
 * The method is the trainable sparse attention of the MiniCPM4 technical
 * report ("MiniCPM4: Ultra-Efficient LLMs on End Devices", section "InfLLM v2:
 * Trainable Sparse Attention for Both Prefilling and Decoding"; cited below as
 * [InfLLM v2 > paragraph, equation]).  Three stages:
 *
 *   1. infllmv2_compress_keys       semantic-kernel key means
 *                                   [InfLLM v2 > Semantic kernels, eq. S_j]
 *   2. infllmv2_select_blocks       per-head kernel softmax, GQA group mean,
 *                                   block max, forced blocks, top-k
 *                                   [InfLLM v2 > Semantic kernels, eqs. r_kernel,
 *                                   r_block; > Query group sharing, eq. r_group;
 *                                   > Top-K implementation and the LSE bottleneck;
 *                                   > Initial and local tokens always selected]
 *   3. infllmv2_sparse_attn_decode  exact softmax attention over the selected
 *      infllmv2_sparse_attn_prefill KV blocks [InfLLM v2 > Block-level key-value
 *                                   partitioning, eq. B_j; > Complexity analysis]
 *
 * Around them: infllmv2_append_kv and infllmv2_decode_step (a whole decode
 * step, one launch for n_q = 1), infllmv2_append_decode_step (both as one
 * launch), infllmv2_coarse_means and
 * infllmv2_select_blocks_coarse_lse (the coarse-kernel LSE approximation),
 * and infllmv2_sparse_attn_backward (gradients of stage 3 with the selection
 * fixed [InfLLM v2 > Training-time considerations]).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer owned by the caller (the few
 *   arguments documented as possibly host memory excepted).  The
 *   library never allocates, frees or synchronises in these calls; all work
 *   is enqueued on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *   default stream) and the calls return before it runs.  (One exception:
 *   the prefill selection past 327360 tokens of capacity reads the device's
 *   SM-identifier bound once per device with a small synchronous query on a
 *   private stream; see infllmv2_select_blocks.)
 * - Shapes (row-major, innermost last; d = head_dim, G = group_size,
 *   Hq = n_kv_heads * G, n_c(L) = floor((L - p)/s) + 1 complete kernels,
 *   n_b(L) = ceil(L / m) blocks):
 *       q          bf16  [batch, n_q, Hq, d]        (heads h*G .. h*G+G-1 share KV head h)
 *       k_cache    bf16  [batch, n_kv_heads, max_kv_len, d]
 *       v_cache    bf16  [batch, n_kv_heads, max_kv_len, d]
 *       kv_lens    int32 [batch]                    (L_b, including the n_q query tokens)
 *       kc         bf16  [batch, n_kv_heads, 2, n_c(max_kv_len), d]
 *                  plane 0 holds hi = bf16(mean), plane 1 lo = bf16(mean - hi):
 *                  hi + lo is the fp32 kernel mean to 16 significant bits.
 *       block_idx  int32 [batch, n_kv_heads, n_q, k_max]   ascending, padded with -1
 *       n_selected int32 [batch, n_kv_heads, n_q]
 *       out        bf16  [batch, n_q, Hq, d]
 *       lse        fp32  [batch, n_q, Hq]           natural-log sum of exp of the
 *                                                   scaled scores of the attended keys
 * - Query t (0 <= t < n_q) of sequence b sits at position i = L_b - n_q + t; it
 *   attends keys 0..i of its selected blocks (inclusive causal mask).  The
 *   same rule serves decode (n_q = 1), speculative verification (small n_q)
 *   and causal prefill (n_q = L_b).
 * - Pointers must be 16-byte aligned.  Supported shape: head_dim 128,
 *   group_size 16, block_size 64, kernel_size 32, kernel_stride 16;
 *   anything else returns INFLLMV2_UNSUPPORTED.
 * - Return codes are INFLLMV2_* below; on failure nothing was launched and
 *   infllmv2_last_error() describes why (thread-local string).  Problems only
 *   the device can see (a kv_len outside [n_q, max_kv_len], a bounded wait
 *   that gave up) are recorded in a device status word read by
 *   infllmv2_get_device_status(); the affected unit writes zeros / an empty
 *   selection instead of reading out of bounds.
 * - No C++ exception crosses this boundary.
 */
#ifndef INFLLMV2_H
#define INFLLMV2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define INFLLMV2_OK                  0
#define INFLLMV2_INVALID_ARGUMENT    1  /* null pointer, bad size, topk < forced count, ... */
#define INFLLMV2_UNSUPPORTED         2  /* shape outside the supported set, misaligned pointer */
#define INFLLMV2_WORKSPACE_TOO_SMALL 3
#define INFLLMV2_CUDA_ERROR          4  /* launch failed; message from the CUDA runtime */

/* Device status bits (infllmv2_get_device_status). */
#define INFLLMV2_DEVICE_BAD_KV_LEN   0x1u  /* kv_lens[b] < n_q or > max_kv_len */
#define INFLLMV2_DEVICE_TIMEOUT      0x2u  /* a bounded mbarrier wait expired */
#define INFLLMV2_DEVICE_BOUNDS       0x4u  /* checked build only: a caller-given index out of range */

/* Workspace kinds for infllmv2_workspace_size. */
#define INFLLMV2_OP_SELECT  1
#define INFLLMV2_OP_DECODE  2
#define INFLLMV2_OP_PREFILL 3
#define INFLLMV2_OP_DECODE_STEP 4
#define INFLLMV2_OP_BACKWARD 5

typedef struct infllmv2_params {
  int32_t batch;                 /* B */
  int32_t n_kv_heads;            /* Hkv */
  int32_t group_size;            /* G, query heads per KV head (16) */
  int32_t head_dim;              /* d (128) */
  int32_t block_size;            /* m (64)  [InfLLM v2 > Block-level key-value partitioning] */
  int32_t kernel_size;           /* p (32)  [InfLLM v2 > Semantic kernels] */
  int32_t kernel_stride;         /* s (16)  [InfLLM v2 > Semantic kernels] */
  int32_t topk;                  /* k, blocks per query group */
  int32_t n_init_blocks;         /* forced initial blocks (1) [InfLLM v2 > Initial and local tokens] */
  int32_t n_local_blocks;        /* forced local blocks ending at the query's block (2) */
  int32_t topk_includes_forced;  /* 1: forced blocks count toward k; 0: k scored blocks on top */
  int32_t max_kv_len;            /* cache capacity per (b, h) in tokens */
  float score_scale;             /* scale inside the kernel softmax (default 1/sqrt(d)) */
  float attn_scale;              /* attention softmax scale (default 1/sqrt(d)) */
} infllmv2_params;

/* Fill `p` with the recommended shape (d 128, G 16, m 64, p 32, s 16, one
 * initial and two local blocks, both scales 1/sqrt(128)). */
void infllmv2_default_params(infllmv2_params* p, int32_t batch, int32_t n_kv_heads,
                             int32_t max_kv_len, int32_t topk, int32_t topk_includes_forced);

/* Width of a block_idx row: topk if forced blocks are included, else
 * topk + n_init_blocks + n_local_blocks.  Negative on invalid params. */
int32_t infllmv2_max_selected(const infllmv2_params* p);

/* n_c(max_kv_len): rows of each kc plane. */
int32_t infllmv2_num_kernels(const infllmv2_params* p);

/* Bytes of scratch that `op` (INFLLMV2_OP_*) needs for n_q query tokens per
 * sequence.  0 on invalid arguments. */
size_t infllmv2_workspace_size(const infllmv2_params* p, int32_t n_q, int32_t op);

/*
 * Stage 1: kc[b, h, :, j, :] = split(Mean(k_cache[b, h, j s : j s + p, :])) for
 * complete kernels j in [kernel_begin, kernel_end) of each sequence.
 * [InfLLM v2 > Semantic kernels for block relevance scoring, eqs. S_j, r_kernel]
 *   kernel_begin >= 0 : absolute first kernel;  < 0 : n_c(L_b) + kernel_begin
 *                       (so -1 recomputes only the newest complete kernel).
 *   kernel_end   >= 0 : absolute end (clipped to n_c(L_b));  < 0 : n_c(L_b).
 * Kernels outside the range are left untouched.  The mean is an fp32 sum of
 * the 32 bf16 keys times 1/32.
 */
int infllmv2_compress_keys(const infllmv2_params* p, const void* k_cache, const int32_t* kv_lens,
                           int32_t kernel_begin, int32_t kernel_end, void* kc, void* stream);

/*
 * Stage 2: choose the KV blocks of every (b, h_kv, t).
 *   z[h, j]  = score_scale * q_h . Mean_j            for kernels j visible to i
 *   g[j]     = (1/G) sum_h softmax_j(z[h, :])         (exact two-pass LSE)
 *   r[blk]   = max of g over visible kernels meeting the block, -inf if none
 *   selected = forced blocks (first n_init, the n_local ending at floor(i/m))
 *              + the best other finite-score blocks ordered by (r desc, index asc):
 *              topk - |forced| of them if topk_includes_forced, else topk.
 * block_scores (nullable) receives r as fp32 [B, Hkv, n_q, n_b(max_kv_len)]
 * (-inf past floor(i/m)).  n_q >= 1; workspace from
 * infllmv2_workspace_size(p, n_q, INFLLMV2_OP_SELECT).  For n_q > 16 the
 * selection keeps 8 tokens' block scores on chip up to max_kv_len 327360
 * (no workspace); above that they take one slot per SM of the workspace
 * (SM identifiers x 8 x n_b(max_kv_len) x 4 bytes), up to about 680K tokens
 * (INFLLMV2_UNSUPPORTED above).  The number of SM identifiers is read from
 * the device once, by a small synchronous query the first time it is
 * needed: make that first call (or the workspace-size query) outside
 * stream capture.
 */
int infllmv2_select_blocks(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                           const int32_t* kv_lens, int32_t* block_idx, int32_t* n_selected,
                           float* block_scores, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * infllmv2_select_blocks without a caller workspace.  The MiniCPM4 pages have
 * no counterpart of this entry point; it exists for embedders that cannot
 * hand the library device scratch at the call site: inference engines whose
 * device memory is laid out once at start-up, and plain C hosts that have no
 * device allocator of their own.
 *   Same arguments and result as infllmv2_select_blocks, minus the
 *   workspace.  Scratch comes from a fixed 8 MiB array inside the library
 *   (held by every device that loads it until the process exits); a
 *   selection whose scratch (infllmv2_workspace_size(p, n_q,
 *   INFLLMV2_OP_SELECT)) exceeds 8 MiB returns INFLLMV2_WORKSPACE_TOO_SMALL
 *   and launches nothing.  It allocates and frees nothing.
 *   The first call on a device looks up that device's address of the array
 *   (once); make that first call before any stream capture.  Every call
 *   shares the one array: calls whose work overlaps on the GPU (different
 *   streams, no ordering) race.  Nothing in the array has to start at zero;
 *   each call writes what it reads first.
 */
int infllmv2_select_blocks_static(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                                  const int32_t* kv_lens, int32_t* block_idx, int32_t* n_selected,
                                  float* block_scores, void* stream);

/*
 * Coarse-grained LSE approximation [InfLLM v2 > Efficient LSE approximation]
 * (off the default path; the exact LSE is the reference selection).
 *
 * infllmv2_coarse_means: kcc[b, h, 0 / 1, j, :] = hi / lo bf16 planes of the
 * mean of keys [j coarse, (j + 1) coarse) for every complete window of
 * sequence b (j < kv_lens[b] / coarse); kcc is bf16
 * [batch, n_kv_heads, 2, max_kv_len / coarse, d].  `coarse` is a multiple of
 * 16 in [32, 4096].
 *
 * infllmv2_select_blocks_coarse_lse: infllmv2_select_blocks for the prefill
 * path (n_q > 16) with each head's kernel-softmax normaliser taken over the
 * visible coarse windows (all keys <= i) instead of the fine kernels; a query
 * with no complete window keeps the exact LSE.  This cuts the first pass over
 * the kernel means by coarse / kernel_stride.  The decode path (n_q <= 16)
 * already computes the exact LSE without a second pass over memory, so it
 * has no coarse form (n_q <= 16 returns INFLLMV2_UNSUPPORTED).  Needs no
 * workspace; max_kv_len up to 327360 (the block scores stay on chip).
 */
int infllmv2_coarse_means(const infllmv2_params* p, const void* k_cache, const int32_t* kv_lens, int32_t coarse,
                          void* kcc, void* stream);
int infllmv2_select_blocks_coarse_lse(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                                      int32_t coarse, const void* kcc, const int32_t* kv_lens,
                                      int32_t* block_idx, int32_t* n_selected, float* block_scores,
                                      void* stream);

/*
 * Stage 3, few queries per sequence (decode n_q = 1, speculative verification
 * n_q <= 16): the selected blocks of each (b, h_kv, t) are dealt to the CTAs
 * of a thread-block cluster; each CTA computes an online-softmax partial and
 * the partials are merged through distributed shared memory.  out/lse as
 * documented above (lse nullable).  Only the first n_selected[b, h, t]
 * entries of block_idx are read; each must lie in [0, floor(i/m)] (entries
 * outside are skipped).  Needs no workspace (infllmv2_workspace_size
 * returns 0; workspace may be NULL).
 */
int infllmv2_sparse_attn_decode(const infllmv2_params* p, const void* q, int32_t n_q,
                                const void* k_cache, const void* v_cache, const int32_t* kv_lens,
                                const int32_t* block_idx, const int32_t* n_selected, void* out,
                                float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Stage 3, many queries per sequence (chunked or full causal prefill): same
 * arguments and result as the decode entry point, any n_q up to max_kv_len.
 */
int infllmv2_sparse_attn_prefill(const infllmv2_params* p, const void* q, int32_t n_q,
                                 const void* k_cache, const void* v_cache, const int32_t* kv_lens,
                                 const int32_t* block_idx, const int32_t* n_selected, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Cache append of a decode step: k_new / v_new (bf16 [batch, n_kv_heads, n_q,
 * d], the keys and values of each sequence's n_q newest tokens) are written
 * to cache rows kv_lens[b] - n_q .. kv_lens[b] - 1 of (b, h), so that kv_lens
 * already counts them [InfLLM v2 > Block-level key-value partitioning: the
 * cache grows by the decoded tokens].  A sequence whose kv_lens[b] lies
 * outside [n_q, max_kv_len] is left untouched and sets
 * INFLLMV2_DEVICE_BAD_KV_LEN.  q_src / q_dst (both NULL, or both given):
 * also copy the step's queries, bf16 [batch, n_q, Hq, d], from q_src to q_dst.
 * k_new, v_new and q_src are read with ordinary loads, so they may be
 * page-locked host memory mapped for the device: a decode step whose inputs
 * sit in host memory then needs no separate copy.  The launch may start
 * while the previous kernel of the stream drains; it writes only after that
 * kernel has finished, and infllmv2_decode_step on the same stream reads
 * what it wrote.
 */
int infllmv2_append_kv(const infllmv2_params* p, int32_t n_q, const void* k_new, const void* v_new,
                       const int32_t* kv_lens, void* k_cache, void* v_cache, const void* q_src, void* q_dst,
                       void* stream);

/*
 * One whole decode step: stages 1-3 for the newest n_q tokens of each
 * sequence, whose keys and values the caller has already written to the
 * caches (kv_lens counts them) [InfLLM v2 > Semantic kernels, eq. S_j;
 * > Top-K implementation and the LSE bottleneck; > Block-level key-value
 * partitioning; > Complexity analysis, stage 2].
 *   kc      in/out: every kernel mean that ends before the step's tokens must
 *           be present; the kernels that end inside them (for n_q = 1: the
 *           newest complete kernel n_c(L) - 1) are recomputed from k_cache
 *           and written back.
 *   block_idx, n_selected, out, lse: as from infllmv2_select_blocks followed
 *           by infllmv2_sparse_attn_decode (lse nullable).  out and lse are
 *           written with ordinary stores, so they may also be page-locked host
 *           memory mapped for the device (e.g. from cudaHostAlloc on a system
 *           with unified addressing): the result then reaches the host without
 *           a separate copy.
 *   n_q in [1, 16].  With n_q = 1 the step is one launch of a thread-block
 *   cluster of C CTAs per (b, h_kv), one CTA per SM, that keeps every
 *   intermediate on chip and needs no workspace.  C (at most 16) is chosen
 *   for the device and batch so that all batch * n_kv_heads clusters are
 *   resident at once; the form applies while the cache holds at most
 *   256 C blocks of 64 tokens and at most 4096 blocks (262144 tokens).
 *   Otherwise the step enqueues the three stages in order.  Workspace:
 *   infllmv2_workspace_size(p, n_q, INFLLMV2_OP_DECODE_STEP) bytes (0 for
 *   the single-launch form; workspace may then be NULL).
 */
int infllmv2_decode_step(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                         const void* v_cache, const int32_t* kv_lens, void* kc, int32_t* block_idx,
                         int32_t* n_selected, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * infllmv2_append_kv followed by infllmv2_decode_step for one new token per
 * sequence (n_q = 1), as a single launch of the decode step's cluster form
 * [InfLLM v2 > Block-level key-value partitioning: the cache grows by the
 * decoded token; the step's stages as for infllmv2_decode_step].
 *   q       bf16 [batch, 1, Hq, d]: the token's queries.
 *   k_new, v_new  bf16 [batch, n_kv_heads, 1, d]: its key and value, written
 *           to cache row kv_lens[b] - 1 of k_cache / v_cache (kv_lens
 *           already counts the token); the step reads the key from k_new
 *           where it needs it before the store is visible.
 *   q, k_new and v_new are read with ordinary loads and out / lse written
 *   with ordinary stores, so any of them may be page-locked host memory mapped
 *   for the device: a step whose inputs and result live in host memory is one
 *   launch and no copy.  kc, block_idx, n_selected, out, lse: as for
 *   infllmv2_decode_step.  No workspace.
 * INFLLMV2_UNSUPPORTED for n_q != 1 or a shape outside the single-launch
 * form (see infllmv2_decode_step): call infllmv2_append_kv and
 * infllmv2_decode_step there.  A sequence whose kv_lens[b] lies outside
 * [1, max_kv_len] is left untouched (no row written, out zero, block_idx
 * -1) and sets INFLLMV2_DEVICE_BAD_KV_LEN.
 */
int infllmv2_append_decode_step(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_new,
                                const void* v_new, void* k_cache, void* v_cache, const int32_t* kv_lens, void* kc,
                                int32_t* block_idx, int32_t* n_selected, void* out, float* lse, void* stream);

/*
 * Backward of stage 3 with the selection held fixed [InfLLM v2 >
 * Training-time considerations: top-k passes no gradient, the keys learn
 * through the gradient of the sparse attention]: for an upstream gradient
 * dout of `out`,
 *     P = exp(attn_scale q.k - lse) over each query's attended keys,
 *     D = rowsum(dout * out),  dS = P * (dout . v - D),
 *     dq = attn_scale sum_k dS k,  dk = attn_scale sum_q dS q,  dv = sum_q P dout.
 *   q, k_cache, v_cache, kv_lens, block_idx, n_selected: as given to the
 *           forward call; out (bf16) and lse (fp32, required) are its results.
 *   dout    bf16 [batch, n_q, Hq, d].
 *   dq      fp32 [batch, n_q, Hq, d], every row written.
 *   dk, dv  fp32 [batch, n_kv_heads, max_kv_len, d], every row written: keys
 *           no query attends get 0 (the call zeroes both, then adds the
 *           contributions of all queries of all heads of the group).
 * The contributions to one key row are added in an order that depends on
 * scheduling, so dk and dv may differ in the last bits from run to run.
 * Workspace: infllmv2_workspace_size(p, n_q, INFLLMV2_OP_BACKWARD) bytes
 * (an inverse block -> query index, D, work lists).
 */
int infllmv2_sparse_attn_backward(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                                  const void* v_cache, const int32_t* kv_lens, const int32_t* block_idx,
                                  const int32_t* n_selected, const void* out, const float* lse, const void* dout,
                                  float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * The checked build.  The library can also be built with INFLLMV2_CHECKED
 * (libinfllmv2_checked.so), in place of a memory checker.  It verifies
 * every index that comes from the caller before use (each counted
 * block_idx entry within [0, floor(i/m)], each n_selected within
 * [0, k_max]) and the start of every K/V tile formed from one; a violation
 * sets INFLLMV2_DEVICE_BOUNDS and the access is skipped (the product build
 * skips the same accesses without reporting them).  Its bounded waits give
 * up after 2^16 polls instead of 2^22.
 *
 * infllmv2_is_checked_build: 1 in the checked build, 0 otherwise.
 *
 * infllmv2_test_hooks: fault injection for the library's own tests, checked
 * build only (the product build returns INFLLMV2_UNSUPPORTED and changes
 * nothing).  flags = 1: in every later infllmv2_decode_step of the
 * single-launch form, one warp per CTA withholds the release of its first
 * ring stage, so a bounded wait expires: the call still returns, sets
 * INFLLMV2_DEVICE_TIMEOUT and leaves no copy in flight.  flags = 0 turns it
 * off.  Process-wide; not for concurrent use with other calls.
 */
int infllmv2_is_checked_build(void);
int infllmv2_test_hooks(uint32_t flags);

/* Human-readable name of an INFLLMV2_* return code. */
const char* infllmv2_status_string(int status);

/* Message of the last failed call on this thread ("" if none). */
const char* infllmv2_last_error(void);

/* Read (and if `clear` is nonzero, reset) the device status word of the
 * current device.  Synchronises the device; not for the hot path.
 * The library looks up the device addresses of its status word and of the
 * built-in selection scratch once per device and keeps them: it assumes the
 * device's primary context (the one the CUDA runtime uses) for the life of
 * the process, and does not support a cudaDeviceReset or a separately
 * created driver context on that device after its first call there. */
int infllmv2_get_device_status(uint32_t* status_out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* INFLLMV2_H */
