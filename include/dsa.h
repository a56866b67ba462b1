/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA sparse-MLA library.
 *
 * The library implements the data-parallel hot path of DeepSeek-style sparse
 * attention (DSA) over multi-head latent attention (MLA) with an FP8 paged KV
 * cache, as described for GLM-5.3-Flash serving:
 *
 *   scores --dsa_topk_select--> idx --dsa_sparse_mla_fwd--> (out, lse)
 *                                              \--(splits)--> partials --dsa_combine--> (out, lse)
 *
 * dsa_topk_sparse_mla_fwd runs the first two calls as two kernels (the top-k
 * also does the attention call's page lookup); dsa_sparse_mla_topk_fwd runs
 * them as one kernel.  Both give the two calls' results bit for bit.
 *
 * Sources (page titles):
 *  [LMSYS]  "Accelerating GLM-5.3-Flash on H200: High-Throughput Disaggregated
 *           Serving": section 1 "Architecture and workloads" (an indexer picks
 *           historical positions, DSA attends to them), section 2 "KV-only
 *           decode RadixCache" (prefix KV pages shared across requests),
 *           section 3 "Larger KV tiles for DSA Partial" and Figure 4 (the
 *           Partial step computes QK^T, online softmax and the weighted value
 *           sum over the selected positions; KV splits need a Combine step).
 *  [vLLM]   "GLM-5.3 Optimizations, Part 2: PCP, DCP, and Hybrid HiSparse on
 *           16 H200s", "Interpretation" (MLA's latent KV row is shared by all
 *           64 heads).
 *  [SGLang] GLM-5.3-Flash cookbook, "Size both memory pools" (paged KV pool)
 *           and "Keep the KV and DSA backends paired" (FP8 E4M3 KV cache on
 *           Blackwell).
 *
 * Conventions shared by every entry point:
 *  - All pointers except those documented as host pointers are DEVICE
 *    pointers.  The caller owns every buffer; the library allocates no device
 *    memory, keeps no per-call state and is reentrant.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; the call returns after argument checks and
 *    kernel launch.
 *  - Argument errors are reported synchronously through the return value and
 *    nothing is launched.  A failed launch returns DSA_ERR_CUDA.
 *  - Data-dependent errors (an index or page id out of range, a bad query
 *    position, an expired wait) never trap the GPU: the kernel ORs a bit
 *    (DSA_DEV_*) into `*dev_status` (an int32 in device memory, may be NULL)
 *    and the offending row contributes nothing.
 *  - Supported (heads, d_latent, d_rope): (16, 64, 16) and (64, 512, 64).
 *    A KV row is d_latent + d_rope FP8 E4M3 bytes (a multiple of 16) with one
 *    fp32 scale per token; K is the whole row, V its first d_latent bytes.
 */
#ifndef DSA_SPARSE_MLA_H_
#define DSA_SPARSE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad alignment */
  DSA_ERR_UNSUPPORTED_SHAPE = 2, /* (heads, d_latent, d_rope) not compiled in */
  DSA_ERR_WORKSPACE_TOO_SMALL = 3,
  DSA_ERR_CUDA = 4, /* a CUDA runtime call or kernel launch failed */
  DSA_ERR_OUT_OF_PAGES = 5 /* the page pool has no free or evictable page left */
} dsa_status;

/* Bits ORed into *dev_status by the kernels. */
#define DSA_DEV_BAD_QPOS 1u  /* q_pos[i] < 0 or >= ld_scores: the row selects nothing */
#define DSA_DEV_BAD_INDEX 2u /* idx entry < -1, or its page slot is past the block table row */
#define DSA_DEV_BAD_PAGE 4u  /* block table entry < 0 or >= num_pages, or q_req out of range */
#define DSA_DEV_TIMEOUT 8u   /* a bounded wait inside a kernel expired */

/* Static description of a status code (never NULL). */
DSA_API const char* dsa_status_string(int32_t status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
DSA_API int32_t dsa_version(void);

/*
 * dsa_topk_select -- causal top-k over fp32 indexer scores.
 * [LMSYS] section 3: the Partial step loads the KV positions the indexer
 * chose; [LMSYS] section 1: the indexer picks relevant historical positions.
 *
 * For each query row i (0 <= i < num_q) the visible positions are
 * 0..q_pos[i] (causal).  The call writes idx[i, 0:k] (int32, row-major,
 * device) = the min(k, q_pos[i] + 1) visible positions with the largest
 * scores[i, :], ranked by (score descending, position ascending) -- equal
 * scores go to the lower position and -0.0 equals +0.0 -- listed in
 * ascending position order, followed by -1 padding.  NaN scores are not
 * allowed (the result is unspecified but stays in range).
 *
 *   scores     fp32 [num_q, ld_scores], row stride ld_scores elements.
 *   q_pos      int32 [num_q]; q_pos[i] must lie in [0, ld_scores).
 *   idx        int32 [num_q, k] output.
 *   workspace  optional device scratch (caller-owned, no alignment beyond
 *              4 bytes).  Rows longer than 65,536 positions use it when
 *              dsa_topk_workspace_size() > 0: each 65,536-position slice
 *              writes its own top k there and a second pass merges them.
 *              NULL with workspace_bytes = 0 selects the slower in-place
 *              path instead; both give the same indices.
 * Errors: num_q < 0, k <= 0, ld_scores <= 0, null pointers -> INVALID_ARG;
 * 0 < workspace_bytes < dsa_topk_workspace_size() -> WORKSPACE_TOO_SMALL;
 * q_pos out of range -> dev bit DSA_DEV_BAD_QPOS and a row of -1.
 */
DSA_API dsa_status dsa_topk_select(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t num_q,
                           int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);

/* Workspace bytes dsa_topk_select can use for these sizes: num_q x slices x k x 8
 * when ld_scores > 65,536 and slices x k <= 65,536 (slices = ceil(ld_scores /
 * 65,536)), else 0. */
DSA_API size_t dsa_topk_workspace_size(int32_t num_q, int64_t ld_scores, int32_t k);

/*
 * dsa_sparse_mla_fwd -- the DSA "Partial" step: sparse MLA attention of every
 * head of each query token over its selected latent-KV rows.
 * [LMSYS] section 3 "Larger KV tiles for DSA Partial": loads the selected KV
 * positions and computes QK^T, online softmax and the weighted value sum;
 * [vLLM] "Interpretation": one latent KV row serves all heads; [SGLang]: FP8
 * E4M3 paged KV.
 *
 * For query token i, request r = q_req[i], head h and every selected
 * position p = idx[i, j] != -1:
 *   slot  = block_table[r * bt_stride + p / page_size] * page_size + p % page_size
 *   x_d   = e4m3(kv[slot, d]) * kv_scale[slot]                 (d < dqk)
 *   z_p   = softmax_scale * sum_d q[i, h, d] * x_d
 *   out[i, h, :] = sum_p softmax(z)_p * x[:d_latent],   lse[i, h] = ln sum_p exp(z_p)
 * A token with no selected rows gets out = 0 and lse = -inf.
 *
 *   q            bf16 [num_q, heads, dqk] (dqk = d_latent + d_rope), 16-byte aligned.
 *   kv           e4m3 bytes [num_pages * page_size, dqk], 16-byte aligned.
 *   kv_scale     fp32 [num_pages * page_size].
 *   block_table  int32 [num_req, bt_stride] page ids; rows may share pages.
 *   q_req        int32 [num_q] request of each query token, in [0, num_req).
 *   idx          int32 [num_q, k] selected positions (-1 = none), any order.
 *   num_splits   1..64.  With 1 the call writes out (bf16 [num_q, heads,
 *                d_latent], 16-byte aligned) and lse (fp32 [num_q, heads]).  With S > 1 the k
 *                entries of each row are cut into S contiguous chunks of whole
 *                KV tiles and the call writes o_part (fp32 [S, num_q, heads,
 *                d_latent]) and lse_part (fp32 [S, num_q, heads]) instead, to
 *                be merged by dsa_combine; out and lse may then be NULL.
 *   workspace    device scratch of at least dsa_sparse_mla_workspace_size()
 *                bytes, 8-byte aligned (NULL allowed when that size is 0).
 *                Its contents are overwritten; no state survives the call.
 * Errors: see the conventions above; a workspace that is too small returns
 * DSA_ERR_WORKSPACE_TOO_SMALL; a pool of 2^31 or more token slots returns
 * DSA_ERR_UNSUPPORTED_SHAPE; page ids or indices out of range set
 * DSA_DEV_BAD_INDEX / DSA_DEV_BAD_PAGE and that row is skipped.
 */
DSA_API dsa_status dsa_sparse_mla_fwd(const void* q, const uint8_t* kv, const float* kv_scale, int64_t num_pages,
                                      const int32_t* block_table, int32_t num_req, int32_t bt_stride,
                                      const int32_t* q_req, const int32_t* idx, int32_t num_q, int32_t num_heads,
                                      int32_t d_latent, int32_t d_rope, int32_t page_size, int32_t k,
                                      float softmax_scale, int32_t num_splits, void* out, float* lse, float* o_part,
                                      float* lse_part, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                      void* stream);

/* Scratch bytes dsa_sparse_mla_fwd needs (8 bytes per selected entry on the
 * tensor-core path: the resolved slot and scale of each position; 0 for
 * shapes served by the CUDA-core kernel). */
DSA_API size_t dsa_sparse_mla_workspace_size(int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope,
                                             int32_t k);

/*
 * dsa_sparse_mla_fwd_noalloc -- dsa_sparse_mla_fwd for callers that cannot
 * allocate device memory.  The pages describe no such call; it exists for
 * callers such as serving loops that reserve all device memory at start-up
 * and forbid later allocations (cudaMalloc can synchronise the device), or
 * plug-in hosts that offer no allocator.
 *
 * Same arguments, layouts, results and errors as dsa_sparse_mla_fwd, minus
 * the workspace: the scratch lives in a fixed 24 MiB array of device memory
 * inside the library (one per GPU, held until the process exits).  Only the
 * tensor-core shape (64, 512, 64) is accepted.  Calls needing more than 24
 * MiB of scratch (dsa_sparse_mla_workspace_size) return
 * DSA_ERR_WORKSPACE_TOO_SMALL without launching anything.  All calls share
 * the array: calls whose GPU work overlaps (unordered streams, concurrent
 * host threads) race and must be serialised by the caller.  The first call on
 * a device, made with that device current, looks up the array's device
 * address; make it before any stream capture on that device.  That address
 * is kept for the life of the process: do not call this entry point again
 * after a device reset (cudaDeviceReset, or a reset of the primary context),
 * which moves the array.  The call allocates nothing.
 */
DSA_API dsa_status dsa_sparse_mla_fwd_noalloc(const void* q, const uint8_t* kv, const float* kv_scale,
                                              int64_t num_pages, const int32_t* block_table, int32_t num_req,
                                              int32_t bt_stride, const int32_t* q_req, const int32_t* idx,
                                              int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope,
                                              int32_t page_size, int32_t k, float softmax_scale, int32_t num_splits,
                                              void* out, float* lse, float* o_part, float* lse_part,
                                              int32_t* dev_status, void* stream);

/*
 * dsa_sparse_mla_topk_fwd -- dsa_topk_select followed by dsa_sparse_mla_fwd
 * with one KV split, in a single kernel: each CTA selects its own query
 * token's top k and then attends to it.  Same results, bit for bit, as the
 * two calls; [LMSYS] section 3 (the indexer's selection feeds the Partial
 * step): the selection of one token's row does not wait for every other
 * row's, and no kernel boundary separates the two steps.  Measured on GB300
 * the two calls are nevertheless faster on every decode, verify and prefill
 * shape tried: this kernel's selection and tile loop run a little slower,
 * and it cannot split the KV range, which small batches need; this call is
 * for callers that want one launch.
 *
 * Arguments are those of the two calls: scores, ld_scores, q_pos and k as
 * for dsa_topk_select (ld_scores at most 65,536), idx is written as that call
 * writes it, the rest as for dsa_sparse_mla_fwd with num_splits = 1 (out is
 * required, lse may be NULL).  Only the tensor-core shape (64, 512, 64) and
 * k <= dsa_sparse_mla_topk_max_k() are accepted; anything else returns
 * DSA_ERR_UNSUPPORTED_SHAPE.  The workspace is dsa_sparse_mla_workspace_size()
 * bytes.  A bad q_pos sets DSA_DEV_BAD_QPOS, gives a row of -1 and that
 * token out = 0, lse = -inf.
 */
DSA_API dsa_status dsa_sparse_mla_topk_fwd(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t k,
                                           int32_t* idx, const void* q, const uint8_t* kv, const float* kv_scale,
                                           int64_t num_pages, const int32_t* block_table, int32_t num_req,
                                           int32_t bt_stride, const int32_t* q_req, int32_t num_q, int32_t num_heads,
                                           int32_t d_latent, int32_t d_rope, int32_t page_size, float softmax_scale,
                                           void* out, float* lse, void* workspace, size_t workspace_bytes,
                                           int32_t* dev_status, void* stream);

/* Largest k dsa_sparse_mla_topk_fwd accepts. */
DSA_API int32_t dsa_sparse_mla_topk_max_k(void);

/*
 * dsa_topk_sparse_mla_fwd -- dsa_topk_select followed by dsa_sparse_mla_fwd,
 * with the attention call's first step (each selected position's page and
 * dequantisation scale, looked up in the block table) done by the top-k
 * kernel as it writes its indices: two kernels instead of three, the
 * attention kernel a programmatic dependent of the top-k.  [LMSYS] section 3:
 * the indexer's selection feeds the Partial step.  Same results, bit for bit,
 * as the two calls, including dev_status: a bad q_pos sets DSA_DEV_BAD_QPOS;
 * a position past the block table row DSA_DEV_BAD_INDEX; a page id or q_req
 * out of range DSA_DEV_BAD_PAGE; such entries are attended as padding.
 *
 * Arguments are those of the two calls: scores, ld_scores, q_pos, k and idx
 * as for dsa_topk_select (ld_scores at most 65,536), the rest as for
 * dsa_sparse_mla_fwd (num_splits = 1 writes out / lse; num_splits > 1 writes
 * o_part / lse_part for dsa_combine).  The workspace is
 * dsa_sparse_mla_workspace_size() bytes (it receives the looked-up entries).
 * Only the tensor-core shape (64, 512, 64) with ld_scores <= 65,536 is
 * accepted; anything else returns DSA_ERR_UNSUPPORTED_SHAPE (the two calls
 * take every shape).
 */
DSA_API dsa_status dsa_topk_sparse_mla_fwd(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t k,
                                           int32_t* idx, const void* q, const uint8_t* kv, const float* kv_scale,
                                           int64_t num_pages, const int32_t* block_table, int32_t num_req,
                                           int32_t bt_stride, const int32_t* q_req, int32_t num_q, int32_t num_heads,
                                           int32_t d_latent, int32_t d_rope, int32_t page_size, float softmax_scale,
                                           int32_t num_splits, void* out, float* lse, float* o_part,
                                           float* lse_part, void* workspace, size_t workspace_bytes,
                                           int32_t* dev_status, void* stream);

/*
 * dsa_combine -- the DSA "Combine" step: exact log-sum-exp merge of split-KV
 * partial results.  [LMSYS] section 3: KV splits add intermediate writes and
 * Combine work.
 *   lse[i, h] = ln sum_s exp(lse_part[s, i, h])
 *   out[i, h, :] = sum_s exp(lse_part[s, i, h] - lse[i, h]) * o_part[s, i, h, :]
 * Splits with lse_part = -inf are empty and ignored; if all are, out = 0 and
 * lse = -inf.  o_part fp32 [S, num_q, heads, d_v]; lse_part fp32 [S, num_q,
 * heads]; out bf16 [num_q, heads, d_v]; lse fp32 [num_q, heads] (may be NULL).
 * d_v must be a multiple of 4 and o_part 16-byte aligned.
 */
DSA_API dsa_status dsa_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t num_q,
                       int32_t num_heads, int32_t d_v, void* out, float* lse, void* stream);

/*
 * dsa_kv_write -- store new latent+rope KV rows into the paged FP8 cache: the
 * write side of the rows that dsa_sparse_mla_fwd gathers.
 *
 * "Accelerating GLM-5.3-Flash on H200", section 2 "KV-only decode
 * RadixCache": rows live in a paged pool, mapped per request by a block
 * table (shared prefix pages appear in several tables).  SGLang cookbook page
 * for GLM-5.3-Flash, "Keep the KV and DSA backends paired": the cache is FP8
 * E4M3.  Row i is quantised with one fp32 scale per token: amax = max |x|,
 * scale = amax / 448, byte_j = E4M3(x_j / scale) rounded to nearest even and
 * saturated (both divisions IEEE fp32); an all-zero row stores scale 0 and
 * zero bytes.  It is stored at slot = block_table[req[i]][pos[i] / page_size]
 * * page_size + pos[i] % page_size.
 *
 *   rows         bf16 [n, d_qk] new rows (latent then rope), 16-byte aligned.
 *   req, pos     int32 [n] request (0..num_req-1) and position of each row.
 *   block_table  int32 [num_req, bt_stride] page ids (0..num_pages-1).
 *   kv           uint8 [num_pages * page_size, d_qk] the cache, 16-byte
 *                aligned; only the rows' slots are written.
 *   kv_scale     fp32 [num_pages * page_size]; only the rows' slots are written.
 *   d_qk         a multiple of 16, at most 2048.
 * Errors: DSA_ERR_INVALID_ARG for bad sizes, null or misaligned pointers
 * (nothing is launched); a request or page id out of range sets
 * DSA_DEV_BAD_PAGE, a position outside the block table row sets
 * DSA_DEV_BAD_INDEX, and that row is skipped.  Rows aimed at the same slot
 * leave one of them there, unspecified which.  Asynchronous on `stream`.
 */
DSA_API dsa_status dsa_kv_write(const void* rows, int32_t n, int32_t d_qk, const int32_t* req, const int32_t* pos,
                                const int32_t* block_table, int32_t num_req, int32_t bt_stride, int32_t page_size,
                                int64_t num_pages, uint8_t* kv, float* kv_scale, int32_t* dev_status, void* stream);

/*
 * KV-only prefix-sharing page allocator (host side, no GPU involved).
 *
 * "Accelerating GLM-5.3-Flash on H200", section 2 "KV-only decode
 * RadixCache": requests sharing a prefix share its KV pages, so N requests
 * with a common prefix of Lp tokens and private suffixes of Ls tokens occupy
 * Lp + N·Ls slots instead of N·(Lp + Ls).  The unit of sharing is a whole
 * page whose tokens, and all tokens before it, match (KV rows depend on the
 * whole causal prefix); the block tables it returns are the ones
 * dsa_kv_write and dsa_sparse_mla_fwd take.
 *
 * dsa_prefix_cache_create: a cache over a pool of num_pages pages of
 *   page_size tokens (page ids 0..num_pages-1).  NULL on bad sizes or when
 *   out of host memory.  The caller owns the handle (dsa_prefix_cache_destroy).
 * dsa_prefix_cache_acquire: pages for a request of n_tokens token ids.
 *   block_table (int32 [max_pages], host memory) receives ceil(n_tokens /
 *   page_size) page ids: the first *n_shared are cached pages of the longest
 *   matching whole-page prefix (their KV is already in the cache), the rest
 *   are fresh (the caller writes their KV rows).  The request's new full pages
 *   are cached for later requests; a partial last page stays private.  Every
 *   page returned is referenced until released.  When no page is free,
 *   unreferenced cached pages are evicted, least recently used first (leaves
 *   of the prefix tree only); if none is left the call changes nothing and
 *   returns DSA_ERR_OUT_OF_PAGES.  max_pages too small: DSA_ERR_INVALID_ARG.
 * dsa_prefix_cache_release: drops the references of a block table acquire
 *   returned (n_pages entries).  Private pages become free; cached pages stay
 *   cached (reusable) until evicted.  An entry that is not a referenced page
 *   returns DSA_ERR_INVALID_ARG and releases nothing.
 * dsa_prefix_cache_stats: pages referenced by live requests, pages cached in
 *   the prefix tree (referenced or not), free pages.
 * The calls are thread-safe (one lock per cache).
 */
typedef struct dsa_prefix_cache dsa_prefix_cache;
DSA_API dsa_prefix_cache* dsa_prefix_cache_create(int32_t page_size, int32_t num_pages);
DSA_API void dsa_prefix_cache_destroy(dsa_prefix_cache* cache);
DSA_API dsa_status dsa_prefix_cache_acquire(dsa_prefix_cache* cache, const int32_t* tokens, int64_t n_tokens,
                                            int32_t* block_table, int32_t max_pages, int32_t* n_pages,
                                            int32_t* n_shared);
DSA_API dsa_status dsa_prefix_cache_release(dsa_prefix_cache* cache, const int32_t* block_table, int32_t n_pages);
DSA_API dsa_status dsa_prefix_cache_stats(dsa_prefix_cache* cache, int32_t* pages_referenced, int32_t* pages_cached,
                                          int32_t* pages_free);

/*
 * Host-side planning helpers (no GPU needed).
 *
 * dsa_kv_tile_count: KV tiles of `tile` entries that cover an index row of
 * `width` entries; the last tile is padded virtually, the index tensor is
 * unchanged ([LMSYS] Figure 4: width 2112 -> 66 tiles of 32 or 17 of 128,
 * 2176 virtual columns of which 64 are padding).
 *
 * dsa_pick_num_splits: KV splits per query token for the given launch.  KV
 * splits are added only while query tokens alone leave SMs idle ([LMSYS]
 * section 3: splits cost intermediate writes and Combine work, so they are
 * used only when query parallelism is insufficient).  num_sms <= 0 queries
 * the current device.
 */
DSA_API int32_t dsa_kv_tile_count(int32_t width, int32_t tile);
DSA_API int32_t dsa_kv_tile_size(int32_t num_heads, int32_t d_latent, int32_t d_rope);
DSA_API int32_t dsa_pick_num_splits(int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope, int32_t k,
                            int32_t num_sms);

#ifdef __cplusplus
}
#endif

#endif /* DSA_SPARSE_MLA_H_ */
