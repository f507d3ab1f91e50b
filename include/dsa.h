/*
 * dsa.h -- C ABI of libdsa.so, the GB300 (sm_103a) decode hot path of
 * DeepSeek Sparse Attention (DSA).
 *
 * The path, for each decode query token t of a batch of requests:
 *   1. lightning indexer: I[t,s] = sum_j w[t,j] * ReLU(q^I[t,j] . k^I[s]) over
 *      64 FP8 heads of 128 dims, for every cached token s it can see
 *      ("MTP and sparse attention: NSA and DSA", section "Sparse attention:
 *      NSA and DSA");
 *   2. top-k: the k (= 2048) highest-scoring tokens (same section; "Multi-layer
 *      Indexer" abstract);
 *   3. sparse MLA over only those tokens against the latent cache (576 dims =
 *      kv_lora_rank 512 + rope 64; V = the first 512 dims), as split-KV
 *      partials Mid_O / Mid_O_LogExpSum ("Deepseek Details", section "DSA",
 *      stage 2; "[SGLang] NSA", section "forward_decode");
 *   4. a cross-split online-softmax merge ("Deepseek Details", section "DSA",
 *      stage 3).
 *
 * Conventions for every call:
 *   - Buffers are owned by the caller.  Pointers marked [dev] are device
 *     pointers on the current CUDA device; the library allocates no memory and
 *     keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  They never synchronise, except
 *     dsa_get_device_error.
 *   - Host-detectable errors (null or misaligned pointers, unsupported sizes,
 *     a short workspace) are returned before anything is launched.  Errors the
 *     kernels detect (a page id outside the cache, an index outside the visible
 *     range, a bounded wait that ran out) are recorded in a device-side error
 *     word and read with dsa_get_device_error; the offending access is skipped.
 *   - Layouts are row-major and contiguous.  Query rows are ordered
 *     request-major: row t = r * q_per_req + i is query i of request r.
 *   - Request r holds seqlens[r] cached tokens, its q_per_req new tokens
 *     included.  Query i of request r sees
 *         vis[t] = seqlens[r] - (q_per_req - 1 - i)
 *     tokens, logical positions [0, vis[t])  ("[SGLang] NSA", section
 *     "init_forward_metadata": 3 query tokens over 10 cached tokens see 8, 9,
 *     10).
 *   - Both caches are paged with 64 tokens per page and share one page table:
 *     logical position s of request r lives in cache row
 *         page_table[r * max_pages + s / 64] * 64 + s % 64.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer or out-of-range size   */
  DSA_ERR_UNSUPPORTED = 2,   /* a size this build does not implement           */
  DSA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required     */
  DSA_ERR_CUDA = 4,          /* a CUDA runtime call failed                      */
  DSA_ERR_DEVICE_CHECK = 5,  /* a kernel found a bad page id / index (skipped)  */
  DSA_ERR_TIMEOUT = 6        /* a kernel's bounded wait ran out                 */
} dsa_status;

#define DSA_INDEX_HEADS 64   /* lightning-indexer heads                     */
#define DSA_INDEX_DIM 128    /* indexer head / key dim (FP8 E4M3 bytes)     */
#define DSA_LATENT_DIM 576   /* latent row: kv_lora_rank 512 + rope 64      */
#define DSA_V_DIM 512        /* value dims: the first 512 of the latent row */
#define DSA_PAGE_SIZE 64     /* tokens per cache page                       */
#define DSA_MAX_TOPK 2048
#define DSA_MAX_BATCH 1024
#define DSA_MAX_Q_PER_REQ 4

/*
 * One decode batch.  Sizes are host integers; seqlens and page_table are
 * device arrays read by the kernels.
 *   batch      B requests, 1 <= B <= DSA_MAX_BATCH.
 *   q_per_req  n_q = 1 + MTP draft tokens, 1 <= n_q <= 4.  T = B * n_q rows.
 *   num_heads  MLA query heads H: 16, 32, 48, ..., 128.
 *   topk       k, 1 <= k <= 2048.
 *   page_size  must be 64.
 *   max_pages  columns of page_table (>= ceil(max seqlen / 64)).
 *   num_pages  pages in each cache; rows = num_pages * 64.  Page ids outside
 *              [0, num_pages) are reported as DSA_ERR_DEVICE_CHECK.
 *   seqlens    [dev] int32 [B], each >= q_per_req (so every query sees itself).
 *   page_table [dev] int32 [B, max_pages].  Entries past a request's last page
 *              are never read.
 */
typedef struct dsa_decode_desc {
  int32_t batch;
  int32_t q_per_req;
  int32_t num_heads;
  int32_t topk;
  int32_t page_size;
  int32_t max_pages;
  int32_t num_pages;
  const int32_t* seqlens;
  const int32_t* page_table;
} dsa_decode_desc;

/*
 * Stage 1 -- lightning-indexer logits ("MTP and sparse attention: NSA and
 * DSA", section "Sparse attention: NSA and DSA", the index score
 * I[t,s] = sum_j w[t,j] ReLU(q^I[t,j] . k^I[s]), computed in FP8).
 *
 * With the FP8 values dequantised by their per-token scales,
 *   logits[t*ld + s] = k_scale[row(s)] * sum_j (w[t,j] * q_scale[t]) *
 *                      ReLU(sum_d q_fp8[t,j,d] * k_fp8[row(s),d])
 * for s < vis[t] (both scales must be positive, so they factor out of the
 * ReLU); fp32 result, FP8 x FP8 products accumulated in fp32 on tensor cores.
 * Entries s >= vis[t] inside the last 128-token tile are written -inf; the rest
 * of the row is not touched.
 *   q_fp8   [dev] uint8 [T, 64, 128]  FP8 E4M3 index queries, 16-B aligned
 *   q_scale [dev] float [T]           per query token, > 0
 *   w       [dev] float [T, 64]       per-head weights
 *   k_fp8   [dev] uint8 [num_pages*64, 128] FP8 E4M3 index-key cache, 16-B aligned
 *   k_scale [dev] float [num_pages*64] per cached token, > 0, 16-B aligned
 *   logits  [dev] float [T, ld_logits]; ld_logits >= max_pages*64, multiple of 4
 */
dsa_status dsa_indexer_logits(const dsa_decode_desc* desc, const uint8_t* q_fp8,
                              const float* q_scale, const float* w,
                              const uint8_t* k_fp8, const float* k_scale,
                              float* logits, int64_t ld_logits, void* stream);

/*
 * Stage 2 -- per-query top-k ("Sparse attention: NSA and DSA": each query keeps
 * the 2048 highest-scoring tokens; "[SGLang] NSA", section "Fused Top-K
 * Transform", top-k over variable-length rows).
 *
 * Row t of topk_idx receives the n = min(k, vis[t]) positions s < vis[t] with
 * the largest logits[t*ld + s]; equal scores go to the lower position, -0.0
 * equals +0.0.  The n positions are written in ascending order at [0, n) and
 * the rest of the row is -1.  Exact: the set equals that of a full sort.
 * No full sort is done (radix select with shared-memory histograms; each row
 * is one cluster of 16 CTAs, launched with the non-portable cluster size).
 *   logits   [dev] float [T, ld_logits] (only s < vis[t] is read),
 *            ld_logits <= 524288 (else DSA_ERR_UNSUPPORTED)
 *   topk_idx [dev] int32 [T, k]
 *   ws       [dev] workspace of dsa_topk_workspace_bytes() bytes, 16-B aligned
 */
dsa_status dsa_topk(const dsa_decode_desc* desc, const float* logits, int64_t ld_logits,
                    int32_t* topk_idx, void* ws, size_t ws_bytes, void* stream);

size_t dsa_topk_workspace_bytes(const dsa_decode_desc* desc, int64_t ld_logits);

/*
 * dsa_topk without a workspace argument.  (A library convenience; the pages
 * have no counterpart.)
 *
 * For callers that cannot allocate device memory where they run the
 * selection: an inference-engine plugin or step function that executes after
 * the engine has reserved all of the device's memory for its caches, or a
 * host runtime without a device allocator of its own, where a cudaMalloc
 * would fail or stall the device.  The histogram and candidate
 * lists then live in a file-scope device array of fixed size (about 16.5 MB)
 * that every GPU loading this library reserves until the process exits.  No
 * call allocates or frees memory.
 *   Limits: T = batch * q_per_req <= 64, T * ld_logits <= 2^21 scores and
 *   ld_logits <= 524288 (as dsa_topk);
 *   larger batches return DSA_ERR_UNSUPPORTED (use dsa_topk with a workspace).
 *   Every call looks up the array's device address on the current device
 *   (the first lookup may load the library's device code); make the first
 *   call on a device before capturing the stream into a graph.
 *   All calls on a device share the one array: each call clears the parts
 *   that must start at zero, and calls that may run at the same time on the
 *   GPU (different streams, no ordering between them) race on it.
 * Arguments and results are those of dsa_topk.
 */
dsa_status dsa_topk_noalloc(const dsa_decode_desc* desc, const float* logits, int64_t ld_logits,
                            int32_t* topk_idx, void* stream);

/*
 * Stage 3 -- sparse MLA split partials ("Deepseek Details", section "DSA",
 * stage 2: each block of the selected tokens runs an online softmax and writes
 * Mid_O[batch, head, block, dim] and Mid_O_LogExpSum[batch, head, block];
 * absorbed MLA as in "[SGLang] NSA", section "forward_decode").
 *
 * Query row t reads positions [0, n) of topk_idx row t, n = min(k, vis[t]);
 * entries there that are < 0 or >= vis[t] are skipped.  Positions are cut into
 * num_splits blocks of C = 64 * ceil(ceil(k / num_splits) / 64) positions;
 * block b covers [b*C, (b+1)*C) clipped to n.  For block b and head h:
 *   x_s   = sm_scale * q[t,h,:] . kv[row(s),:]            (576 dims)
 *   Mid_O[t,h,b,:]  = sum_s softmax_b(x)_s * kv[row(s), 0:512]
 *   Mid_LSE[t,h,b]  = log(sum_s exp(x_s))                  (natural log)
 * An empty block writes Mid_O = 0 and Mid_LSE = -inf.  QK^T and PV run on
 * tcgen05 tensor cores in bf16 with fp32 accumulation; softmax in fp32.
 *   q        [dev] bf16 [T, H, 576] (q_nope 512 then q_rope 64), 16-B aligned
 *   kv       [dev] bf16 [num_pages*64, 576] latent cache, 16-B aligned
 *   topk_idx [dev] int32 [T, k] logical positions
 *   num_splits 1 .. ceil(k/64), or 0 for dsa_num_splits_auto()
 *   mid_o    [dev] float [T, H, num_splits, 512]
 *   mid_lse  [dev] float [T, H, num_splits]
 * With num_splits == 1, mid_o already is the final output.
 */
dsa_status dsa_sparse_mla_decode_split(const dsa_decode_desc* desc, const uint16_t* q,
                                       const uint16_t* kv, const int32_t* topk_idx,
                                       int32_t num_splits, float sm_scale, float* mid_o,
                                       float* mid_lse, void* stream);

/*
 * The step before stage 1 -- the cache write: every new token's latent row is
 * written into the paged MLA cache and its indexer key, quantised to FP8 E4M3
 * with one fp32 scale per token, into the indexer's key cache ("[SGLang] NSA
 * (Narrow Sparse Attention)", section "forward_decode": set_mla_kv_buffer
 * before the attention; its module list: quant_k_cache, the NSA-specific FP8
 * quantisation of the K cache; "MTP and sparse attention: NSA and DSA":
 * the indexer key, FP8 + scale).
 *   new_latent  [dev] bf16 [T, 576] (kv_lora 512 + rope 64), 16-byte aligned
 *   new_index_k [dev] bf16 [T, 128], 8-byte aligned
 *   kv          [dev] bf16 [num_pages * 64, 576], 16-byte aligned (written)
 *   k_fp8       [dev] E4M3 [num_pages * 64, 128], 4-byte aligned (written)
 *   k_scale     [dev] float [num_pages * 64] (written)
 * Row t = r * q_per_req + i is request r's token S_r - q_per_req + i (the
 * new tokens are the last q_per_req of seqlens[r]); its cache row is
 * page_table[r][pos / 64] * 64 + pos % 64.  Key: scale = amax / 448 over its
 * 128 values, codes = E4M3(k / scale) rounded to nearest even and saturated
 * at 448, in fp32 (a key of zeros: scale 1, zero codes).  Only those rows
 * are written.  A position outside the page table or a page id outside
 * [0, num_pages) skips the row and sets DSA_ERR_DEVICE_CHECK (read by
 * dsa_get_device_error).  Host-detected errors return before any launch.
 */
dsa_status dsa_cache_write(const dsa_decode_desc* desc, const uint16_t* new_latent,
                           const uint16_t* new_index_k, uint16_t* kv, uint8_t* k_fp8,
                           float* k_scale, void* stream);

/*
 * Stage 4 -- cross-split merge ("Deepseek Details", section "DSA", stage 3:
 * an online-softmax merge of the blocks' Mid_O and Mid_O_LogExpSum).
 * For each of the num_rows = T*H rows, with L = max_b mid_lse[b]:
 *   out = sum_b exp(mid_lse[b] - L) * mid_o[b] / sum_b exp(mid_lse[b] - L)
 *   out_lse = L + log(sum_b exp(mid_lse[b] - L))
 * Blocks with mid_lse = -inf are skipped; a row with none gives out = 0,
 * out_lse = -inf.
 *   mid_o [dev] float [num_rows, num_splits, 512]; mid_lse [dev] [num_rows, num_splits]
 *   out   [dev] float [num_rows, 512]; out_lse [dev] float [num_rows] or NULL
 */
dsa_status dsa_merge(int32_t num_rows, int32_t num_splits, const float* mid_o,
                     const float* mid_lse, float* out, float* out_lse, void* stream);

/*
 * The whole decode layer, stages 1-4 on one stream.
 * If topk_in is non-NULL, stages 1-2 are skipped and the layer attends the
 * given selection (the layer reuses another layer's top-k: "Multi-layer
 * Indexer" abstract, and "Sparse attention: NSA and DSA", section "New demands
 * on inference engines", reusing selections).  Otherwise the indexer and top-k
 * run and, if topk_out is non-NULL, the selection is also written there.
 * Requests whose every query sees <= k tokens select all of them, so their
 * indexer scan is skipped (the short-context dense fallback of the same page).
 *   out [dev] float [T, H, 512]
 *   ws  [dev] workspace of dsa_workspace_bytes(desc, max_seqlen, num_splits)
 * Other arguments as in the stage calls; max_seqlen bounds every seqlens[r].
 */
dsa_status dsa_decode_fused(const dsa_decode_desc* desc,
                            const uint8_t* q_fp8, const float* q_scale, const float* w,
                            const uint8_t* k_fp8, const float* k_scale,
                            const uint16_t* q, const uint16_t* kv,
                            const int32_t* topk_in, int32_t* topk_out,
                            float sm_scale, int32_t num_splits, int32_t max_seqlen,
                            float* out, void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_decode_fused with per-stage timing: stage_events[0..4] (cudaEvent_t
 * handles passed as void*, any of them NULL) are recorded on `stream` before
 * stage 1 (after the workspace clear that precedes the indexer), after stage 1
 * (indexer), after stage 2 (top-k), after stage 3 (sparse MLA) and after
 * stage 4 (merge).  With stage_events == NULL this is dsa_decode_fused.  When
 * topk_in is given, events 0, 1 and 2 mark the same point.
 */
dsa_status dsa_decode_fused_timed(const dsa_decode_desc* desc,
                                  const uint8_t* q_fp8, const float* q_scale, const float* w,
                                  const uint8_t* k_fp8, const float* k_scale,
                                  const uint16_t* q, const uint16_t* kv,
                                  const int32_t* topk_in, int32_t* topk_out,
                                  float sm_scale, int32_t num_splits, int32_t max_seqlen,
                                  float* out, void* ws, size_t ws_bytes, void* stream,
                                  void* const* stage_events);

/*
 * The cache write of the step's new tokens, then the layer: dsa_cache_write
 * followed by dsa_decode_fused on the same caches, in one call (the new
 * tokens' latent rows and FP8 index keys are written before the indexer reads
 * them: "[SGLang] NSA (Narrow Sparse Attention)", section "forward_decode",
 * set_mla_kv_buffer before the attention; "MTP and sparse attention: NSA and
 * DSA", section "Sparse attention: NSA and DSA", the indexer key in FP8 with
 * a scale).  The write shares a kernel with the workspace clear, and the
 * indexer waits for it only before the tiles that hold new tokens (a
 * request's last two 128-token tiles, since q_per_req <= 4).
 * Arguments: those of dsa_cache_write (new_latent, new_index_k; kv, k_fp8 and
 * k_scale are written, then read) and of dsa_decode_fused; the same alignment
 * rules and errors.  topk_in non-NULL: the write, then the attention over the
 * given selection.
 */
dsa_status dsa_decode_fused_write(const dsa_decode_desc* desc, const uint16_t* new_latent,
                                  const uint16_t* new_index_k,
                                  const uint8_t* q_fp8, const float* q_scale, const float* w,
                                  uint8_t* k_fp8, float* k_scale,
                                  const uint16_t* q, uint16_t* kv,
                                  const int32_t* topk_in, int32_t* topk_out,
                                  float sm_scale, int32_t num_splits, int32_t max_seqlen,
                                  float* out, void* ws, size_t ws_bytes, void* stream);

/*
 * FP8 latent cache ("[SGLang] NSA (Narrow Sparse Attention)", its module
 * list: quant_k_cache / dequant_k_cache, the NSA cache's own FP8
 * quantisation, read as FP8 by the attention to save bandwidth; "Deepseek
 * Details", section "FP8 Training": E4M3 with one scale per 1 x 128 tile).
 * Row layout, 656 bytes: bytes 0..511 the value dims 0..511 as E4M3 codes in
 * four 128-dim tiles, tile scale = amax / 448 in fp32 (a tile of zeros:
 * scale 1), codes = E4M3(x / scale) rounded to nearest even and saturated;
 * bytes 512..527 the four fp32 scales; bytes 528..655 the 64 rope dims as
 * bf16, unchanged.  The attention over such rows is the attention over their
 * dequantised values (code x scale).
 */

/*
 * Quantises `rows` bf16 latent rows kv [rows, 576] (16-byte aligned) into
 * FP8 rows kv8 [rows, 656] (16-byte aligned, written).  Both [dev].
 */
dsa_status dsa_latent_to_fp8(const uint16_t* kv, int64_t rows, uint8_t* kv8, void* stream);

/*
 * dsa_sparse_mla_decode_split over the FP8 latent cache kv8 [num_pages * 64,
 * 656] (16-byte aligned): the selected rows are gathered as FP8 and
 * dequantised in shared memory to bf16 for the tensor cores (each value
 * rounded once to bf16).  Other arguments, outputs and errors as there.
 */
dsa_status dsa_sparse_mla_decode_split_fp8(const dsa_decode_desc* desc, const uint16_t* q,
                                           const uint8_t* kv8, const int32_t* topk_idx,
                                           int32_t num_splits, float sm_scale, float* mid_o,
                                           float* mid_lse, void* stream);

/*
 * dsa_decode_fused with the latent cache in FP8 rows (kv8 as in
 * dsa_sparse_mla_decode_split_fp8); every other argument as there.
 */
dsa_status dsa_decode_fused_fp8kv(const dsa_decode_desc* desc,
                                  const uint8_t* q_fp8, const float* q_scale, const float* w,
                                  const uint8_t* k_fp8, const float* k_scale,
                                  const uint16_t* q, const uint8_t* kv8,
                                  const int32_t* topk_in, int32_t* topk_out,
                                  float sm_scale, int32_t num_splits, int32_t max_seqlen,
                                  float* out, void* ws, size_t ws_bytes, void* stream);

/*
 * One layer of the Multi-layer Indexer schedule ("Multi-layer Indexer:
 * Overlapping Selection and Attention in DeepSeek Sparse Attention",
 * abstract; "MTP and sparse attention: NSA and DSA", section "New demands on
 * inference engines", reusing selections): the layer's attention runs over
 * an earlier layer's selection (topk_prev) while the layer's own indexer and
 * top-k run and write the selection a later layer reuses (topk_next).  On
 * one stream: the workspace clear; the indexer (one CTA per SM) and its
 * top-k into topk_next, as in dsa_decode_fused; the attention over
 * topk_prev with num_splits splits (0: dsa_num_splits_mli), launched as the
 * top-k's programmatic dependent so that it runs on the SMs the
 * latency-bound top-k leaves free, beside it; the merge of its splits.
 *   topk_prev [dev] int32 [T, k]  the selection attended (like topk_in);
 *             complete before the call (written by earlier work on `stream`)
 *   topk_next [dev] int32 [T, k]  this layer's selection (like topk_out)
 *   ws        [dev] dsa_workspace_bytes(desc, max_seqlen, num_splits)
 *             (num_splits 0 there covers the split count chosen here)
 * Other arguments and errors as in dsa_decode_fused; the indexer inputs are
 * required.  `out` equals dsa_decode_fused with topk_in = topk_prev up to the
 * rounding of another split count, and topk_next equals the selection
 * dsa_decode_fused writes to topk_out, bit for bit.
 */
dsa_status dsa_decode_mli(const dsa_decode_desc* desc,
                          const uint8_t* q_fp8, const float* q_scale, const float* w,
                          const uint8_t* k_fp8, const float* k_scale,
                          const uint16_t* q, const uint16_t* kv,
                          const int32_t* topk_prev, int32_t* topk_next,
                          float sm_scale, int32_t num_splits, int32_t max_seqlen,
                          float* out, void* ws, size_t ws_bytes, void* stream);

/* The attention's split count dsa_decode_mli picks when 0 is passed: its CTAs
 * (two per split and row) take about 58 % of the SMs (the top-k beside it
 * holds up to ~40 %), at least one split per row, at most ceil(k/64). */
int32_t dsa_num_splits_mli(const dsa_decode_desc* desc);

/*
 * A decode step whose inputs start in host memory and whose output ends
 * there.  What changes from one step to the next (index queries and their
 * scales, head weights, MLA queries, seqlens, page table) is packed in one
 * block, so that it crosses the host link in one copy; the caches and the
 * workspace stay in device memory (model state and scratch).  The pages
 * give no host interface; this packing is the library's.
 *
 * dsa_step_layout_get: byte offsets of each input in the block, for
 * B = batch requests, T = B * q_per_req rows, H = num_heads:
 *   q_fp8      uint8 [T, 64, 128]        q_scale  float [T]
 *   w          float [T, 64]             q        bf16  [T, H, 576]
 *   seqlens    int32 [B]                 page_table int32 [B, max_pages]
 * Every offset is a multiple of 256; `bytes` is the block size.
 * DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED for sizes the decode calls reject.
 */
typedef struct dsa_step_layout {
  size_t q_fp8, q_scale, w, q, seqlens, page_table;
  size_t bytes;
} dsa_step_layout;

dsa_status dsa_step_layout_get(int32_t batch, int32_t q_per_req, int32_t num_heads,
                               int32_t max_pages, dsa_step_layout* layout);

/*
 * One decode layer from host buffers, queued on `stream`:
 *   1. host_in -> dev_in, one copy of layout.bytes;
 *   2. dsa_decode_fused over the inputs in dev_in (the seqlens and page_table
 *      fields of desc are ignored: they are taken from dev_in);
 *   3. out -> host_out, one copy of T * H * 512 floats (skipped if host_out
 *      is NULL).
 *   host_in   [host] the block laid out by dsa_step_layout_get(desc's sizes).
 *             Page-locked memory (cudaHostAlloc, cudaHostRegister) keeps the
 *             copies asynchronous; with pageable memory they still happen but
 *             the call may block until they are done.
 *   dev_in    [dev]  layout.bytes, 256-byte aligned; overwritten by the copy.
 *   host_out  [host] float [T, H, 512]; valid once `stream` has passed the call.
 * k_fp8, k_scale, kv, sm_scale, num_splits, max_seqlen, out, ws and ws_bytes
 * as in dsa_decode_fused.  Every argument is checked before the first copy
 * is queued; the errors are those of dsa_decode_fused.
 */
dsa_status dsa_decode_step_host(const dsa_decode_desc* desc, const void* host_in, void* dev_in,
                                const uint8_t* k_fp8, const float* k_scale, const uint16_t* kv,
                                float sm_scale, int32_t num_splits, int32_t max_seqlen,
                                float* out, float* host_out, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * Decode steps from host buffers with the copies of one step overlapping the
 * layers of its neighbours (the pages give no host interface; this is the
 * library's).  Every resource is the caller's: two device input blocks and
 * two device outputs that alternate between steps, the workspace, a stream
 * for the host-to-device copies, one for the device-to-host copies, and six
 * events (cudaEvent_t, e.g. created with cudaEventDisableTiming).  Step i
 * uses slot b = i % 2:
 *   1. on copy_in_stream: wait for the layer of step i - 2 (ev_done[b]), copy
 *      host_in -> dev_in[b] (layout.bytes), record ev_in[b];
 *   2. on `stream`: wait for ev_in[b] and for the output copy of step i - 2
 *      (ev_out[b]), run dsa_decode_fused over dev_in[b] into out[b], record
 *      ev_done[b];
 *   3. on copy_out_stream: wait for ev_done[b], copy out[b] -> host_out
 *      (T * H * 512 floats), record ev_out[b].
 * So while the layer of step i runs, the inputs of step i + 1 come in and
 * the output of step i - 1 goes out.  host_in may be rewritten once ev_in[b]
 * has completed; host_out is valid once ev_out[b] has.  `step` is the count
 * of steps submitted so far (start at 0; the call increments it); every step
 * of one ring runs its layer on the same `stream` (the steps share one
 * workspace).
 */
typedef struct dsa_step_ring {
  void* dev_in[2];          /* [dev] layout.bytes each, 256-byte aligned          */
  float* out[2];            /* [dev] float [T, H, 512] each, 16-byte aligned       */
  void* ws;                 /* [dev] dsa_workspace_bytes(desc, max_seqlen, splits) */
  size_t ws_bytes;
  void* copy_in_stream;     /* cudaStream_t of the host-to-device copies           */
  void* copy_out_stream;    /* cudaStream_t of the device-to-host copies           */
  void* ev_in[2];           /* cudaEvent_t: input block b copied in                */
  void* ev_done[2];         /* cudaEvent_t: the layer of slot b done               */
  void* ev_out[2];          /* cudaEvent_t: output b copied out                    */
  int64_t step;             /* steps submitted so far                              */
} dsa_step_ring;

/*
 * Queues one step of `ring` as described above.  desc gives the sizes (its
 * seqlens and page_table fields are ignored: they are taken from dev_in[b]);
 * host_in [host] is the step's block laid out by dsa_step_layout_get,
 * host_out [host] float [T, H, 512] (page-locked memory keeps the copies
 * asynchronous).  Other arguments as in dsa_decode_fused.  Every argument is
 * checked before anything is queued; DSA_ERR_INVALID_ARG for a null event,
 * buffer or misaligned block, else the errors of dsa_decode_fused.
 */
dsa_status dsa_decode_step_ring(const dsa_decode_desc* desc, dsa_step_ring* ring,
                                const void* host_in, float* host_out, const uint8_t* k_fp8,
                                const float* k_scale, const uint16_t* kv, float sm_scale,
                                int32_t num_splits, int32_t max_seqlen, void* stream);

/* Workspace bytes dsa_decode_fused needs (num_splits 0 = auto). */
size_t dsa_workspace_bytes(const dsa_decode_desc* desc, int32_t max_seqlen,
                           int32_t num_splits);

/* The split count the library picks when 0 is passed: enough CTAs to cover the
 * GPU's SMs at one CTA per SM, at most ceil(k/64). */
int32_t dsa_num_splits_auto(const dsa_decode_desc* desc);

/* Human-readable name of a status code (static storage). */
const char* dsa_status_str(dsa_status status);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: DSA_OK, DSA_ERR_DEVICE_CHECK or DSA_ERR_TIMEOUT (or
 * DSA_ERR_CUDA if the synchronisation itself failed). */
dsa_status dsa_get_device_error(void* stream);

/*
 * Test hook for the timeout path (a library facility; the pages have no
 * counterpart).  Sets the bound, in SM cycles, on the waits of the indexer
 * kernel's pipeline (copy engine -> tensor cores -> epilogue) for the
 * launches that follow; 0 restores the default (about 1.5 s of SM cycles).
 * With a bound of a few cycles a wait runs out: the kernel records
 * DSA_ERR_TIMEOUT (read with dsa_get_device_error), stops its pipeline, waits
 * with the default bound for its copies already in flight, frees its tensor
 * memory and returns, and the CUDA context stays usable.  Process-wide;
 * DSA_ERR_INVALID_ARG for a negative value.
 */
dsa_status dsa_debug_set_wait_cycles(int64_t cycles);

/* Library version string. */
const char* dsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
