/*
 * bskv.h - C ABI of libbskv: attention restricted to a CSR-indexed key set on one GB300.
 *
 * Three index forms, one idea: each query row (or row block) attends only to the keys
 * named by a CSR-style index.
 *   - paged-KV decode page table (kv_indptr, kv_indices, kv_last_page_len, page_size),
 *     with split-KV partial states merged by log-sum-exp;
 *   - BSR block-sparse mask (indptr, indices, M, N, R, C) with grouped-query heads;
 *   - sparse MLA decode over FP8 E4M3 rows of 576 values (512 latent + 64 rotated),
 *     fed by the fused RoPE + FP8 prologue.
 *
 * Sources (web pages, by title and section):
 *   [SPARSE]  "flashinfer.sparse - FlashInfer 0.7.4 documentation",
 *             BlockSparseAttentionWrapper (__init__, plan, run).
 *   [MLA]     "Sparse MLA" (MATE 0.2.6 API docs): mla_rope_quantize_fp8,
 *             sparse_mla_fp8_decode, get_batch_decode_metadata_mla.
 *   [WRAP]    "FlashInfer Compatibility Wrapper" (MATE 0.2.6 docs): RoPE and FP8
 *             quantization; Sparse MLA decode; Metadata reuse.
 *   [SKILL]   "FlashInfer" agent-skill summary: KV-Cache Formats (paged KV-cache),
 *             Cascade Inference, Roofline Analysis.
 *   [CHEAT]   FlashInfer cheat page: docs/api/cascade.rst (merge_state(s)); README
 *             (its production notes: the library is meant to run under CUDA graphs).
 *
 * Conventions (all entry points):
 *   - Every function returns a bskv_status. Unsupported shapes, dtypes, layouts and
 *     sizes fail explicitly ([WRAP] Sparse MLA decode) with a status and a message
 *     readable through bskv_last_error_message(); nothing is launched then.
 *   - All device memory is owned by the caller: inputs, outputs and the int/float
 *     workspaces ([SPARSE] __init__: a user-reserved float workspace holds the
 *     intermediate results of the split-k algorithm). The library allocates no device
 *     memory and never synchronises inside bskv_run_* / bskv_rope_quantize_fp8 /
 *     bskv_merge_states; all work is enqueued on the caller's stream (a cudaStream_t
 *     passed as void*, NULL = legacy default stream).
 *   - Tensors are passed as a pointer plus element strides of the leading dims; the
 *     last dim must be contiguous. Device pointers must be 16-byte aligned, and every
 *     stride times the element size must be a multiple of 16 bytes.
 *   - A plan (bskv_plan*) is an opaque host object made by bskv_plan_* from host copies
 *     of the index arrays ([SPARSE] plan(): the plan step builds its helper structures
 *     once and later runs reuse them). It is re-made whenever
 *     the index arrays, lengths or shapes change, and must not be shared between
 *     overlapping runs ([WRAP] Metadata reuse). bskv_plan_upload copies its metadata
 *     into the caller's int workspace on a stream; runs read it from there.
 *   - LSE is the natural-log log-sum-exp of the scaled logits ([SPARSE] run(), its
 *     optional second output); a row that sees no key gets out = 0 and
 *     lse = -inf.
 *   - sm_scale (decode, prefill and BSR runs) multiplies q.k before the softmax; the value
 *     0 selects the pages' default 1/sqrt(head_dim) ([SPARSE] plan(): sm_scale defaults to
 *     1/sqrt(head_dim)). The MLA runs take their scales explicitly (bmm1/bmm2).
 *   - Setting the environment variable BSKV_LOGLEVEL to 1 makes every bskv_plan_* call print
 *     one line about its decisions (units, workers, split pieces, kernel, workspace bytes) to
 *     stderr; 2 adds the per-worker load spread. Every bskv_run_* / bskv_rope_* /
 *     bskv_merge_states call opens an NVTX range of its own name around its launches (a
 *     no-op unless a profiler is attached).
 */
#ifndef BSKV_H_
#define BSKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bskv_status {
  BSKV_OK = 0,
  BSKV_ERR_INVALID_ARG = 1,          /* bad pointer, size, index array or stride    */
  BSKV_ERR_UNSUPPORTED = 2,          /* valid but not implemented (dtype, dims, ...) */
  BSKV_ERR_WORKSPACE_TOO_SMALL = 3,  /* a caller workspace is smaller than needed    */
  BSKV_ERR_CUDA = 4,                 /* a CUDA runtime call failed                    */
  BSKV_ERR_TIMEOUT = 5,              /* a device wait gave up (reported on device)    */
  BSKV_ERR_DEVICE_INDEX = 6          /* a device-side index or position out of range  */
} bskv_status;

typedef enum bskv_dtype {
  BSKV_FP16 = 0,
  BSKV_BF16 = 1,
  BSKV_FP32 = 2,
  BSKV_E4M3 = 3,
  BSKV_INT32 = 4,
  BSKV_INT64 = 5
} bskv_dtype;

typedef struct bskv_plan bskv_plan;

/* Library version (major*10000 + minor*100 + patch). */
int32_t bskv_version(void);

/* Text of the last error raised on the calling thread ("" if none). Owned by the library. */
const char* bskv_last_error_message(void);

/* ---------------------------------------------------------------------------------
 * Plans (host only: no CUDA call, so they also run on a machine without a GPU)
 * --------------------------------------------------------------------------------- */

/*
 * Paged-KV batch decode plan ([SKILL] KV-Cache Formats: page table kv_indptr (batch+1),
 * kv_indices, kv_last_page_len (batch); [CHEAT] BatchDecodeWithPagedKVCacheWrapper:
 * plan once per step, run per layer).
 *   kv_indptr[batch+1], kv_indices[kv_indptr[batch]], kv_last_page_len[batch]: HOST
 *     int32 arrays, read during the call only. Request b owns pages
 *     kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in order; its length is
 *     (n_pages-1)*page_size + kv_last_page_len[b] (0 when it has no page), with
 *     1 <= kv_last_page_len[b] <= page_size when n_pages > 0.
 *   num_pages: pages in the pool; every kv_indices value must be in [0, num_pages).
 *   num_qo_heads % num_kv_heads == 0 (query head h reads kv head h / group).
 *   dtype: BSKV_BF16 or BSKV_FP16 (q, kv_cache and out share it).
 *   num_sms: SM count of the target GPU; max_workers: 0 = one worker per decode warp
 *     slot of the GPU, else an upper bound on the number of workers (split-KV pieces).
 * Errors: BSKV_ERR_INVALID_ARG for malformed arrays; BSKV_ERR_UNSUPPORTED for
 *   head_dim not in {64, 128} or more than 16 query heads per kv head.
 */
bskv_status bskv_plan_decode(const int32_t* kv_indptr, const int32_t* kv_indices,
                             const int32_t* kv_last_page_len, int32_t batch, int32_t num_pages,
                             int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t dtype, int32_t num_sms,
                             int32_t max_workers, bskv_plan** out_plan);

/*
 * BSR block-sparse attention plan ([SPARSE] plan(indptr, indices, M, N, R, C,
 * num_qo_heads, num_kv_heads, head_dim, causal, ...)).
 *   indptr[MB+1] (MB = ceil(M/R)), indices[indptr[MB]]: HOST int32 CSR arrays of the
 *     block mask (SciPy bsr_matrix semantics); indices < NB = N / C; N % C == 0.
 *     A column block listed twice in one row block is rejected (mask semantics).
 *   causal: token-level mask key j visible to query i iff j <= i + (N - M).
 *   dtype: BSKV_FP16 or BSKV_BF16 (q, k, v, out).
 *   num_sms: SM count of the target GPU.
 * The plan picks the tensor-core (tcgen05) kernel when R == 64, C == 64,
 * head_dim == 128 and the grouped rows R*(num_qo_heads/num_kv_heads) are 128 or 256;
 * any other shape runs the general kernel (head_dim 64 or 128, any R and C).
 */
bskv_status bskv_plan_bsr(const int32_t* indptr, const int32_t* indices, int32_t M, int32_t N,
                          int32_t R, int32_t C, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t causal, int32_t dtype, int32_t num_sms,
                          bskv_plan** out_plan);

/*
 * BSR plan for runs with a per-block token mask ([SPARSE] plan(..., mask, packed_mask):
 * a mask of shape (nnz, R, C) selects the visible (query, key) pairs inside each listed
 * block; causal applies only when no mask is given, so this plan has no causal flag).
 * Arguments and kernel choice as for bskv_plan_bsr.
 */
bskv_status bskv_plan_bsr_masked(const int32_t* indptr, const int32_t* indices, int32_t M,
                                 int32_t N, int32_t R, int32_t C, int32_t num_qo_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                                 int32_t num_sms, bskv_plan** out_plan);

/*
 * Variable-block sparse attention plan ([SPARSE] VariableBlockSparseAttentionWrapper.plan:
 * block sizes given by block_row_sz and block_col_sz, and each kv head with its own block
 * mask; the query heads of a group share their kv head's pattern).
 *   block_mask_map [num_kv_heads, MB, NB] (HOST bytes, nonzero = the block is visible),
 *   block_row_sz [num_kv_heads, MB] and block_col_sz [num_kv_heads, NB] (HOST int32, all
 *   positive): kv head h splits the qo_len query tokens into MB consecutive row blocks and the
 *   kv_len keys into NB consecutive column blocks; every head must cover the same qo_len and
 *   kv_len. Query token i of row block a sees key j of column block c of its kv head iff
 *   block_mask_map[h][a][c] (and, when causal, j <= i + kv_len - qo_len).
 *   head_dim 64 or 128; dtype BSKV_FP16 or BSKV_BF16; the general kernel serves these plans.
 */
bskv_status bskv_plan_bsr_variable(const uint8_t* block_mask_map, const int32_t* block_row_sz,
                                   const int32_t* block_col_sz, int32_t MB, int32_t NB,
                                   int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t causal, int32_t dtype, int32_t num_sms,
                                   bskv_plan** out_plan);

/*
 * Batch prefill over a paged KV cache ([CHEAT] benchmark README:
 * BatchPrefillWithPagedKVCacheWrapper, the paged-cache prefill wrapper; [SKILL]
 * KV-Cache Formats and Batch prefill / Append): request b owns query tokens
 * [qo_indptr[b], qo_indptr[b+1]) (the last qo_len_b tokens of its sequence) and the pages of
 * its kv_indptr/kv_indices/kv_last_page_len entry (L_b tokens, as for bskv_plan_decode).
 *   qo_indptr[batch+1], kv_indptr[batch+1], kv_indices, kv_last_page_len[batch]: HOST int32;
 *   page ids in [0, num_pages). causal: query token t of request b (0-based within its
 *   queries) sees key j iff j <= t + L_b - qo_len_b (bottom-right aligned).
 *   head_dim 64 or 128; dtype BSKV_FP16 or BSKV_BF16; the general kernel serves these plans.
 */
bskv_status bskv_plan_prefill_paged(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                    const int32_t* kv_indices, const int32_t* kv_last_page_len,
                                    int32_t batch, int32_t num_pages, int32_t page_size,
                                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t causal, int32_t dtype, int32_t num_sms,
                                    bskv_plan** out_plan);

/*
 * Sparse MLA FP8 decode plan ([MLA] get_batch_decode_metadata_mla(query, seq_lens,
 * sparse_mla_top_k): reusable while seq_lens, the query shape and top_k are unchanged).
 *   seq_lens[batch]: HOST int32 valid sparse lengths, 0 <= seq_lens[b] <= top_k.
 *   q_len >= 1 query tokens per request; num_heads in [1, 128]; top_k a positive
 *   multiple of 64 ([MLA] sparse_mla_top_k).
 */
bskv_status bskv_plan_mla_sparse(const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                 int32_t num_heads, int32_t top_k, int32_t num_sms,
                                 bskv_plan** out_plan);

/*
 * Dense paged MLA FP8 decode plan ([SKILL] Multi-Head Latent Attention (MLA):
 * BatchMLAPagedAttentionWrapper and trtllm_batch_decode_with_kv_cache_mla over a latent
 * KV cache; [CHEAT] benchmark README: BatchMLAPagedAttentionWrapper, MLA attention of the
 * DeepSeek models; page table as in [SKILL] KV-Cache Formats). One query token per
 * request attends to every token of its request.
 *   kv_indptr[batch+1], kv_indices[kv_indptr[batch]], kv_last_page_len[batch]: HOST int32
 *     page table; request b owns pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in
 *     order and L_b = (n_b - 1) * page_size + kv_last_page_len[b] tokens (0 when it owns
 *     no page); kv_indptr[0] == 0 and non-decreasing, page ids in [0, num_pages),
 *     1 <= kv_last_page_len[b] <= page_size for a request with pages.
 *   Token t of request b is cache row kv_indices[kv_indptr[b] + t / page_size] *
 *   page_size + t % page_size; num_pages * page_size must stay below 2^31.
 *   num_heads in [1, 128]; num_sms: SM count of the target GPU.
 * The plan copies the page table into its metadata; runs read each token's cache row from
 * it while they gather the rows (no separate row list).
 */
bskv_status bskv_plan_mla_paged(const int32_t* kv_indptr, const int32_t* kv_indices,
                                const int32_t* kv_last_page_len, int32_t batch,
                                int32_t num_pages, int32_t page_size, int32_t num_heads,
                                int32_t num_sms, bskv_plan** out_plan);

/* Free a plan (NULL is accepted). */
bskv_status bskv_plan_destroy(bskv_plan* plan);

/*
 * Host view of the plan's int32 metadata (the exact words bskv_plan_upload copies).
 * *meta stays valid until the plan is destroyed. Layout: a 16-word header
 * {magic, kind, units, workers, chunks, slots, merges, tile, off_workers, off_chunks,
 * off_merges, off_aux0, off_aux1, grid, total_words, variant} then the sections.
 */
bskv_status bskv_plan_metadata(const bskv_plan* plan, const int32_t** meta, int64_t* num_words);

/*
 * Bytes of int workspace (the metadata, then at the next 256-byte boundary the int32 merge
 * counters of a decode plan, one per merge item and kv head of the unit) and of float
 * workspace (split-KV partials) a run needs.
 */
bskv_status bskv_plan_workspace_sizes(const bskv_plan* plan, size_t* int_ws_bytes,
                                      size_t* float_ws_bytes);

/*
 * Copy the metadata into the caller's device int workspace (cudaMemcpyAsync on
 * `stream`; the host copy lives in the plan, so it must outlive the copy) and zero the
 * merge counters after it (cudaMemsetAsync). Later runs with this plan read that
 * workspace, which must not be changed meanwhile. A complete bskv_run_decode leaves the
 * counters at zero again; after a run that reported a device error (bskv_get_device_status)
 * upload the plan again before reusing it.
 */
bskv_status bskv_plan_upload(bskv_plan* plan, void* int_ws, size_t int_ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Runs (device work on `stream`; no allocation, no synchronisation)
 * --------------------------------------------------------------------------------- */

/*
 * Paged-KV batch decode, one query token per request ([SKILL] KV-Cache Formats):
 *   out[b, h, :] = sum_j softmax_j(sm_scale * q[b,h,:].k_j) v_j over the L_b tokens of
 *   request b's pages, kv head h / group.
 *   q     [batch, num_qo_heads, head_dim], strides q_strides = {batch, head} (elements).
 *   kv_cache: pages of K and V; element (page p, t in {0=K,1=V}, kv head k, token s, d)
 *         at p*kv_strides[0] + t*kv_strides[1] + k*kv_strides[2] + s*kv_strides[3] + d.
 *         The layout (num_pages, 2, num_kv_heads, page_size, head_dim) is the
 *         contiguous case ([SKILL] paged KV-cache).
 *   out   [batch, num_qo_heads, head_dim] in the plan dtype, strides out_strides.
 *   lse   [batch, num_qo_heads] float32 contiguous, or NULL.
 *   float_ws: at least bskv_plan_workspace_sizes().float_ws_bytes (may be NULL if 0).
 * When no unit (request and kv head, or request and group of kv heads) is cut into more
 * than 8 pieces, one kernel launch: a split unit is merged by the worker that finishes
 * its last piece (per kv head), which it learns from an atomic counter in the int
 * workspace. Otherwise the attention kernel and then the merge kernel. Either way the
 * merge is the one bskv_decode_merge applies ([CHEAT] merge_state), in the same order, so
 * the result is bit-identical to bskv_run_decode_partial followed by bskv_decode_merge.
 */
bskv_status bskv_run_decode(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                            const void* kv_cache, const int64_t* kv_strides, void* out,
                            const int64_t* out_strides, float* lse, float sm_scale,
                            void* float_ws, size_t float_ws_bytes, void* stream);

/*
 * The two halves of bskv_run_decode, for callers that want the split-KV partial states
 * or to time the kernels apart. bskv_run_decode_partial runs the attention kernel only:
 * requests computed in one piece are written to out/lse, split ones leave normalised
 * partial outputs and LSE in float_ws. bskv_decode_merge then merges those into out/lse
 * (and zero-fills requests without tokens); it is a no-op when the plan split nothing.
 * Same arguments and errors as bskv_run_decode.
 */
bskv_status bskv_run_decode_partial(const bskv_plan* plan, const void* q,
                                    const int64_t* q_strides, const void* kv_cache,
                                    const int64_t* kv_strides, void* out,
                                    const int64_t* out_strides, float* lse, float sm_scale,
                                    void* float_ws, size_t float_ws_bytes, void* stream);
bskv_status bskv_decode_merge(const bskv_plan* plan, void* out, const int64_t* out_strides,
                              float* lse, void* float_ws, size_t float_ws_bytes, void* stream);

/*
 * Allocation-free paged decode. The pages have no counterpart: this entry point exists for
 * callers that cannot allocate device memory -- code embedded in a host framework that
 * hands it only tensors and a stream, processes whose device memory is all reserved by
 * another allocator, or latency-critical loops where cudaMalloc/cudaFree (which can
 * synchronise the device) is not acceptable. It computes exactly what bskv_run_decode
 * computes, with the same arguments minus the float workspace, and needs no
 * bskv_plan_upload: the plan metadata (at most 1 MiB) is copied on `stream` into a
 * library-owned static device array, and the split-KV partial states (at most 8 MiB) live
 * in a second one. Every GPU that loads the library holds these 9 MiB until the process
 * exits. A plan that needs more returns BSKV_ERR_UNSUPPORTED and launches nothing.
 * The first call on a device looks up the arrays' device addresses (cudaGetSymbolAddress).
 * All calls share the two arrays, and each call overwrites what the previous one left
 * there, so calls that overlap on the GPU (e.g. on two streams) race: serialise them. No call allocates or frees device memory.
 * The metadata copy reads the plan's own host memory, which is pageable: the call can wait
 * while the driver stages those bytes, and the plan is no longer read once the call returns.
 */
bskv_status bskv_run_decode_noalloc(const bskv_plan* plan, const void* q,
                                    const int64_t* q_strides, const void* kv_cache,
                                    const int64_t* kv_strides, void* out,
                                    const int64_t* out_strides, float* lse, float sm_scale,
                                    void* stream);

/*
 * BSR block-sparse attention ([SPARSE] run(q, k, v, out, lse)):
 *   q [M, num_qo_heads, head_dim], k and v [N, num_kv_heads, head_dim] (strides {row,
 *   head} in elements); out like q; lse [M, num_qo_heads] float32 contiguous or NULL.
 */
bskv_status bskv_run_bsr(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                         const void* k, const int64_t* k_strides, const void* v,
                         const int64_t* v_strides, void* out, const int64_t* out_strides,
                         float* lse, float sm_scale, void* float_ws, size_t float_ws_bytes,
                         void* stream);

/*
 * BSR block-sparse attention with a per-block token mask ([SPARSE] run() of a plan made
 * with mask / packed_mask), for a plan of bskv_plan_bsr_masked:
 *   q, k, v, out, lse as for bskv_run_bsr.
 *   packed_mask: device bytes holding the (nnz, R, C) boolean mask flattened in that order
 *     (nnz in the order of indices), eight entries per byte, entry t in bit t % 8 of byte
 *     t / 8 (numpy.packbits(..., bitorder="little")); packed_mask_bytes >= ceil(nnz*R*C/8);
 *     16-byte aligned.
 *   Query i sees key j iff the block (i / R, j / C) is listed and its mask entry
 *   (i % R, j % C) is set; a row that sees nothing gets out = 0 and lse = -inf.
 */
bskv_status bskv_run_bsr_masked(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                                const void* k, const int64_t* k_strides, const void* v,
                                const int64_t* v_strides, const void* packed_mask,
                                size_t packed_mask_bytes, void* out, const int64_t* out_strides,
                                float* lse, float sm_scale, void* stream);

/*
 * Variable-block sparse attention ([SPARSE] VariableBlockSparseAttentionWrapper.run), for a
 * plan of bskv_plan_bsr_variable:
 *   q [num_qo_heads, qo_len, head_dim], k and v [num_kv_heads, kv_len, head_dim], out like
 *   q; strides are given as {token, head} in elements (the pages' head-major tensors have
 *   token stride head_dim and head stride len * head_dim); lse [num_qo_heads, qo_len]
 *   float32 contiguous, or NULL. A token that sees no key gets out = 0 and lse = -inf.
 */
bskv_status bskv_run_bsr_variable(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                                  const void* k, const int64_t* k_strides, const void* v,
                                  const int64_t* v_strides, void* out,
                                  const int64_t* out_strides, float* lse, float sm_scale,
                                  void* stream);

/*
 * Batch prefill over a paged KV cache, for a plan of bskv_plan_prefill_paged:
 *   q [total_qo, num_qo_heads, head_dim], strides {token, head}; kv_cache and kv_strides as
 *   for bskv_run_decode (4 strides: page, K/V, kv head, slot); out like q; lse
 *   [total_qo, num_qo_heads] float32 contiguous, or NULL. A query that sees no key gets
 *   out = 0 and lse = -inf.
 */
bskv_status bskv_run_prefill_paged(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                                   const void* kv_cache, const int64_t* kv_strides, void* out,
                                   const int64_t* out_strides, float* lse, float sm_scale,
                                   void* stream);

/*
 * Sparse MLA FP8 decode ([MLA] sparse_mla_fp8_decode; [WRAP] scale folding):
 *   query   [batch, q_len, num_heads, 576] E4M3, contiguous.
 *   kv_rows [num_rows, 576] E4M3, contiguous (a [pages, page_size, 576] cache viewed as
 *           rows; indices are physical token ids = page * page_size + slot).
 *   indices [batch, q_len, top_k] int32 on the device, shared by all heads; entries
 *           [0, seq_lens[b]) are used and must lie in [0, num_rows). An entry outside
 *           that range is never read (its row is taken as zeros), the output of that query
 *           is unspecified, and BSKV_ERR_DEVICE_INDEX is raised in the device status word
 *           (bskv_get_device_status).
 *   s_j = bmm1_scale * <q, kv_j> over 576 values; out = bmm2_scale * sum_j softmax(s)_j
 *   kv_j[:512] (V = the 512 latent values); out bf16 [batch, q_len, num_heads, 512];
 *   lse float32 [batch, q_len, num_heads] of the bmm1-scaled logits, or NULL.
 *   bmm1_scale = attention_scale * q_descale * kv_descale, bmm2_scale = kv_descale.
 */
bskv_status bskv_run_mla_sparse(const bskv_plan* plan, const void* query, const void* kv_rows,
                                int64_t num_rows, const int32_t* indices, float bmm1_scale,
                                float bmm2_scale, void* out, float* lse, void* float_ws,
                                size_t float_ws_bytes, void* stream);

/*
 * Dense paged MLA FP8 decode (the plan of bskv_plan_mla_paged):
 *   query    [batch, num_heads, 576] E4M3, contiguous (one token per request).
 *   kv_pages [num_pages, page_size, 576] E4M3, contiguous: the latent cache, one row of
 *            512 latent + 64 rotated values per token (the layout the prologue writes).
 *   s_j, out and lse as for bskv_run_mla_sparse over the L_b tokens of request b:
 *   out bf16 [batch, num_heads, 512]; lse float32 [batch, num_heads] or NULL. A request
 *   with no token gets out = 0 and lse = -inf.
 *   float_ws: at least bskv_plan_workspace_sizes' float bytes (split-KV partials; 0 bytes,
 *   and NULL allowed, when the plan assigns whole requests), 16-byte aligned.
 */
bskv_status bskv_run_mla_paged(const bskv_plan* plan, const void* query, const void* kv_pages,
                               float bmm1_scale, float bmm2_scale, void* out, float* lse,
                               void* float_ws, size_t float_ws_bytes, void* stream);

/*
 * RoPE + FP8 E4M3 quantisation of MLA query/key rows ([MLA] mla_rope_quantize_fp8;
 * [WRAP] RoPE and FP8 quantization). Rotary arithmetic in float32 on the 64-value
 * tail; is_neox != 0 pairs tail value i with value i + 32 (NeoX layout), 0 pairs values
 * 2i and 2i + 1 (interleaved layout); pair i uses cos = cos_sin[pos, i], sin = cos_sin[pos, 32 + i].
 * Outputs: Q_fp8 = cast(Q * quant_scale_q), K_fp8 = cast(K * quant_scale_kv), round to
 * nearest even, saturating to +-448.
 *   Query group (all NULL to skip): q_rope [nnz_q, num_heads, 64], q_nope [nnz_q,
 *     num_heads, 512] bf16 with strides {token, head}; pos_q [nnz_q];
 *     q_rope_out / q_nope_out E4M3 with strides {token, head} (e.g. slices [..., 512:]
 *     and [..., :512] of a [nnz_q, num_heads, 576] buffer).
 *   Key group (all NULL to skip): k_rope [nnz_k, 64], k_nope [nnz_k, 512] bf16 with row
 *     strides; pos_k [nnz_k]; k_rope_out / k_nope_out E4M3 with row strides.
 *   pos_dtype: BSKV_INT32 or BSKV_INT64; cos_sin [max_seq_len, 64] contiguous,
 *     BSKV_FP32 or BSKV_BF16. A position outside [0, max_seq_len) leaves its row
 *     unwritten and raises BSKV_ERR_DEVICE_INDEX in the device status word.
 */
bskv_status bskv_rope_quantize_fp8(
    const void* q_rope, const int64_t* q_rope_strides, const void* q_nope,
    const int64_t* q_nope_strides, const void* pos_q, int64_t nnz_q, int32_t num_heads,
    void* q_rope_out, const int64_t* q_rope_out_strides, void* q_nope_out,
    const int64_t* q_nope_out_strides,
    const void* k_rope, int64_t k_rope_stride, const void* k_nope, int64_t k_nope_stride,
    const void* pos_k, int64_t nnz_k, void* k_rope_out, int64_t k_rope_out_stride,
    void* k_nope_out, int64_t k_nope_out_stride,
    int32_t pos_dtype, const void* cos_sin, int32_t cos_sin_dtype, int64_t max_seq_len,
    int32_t is_neox, float quant_scale_q, float quant_scale_kv, void* stream);

/*
 * RoPE + FP8 quantisation with the key rows appended to a paged latent cache ([CHEAT]
 * benchmark README: rope_quantize_fp8_append_paged_kv_cache, which rotates, quantises and
 * writes the key rows into a paged cache in one call; page table as in [SKILL] KV-Cache
 * Formats). The arithmetic is that
 * of bskv_rope_quantize_fp8; only the destination of a key row differs.
 *   Query group: exactly as bskv_rope_quantize_fp8 (all NULL to skip).
 *   Key rows: k_rope [nnz_k, 64], k_nope [nnz_k, 512] bf16 with row strides; pos_k [nnz_k]
 *     rotary positions (pos_dtype).
 *   Destination, all int32 on the device: key row i belongs to request batch_indices[i]
 *     (in [0, batch)) at token position positions[i] (>= 0) of that request; the request's
 *     pages are kv_indices[kv_indptr[b] .. kv_indptr[b+1]) and the row is written to page
 *     kv_indices[kv_indptr[b] + positions[i] / page_size], slot positions[i] % page_size of
 *     kv_pages [num_pages, page_size, 576] E4M3 (512 NoPE then 64 rotated values), the
 *     layout the paged MLA decode reads. A row whose position lies past the request's pages,
 *     whose page id lies outside [0, num_pages), whose request lies outside [0, batch) or
 *     whose rotary position lies outside [0, max_seq_len) is not written and raises
 *     BSKV_ERR_DEVICE_INDEX in the device status word. Other cache bytes are not touched.
 *   Rows that share a destination race (the last writer wins).
 */
bskv_status bskv_rope_quantize_fp8_append_paged(
    const void* q_rope, const int64_t* q_rope_strides, const void* q_nope,
    const int64_t* q_nope_strides, const void* pos_q, int64_t nnz_q, int32_t num_heads,
    void* q_rope_out, const int64_t* q_rope_out_strides, void* q_nope_out,
    const int64_t* q_nope_out_strides,
    const void* k_rope, int64_t k_rope_stride, const void* k_nope, int64_t k_nope_stride,
    const void* pos_k, int64_t nnz_k, const int32_t* batch_indices, const int32_t* positions,
    const int32_t* kv_indptr, const int32_t* kv_indices, int32_t batch, int32_t page_size,
    int64_t num_pages, void* kv_pages,
    int32_t pos_dtype, const void* cos_sin, int32_t cos_sin_dtype, int64_t max_seq_len,
    int32_t is_neox, float quant_scale_q, float quant_scale_kv, void* stream);

/*
 * Merge attention states ([CHEAT] cascade.rst merge_states; [SKILL] Cascade Inference):
 *   v [seq_len, num_states, num_heads, head_dim] float32 (normalised partial outputs),
 *   s [seq_len, num_states, num_heads] float32 natural-log LSE, both contiguous;
 *   lse = log sum_c exp(s_c); v_out = sum_c exp(s_c - lse) v_c.
 *   v_out [seq_len, num_heads, head_dim] in out_dtype (BSKV_FP32, BSKV_BF16, BSKV_FP16);
 *   s_out [seq_len, num_heads] float32 or NULL. head_dim % 4 == 0.
 */
bskv_status bskv_merge_states(const float* v, const float* s, int64_t seq_len,
                              int32_t num_states, int32_t num_heads, int32_t head_dim,
                              void* v_out, int32_t out_dtype, float* s_out, void* stream);

/*
 * Read (and optionally clear) the device status word of the current device: BSKV_OK,
 * or the first device-side error a kernel recorded (BSKV_ERR_TIMEOUT when a bounded
 * wait gave up, BSKV_ERR_DEVICE_INDEX for an index or position out of range).
 * Synchronous (cudaMemcpy); not for use inside stream capture.
 */
bskv_status bskv_get_device_status(int32_t* status, int32_t reset);

/* Testing hook: a nonzero value makes every bounded device wait give up at once, so
 * the timeout path can be exercised without stalling a GPU. Default 0. */
bskv_status bskv_set_debug_force_timeout(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* BSKV_H_ */
