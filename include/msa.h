/*
 * msa.h -- C ABI of the GB300 (sm_103a) block-sparse top-k GQA attention library (libmsa.so).
 *
 * What the library computes (MSA sparse attention pages):
 *   For batch b, KV head h, query s and query head hq = h*qhead_per_kv + g,
 *   the query attends to the union of the 128-token KV blocks listed in
 *   q2k[b][h][s][0..topk) (entries < 0 are padding), restricted to keys below
 *   the used KV length and, when causal, to keys t <= s + (kv_len - Sq)
 *   (bottom-right alignment).  Scores are softmax_scale * q.k, the output row
 *   is softmax-weighted V (bf16) and LSE is the natural-log logsumexp of the
 *   visible scores (fp32).  A row with no visible key gets O = 0, LSE = -inf.
 *   Sources: test_sparse_atten.py (sparse_attention_ref,
 *   _bottom_right_causal_visible_blocks, pack_paged_kv) and interface.py
 *   (sparse_atten_func, sparse_decode_atten_func, build_k2q_csr docstring).
 *
 * Conventions for every entry point:
 *   - pointers named *_dev or documented as device are device pointers; the
 *     caller owns every buffer (inputs, outputs, plan, workspace);
 *   - calls are asynchronous on `stream`, never synchronise the device and
 *     never allocate memory;
 *   - the attention, combine and paged-plan kernels are launched with
 *     programmatic stream serialization: one may start its prologue while the
 *     previous kernel on `stream` drains, but reads and writes nothing in
 *     global memory before that kernel has completed, so stream order holds
 *     for the caller's own work on either side of a call;
 *   - the return value is an MSA_* status; on any error nothing is launched;
 *   - workspaces are caller-allocated, 256-byte aligned, sized by the
 *     matching *_workspace_size() query;
 *   - `status_dev` (may be NULL) is a device uint32 the kernels OR MSA_STATUS_*
 *     bits into; the caller zeroes it before the call and, once the stream is
 *     synchronised, checks the word with msa_check_status() (or reads and
 *     checks it in one call with msa_read_status());
 *   - layouts are dense row-major C arrays in the shapes given;
 *   - bf16 tensors are passed as void* (IEEE bfloat16 bit patterns).
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ---- */
#define MSA_OK 0
#define MSA_ERR_INVALID_ARG (-1) /* null pointer, negative size, inconsistent shape */
#define MSA_ERR_UNSUPPORTED (-2) /* D != 128, qhead_per_kv not in {1,2,4,8,16},
                                    topk not in {4,8,16,32}, page_size != blk_kv != 128 */
#define MSA_ERR_WORKSPACE (-3)   /* workspace or plan buffer too small or misaligned */
#define MSA_ERR_CUDA (-4)        /* a kernel launch or CUDA runtime call failed */
#define MSA_ERR_DEVICE (-5)      /* msa_check_status found a fatal device status bit */

/* ---- device status bits (ORed into *status_dev by the kernels) ---- */
#define MSA_STATUS_INDEX_RANGE 0x1u  /* a q2k id >= the sequence's block count: treated as padding */
#define MSA_STATUS_DUPLICATE 0x2u    /* a query named one block twice: counted once */
#define MSA_STATUS_PAGE_RANGE 0x4u   /* a page_table entry outside [0, num_pages): block skipped (fatal) */
#define MSA_STATUS_PLAN_OVERFLOW 0x8u /* the plan buffer could not hold the schedule (fatal) */
#define MSA_STATUS_TIMEOUT 0x10u      /* a bounded wait inside a kernel gave up; output invalid (fatal) */
#define MSA_STATUS_LAUNCH 0x20u       /* a kernel found its shared memory misaligned; nothing written (fatal) */
#define MSA_STATUS_SHAPE 0x40u        /* cu_seqlens disagree with the declared sizes; sequence dropped (fatal) */
#define MSA_STATUS_FATAL_MASK \
    (MSA_STATUS_PAGE_RANGE | MSA_STATUS_PLAN_OVERFLOW | MSA_STATUS_TIMEOUT | MSA_STATUS_LAUNCH | MSA_STATUS_SHAPE)

/* K/V storage formats of msa_sparse_attn_fwd (and, bf16 / fp8, of the paged decode pools) */
#define MSA_KV_BF16 0
#define MSA_KV_NVFP4 1
#define MSA_KV_FP8 2 /* e4m3 bytes [..][Hkv][D], staged to bf16 on load (exact) for both MMAs */

/* Storage type of the split partials (msa_fwd_options.partial_dtype) */
#define MSA_PARTIAL_BF16 0
#define MSA_PARTIAL_FP16 1
#define MSA_PARTIAL_FP32 2

/*
 * Options of msa_sparse_attn_fwd_varlen; NULL selects the defaults (bf16
 * partials, no temperature LSE).  Source: interface.py sparse_atten_func
 * (partial_dtype, lse_temperature_scale, return_temperature_lse).
 *   partial_dtype          MSA_PARTIAL_*: storage of each split's partial output.
 *   lse_temperature_scale  T > 0, finite: used when lse_temperature != NULL.
 *   lse_temperature        [total_q][Hq] fp32 device output or NULL: the LSE of
 *                          the visible scores divided by T, log sum_t
 *                          exp(scale q.k_t / T) (-inf for a row with no key).
 *   qk_fp8                 1: q is e4m3 bytes [total_q][Hq][D] and, with
 *                          kv_format MSA_KV_FP8, S = Q K^T runs as an e4m3 MMA
 *                          (fp32 accumulate) while V is staged to bf16 for the
 *                          bf16 P V MMA (interface.py qk_dtype = fp8, pv_dtype =
 *                          bf16); 0: q is bf16.
 */
typedef struct msa_fwd_options {
    int partial_dtype;
    float lse_temperature_scale;
    float *lse_temperature;
    int qk_fp8;
} msa_fwd_options;

/* Human-readable name of an MSA_* status code (static string). */
const char *msa_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int msa_version(void);

/*
 * Checks a status word that the caller has already brought back: a host copy
 * of *status_dev taken after the stream was synchronised, or the word itself
 * when status_dev lives in host-mapped or managed memory.  Makes no CUDA
 * call and does not synchronise.  Returns MSA_ERR_DEVICE if a bit of
 * MSA_STATUS_FATAL_MASK is set, MSA_ERR_INVALID_ARG for NULL, else MSA_OK
 * (the non-fatal bits MSA_STATUS_INDEX_RANGE / MSA_STATUS_DUPLICATE only
 * report that padding rules were applied).
 */
int msa_check_status(const uint32_t *status_word);

/*
 * Convenience form: copies *status_dev to *status_host on `stream`,
 * synchronises the stream, then returns msa_check_status(status_host).
 * A diagnostic call, not part of the hot path.
 */
int msa_read_status(const uint32_t *status_dev, uint32_t *status_host, cudaStream_t stream);

/* =========================================================================
 * (a1, a2) k->q CSR inversion and work plan
 * =========================================================================
 * Source: interface.py module docstring (q2k [Hkv,total_q,topK] ->
 * k2q_row_ptr [Hkv,total_rows+1], k2q_q_indices [Hkv,total_q*topK]) and
 * test_sparse_atten.py test_scheduler_builds_packed_qsplit_metadata (packed
 * q | split << 24, split ids of a query are 0..count-1, every row covered,
 * no work item above the per-CTA query target).
 *
 * Inputs
 *   q2k      [B][Hkv][Sq][topk] int32, device.  Block ids; < 0 is padding.
 *   seqused  [B] int32 device or NULL: used KV length per sequence (default
 *            Skv).  Ids >= ceil(kv_len_b / blk_kv) are padding and set
 *            MSA_STATUS_INDEX_RANGE.  A repeated id of one query counts once
 *            and sets MSA_STATUS_DUPLICATE.
 *   qhead_per_kv  query heads per KV head; sizes the plan's work items.
 * Outputs (device, written in full, bit-deterministic)
 *   row_ptr      [Hkv][B*nblk + 1], nblk = ceil(Skv / blk_kv); row r = b*nblk + j.
 *   q_indices    [Hkv][B*Sq*topk]: per row, global query ids b*Sq+s ascending;
 *                entries past row_ptr[h][B*nblk] are -1.
 *   qsplit       [Hkv][B*Sq*topk]: q | (split << 24); split = rank of the block
 *                among the query's distinct valid slots (slot order); tail -1.
 *   split_counts [B*Sq][Hkv]: number of distinct valid blocks of the query.
 *   plan         opaque work plan for msa_sparse_attn_fwd (may be NULL), of
 *                msa_plan_size() bytes; its item count stays on the device.
 * Limits: B*Sq < 2^24, ceil(Skv/blk_kv) <= 8192.
 */
size_t msa_k2q_csr_workspace_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv);
size_t msa_plan_size(int B, int Hkv, int Sq, int Skv, int topk, int blk_kv, int qhead_per_kv);
int msa_build_k2q_csr(const int32_t *q2k, int B, int Hkv, int Sq, int Skv, int topk, int blk_kv,
                      int qhead_per_kv, const int32_t *seqused, int32_t *row_ptr, int32_t *q_indices,
                      int32_t *qsplit, int32_t *split_counts, void *plan, size_t plan_bytes,
                      void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream);

/* =========================================================================
 * Ragged batches: k->q CSR and work plan
 * =========================================================================
 * Source: interface.py sparse_atten_func and _validate_csr_varlen_inputs
 * (cu_seqlens_q / cu_seqlens_k [B+1] int32 prefix sums, q2k
 * [Hkv][total_q][topK], k2q_row_ptr [Hkv][total_rows+1]).
 *
 *   q2k          [Hkv][total_q][topk] int32, device; ids are blocks of the
 *                query's own sequence (0 .. ceil(keys_b/blk_kv)-1), < 0 padding.
 *   cu_seqlens_q, cu_seqlens_k  [B+1] int32, device: sequence b holds queries
 *                cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and keys
 *                cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1.
 *   total_q      rows of q2k (cu_seqlens_q[B] must equal it).
 *   max_seqlen_q, max_seqlen_k  per-sequence maxima (size the builder's tiles).
 *   total_rows   row capacity of row_ptr: >= sum_b ceil(keys_b / blk_kv).
 *   seqused      [B] or NULL: used key count per sequence (<= keys_b).
 * Outputs as msa_build_k2q_csr with rows r = row0_b + j, row0_b = sum over
 * earlier sequences of ceil(keys/blk_kv); rows past the last sequence's are
 * empty; query ids are global (cu_seqlens_q[b] + local index).  A sequence
 * whose ranges decrease, start below 0, exceed total_q / total_rows or the
 * maxima is dropped (its queries see nothing) and MSA_STATUS_SHAPE is set.
 * Limits: total_q < 2^24, ceil(max_seqlen_k/blk_kv) <= 8192, B <= 65535.
 */
size_t msa_k2q_csr_varlen_workspace_size(int B, int Hkv, int total_q, int max_seqlen_q, int max_seqlen_k,
                                         int total_rows, int topk, int blk_kv);
size_t msa_plan_varlen_size(int Hkv, int total_q, int total_rows, int topk, int blk_kv, int qhead_per_kv);
int msa_build_k2q_csr_varlen(const int32_t *q2k, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B,
                             int Hkv, int total_q, int max_seqlen_q, int max_seqlen_k, int total_rows, int topk,
                             int blk_kv, int qhead_per_kv, const int32_t *seqused, int32_t *row_ptr,
                             int32_t *q_indices, int32_t *qsplit, int32_t *split_counts, void *plan,
                             size_t plan_bytes, void *workspace, size_t ws_bytes, uint32_t *status_dev,
                             cudaStream_t stream);

/* =========================================================================
 * (a3, a4, a6) block-sparse prefill forward, dense KV
 * =========================================================================
 * Source: interface.py sparse_atten_func / sparse_atten_nvfp4_kv_func and
 * _sparse_atten_csr_varlen_forward (KV-block-major work over the CSR, one
 * partial (O, LSE) per (query, split, head), then an LSE combine:
 * O = sum_s exp(lse_s - LSE) O_s, LSE = logsumexp_s lse_s, a split with a
 * non-finite lse has weight 0; test_sparse_atten.py sparse_attention_ref).
 *
 *   q       [B][Sq][Hq][D] bf16, device.
 *   k, v    kv_format MSA_KV_BF16: [B][Skv][Hkv][D] bf16.
 *           kv_format MSA_KV_FP8: [B][Skv][Hkv][D] e4m3 bytes, staged to bf16 on load.
 *           kv_format MSA_KV_NVFP4: [B][Skv][Hkv][D/2] uint8, e2m1 codes, element
 *           2i in the low nibble; k_scales / v_scales [B][Skv][Hkv][D/16] e4m3
 *           bytes, one per 16 elements along D; value = e2m1 * e4m3 (no global scale).
 *   row_ptr, q_indices, qsplit, split_counts, plan: from msa_build_k2q_csr
 *           with the same q2k, shapes and qhead_per_kv = Hq / Hkv.
 *   causal  0/1, bottom-right aligned.  softmax_scale <= 0 selects 1/sqrt(D).
 *   o       [B][Sq][Hq][D] bf16, device (written in full).
 *   lse     [B][Sq][Hq] fp32, device, or NULL.
 *   workspace  msa_sparse_attn_fwd_workspace_size() bytes (split partials).
 */
size_t msa_sparse_attn_fwd_workspace_size(int B, int Sq, int Hq, int topk, int D);
int msa_sparse_attn_fwd(const void *q, const void *k, const void *v, int kv_format, const void *k_scales,
                        const void *v_scales, const int32_t *row_ptr, const int32_t *q_indices,
                        const int32_t *qsplit, const int32_t *split_counts, const void *plan, int B, int Sq,
                        int Skv, int Hq, int Hkv, int D, int blk_kv, int topk, int causal, float softmax_scale,
                        void *o, float *lse, void *workspace, size_t ws_bytes, uint32_t *status_dev,
                        cudaStream_t stream);

/*
 * The two halves of msa_sparse_attn_fwd, for callers that schedule or time
 * them separately (same arguments and workspace):
 *   msa_sparse_attn_fwd_partial  -- the attention tiles: writes one partial
 *                                   (O_s bf16, lse_s fp32) per (query, split,
 *                                   query head) into the workspace;
 *   msa_sparse_attn_combine      -- the LSE combine of those partials into o
 *                                   and lse.
 * Calling partial then combine on one stream equals msa_sparse_attn_fwd.
 */
int msa_sparse_attn_fwd_partial(const void *q, const void *k, const void *v, int kv_format, const void *k_scales,
                                const void *v_scales, const int32_t *q_indices, const int32_t *qsplit,
                                const void *plan, int B, int Sq, int Skv, int Hq, int Hkv, int D, int blk_kv,
                                int topk, int causal, float softmax_scale, void *workspace, size_t ws_bytes,
                                uint32_t *status_dev, cudaStream_t stream);
int msa_sparse_attn_combine(const int32_t *split_counts, int B, int Sq, int Hq, int Hkv, int D, int topk, void *o,
                            float *lse, const void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * Ragged-batch forward: msa_sparse_attn_fwd over sequences of different
 * lengths (the tiles and then the LSE combine, one call).
 *   q       [total_q][Hq][D] bf16.
 *   k, v    [total_k][Hkv][D] bf16 (MSA_KV_NVFP4: [total_k][Hkv][D/2] codes and
 *           [total_k][Hkv][D/16] scales).
 *   q_indices, qsplit, split_counts, plan: from msa_build_k2q_csr_varlen with
 *           the same q2k, cu_seqlens and qhead_per_kv = Hq / Hkv.
 *   cu_seqlens_q, cu_seqlens_k [B+1] device, as given to the builder; causal
 *           masking is bottom-right per sequence (key t <= s + keys_b - queries_b).
 *   opts    NULL or msa_fwd_options (partial dtype, temperature LSE).
 *   o       [total_q][Hq][D] bf16; lse [total_q][Hq] fp32 or NULL.
 *   workspace  msa_sparse_attn_fwd_varlen_workspace_size() bytes.
 */
size_t msa_sparse_attn_fwd_varlen_workspace_size(int total_q, int Hq, int topk, int D, const msa_fwd_options *opts);
int msa_sparse_attn_fwd_varlen(const void *q, const void *k, const void *v, int kv_format, const void *k_scales,
                               const void *v_scales, const int32_t *q_indices, const int32_t *qsplit,
                               const int32_t *split_counts, const void *plan, const int32_t *cu_seqlens_q,
                               const int32_t *cu_seqlens_k, int B, int total_q, int total_k, int Hq, int Hkv, int D,
                               int blk_kv, int topk, int causal, float softmax_scale, const msa_fwd_options *opts,
                               void *o, float *lse, void *workspace, size_t ws_bytes, uint32_t *status_dev,
                               cudaStream_t stream);

/* =========================================================================
 * (a5) block-sparse paged decode
 * =========================================================================
 * Source: interface.py sparse_decode_atten_func and
 * SparseDecodePagedAttentionWrapper (paged KV through page_table, seqused_k,
 * uniform seqlen_q per request, split-KV partials merged by LSE);
 * test_sparse_atten.py _decode_paged_kv_chunk (logical block j of sequence b
 * is physical page page_table[b][j]).
 *
 *   q          [B*Sq][Hq][D] bf16, device; query i of sequence b sits at
 *              position seqused_k[b] - Sq + i.
 *   k_pool, v_pool  [num_pages][page_size][Hkv][D] bf16, device.
 *   page_table [B][max_pages] int32, device.
 *   seqused_k  [B] int32, device (1 <= seqused_k[b] <= max_pages*page_size).
 *   q2k        [B][Hkv][Sq][topk] int32, device; ids >= ceil(seqused_k/page) are padding.
 *   o          [B*Sq][Hq][D] bf16; lse [B*Sq][Hq] fp32 or NULL.
 *   workspace  msa_sparse_attn_paged_fwd_workspace_size() bytes: per group
 *              its union of selected blocks with their pages and query
 *              masks, and per SM two 128-row pieces (O and LSE) of the
 *              groups the partition cuts.  The size depends on the current
 *              device's SM count.
 * The work, in two launches (one when there are at most as many groups as
 * SMs and no union can exceed 16 blocks: each CTA of the decode kernel then
 * plans its own group): per group (sequence b, KV head h, 128/(Hq/Hkv)
 * consecutive queries) the ascending union of the blocks its queries
 * selected (ids at or past ceil(seqused_k[b]/page) are padding and set
 * MSA_STATUS_INDEX_RANGE; repeats of one query set MSA_STATUS_DUPLICATE and
 * count once), each block's physical page (entries outside [0, num_pages)
 * set MSA_STATUS_PAGE_RANGE and the block is skipped) and the queries that
 * selected it; then one persistent kernel that streams each group's union
 * blocks through tensor-core attention with one accumulator per group (rows
 * of queries that did not select a block get no weight from it) and writes O
 * and LSE; a group split between CTAs is merged by LSE by the CTA that
 * finishes it last.  Max max_pages: 8192; at most 49152 groups.
 */
size_t msa_sparse_attn_paged_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages);
/*
 * Kernel launches one msa_sparse_attn_paged_fwd (topk > 0) or
 * msa_paged_attn_fwd (topk = 0: the dense mode) call of this shape makes on
 * the current device: 1 (the decode kernel plans each group itself) or 2
 * (the plan kernel, then the decode kernel).  Depends only on the shape and
 * the device's SM count, never on the data.  Returns MSA_ERR_INVALID_ARG or
 * MSA_ERR_UNSUPPORTED for a shape the calls reject.  Launches nothing.
 */
int msa_sparse_attn_paged_fwd_launches(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages);
int msa_sparse_attn_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                              const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                              const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size,
                              int topk, int causal, float softmax_scale, void *o, float *lse, void *workspace,
                              size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream);

/*
 * General paged decode: as msa_sparse_attn_paged_fwd, plus
 *   kv_format  MSA_KV_BF16, or MSA_KV_FP8 (pools of e4m3 bytes, staged to bf16
 *              on load, exact);
 *   q2k        NULL selects the dense mode (interface.py sparse_decode_atten_func
 *              with q2k_indices = None): every block of each sequence, i.e.
 *              causal attention over all seqused_k[b] keys; topk is then ignored.
 * The workspace is msa_paged_attn_fwd_workspace_size(..., topk, ...), with
 * topk = 0 for the dense mode.
 */
size_t msa_paged_attn_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages);
int msa_paged_attn_fwd(const void *q, const void *k_pool, const void *v_pool, int kv_format, int num_pages,
                       const int32_t *page_table, int max_pages, const int32_t *seqused_k, const int32_t *q2k, int B,
                       int Sq, int Hq, int Hkv, int D, int page_size, int topk, int causal, float softmax_scale,
                       void *o, float *lse, void *workspace, size_t ws_bytes, uint32_t *status_dev,
                       cudaStream_t stream);

/*
 * msa_sparse_attn_paged_fwd without a workspace argument: the same paged
 * decode (same arguments and output) computed by a per-group block-union
 * kernel whose scratch is small, with that scratch (unions, split counters
 * and partials) in a static device array of 32 MiB that every GPU loading
 * the library holds until exit.  The
 * source pages have no counterpart; it exists for callers that cannot
 * allocate device memory when they run a decode step (memory fixed at
 * start-up, or no cudaMalloc allowed while work is queued).
 *   - The first call on a device looks up the array's address on that
 *     device (make it before any stream capture); later calls allocate
 *     nothing and call no allocating routine.
 *   - Argument and support checks are those of msa_sparse_attn_paged_fwd
 *     and come first.  Then MSA_ERR_WORKSPACE is returned when the shape's
 *     union scratch needs more than 32 MiB.  With n = min(Sq,
 *     128/qhead_per_kv) queries per group, G = B * Hkv * ceil(Sq / n) groups
 *     and U = min(n * topk, max_pages) union slots per group, the scratch is
 *     G * U * (4 + 4 * ceil(n / 32)) bytes (block ids and query masks), plus
 *     8 bytes per group, plus 129 KB per SM (cut-group partials), each part
 *     rounded up to 256 bytes.
 *   - All calls share the one array: it keeps the last call's contents, the
 *     split counters are cleared on `stream` at the start of each call, and
 *     calls that overlap on the GPU (other streams, other host threads) race.
 */
int msa_sparse_attn_paged_fwd_noalloc(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                                      const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                      const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                      int topk, int causal, float softmax_scale, void *o, float *lse,
                                      uint32_t *status_dev, cudaStream_t stream);

/* =========================================================================
 * NVFP4 encoder for K/V rows (input side of MSA_KV_NVFP4)
 * =========================================================================
 * Source: interface.py sparse_atten_nvfp4_kv_func docstring (e2m1 data packed
 * two per byte, one e4m3 scale per 16 elements along D) and the vLLM
 * sparse-MLA test page (_E2M1_TABLE, unpack_e2m1).  Per group of 16:
 * scale = e4m3_rne_satfinite(amax / 6) (binary32 quotient), code =
 * e2m1_rne_satfinite(x / scale) (binary32 quotient); scale 0 -> codes 0.
 *   x       [rows][D] bf16, device; packed [rows][D/2]; scales [rows][D/16].
 */
int msa_nvfp4_quantize(const void *x, int64_t rows, int D, uint8_t *packed, uint8_t *scales,
                       cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H */
