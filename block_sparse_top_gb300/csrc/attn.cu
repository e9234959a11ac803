// attn.cu -- block-sparse prefill forward over the k->q CSR: per work unit
// (KV head h, KV block j of sequence b, a run of the queries that selected
// j) the K/V block is staged once in shared memory and every chunk of
// 128/qhead_per_kv queries (128 query-head rows, gathered from all heads of
// the GQA group) computes S = scale Q K^T, the single-block softmax
// (bottom-right causal mask on the diagonal block), O_p = P V / l and
// lse_p = m + ln l; the result goes to the query's split slot.  The LSE
// combine then merges the splits of every (query, head).
//
// Source: interface.py _sparse_atten_csr_varlen_forward (O_partial
// [topK,total_q,Hq,D] + LSE_partial, then combine) and
// test_sparse_atten.py sparse_attention_ref (mask, scale, LSE, empty rows).
// Here the partials are laid out [total_q][topk][D/8][Hq][8]: one query's
// splits are contiguous, and for a fixed 8-dim chunk the heads are
// contiguous, which makes both the tile stores and the combine reads whole
// runs.
#include <algorithm>
#include <cstring>

#include "attn_tc.cuh"

namespace msa {
namespace {

// LSE combine.  Partials are laid out [query][split][chunk c][query head][8
// dims]; one thread handles one (query, c, query head) item, so for each split
// the threads of a CTA read contiguous 16-byte pieces.
// O = sum_s exp(lse_s - LSE) O_s, LSE = logsumexp_s lse_s; a split with a
// non-finite lse has weight 0; no finite split -> O = 0, LSE = -inf.  All of
// an item's split pieces are loaded before they are summed.
template <int MAXS>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16 *__restrict__ o_part,
                                                      const float *__restrict__ lse_part,
                                                      const int32_t *__restrict__ split_counts, int64_t total_q,
                                                      int Hq, int Hkv, int topk, __nv_bfloat16 *__restrict__ o,
                                                      float *__restrict__ lse) {
    const int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t per_q = 16 * (int64_t)Hq;
    if (item >= total_q * per_q) return;
    const int64_t gq = item / per_q;
    const int rem = (int)(item % per_q);
    const int c = rem / Hq, hq = rem % Hq;
    const int h = hq / (Hq / Hkv);
    const int n = split_counts[gq * Hkv + h];
    const uint4 *src = reinterpret_cast<const uint4 *>(o_part) + (gq * topk * 16 + c) * Hq + hq;
    const int64_t split_stride = 16 * (int64_t)Hq;
    uint4 v[MAXS];
    float ls[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
        if (s < n) {
            v[s] = __ldcs(src + s * split_stride);
            ls[s] = __ldg(lse_part + (gq * topk + s) * Hq + hq);
        }
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
        if (s < n && isfinite(ls[s])) mx = fmaxf(mx, ls[s]);
    float den = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < MAXS; ++s) {
        if (s < n && isfinite(ls[s])) {
            const float w = __expf(ls[s] - mx);
            den += w;
            acc[0] += w * bf16_lo(v[s].x);
            acc[1] += w * bf16_hi(v[s].x);
            acc[2] += w * bf16_lo(v[s].y);
            acc[3] += w * bf16_hi(v[s].y);
            acc[4] += w * bf16_lo(v[s].z);
            acc[5] += w * bf16_hi(v[s].z);
            acc[6] += w * bf16_lo(v[s].w);
            acc[7] += w * bf16_hi(v[s].w);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint4 out;
    out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    reinterpret_cast<uint4 *>(o)[(gq * Hq + hq) * 16 + c] = out;
    if (c == 0 && lse) lse[gq * Hq + hq] = den > 0.f ? mx + logf(den) : -INFINITY;
}

struct FwdWorkspace {
    size_t o_part, lse_part, bytes;
};

FwdWorkspace fwd_workspace_layout(int B, int Sq, int Hq, int topk, int D) {
    FwdWorkspace w;
    size_t rows = (size_t)B * Sq * topk * Hq;
    w.o_part = 0;
    w.lse_part = align_up(rows * D * sizeof(__nv_bfloat16), 256);
    w.bytes = align_up(w.lse_part + rows * sizeof(float), 256);
    return w;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_attn_fwd_workspace_size(int B, int Sq, int Hq, int topk, int D) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || topk <= 0 || D != kD) return 0;
    return fwd_workspace_layout(B, Sq, Hq, topk, D).bytes;
}

extern "C" int msa_sparse_attn_fwd_partial(const void *q, const void *k, const void *v, int kv_format,
                                           const void *k_scales, const void *v_scales, const int32_t *q_indices,
                                           const int32_t *qsplit, const void *plan, int B, int Sq, int Skv, int Hq,
                                           int Hkv, int D, int blk_kv, int topk, int causal, float softmax_scale,
                                           void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                           cudaStream_t stream) {
    if (!q || !k || !v || !q_indices || !qsplit || !plan || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Skv <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv) return MSA_ERR_INVALID_ARG;
    if (kv_format != MSA_KV_BF16 && kv_format != MSA_KV_NVFP4) return MSA_ERR_INVALID_ARG;
    if (kv_format == MSA_KV_NVFP4 && (!k_scales || !v_scales)) return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || blk_kv != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)B * Sq >= (1 << 24)) return MSA_ERR_UNSUPPORTED;
    FwdWorkspace w = fwd_workspace_layout(B, Sq, Hq, topk, D);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(plan, 16)) return MSA_ERR_INVALID_ARG;

    const FwdWorkspace w_ = w;
    char *ws = static_cast<char *>(workspace);
    TcParams t;
    t.k_packed = static_cast<const uint8_t *>(k);
    t.v_packed = static_cast<const uint8_t *>(v);
    t.k_scales = static_cast<const uint8_t *>(k_scales);
    t.v_scales = static_cast<const uint8_t *>(v_scales);
    t.qsplit = qsplit;
    t.plan = static_cast<const PlanHeader *>(plan);
    t.units = reinterpret_cast<const PlanUnit *>(t.plan + 1);
    t.o_part = reinterpret_cast<__nv_bfloat16 *>(ws + w_.o_part);
    t.lse_part = reinterpret_cast<float *>(ws + w_.lse_part);
    t.status = status_dev;
    t.B = B; t.Sq = Sq; t.Skv = Skv; t.Hq = Hq; t.Hkv = Hkv; t.qpk = qpk; t.topk = topk;
    t.nblk = (int)ceil_div(Skv, kBlk);
    t.causal = causal ? 1 : 0;
    t.cap = (int64_t)B * Sq * topk;
    t.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    t.scale_log2 = t.scale * 1.4426950408889634f;
    (void)q_indices;

    const int sms = num_sms();
    int64_t capacity = plan_capacity(B, Hkv, Sq, Skv, topk, qpk);
    int grid = (int)std::min<int64_t>(capacity, (int64_t)sms);
    if (grid < 1) grid = 1;
    CUtensorMap mk, mv, mq;
    memset(&mk, 0, sizeof mk);
    memset(&mv, 0, sizeof mv);
    if (!make_q_map(&mq, q, (int64_t)B * Sq * Hq, qpk >= 8 ? qpk : 1)) return MSA_ERR_CUDA;
    const size_t smem = tck::kSmAlloc;
    if (kv_format == MSA_KV_BF16) {
        if (!make_kv_map(&mk, k, Hkv, (int64_t)B * Skv, (int64_t)Hkv * kD) ||
            !make_kv_map(&mv, v, Hkv, (int64_t)B * Skv, (int64_t)Hkv * kD))
            return MSA_ERR_CUDA;
        MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_tc_kernel<MSA_KV_BF16>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sparse_fwd_tc_kernel<MSA_KV_BF16><<<grid, tck::kThreads, smem, stream>>>(mk, mv, mq, t);
    } else {
        MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_tc_kernel<MSA_KV_NVFP4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sparse_fwd_tc_kernel<MSA_KV_NVFP4><<<grid, tck::kThreads, smem, stream>>>(mk, mv, mq, t);
    }
    MSA_LAUNCH_CHECK();
    return MSA_OK;
}

extern "C" int msa_sparse_attn_combine(const int32_t *split_counts, int B, int Sq, int Hq, int Hkv, int D, int topk,
                                       void *o, float *lse, const void *workspace, size_t ws_bytes,
                                       cudaStream_t stream) {
    if (!split_counts || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv) return MSA_ERR_INVALID_ARG;
    if (D != kD || !supported_topk(topk)) return MSA_ERR_UNSUPPORTED;
    FwdWorkspace w = fwd_workspace_layout(B, Sq, Hq, topk, D);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (!aligned(o, 16)) return MSA_ERR_INVALID_ARG;
    const char *ws = static_cast<const char *>(workspace);
    int64_t items = (int64_t)B * Sq * Hq * 16;
    int64_t blocks = ceil_div(items, 256);
    const __nv_bfloat16 *op = reinterpret_cast<const __nv_bfloat16 *>(ws + w.o_part);
    const float *lp = reinterpret_cast<const float *>(ws + w.lse_part);
    __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(o);
    if (topk <= 16)
        combine_kernel<16><<<(unsigned)blocks, 256, 0, stream>>>(op, lp, split_counts, (int64_t)B * Sq, Hq, Hkv,
                                                                 topk, ob, lse);
    else
        combine_kernel<32><<<(unsigned)blocks, 256, 0, stream>>>(op, lp, split_counts, (int64_t)B * Sq, Hq, Hkv,
                                                                 topk, ob, lse);
    MSA_LAUNCH_CHECK();
    return MSA_OK;
}

extern "C" int msa_sparse_attn_fwd(const void *q, const void *k, const void *v, int kv_format, const void *k_scales,
                                   const void *v_scales, const int32_t *row_ptr, const int32_t *q_indices,
                                   const int32_t *qsplit, const int32_t *split_counts, const void *plan, int B,
                                   int Sq, int Skv, int Hq, int Hkv, int D, int blk_kv, int topk, int causal,
                                   float softmax_scale, void *o, float *lse, void *workspace, size_t ws_bytes,
                                   uint32_t *status_dev, cudaStream_t stream) {
    (void)row_ptr;
    if (!split_counts || !o) return MSA_ERR_INVALID_ARG;
    int rc = msa_sparse_attn_fwd_partial(q, k, v, kv_format, k_scales, v_scales, q_indices, qsplit, plan, B, Sq, Skv,
                                         Hq, Hkv, D, blk_kv, topk, causal, softmax_scale, workspace, ws_bytes,
                                         status_dev, stream);
    if (rc != MSA_OK) return rc;
    return msa_sparse_attn_combine(split_counts, B, Sq, Hq, Hkv, D, topk, o, lse, workspace, ws_bytes, stream);
}
