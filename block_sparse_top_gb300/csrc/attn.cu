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
// Here the partials are laid out [total_q][topk][Hq][D] so that one
// query's splits are contiguous for the combine.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "attn_mma.cuh"
#include "attn_tc.cuh"

namespace msa {
namespace {

struct FwdParams {
    const __nv_bfloat16 *q;
    const void *k, *v;            // bf16 [B][Skv][Hkv][D] or packed NVFP4 [B][Skv][Hkv][D/2]
    const uint8_t *k_scales, *v_scales;
    const int32_t *q_indices, *qsplit;
    const PlanHeader *plan;
    const PlanUnit *units;
    __nv_bfloat16 *o_part;        // [B*Sq][topk][Hq][D]
    float *lse_part;              // [B*Sq][topk][Hq]
    int B, Sq, Skv, Hq, Hkv, qpk, topk, nblk, causal;
    int64_t cap;                  // q_indices row length
    float scale_log2;             // softmax_scale * log2(e)
    float scale;
};

// Stages the K or V block (128 tokens of one KV head) into a swizzled tile;
// tokens past Skv are zero-filled (masked later).
template <int KV_FORMAT>
__device__ void load_kv_tile(uint32_t dst, const void *src, const uint8_t *scales, const FwdParams &p, int b, int h,
                             int tok0) {
    if (KV_FORMAT == MSA_KV_BF16) {
        const __nv_bfloat16 *base = static_cast<const __nv_bfloat16 *>(src);
        for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
            int r = i >> 4, c = i & 15;
            int t = tok0 + r;
            bool ok = t < p.Skv;
            const __nv_bfloat16 *g = base + (((int64_t)b * p.Skv + (ok ? t : 0)) * p.Hkv + h) * kD + c * 8;
            cp_async16(dst + swz_off(r, c), g, ok);
        }
    } else {
        const uint8_t *base = static_cast<const uint8_t *>(src);
        for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
            int r = i >> 3, g = i & 7;
            int t = tok0 + r;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (t < p.Skv) {
                int64_t row = ((int64_t)b * p.Skv + t) * p.Hkv + h;
                uint2 pk = *reinterpret_cast<const uint2 *>(base + row * (kD / 2) + g * 8);
                uint32_t sb = scales[row * (kD / 16) + g];
                nvfp4_group_to_bf16(pk, sb, lo, hi);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst + swz_off(r, 2 * g)), "r"(lo.x),
                         "r"(lo.y), "r"(lo.z), "r"(lo.w));
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst + swz_off(r, 2 * g + 1)), "r"(hi.x),
                         "r"(hi.y), "r"(hi.z), "r"(hi.w));
        }
    }
}

// Warp-MMA prefill kernel (8 warps, one 16-row slice of the 128-row chunk each).
template <int KV_FORMAT>
__global__ void __launch_bounds__(256, 1) sparse_fwd_mma_kernel(FwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t k_s = smem_u32(smem), v_s = k_s + 32768, q_s = k_s + 65536;
    __shared__ int32_t row_q[128];      // global query id of each chunk row (-1: empty)
    __shared__ int32_t row_split[128];  // split slot of each chunk row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qc = 128 / p.qpk;         // queries per chunk
    const int work = p.plan->work_count;

    for (int u = blockIdx.x; u < work; u += gridDim.x) {
        const PlanUnit unit = p.units[u];
        const int h = unit.head, b = unit.row / p.nblk, j = unit.row % p.nblk;
        const int tok0 = j * kBlk;
        __syncthreads();  // previous unit done with K/V
        load_kv_tile<KV_FORMAT>(k_s, p.k, p.k_scales, p, b, h, tok0);
        load_kv_tile<KV_FORMAT>(v_s, p.v, p.v_scales, p, b, h, tok0);
        cp_async_commit();
        const int nchunks = (unit.count + qc - 1) / qc;
        for (int c = 0; c < nchunks; ++c) {
            __syncthreads();  // previous chunk done with Q and row tables
            if (threadIdx.x < 128) {
                int R = threadIdx.x, qi = R / p.qpk;
                int idx = c * qc + qi;
                int gq = -1, sp = 0;
                if (idx < unit.count) {
                    int packed = p.qsplit[(int64_t)h * p.cap + unit.start + idx];
                    gq = packed & 0xFFFFFF;
                    sp = (packed >> 24) & 0xFF;
                }
                row_q[R] = gq;
                row_split[R] = sp;
            }
            __syncthreads();
            for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
                int R = i >> 4, ch = i & 15;
                int gq = row_q[R];
                int hq = h * p.qpk + (R % p.qpk);
                const __nv_bfloat16 *g = p.q + ((int64_t)(gq < 0 ? 0 : gq) * p.Hq + hq) * kD + ch * 8;
                cp_async16(q_s + swz_off(R, ch), g, gq >= 0);
            }
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();

            const int row0 = warp * 16;
            float s[16][4];
            warp_qk(q_s, k_s, row0, s);

            // per-row visibility: keys tok0 + k with k < nvis
            const int g = lane >> 2, t = lane & 3;
            int nvis[2];
            float m[2], l[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                int R = row0 + g + 8 * hr;
                int gq = row_q[R];
                int n = 0;
                if (gq >= 0) {
                    int sq = gq % p.Sq;
                    int64_t limit = (int64_t)p.Skv - 1;
                    if (p.causal) limit = std::min<int64_t>(limit, (int64_t)sq + (p.Skv - p.Sq));
                    int64_t nv = limit - tok0 + 1;
                    n = (int)std::max<int64_t>(0, std::min<int64_t>(128, nv));
                }
                nvis[hr] = n;
                m[hr] = -INFINITY;
            }
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int hr = e >> 1;
                    int key = nt * 8 + 2 * t + (e & 1);
                    if (key >= nvis[hr]) s[nt][e] = -INFINITY;
                    m[hr] = fmaxf(m[hr], s[nt][e]);
                }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                m[hr] = fmaxf(m[hr], __shfl_xor_sync(0xffffffffu, m[hr], 1));
                m[hr] = fmaxf(m[hr], __shfl_xor_sync(0xffffffffu, m[hr], 2));
                l[hr] = 0.f;
            }
            uint32_t pk[16][2];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                float pe[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int hr = e >> 1;
                    float x = (m[hr] == -INFINITY) ? 0.f : ex2_approx((s[nt][e] - m[hr]) * p.scale_log2);
                    pe[e] = x;
                    l[hr] += x;
                }
                pk[nt][0] = pack_bf16x2(pe[0], pe[1]);
                pk[nt][1] = pack_bf16x2(pe[2], pe[3]);
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
                l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
            }
            float o[16][4];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
            warp_pv(v_s, pk, o);

#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                int R = row0 + g + 8 * hr;
                int gq = row_q[R];
                if (gq < 0) continue;
                int hq = h * p.qpk + (R % p.qpk);
                int64_t slot = ((int64_t)gq * p.topk + row_split[R]) * p.Hq + hq;
                float inv = l[hr] > 0.f ? 1.f / l[hr] : 0.f;
                __nv_bfloat16 *orow = p.o_part + slot * kD;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    uint32_t w = pack_bf16x2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
                    *reinterpret_cast<uint32_t *>(orow + nt * 8 + 2 * t) = w;
                }
                if (t == 0)
                    p.lse_part[slot] = (l[hr] > 0.f) ? (m[hr] * p.scale + logf(l[hr])) : -INFINITY;
            }
        }
    }
}

// LSE combine: one warp per (query, query head); lane covers 4 of the 128 dims.
// O = sum_s exp(lse_s - LSE) O_s, LSE = logsumexp_s lse_s; a split with a
// non-finite lse has weight 0; no finite split -> O = 0, LSE = -inf.
__global__ void combine_kernel(const __nv_bfloat16 *__restrict__ o_part, const float *__restrict__ lse_part,
                               const int32_t *__restrict__ split_counts, int64_t total_q, int Hq, int Hkv,
                               int topk, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
    int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (wid >= total_q * Hq) return;
    int64_t gq = wid / Hq;
    int hq = (int)(wid % Hq);
    int h = hq / (Hq / Hkv);
    int n = split_counts[gq * Hkv + h];
    float ls = -INFINITY;
    if (lane < n) ls = lse_part[(gq * topk + lane) * Hq + hq];
    float mx = ls;
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o_));
    float w = (isfinite(ls) && isfinite(mx)) ? __expf(ls - mx) : 0.f;
    float den = w;
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o_);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float inv = den > 0.f ? 1.f / den : 0.f;
    for (int s = 0; s < n; ++s) {
        float ws = __shfl_sync(0xffffffffu, w, s) * inv;
        if (ws == 0.f) continue;
        uint2 v = *reinterpret_cast<const uint2 *>(o_part + ((gq * topk + s) * Hq + hq) * kD + lane * 4);
        acc[0] += ws * bf16_lo(v.x);
        acc[1] += ws * bf16_hi(v.x);
        acc[2] += ws * bf16_lo(v.y);
        acc[3] += ws * bf16_hi(v.y);
    }
    uint2 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[2], acc[3]);
    *reinterpret_cast<uint2 *>(o + (gq * Hq + hq) * kD + lane * 4) = out;
    if (lane == 0 && lse) lse[gq * Hq + hq] = den > 0.f ? mx + logf(den) : -INFINITY;
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

// The warp-MMA kernel stays selectable while the tensor-core kernel is
// validated: MSA_PREFILL_KERNEL=mma.
bool use_legacy_mma() {
    const char *e = getenv("MSA_PREFILL_KERNEL");
    return e && e[0] == 'm';
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

    FwdParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = k;
    p.v = v;
    p.k_scales = static_cast<const uint8_t *>(k_scales);
    p.v_scales = static_cast<const uint8_t *>(v_scales);
    p.q_indices = q_indices;
    p.qsplit = qsplit;
    p.plan = static_cast<const PlanHeader *>(plan);
    p.units = reinterpret_cast<const PlanUnit *>(p.plan + 1);
    char *ws = static_cast<char *>(workspace);
    p.o_part = reinterpret_cast<__nv_bfloat16 *>(ws + w.o_part);
    p.lse_part = reinterpret_cast<float *>(ws + w.lse_part);
    p.B = B; p.Sq = Sq; p.Skv = Skv; p.Hq = Hq; p.Hkv = Hkv; p.qpk = qpk; p.topk = topk;
    p.nblk = (int)ceil_div(Skv, kBlk);
    p.causal = causal ? 1 : 0;
    p.cap = (int64_t)B * Sq * topk;
    float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;

    const int sms = num_sms();
    int64_t capacity = plan_capacity(B, Hkv, Sq, Skv, topk, qpk);
    int grid = (int)std::min<int64_t>(capacity, (int64_t)sms);
    if (grid < 1) grid = 1;
    if (use_legacy_mma()) {
        const size_t smem = 3 * 32768 + 1024;
        if (kv_format == MSA_KV_BF16) {
            MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_mma_kernel<MSA_KV_BF16>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            sparse_fwd_mma_kernel<MSA_KV_BF16><<<grid, 256, smem, stream>>>(p);
        } else {
            MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_mma_kernel<MSA_KV_NVFP4>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            sparse_fwd_mma_kernel<MSA_KV_NVFP4><<<grid, 256, smem, stream>>>(p);
        }
        MSA_LAUNCH_CHECK();
        return MSA_OK;
    }
    TcParams t;
    t.q = p.q;
    t.k_packed = static_cast<const uint8_t *>(k);
    t.v_packed = static_cast<const uint8_t *>(v);
    t.k_scales = p.k_scales;
    t.v_scales = p.v_scales;
    t.qsplit = qsplit;
    t.plan = p.plan;
    t.units = p.units;
    t.o_part = p.o_part;
    t.lse_part = p.lse_part;
    t.status = status_dev;
    t.B = B; t.Sq = Sq; t.Skv = Skv; t.Hq = Hq; t.Hkv = Hkv; t.qpk = qpk; t.topk = topk;
    t.nblk = p.nblk; t.causal = p.causal; t.cap = p.cap; t.scale = p.scale; t.scale_log2 = p.scale_log2;
    CUtensorMap mk, mv;
    memset(&mk, 0, sizeof mk);
    memset(&mv, 0, sizeof mv);
    const size_t smem = tck::kSmAlloc;
    if (kv_format == MSA_KV_BF16) {
        if (!make_kv_map(&mk, k, Hkv, (int64_t)B * Skv, (int64_t)Hkv * kD) ||
            !make_kv_map(&mv, v, Hkv, (int64_t)B * Skv, (int64_t)Hkv * kD))
            return MSA_ERR_CUDA;
        MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_tc_kernel<MSA_KV_BF16>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sparse_fwd_tc_kernel<MSA_KV_BF16><<<grid, tck::kThreads, smem, stream>>>(mk, mv, t);
    } else {
        MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_tc_kernel<MSA_KV_NVFP4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sparse_fwd_tc_kernel<MSA_KV_NVFP4><<<grid, tck::kThreads, smem, stream>>>(mk, mv, t);
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
    int64_t warps = (int64_t)B * Sq * Hq;
    int64_t blocks = ceil_div(warps * 32, 256);
    combine_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16 *>(ws + w.o_part), reinterpret_cast<const float *>(ws + w.lse_part),
        split_counts, (int64_t)B * Sq, Hq, Hkv, topk, static_cast<__nv_bfloat16 *>(o), lse);
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
