// decode.cu -- block-sparse paged decode: for every (sequence b, KV head h,
// group of 128/qhead_per_kv queries) the union of the KV blocks the group's
// queries selected is split over `nsplit` CTAs.  Each CTA streams its share
// of the union from the paged pool (logical block j -> physical page
// page_table[b][j], token rows of Hkv*D bf16) through a two-stage cp.async
// pipeline, and every warp runs an online softmax over the blocks its
// queries selected (rows of queries that did not select a block are masked).
// The CTA that finishes last (atomic counter) merges the split partials by
// LSE and writes O and LSE.
//
// Source: interface.py sparse_decode_atten_func and
// SparseDecodePagedAttentionWrapper (paged KV, seqused_k, uniform seqlen_q,
// split-KV partials merged by LSE); test_sparse_atten.py
// _decode_paged_dense_reference (running max/sum per chunk, lse = m + log l,
// -inf for empty rows) and _decode_paged_kv_chunk (page-table addressing).
#include <algorithm>

#include "attn_mma.cuh"

namespace msa {
namespace {

constexpr int kMaxPagesDecode = 8192;  // union bitmap bound (1M tokens per sequence)

struct DecParams {
    const __nv_bfloat16 *q, *k_pool, *v_pool;
    const int32_t *page_table, *seqused, *q2k;
    __nv_bfloat16 *o;
    float *lse;
    float *o_part;         // [B][Hkv][qgroups][nsplit][128][D]
    float *lse_part;       // [B][Hkv][qgroups][nsplit][128]
    int32_t *counters;     // [B][Hkv][qgroups]
    uint32_t *status;
    int B, Sq, Hq, Hkv, qpk, topk, num_pages, max_pages, causal, qgroups, nsplit;
    float scale, scale_log2;
};

__global__ void __launch_bounds__(256, 1) sparse_decode_kernel(DecParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t q_s = smem_u32(smem);
    const uint32_t kv_s = q_s + 32768;  // stage s: K at kv_s + s*65536, V at +32768
    __shared__ uint32_t bitmap[kMaxPagesDecode / 32];
    __shared__ int32_t ulist[128 * 32];    // union of the group's blocks (<= queries x topk)
    __shared__ int32_t qsel[128 * 32];  // per query of the group: its valid block ids (-1 pad)
    __shared__ int32_t warp_tot[8];
    __shared__ int32_t s_nu;
    __shared__ int32_t s_last;

    const int split = blockIdx.x, h = blockIdx.y % p.Hkv, grp = blockIdx.y / p.Hkv, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qg = 128 / p.qpk;                    // queries per group
    const int q0 = grp * qg;                       // first local query of the group
    const int nq = min(qg, p.Sq - q0);
    const int seqused = p.seqused[b];
    const int nvalid = (int)(ceil_div(seqused, kBlk) < p.max_pages ? ceil_div(seqused, kBlk) : p.max_pages);
    const int nwords = (nvalid + 31) / 32;

    // 1. per-query valid block lists and the union bitmap
    for (int i = threadIdx.x; i < nwords; i += blockDim.x) bitmap[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < qg * p.topk; i += blockDim.x) {
        int qi = i / p.topk, t = i % p.topk;
        int j = -1;
        if (qi < nq) {
            const int32_t *sel = p.q2k + (((int64_t)b * p.Hkv + h) * p.Sq + q0 + qi) * p.topk;
            j = sel[t];
            if (j >= nvalid) {
                set_status(p.status, MSA_STATUS_INDEX_RANGE);
                j = -1;
            }
            if (j >= 0)
                for (int u = 0; u < t; ++u)
                    if (sel[u] == j) {
                        set_status(p.status, MSA_STATUS_DUPLICATE);
                        j = -1;
                        break;
                    }
            if (j >= 0) atomicOr(&bitmap[j >> 5], 1u << (j & 31));
        }
        qsel[qi * 32 + t] = j;
    }
    __syncthreads();
    // 2. compact the union in ascending block order
    {
        int per = (nwords + blockDim.x - 1) / blockDim.x;
        int w0 = threadIdx.x * per, w1 = min(w0 + per, nwords);
        int cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(bitmap[w]);
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += warp_tot[w];
        int pos = base + x - cnt;
        for (int w = w0; w < w1; ++w) {
            uint32_t m = bitmap[w];
            while (m) {
                int bit = __ffs(m) - 1;
                m &= m - 1;
                ulist[pos++] = w * 32 + bit;
            }
        }
        if (threadIdx.x == blockDim.x - 1) s_nu = pos;
    }
    __syncthreads();
    const int nu = s_nu;
    const int per_split = (nu + p.nsplit - 1) / p.nsplit;
    const int e0 = min(nu, split * per_split), e1 = min(nu, e0 + per_split);

    // 3. Q rows of the group (row R = qi*qpk + g)
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
        int R = i >> 4, ch = i & 15;
        int qi = R / p.qpk;
        bool ok = qi < nq;
        int64_t gq = (int64_t)b * p.Sq + q0 + (ok ? qi : 0);
        const __nv_bfloat16 *g = p.q + (gq * p.Hq + h * p.qpk + R % p.qpk) * kD + ch * 8;
        cp_async16(q_s + swz_off(R, ch), g, ok);
    }
    cp_async_commit();

    auto issue_block = [&](int e, int stage) {
        int j = ulist[e];
        int page = p.page_table[(int64_t)b * p.max_pages + j];
        bool pok = page >= 0 && page < p.num_pages;
        if (!pok && threadIdx.x == 0) set_status(p.status, MSA_STATUS_PAGE_RANGE);
        uint32_t ks = kv_s + stage * 65536, vs = ks + 32768;
        for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
            int r = i >> 4, ch = i & 15;
            bool ok = pok && (j * kBlk + r) < seqused;
            int64_t off = (((int64_t)(ok ? page : 0) * kBlk + r) * p.Hkv + h) * kD + ch * 8;
            cp_async16(ks + swz_off(r, ch), p.k_pool + off, ok);
            cp_async16(vs + swz_off(r, ch), p.v_pool + off, ok);
        }
    };

    // per-thread online softmax state for rows g and g + 8 of the warp slice
    const int g = lane >> 2, t = lane & 3;
    const int row0 = warp * 16;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    int qi_row[2], limit_row[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        int R = row0 + g + 8 * hr;
        qi_row[hr] = R / p.qpk;
        int pos = seqused - p.Sq + q0 + qi_row[hr];   // position of the query
        limit_row[hr] = p.causal ? min(pos, seqused - 1) : seqused - 1;
    }
    const int wq0 = row0 / p.qpk, wq1 = (row0 + 15) / p.qpk;  // queries of this warp

    if (e0 < e1) issue_block(e0, 0);
    cp_async_commit();
    for (int e = e0; e < e1; ++e) {
        const int stage = (e - e0) & 1;
        if (e + 1 < e1) issue_block(e + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int j = ulist[e];
        const int page = p.page_table[(int64_t)b * p.max_pages + j];
        const bool pok = page >= 0 && page < p.num_pages;
        // does any query of this warp select block j?
        bool any = false;
        for (int qi = wq0; qi <= wq1 && qi < nq; ++qi)
            for (int tt = 0; tt < p.topk; ++tt) any |= (qsel[qi * 32 + tt] == j);
        if (pok && any) {
            uint32_t ks = kv_s + stage * 65536, vs = ks + 32768;
            float s[16][4];
            warp_qk(q_s, ks, row0, s);
            int nvis[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                bool sel = false;
                if (qi_row[hr] < nq)
                    for (int tt = 0; tt < p.topk; ++tt) sel |= (qsel[qi_row[hr] * 32 + tt] == j);
                nvis[hr] = sel ? max(0, min(128, limit_row[hr] - j * kBlk + 1)) : 0;
            }
            float mnew[2] = {m[0], m[1]};
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int ee = 0; ee < 4; ++ee) {
                    int hr = ee >> 1;
                    int key = nt * 8 + 2 * t + (ee & 1);
                    if (key >= nvis[hr]) s[nt][ee] = -INFINITY;
                    mnew[hr] = fmaxf(mnew[hr], s[nt][ee]);
                }
            float corr[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                mnew[hr] = fmaxf(mnew[hr], __shfl_xor_sync(0xffffffffu, mnew[hr], 1));
                mnew[hr] = fmaxf(mnew[hr], __shfl_xor_sync(0xffffffffu, mnew[hr], 2));
                corr[hr] = (m[hr] == -INFINITY) ? 0.f : ex2_approx((m[hr] - mnew[hr]) * p.scale_log2);
                if (mnew[hr] == -INFINITY) corr[hr] = 1.f;
                l[hr] *= corr[hr];
                m[hr] = mnew[hr];
            }
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= corr[0];
                o[nt][1] *= corr[0];
                o[nt][2] *= corr[1];
                o[nt][3] *= corr[1];
            }
            uint32_t pk[16][2];
            float lsum[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                float pe[4];
#pragma unroll
                for (int ee = 0; ee < 4; ++ee) {
                    int hr = ee >> 1;
                    float x = (m[hr] == -INFINITY) ? 0.f : ex2_approx((s[nt][ee] - m[hr]) * p.scale_log2);
                    pe[ee] = x;
                    lsum[hr] += x;
                }
                pk[nt][0] = pack_bf16x2(pe[0], pe[1]);
                pk[nt][1] = pack_bf16x2(pe[2], pe[3]);
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                lsum[hr] += __shfl_xor_sync(0xffffffffu, lsum[hr], 1);
                lsum[hr] += __shfl_xor_sync(0xffffffffu, lsum[hr], 2);
                l[hr] += lsum[hr];
            }
            warp_pv(vs, pk, o);
        }
        __syncthreads();  // stage may be overwritten next iteration
    }
    cp_async_wait<0>();

    // 4. write this split's partial (normalised O, lse) or the final result
    const int64_t grp_id = ((int64_t)b * p.Hkv + h) * p.qgroups + grp;
    const bool direct = (p.nsplit == 1);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        int R = row0 + g + 8 * hr;
        float inv = l[hr] > 0.f ? 1.f / l[hr] : 0.f;
        float lse_v = l[hr] > 0.f ? m[hr] * p.scale + logf(l[hr]) : -INFINITY;
        if (direct) {
            if (qi_row[hr] >= nq) continue;
            int64_t gq = (int64_t)b * p.Sq + q0 + qi_row[hr];
            int hq = h * p.qpk + R % p.qpk;
            __nv_bfloat16 *orow = p.o + (gq * p.Hq + hq) * kD;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<uint32_t *>(orow + nt * 8 + 2 * t) =
                    pack_bf16x2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            if (t == 0 && p.lse) p.lse[gq * p.Hq + hq] = lse_v;
        } else {
            float *orow = p.o_part + ((grp_id * p.nsplit + split) * 128 + R) * kD;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<float2 *>(orow + nt * 8 + 2 * t) =
                    make_float2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            if (t == 0) p.lse_part[(grp_id * p.nsplit + split) * 128 + R] = lse_v;
        }
    }
    if (direct) return;

    // 5. last-arriving split merges all partials of the group
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        int prev = atomicAdd(&p.counters[grp_id], 1);
        s_last = (prev == p.nsplit - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    {
        int R = threadIdx.x >> 1, half = threadIdx.x & 1;
        int qi = R / p.qpk;
        float mx = -INFINITY;
        for (int sp = 0; sp < p.nsplit; ++sp)
            mx = fmaxf(mx, __ldcg(p.lse_part + (grp_id * p.nsplit + sp) * 128 + R));
        float den = 0.f;
        float acc[64];
#pragma unroll
        for (int d = 0; d < 64; ++d) acc[d] = 0.f;
        for (int sp = 0; sp < p.nsplit; ++sp) {
            float ls = __ldcg(p.lse_part + (grp_id * p.nsplit + sp) * 128 + R);
            if (!(ls > -INFINITY) || !(mx > -INFINITY)) continue;
            float w = __expf(ls - mx);
            den += w;
            const float4 *src =
                reinterpret_cast<const float4 *>(p.o_part + ((grp_id * p.nsplit + sp) * 128 + R) * kD + half * 64);
#pragma unroll
            for (int d4 = 0; d4 < 16; ++d4) {
                float4 v = __ldcg(src + d4);
                acc[4 * d4] += w * v.x;
                acc[4 * d4 + 1] += w * v.y;
                acc[4 * d4 + 2] += w * v.z;
                acc[4 * d4 + 3] += w * v.w;
            }
        }
        if (qi < nq) {
            int64_t gq = (int64_t)b * p.Sq + q0 + qi;
            int hq = h * p.qpk + R % p.qpk;
            float inv = den > 0.f ? 1.f / den : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + (gq * p.Hq + hq) * kD + half * 64);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                dst[c] = make_uint4(pack_bf16x2(acc[8 * c] * inv, acc[8 * c + 1] * inv),
                                    pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv),
                                    pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv),
                                    pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv));
            if (half == 0 && p.lse) p.lse[gq * p.Hq + hq] = den > 0.f ? mx + logf(den) : -INFINITY;
        }
    }
    if (threadIdx.x == 0) p.counters[grp_id] = 0;  // ready for the next call
}

struct DecWorkspace {
    size_t counters, lse_part, o_part, bytes;
};

DecWorkspace dec_workspace_layout(int B, int Hkv, int qgroups, int nsplit) {
    DecWorkspace w;
    size_t groups = (size_t)B * Hkv * qgroups;
    w.counters = 0;
    w.lse_part = align_up(groups * sizeof(int32_t), 256);
    w.o_part = align_up(w.lse_part + groups * nsplit * 128 * sizeof(float), 256);
    w.bytes = align_up(w.o_part + groups * nsplit * 128 * (size_t)kD * sizeof(float), 256);
    return w;
}

int decode_num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

// Splits per group: enough CTAs for about two per SM, never more than the
// largest possible union of blocks.
int choose_nsplit(int B, int Hkv, int qgroups, int Sq, int qpk, int topk, int max_pages) {
    int64_t groups = (int64_t)B * Hkv * qgroups;
    int64_t target = 2 * (int64_t)decode_num_sms();
    int64_t ns = ceil_div(target, groups);
    int64_t max_union = std::min<int64_t>((int64_t)std::min(Sq, 128 / qpk) * topk, max_pages);
    ns = std::max<int64_t>(1, std::min<int64_t>(ns, std::max<int64_t>(1, max_union)));
    return (int)std::min<int64_t>(ns, 64);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_attn_paged_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk,
                                                           int max_pages) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || D != kD || topk <= 0 || max_pages <= 0 || Hq % Hkv) return 0;
    int qpk = Hq / Hkv;
    if (!supported_qpk(qpk)) return 0;
    int qgroups = (int)ceil_div(Sq, 128 / qpk);
    int ns = choose_nsplit(B, Hkv, qgroups, Sq, qpk, topk, max_pages);
    return dec_workspace_layout(B, Hkv, qgroups, ns).bytes;
}

extern "C" int msa_sparse_attn_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                                         const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                         const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                         int topk, int causal, float softmax_scale, void *o, float *lse,
                                         void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                         cudaStream_t stream) {
    if (!q || !k_pool || !v_pool || !page_table || !seqused_k || !q2k || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pages <= 0 || topk <= 0 || Hq % Hkv)
        return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || page_size != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if (max_pages > kMaxPagesDecode) return MSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return MSA_ERR_INVALID_ARG;
    const int qgroups = (int)ceil_div(Sq, 128 / qpk);
    const int nsplit = choose_nsplit(B, Hkv, qgroups, Sq, qpk, topk, max_pages);
    DecWorkspace w = dec_workspace_layout(B, Hkv, qgroups, nsplit);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);

    DecParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.page_table = page_table;
    p.seqused = seqused_k;
    p.q2k = q2k;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.counters = reinterpret_cast<int32_t *>(ws + w.counters);
    p.lse_part = reinterpret_cast<float *>(ws + w.lse_part);
    p.o_part = reinterpret_cast<float *>(ws + w.o_part);
    p.status = status_dev;
    p.B = B; p.Sq = Sq; p.Hq = Hq; p.Hkv = Hkv; p.qpk = qpk; p.topk = topk;
    p.num_pages = num_pages; p.max_pages = max_pages; p.causal = causal ? 1 : 0;
    p.qgroups = qgroups; p.nsplit = nsplit;
    float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;

    if (nsplit > 1)
        MSA_CUDA_TRY(cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * (size_t)B * Hkv * qgroups, stream));
    const size_t smem = 32768 + 2 * 65536;
    MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid(nsplit, Hkv * qgroups, B);
    sparse_decode_kernel<<<grid, 256, smem, stream>>>(p);
    MSA_LAUNCH_CHECK();
    return MSA_OK;
}

// ---------------------------------------------------------------------------
// Paged decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: a serving loop whose memory is fixed at start-up, or code that
// must not call cudaMalloc while other work is queued.  This variant keeps
// its scratch (split counters and partials) in one file-scope device array of
// kNoAllocScratchBytes, which every GPU that loads the library holds until
// the process exits.  The array's address is looked up once per device with
// that device current (cudaGetSymbolAddress), on the first call made on that
// device.  Calls share the array: the split counters are cleared on the
// stream at the start of each call, and calls that overlap on the GPU race
// for it.
// ---------------------------------------------------------------------------
#include <mutex>

namespace msa {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_paged_scratch[kNoAllocScratchBytes];

// Device address of g_paged_scratch on the current device; nullptr on error.
void *paged_scratch_for_current_device() {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_paged_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace
}  // namespace msa

extern "C" int msa_sparse_attn_paged_fwd_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                                 int num_pages, const int32_t *page_table, int max_pages,
                                                 const int32_t *seqused_k, const int32_t *q2k, int B, int Sq,
                                                 int Hq, int Hkv, int D, int page_size, int topk, int causal,
                                                 float softmax_scale, void *o, float *lse, uint32_t *status_dev,
                                                 cudaStream_t stream) {
    size_t need = msa_sparse_attn_paged_fwd_workspace_size(B, Sq, Hq, Hkv, D, topk, max_pages);
    if (need == 0) return MSA_ERR_UNSUPPORTED;
    if (need > msa::kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // shape needs more than the static scratch
    void *scratch = msa::paged_scratch_for_current_device();
    if (!scratch) return MSA_ERR_CUDA;
    return msa_sparse_attn_paged_fwd(q, k_pool, v_pool, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq, Hq,
                                     Hkv, D, page_size, topk, causal, softmax_scale, o, lse, scratch,
                                     msa::kNoAllocScratchBytes, status_dev, stream);
}
