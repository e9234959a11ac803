// paged.cu -- block-sparse and dense paged decode (msa_sparse_attn_paged_fwd,
// msa_paged_attn_fwd): the union plan kernel and the host side of the
// two-launch decode whose kernel is in paged_tc.cuh.
#include <algorithm>
#include <cstring>

#include "paged_tc.cuh"
#include "tiles.h"  // num_sms

namespace msa {

// ---------------------------------------------------------------------------
// plan: one CTA (256 threads) per group; the plan itself is plan_group
// (paged_tc.cuh), which the decode kernel's local-plan mode runs too.
// Dynamic shared memory: plan_scratch_words words.
__global__ void __launch_bounds__(256) paged_plan_kernel(DecodeParams p) {
    extern __shared__ uint32_t dsm[];
    grid_dependency_wait();  // the previous call's decode kernel may still read this workspace
    grid_dependents_launch();
    pdk::plan_group<256>(p, blockIdx.x, dsm);
}

namespace {

struct DecodeShape {
    int qpk, qc, qgroups, G, maxu, wq, grid;
};

// sparse: topk > 0; dense: topk == 0 (every block)
DecodeShape decode_shape(int B, int Sq, int Hq, int Hkv, int topk, int max_pages) {
    DecodeShape d;
    d.qpk = Hq / Hkv;
    d.qc = 128 / d.qpk;
    d.qgroups = (int)ceil_div(Sq, d.qc);
    d.G = B * Hkv * d.qgroups;
    d.maxu = topk > 0 ? std::min(std::min(Sq, d.qc) * topk, max_pages) : max_pages;
    d.wq = (d.qc + 31) / 32;
    d.grid = num_sms();
    return d;
}

struct DecodeWorkspace {
    size_t nunits, merge_cnt, ublk, upage, umask, slot_o, slot_lse, bytes;
};

DecodeWorkspace decode_workspace_layout(const DecodeShape &d) {
    DecodeWorkspace w;
    const size_t units = (size_t)d.G * d.maxu;
    size_t o = 0;
    w.nunits = o;
    o = align_up(o + sizeof(int32_t) * d.G, 256);
    w.merge_cnt = o;
    o = align_up(o + sizeof(int32_t) * d.G, 256);
    w.ublk = o;
    o = align_up(o + sizeof(int32_t) * units, 256);
    w.upage = o;
    o = align_up(o + sizeof(int32_t) * units, 256);
    w.umask = o;
    o = align_up(o + sizeof(uint32_t) * units * d.wq, 256);
    w.slot_o = o;
    o = align_up(o + sizeof(float) * (size_t)d.grid * 2 * 128 * kD, 256);
    w.slot_lse = o;
    o = align_up(o + sizeof(float) * (size_t)d.grid * 2 * 128, 256);
    w.bytes = o;
    return w;
}

// Shape checks shared by the size query and the call (sparse: topk > 0).
int check_decode_shape(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || max_pages <= 0 || topk < 0 || Hq % Hkv) return MSA_ERR_INVALID_ARG;
    if (D != kD || !supported_qpk(Hq / Hkv) || (topk > 0 && !supported_topk(topk))) return MSA_ERR_UNSUPPORTED;
    if (max_pages > kMaxNblk || (int64_t)B * Sq >= (1 << 24) || Hkv > kMaxHkv) return MSA_ERR_UNSUPPORTED;
    const int qc = 128 / (Hq / Hkv);
    if ((int64_t)B * Hkv * ceil_div(Sq, qc) > pdk::kMaxGroups) return MSA_ERR_UNSUPPORTED;
    return MSA_OK;
}

// Local plan: when every group has a CTA of its own and no union can exceed
// twice the smallest share (kMinShare units), each CTA plans its own group
// and holds it whole, and the plan kernel is not launched.  Up to a quarter
// over the smallest share the partition would give each group to one CTA
// whatever the data; beyond that, on very uneven unions, a CTA may hold up to
// twice an equal share, which still costs less than cutting groups this
// short (the merge of a cut group's pieces and the plan launch).
bool decode_local_plan(const DecodeShape &d, int max_pages, int topk) {
    return d.G <= d.grid && d.maxu <= 2 * pdk::kMinShare &&
           pdk::plan_scratch_words(max_pages, topk > 0, d.qc, topk, d.maxu, d.wq) * 4 <= pdk::Layout::Q;
}

size_t decode_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    if (check_decode_shape(B, Sq, Hq, Hkv, D, topk, max_pages) != MSA_OK) return 0;
    return decode_workspace_layout(decode_shape(B, Sq, Hq, Hkv, topk, max_pages)).bytes;
}

// The paged decode: plan kernel, then the decode kernel (q2k null: dense).
int paged_decode(const void *q, const void *k_pool, const void *v_pool, int kv_format, int num_pages,
                 const int32_t *page_table, int max_pages, const int32_t *seqused_k, const int32_t *q2k, int B, int Sq,
                 int Hq, int Hkv, int D, int page_size, int topk, int causal, float softmax_scale, void *o, float *lse,
                 void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    if (kv_format != MSA_KV_BF16 && kv_format != MSA_KV_FP8) return MSA_ERR_INVALID_ARG;
    if (!q || !k_pool || !v_pool || !page_table || !seqused_k || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (num_pages <= 0) return MSA_ERR_INVALID_ARG;
    if (q2k && topk <= 0) return MSA_ERR_INVALID_ARG;
    if (!q2k) topk = 0;
    const int rc0 = check_decode_shape(B, Sq, Hq, Hkv, D, topk, max_pages);
    if (rc0 != MSA_OK) return rc0;
    if (page_size != kBlk) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)num_pages * kBlk >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return MSA_ERR_INVALID_ARG;
    const DecodeShape d = decode_shape(B, Sq, Hq, Hkv, topk, max_pages);
    const DecodeWorkspace w = decode_workspace_layout(d);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);

    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.q2k = q2k;
    p.seqused = seqused_k;
    p.page_table = page_table;
    p.k8 = static_cast<const uint8_t *>(k_pool);
    p.v8 = static_cast<const uint8_t *>(v_pool);
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.nunits = reinterpret_cast<int32_t *>(ws + w.nunits);
    p.merge_cnt = reinterpret_cast<int32_t *>(ws + w.merge_cnt);
    p.ublk = reinterpret_cast<int32_t *>(ws + w.ublk);
    p.upage = reinterpret_cast<int32_t *>(ws + w.upage);
    p.umask = reinterpret_cast<uint32_t *>(ws + w.umask);
    p.slot_o = reinterpret_cast<float *>(ws + w.slot_o);
    p.slot_lse = reinterpret_cast<float *>(ws + w.slot_lse);
    p.status = status_dev;
    p.B = B; p.Sq = Sq; p.Hq = Hq; p.Hkv = Hkv; p.qpk = d.qpk; p.topk = topk;
    p.max_pages = max_pages; p.num_pages = num_pages; p.causal = causal ? 1 : 0;
    p.qc = d.qc; p.qgroups = d.qgroups; p.G = d.G; p.maxu = d.maxu; p.wq = d.wq;
    p.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.p_bound = 64.f;

    CUtensorMap mk, mv, mq;
    if (!make_q_heads_map(&mq, q, (int64_t)B * Sq, Hq, d.qpk)) return MSA_ERR_CUDA;
    if (kv_format == MSA_KV_BF16) {
        if (!make_kv_map(&mk, k_pool, Hkv, (int64_t)num_pages * kBlk) ||
            !make_kv_map(&mv, v_pool, Hkv, (int64_t)num_pages * kBlk))
            return MSA_ERR_CUDA;
    } else {
        mk = mv = mq;  // unused: the staging warp reads the e4m3 pools
    }
    const bool local = decode_local_plan(d, max_pages, topk);
    p.local_plan = local ? 1 : 0;
    if (!local) {
        const size_t psmem =
            sizeof(uint32_t) * pdk::plan_scratch_words(max_pages, q2k != nullptr, d.qc, topk, d.maxu, d.wq);
        MSA_CUDA_TRY(cudaFuncSetAttribute(paged_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem));
        MSA_CUDA_TRY(launch_pdl(paged_plan_kernel, dim3(d.G), dim3(256), psmem, stream, p));
    }
    return kv_format == MSA_KV_BF16 ? launch_paged_decode_bf16(mk, mv, mq, p, d.grid, stream)
                                    : launch_paged_decode_fp8(mk, mv, mq, p, d.grid, stream);
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_attn_paged_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk,
                                                           int max_pages) {
    if (topk <= 0) return 0;
    return decode_workspace_size(B, Sq, Hq, Hkv, D, topk, max_pages);
}

extern "C" int msa_sparse_attn_paged_fwd_launches(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    if (topk < 0) return MSA_ERR_INVALID_ARG;
    const int rc = check_decode_shape(B, Sq, Hq, Hkv, D, topk, max_pages);
    if (rc != MSA_OK) return rc;
    return decode_local_plan(decode_shape(B, Sq, Hq, Hkv, topk, max_pages), max_pages, topk) ? 1 : 2;
}

extern "C" int msa_sparse_attn_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                                         const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                         const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                         int topk, int causal, float softmax_scale, void *o, float *lse,
                                         void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                         cudaStream_t stream) {
    if (!q2k) return MSA_ERR_INVALID_ARG;
    return paged_decode(q, k_pool, v_pool, MSA_KV_BF16, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq, Hq,
                        Hkv, D, page_size, topk, causal, softmax_scale, o, lse, workspace, ws_bytes, status_dev,
                        stream);
}

extern "C" size_t msa_paged_attn_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    return decode_workspace_size(B, Sq, Hq, Hkv, D, topk, max_pages);
}

extern "C" int msa_paged_attn_fwd(const void *q, const void *k_pool, const void *v_pool, int kv_format,
                                  int num_pages, const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                  const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size, int topk,
                                  int causal, float softmax_scale, void *o, float *lse, void *workspace,
                                  size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    return paged_decode(q, k_pool, v_pool, kv_format, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq, Hq,
                        Hkv, D, page_size, topk, causal, softmax_scale, o, lse, workspace, ws_bytes, status_dev,
                        stream);
}
