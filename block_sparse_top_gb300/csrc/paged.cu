// paged.cu -- block-sparse paged decode (msa_sparse_attn_paged_fwd).
//
// A group is (sequence b, KV head h, qg = 128/qhead_per_kv consecutive
// queries): the 128 query-head rows one attention tile holds.  Three small
// launches turn the selections into the tile kernel's work plan directly:
//   1. union: per group, the ascending union of the blocks its queries
//      selected (ids >= ceil(seqused/page) are padding, repeats count once),
//      every valid slot's split id, every query's split count, and the split
//      id of each (union block, query of the group), 255 where the query did
//      not select the block;
//   2. scan:  exclusive prefixes of the groups' union sizes and selection
//      counts -> one global unit list;
//   3. write: one plan unit per union block (its page looked up once), and
//      the unit's query table: every query of the group, packed query id |
//      split << 24, split 255 for a query that did not select the block (the
//      tile kernel masks its rows and keeps the group's Q tile for all of the
//      group's units).
// The tcgen05 tile kernel then streams each unit's page and applies the
// causal limit of each query's own position seqused[b] - Sq + i, and the LSE
// combine merges every query head's splits.
//
// Source: interface.py sparse_decode_atten_func and
// SparseDecodePagedAttentionWrapper (paged KV, seqused_k, uniform seqlen_q,
// split-KV partials merged by LSE); test_sparse_atten.py
// _decode_paged_dense_reference (lse = m + log l, -inf for empty rows) and
// _decode_paged_kv_chunk (logical block j of sequence b is page
// page_table[b][j]).
#include <algorithm>
#include <cstring>

#include "tiles.h"

namespace msa {
namespace {

struct PagedShape {
    int qg, qgroups, groups, maxu;
};

PagedShape paged_shape(int B, int Sq, int Hkv, int qpk, int topk, int max_pages) {
    PagedShape d;
    d.qg = 128 / qpk;
    d.qgroups = (int)ceil_div(Sq, d.qg);
    d.groups = B * Hkv * d.qgroups;
    d.maxu = std::min(std::min(Sq, d.qg) * topk, max_pages);
    return d;
}

struct PlanArgs {
    const int32_t *q2k, *seqused, *page_table;
    int32_t *ulist;        // [groups][maxu] union block ids, ascending
    uint8_t *usplit;       // [groups][maxu][qg] split id of (union block, query of the group), 255: not selected
    int2 *ucount;          // [groups + 1] (union size, valid selections), then exclusive prefixes
    int32_t *slot_split;   // [B][Hkv][Sq][topk] split id of each slot, -1 for padding and repeats
    int32_t *split_counts; // [B*Sq][Hkv]
    int32_t *qlist;        // [groups * maxu][qg] per unit: packed query id | split << 24 (255: not selected)
    PlanHeader *plan;
    PlanUnit *units;
    int32_t *unit_page;
    uint32_t *status;
    int B, Sq, Hkv, qpk, topk, num_pages, max_pages, qg, qgroups, groups, maxu;
    int grid;  // CTAs of the tile kernel (its partition of the unit list)
};

struct Group {
    int b, h, q0, nq, nvalid;
};

__device__ __forceinline__ Group group_of(const PlanArgs &a, int g) {
    Group x;
    x.b = g / (a.Hkv * a.qgroups);
    const int rem = g % (a.Hkv * a.qgroups);
    x.h = rem / a.qgroups;
    x.q0 = (rem % a.qgroups) * a.qg;
    x.nq = min(a.qg, a.Sq - x.q0);
    const int64_t kv = a.seqused[x.b];
    x.nvalid = kv <= 0 ? 0 : (int)min(ceil_div(kv, kBlk), (int64_t)a.max_pages);
    return x;
}

// ---------------------------------------------------------------- 1. unions
__global__ void __launch_bounds__(256) paged_union_kernel(PlanArgs a) {
    extern __shared__ uint32_t dsm[];
    const int nwords = (a.max_pages + 31) / 32;
    uint32_t *bitmap = dsm;                                        // [nwords]
    int32_t *ul = reinterpret_cast<int32_t *>(bitmap + nwords);    // [maxu]
    int32_t *spl = ul + a.maxu;                                    // [qg * topk]
    __shared__ int32_t warp_tot[8];
    __shared__ int32_t s_nu, s_nsel;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();  // the previous call's kernels may still read this workspace
    grid_dependents_launch();
    const Group x = group_of(a, g);
    for (int i = tid; i < nwords; i += blockDim.x) bitmap[i] = 0u;
    if (tid == 0) s_nsel = 0;
    __syncthreads();
    // split id of a slot: the number of distinct valid ids in the earlier slots
    const int nslots = x.nq * a.topk;
    for (int i = tid; i < nslots; i += blockDim.x) {
        const int qi = i / a.topk, t = i % a.topk;
        const int32_t *sel = a.q2k + (((int64_t)x.b * a.Hkv + x.h) * a.Sq + x.q0 + qi) * a.topk;
        const int j = sel[t];
        int split = -1;
        if (j >= 0 && j >= x.nvalid) {
            set_status(a.status, MSA_STATUS_INDEX_RANGE);
        } else if (j >= 0) {
            bool dup = false;
            int distinct = 0;
            for (int u = 0; u < t; ++u) {
                const int ju = sel[u];
                if (ju == j) dup = true;
                if (ju < 0 || ju >= x.nvalid) continue;
                bool first = true;
                for (int w = 0; w < u; ++w) first &= (sel[w] != ju);
                distinct += first ? 1 : 0;
            }
            if (dup) {
                set_status(a.status, MSA_STATUS_DUPLICATE);
            } else {
                split = distinct;
                atomicOr(&bitmap[j >> 5], 1u << (j & 31));
                atomicAdd(&s_nsel, 1);
            }
        }
        spl[i] = split;
        a.slot_split[(((int64_t)x.b * a.Hkv + x.h) * a.Sq + x.q0 + qi) * a.topk + t] = split;
    }
    __syncthreads();
    // per query: its number of valid splits
    for (int qi = tid; qi < x.nq; qi += blockDim.x) {
        int n = 0;
        for (int t = 0; t < a.topk; ++t) n += spl[qi * a.topk + t] >= 0 ? 1 : 0;
        a.split_counts[((int64_t)x.b * a.Sq + x.q0 + qi) * a.Hkv + x.h] = n;
    }
    // compact the bitmap in ascending block order
    {
        const int per = (nwords + blockDim.x - 1) / blockDim.x;
        const int w0 = tid * per, w1 = min(w0 + per, nwords);
        int cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(bitmap[w]);
        int v = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane == 31) warp_tot[warp] = v;
        __syncthreads();
        int pos = v - cnt;
        for (int w = 0; w < warp; ++w) pos += warp_tot[w];
        for (int w = w0; w < w1; ++w) {
            uint32_t m = bitmap[w];
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                ul[pos++] = w * 32 + bit;
            }
        }
        if (tid == blockDim.x - 1) s_nu = pos;
    }
    __syncthreads();
    const int nu = s_nu;
    // split table: 255 (not selected) for every (union block, query), then each
    // valid slot's split id at its block's union position
    uint8_t *us = a.usplit + (int64_t)g * a.maxu * a.qg;
    for (int i = tid; i < nu * a.qg; i += blockDim.x) us[i] = 255;
    __syncthreads();
    for (int i = tid; i < nslots; i += blockDim.x) {
        if (spl[i] < 0) continue;
        const int qi = i / a.topk;
        const int j = a.q2k[(((int64_t)x.b * a.Hkv + x.h) * a.Sq + x.q0 + qi) * a.topk + i % a.topk];
        int lo = 0, hi = nu;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (ul[mid] < j) lo = mid + 1;
            else hi = mid;
        }
        us[lo * a.qg + qi] = (uint8_t)spl[i];
    }
    for (int e = tid; e < nu; e += blockDim.x) a.ulist[(int64_t)g * a.maxu + e] = ul[e];
    if (tid == 0) a.ucount[g] = make_int2(nu, s_nsel);
}

// ---------------------------------------------------------------- 2. scan
// In place: ucount[0..groups) -> exclusive prefixes of both counts,
// ucount[groups] = totals; the plan header is filled from the totals.
__global__ void __launch_bounds__(1024) paged_scan_kernel(PlanArgs a) {
    __shared__ int2 warp_sums[32];
    __shared__ int2 carry_s;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_s = make_int2(0, 0);
    grid_dependency_wait();
    grid_dependents_launch();
    __syncthreads();
    for (int base = 0; base < a.groups; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int2 v = (i < a.groups) ? a.ucount[i] : make_int2(0, 0);
        int2 x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(0xffffffffu, x.x, o), yy = __shfl_up_sync(0xffffffffu, x.y, o);
            if (lane >= o) x = make_int2(x.x + yx, x.y + yy);
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int2 w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yx = __shfl_up_sync(0xffffffffu, w.x, o), yy = __shfl_up_sync(0xffffffffu, w.y, o);
                if (lane >= o) w = make_int2(w.x + yx, w.y + yy);
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int2 c = carry_s;
        const int2 before = warp > 0 ? warp_sums[warp - 1] : make_int2(0, 0);
        const int2 incl = make_int2(x.x + before.x + c.x, x.y + before.y + c.y);
        if (i < a.groups) a.ucount[i] = make_int2(incl.x - v.x, incl.y - v.y);
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry_s = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.ucount[a.groups] = carry_s;
        a.plan->work_count = carry_s.x;
        a.plan->capacity = a.groups * a.maxu;
        a.plan->qhead_per_kv = a.qpk;
        a.plan->q_per_unit = a.qg;
        a.plan->wave_queries = 0;
        a.plan->nwaves = 0;
    }
}

// ---------------------------------------------------------------- 3. write
// One unit per union block of group g (global index u = ucount[g].x + e); its
// query table (all queries of the group, ascending) is qlist[u*qg .. + nq).
__global__ void __launch_bounds__(128) paged_write_kernel(PlanArgs a) {
    const int g = blockIdx.x;
    grid_dependency_wait();
    grid_dependents_launch();
    const Group x = group_of(a, g);
    const int off = a.ucount[g].x;
    const int nu = a.ucount[g + 1].x - off;
    for (int e = threadIdx.x; e < nu; e += blockDim.x) {
        const uint8_t *us = a.usplit + ((int64_t)g * a.maxu + e) * a.qg;
        const int j = a.ulist[(int64_t)g * a.maxu + e];
        const int64_t u = off + e;
        const int start = (int)(u * a.qg);
        PlanUnit pu;
        pu.head = (int16_t)x.h;
        pu.blk = (int16_t)j;
        pu.seq = x.b;
        pu.start = start;
        pu.count = x.nq;
        a.units[u] = pu;
        int pg = a.page_table[(int64_t)x.b * a.max_pages + j];
        if (pg < 0 || pg >= a.num_pages) {
            set_status(a.status, MSA_STATUS_PAGE_RANGE);
            pg = -1;  // the tile kernel skips the block
        }
        a.unit_page[u] = pg;
    }
    // Query tables.  The tile kernel's CTA c runs units [work c / G, work (c+1) / G)
    // and, inside its run, alternates them between its two softmax warpgroups;
    // a warpgroup accumulates O over consecutive units of one group, so a
    // query's partials are its pieces: the distinct (CTA, warpgroup) pairs
    // that hold a unit it selected, numbered in order of first appearance
    // (at most one per selected block, so at most topk).  The table holds the
    // query's piece for each unit it selected, 255 for the others, and the
    // piece count becomes the query's split count.  One warp per query: lane
    // l takes units l, l + 32, ...; the order of first appearance runs over
    // the selected units only (a ballot per 32 units), so the serial steps are
    // at most topk.
    const int64_t work = a.ucount[a.groups].x, G = a.grid;
    const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int qi = threadIdx.x >> 5; qi < x.nq; qi += nwarps) {
        const int gq = x.b * a.Sq + x.q0 + qi;
        int cur_c = -1, pw0 = -1, pw1 = -1, pieces = 0;
        for (int e0 = 0; e0 < nu; e0 += 32) {
            const int e = e0 + lane;
            const int64_t u = off + e;
            const bool sel = e < nu && a.usplit[((int64_t)g * a.maxu + e) * a.qg + qi] != 255;
            int c = 0, w = 0;
            if (sel) {
                c = (int)(((u + 1) * G - 1) / work);  // CTA holding unit u
                w = (int)((u - work * c / G) & 1);     // its warpgroup there
            }
            int mine = 255;
            uint32_t m = __ballot_sync(0xffffffffu, sel);
            while (m) {
                const int l = __ffs(m) - 1;
                m &= m - 1;
                const int cl = __shfl_sync(0xffffffffu, c, l), wl = __shfl_sync(0xffffffffu, w, l);
                if (cl != cur_c) {
                    cur_c = cl;
                    pw0 = pw1 = -1;
                }
                int &pw = wl ? pw1 : pw0;
                if (pw < 0) pw = pieces++;
                if (lane == l) mine = pw;
            }
            if (e < nu) a.qlist[u * a.qg + qi] = gq | (mine << 24);
        }
        if (lane == 0) a.split_counts[(int64_t)gq * a.Hkv + x.h] = pieces;
    }
}

// Workspace of msa_sparse_attn_paged_fwd: the union plan, then the split partials.
struct PagedWorkspace {
    size_t ulist, usplit, ucount, slot_split, split_counts, qlist, plan, unit_page, fwd, fwd_bytes, bytes;
};

PagedWorkspace paged_workspace_layout(const PagedShape &d, int B, int Sq, int Hq, int Hkv, int topk) {
    PagedWorkspace w;
    const size_t slots = (size_t)B * Hkv * Sq * topk;
    size_t o = 0;
    w.ulist = o;
    o = align_up(o + sizeof(int32_t) * (size_t)d.groups * d.maxu, 256);
    w.usplit = o;
    o = align_up(o + (size_t)d.groups * d.maxu * d.qg, 256);
    w.ucount = o;
    o = align_up(o + sizeof(int2) * ((size_t)d.groups + 1), 256);
    w.slot_split = o;
    o = align_up(o + sizeof(int32_t) * slots, 256);
    w.split_counts = o;
    o = align_up(o + sizeof(int32_t) * (size_t)B * Sq * Hkv, 256);
    w.qlist = o;
    o = align_up(o + sizeof(int32_t) * (size_t)d.groups * d.maxu * d.qg, 256);
    w.plan = o;
    o = align_up(o + sizeof(PlanHeader) + sizeof(PlanUnit) * (size_t)d.groups * d.maxu, 256);
    w.unit_page = o;
    o = align_up(o + sizeof(int32_t) * (size_t)d.groups * d.maxu, 256);
    w.fwd = o;
    w.fwd_bytes = fwd_workspace_layout((int64_t)B * Sq, Hq, topk, kD, MSA_PARTIAL_FP32).bytes;
    o = align_up(o + w.fwd_bytes, 256);
    w.bytes = o;
    return w;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_attn_paged_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk,
                                                           int max_pages) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || D != kD || topk <= 0 || max_pages <= 0 || Hq % Hkv) return 0;
    const int qpk = Hq / Hkv;
    if (!supported_qpk(qpk) || !supported_topk(topk) || max_pages > kMaxNblk) return 0;
    if ((int64_t)B * Sq >= (1 << 24)) return 0;
    const PagedShape d = paged_shape(B, Sq, Hkv, qpk, topk, max_pages);
    return paged_workspace_layout(d, B, Sq, Hq, Hkv, topk).bytes;
}

namespace msa {
// Paged decode over the tile pipeline for K/V pools of kv_format (bf16, or
// e4m3 staged to bf16 on load).
int paged_tiles_fwd(const void *q, const void *k_pool, const void *v_pool, int kv_format, int num_pages,
                    const int32_t *page_table, int max_pages, const int32_t *seqused_k, const int32_t *q2k, int B,
                    int Sq, int Hq, int Hkv, int D, int page_size, int topk, int causal, float softmax_scale, void *o,
                    float *lse, void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    if (!q || !k_pool || !v_pool || !page_table || !seqused_k || !q2k || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pages <= 0 || topk <= 0 || Hq % Hkv)
        return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || page_size != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if (max_pages > kMaxNblk || (int64_t)B * Sq >= (1 << 24) || Hkv > kMaxHkv) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)num_pages * kBlk >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return MSA_ERR_INVALID_ARG;
    const PagedShape d = paged_shape(B, Sq, Hkv, qpk, topk, max_pages);
    const PagedWorkspace w = paged_workspace_layout(d, B, Sq, Hq, Hkv, topk);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);

    PlanArgs a;
    a.q2k = q2k;
    a.seqused = seqused_k;
    a.page_table = page_table;
    a.ulist = reinterpret_cast<int32_t *>(ws + w.ulist);
    a.usplit = reinterpret_cast<uint8_t *>(ws + w.usplit);
    a.ucount = reinterpret_cast<int2 *>(ws + w.ucount);
    a.slot_split = reinterpret_cast<int32_t *>(ws + w.slot_split);
    a.split_counts = reinterpret_cast<int32_t *>(ws + w.split_counts);
    a.qlist = reinterpret_cast<int32_t *>(ws + w.qlist);
    a.plan = reinterpret_cast<PlanHeader *>(ws + w.plan);
    a.units = reinterpret_cast<PlanUnit *>(a.plan + 1);
    a.unit_page = reinterpret_cast<int32_t *>(ws + w.unit_page);
    a.status = status_dev;
    a.B = B; a.Sq = Sq; a.Hkv = Hkv; a.qpk = qpk; a.topk = topk; a.num_pages = num_pages;
    a.max_pages = max_pages; a.qg = d.qg; a.qgroups = d.qgroups; a.groups = d.groups; a.maxu = d.maxu;
    a.grid = (int)std::min<int64_t>((int64_t)d.groups * d.maxu, (int64_t)num_sms());  // as tiles_launch

    const size_t usmem = sizeof(uint32_t) * (((size_t)max_pages + 31) / 32) + sizeof(int32_t) * (size_t)d.maxu +
                         sizeof(int32_t) * (size_t)d.qg * topk;
    MSA_CUDA_TRY(cudaFuncSetAttribute(paged_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)usmem));
    MSA_CUDA_TRY(launch_pdl(paged_union_kernel, dim3(d.groups), dim3(256), usmem, stream, a));
    MSA_CUDA_TRY(launch_pdl(paged_scan_kernel, dim3(1), dim3(1024), 0, stream, a));
    MSA_CUDA_TRY(launch_pdl(paged_write_kernel, dim3(d.groups), dim3(128), 0, stream, a));

    // fp32 pieces: an accumulated piece is a sum over many keys, kept exact
    // until the combine's single rounding to bf16
    const FwdWorkspace fw = fwd_workspace_layout((int64_t)B * Sq, Hq, topk, D, MSA_PARTIAL_FP32);
    char *fws = ws + w.fwd;
    TcParams t;
    memset(&t, 0, sizeof t);
    t.k_packed = static_cast<const uint8_t *>(k_pool);
    t.v_packed = static_cast<const uint8_t *>(v_pool);
    t.k_scales = nullptr;
    t.v_scales = nullptr;
    t.qsplit = a.qlist;
    t.plan = a.plan;
    t.units = a.units;
    t.o_part = fws + fw.o_part;
    t.stat_part = reinterpret_cast<float2 *>(fws + fw.stat_part);
    t.part_dtype = MSA_PARTIAL_FP32;
    t.inv_temp = 1.f;
    t.seqused = seqused_k;
    t.unit_page = a.unit_page;
    t.cu_q = t.cu_k = nullptr;
    t.kv_rows = (int64_t)num_pages * kBlk;
    t.total_q = (int64_t)B * Sq;
    t.status = status_dev;
    t.B = B; t.Sq = Sq; t.Skv = max_pages * kBlk; t.Hq = Hq; t.Hkv = Hkv; t.qpk = qpk; t.topk = topk;
    t.nblk = max_pages;
    t.causal = causal ? 1 : 0;
    t.cap = 0;  // unit starts index qlist directly
    t.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    t.scale_log2 = t.scale * 1.4426950408889634f;
    t.p_bound = 64.f;
    const int rc = tiles_launch(t, (int64_t)d.groups * d.maxu, q, k_pool, v_pool, (int64_t)num_pages * kBlk,
                                kv_format, false, stream);
    if (rc != MSA_OK) return rc;
    return combine_launch(a.split_counts, (int64_t)B * Sq * Hkv, qpk, topk, o, lse, nullptr, fws, fw,
                          MSA_PARTIAL_FP32, stream);
}

// The per-group union decode of decode.cu (dense mode when q2k is NULL) and its scratch.
int union_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages, const int32_t *page_table,
                    int max_pages, const int32_t *seqused_k, const int32_t *q2k, int B, int Sq, int Hq, int Hkv,
                    int D, int page_size, int topk, int causal, float softmax_scale, void *o, float *lse,
                    void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream);
size_t union_paged_fwd_scratch(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages);
}  // namespace msa

extern "C" int msa_sparse_attn_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages,
                                         const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                         const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                         int topk, int causal, float softmax_scale, void *o, float *lse,
                                         void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                         cudaStream_t stream) {
    if (!q2k) return MSA_ERR_INVALID_ARG;
    return paged_tiles_fwd(q, k_pool, v_pool, MSA_KV_BF16, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq,
                           Hq, Hkv, D, page_size, topk, causal, softmax_scale, o, lse, workspace, ws_bytes,
                           status_dev, stream);
}

extern "C" size_t msa_paged_attn_fwd_workspace_size(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    if (topk == 0) return union_paged_fwd_scratch(B, Sq, Hq, Hkv, D, max_pages, max_pages);
    return msa_sparse_attn_paged_fwd_workspace_size(B, Sq, Hq, Hkv, D, topk, max_pages);
}

extern "C" int msa_paged_attn_fwd(const void *q, const void *k_pool, const void *v_pool, int kv_format,
                                  int num_pages, const int32_t *page_table, int max_pages, const int32_t *seqused_k,
                                  const int32_t *q2k, int B, int Sq, int Hq, int Hkv, int D, int page_size, int topk,
                                  int causal, float softmax_scale, void *o, float *lse, void *workspace,
                                  size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    if (kv_format != MSA_KV_BF16 && kv_format != MSA_KV_FP8) return MSA_ERR_INVALID_ARG;
    if (!q2k) {
        // dense: every block of each sequence, by the per-group union decode (bf16 pools)
        if (kv_format != MSA_KV_BF16) return MSA_ERR_UNSUPPORTED;
        if ((int64_t)B * Sq >= (1 << 24) || Hkv > kMaxHkv) return MSA_ERR_UNSUPPORTED;
        return union_paged_fwd(q, k_pool, v_pool, num_pages, page_table, max_pages, seqused_k, nullptr, B, Sq, Hq,
                               Hkv, D, page_size, max_pages, causal, softmax_scale, o, lse, workspace, ws_bytes,
                               status_dev, stream);
    }
    return paged_tiles_fwd(q, k_pool, v_pool, kv_format, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq, Hq,
                           Hkv, D, page_size, topk, causal, softmax_scale, o, lse, workspace, ws_bytes, status_dev,
                           stream);
}
