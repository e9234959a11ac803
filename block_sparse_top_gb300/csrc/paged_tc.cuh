// paged_tc.cuh -- block-sparse paged decode in two launches: a union plan
// kernel and a persistent tcgen05 decode kernel (one launch when each decode
// CTA can plan its own group, see local_plan).
//
// A group is (sequence b, KV head h, qc = 128/qhead_per_kv consecutive
// queries): the 128 query-head rows (row R = query R / qpk of the group, head
// R % qpk of the KV head's GQA group) that share the KV head's blocks.
//
//   paged_plan_kernel (paged.cu), one CTA per group: the ascending union of the blocks
//     the group's queries selected (ids >= ceil(seqused/page) are padding,
//     repeats of one query count once), each union block's page, and the
//     mask of the queries that selected it.  Dense mode (no selection): every
//     block below ceil(seqused/page), selected by every query.  A group with
//     an empty union writes O = 0, LSE = -inf at once.
//
//   paged_decode_kernel, persistent, one CTA per SM: every CTA takes the
//     prefix of the groups' union sizes, which orders all (group, union block)
//     units, and takes a contiguous run of them -- a whole group per CTA when
//     the groups fit the grid about evenly, else an equal share of the units.
//     Per CTA:
//       warp 0      TMA: each group's 128 Q rows (two boxes), each unit's K and
//                   V block from its page through a 3-stage ring;
//       warp 1      MMA issuer: S = Q K^T into tensor memory (two S buffers),
//                   O += P V into the group's O buffer (two, alternating by
//                   group), P read from tensor memory;
//       warp 2      e4m3 pools only: stages K and V to bf16 in the ring;
//       warps 4-11  softmax, two warpgroups splitting each S row (keys 0-63
//                   and 64-127 of the same TMEM lanes) and agreeing on one
//                   reference max per row: rows whose query did not select
//                   the block get P = 0, and a row's O is rescaled only when
//                   a block's max exceeds the reference by more than
//                   2^p_bound.  At the end of a group they write O / (sum of
//                   P) and the LSE: a group the CTA holds whole goes straight
//                   to the output; a group cut by the partition leaves one
//                   piece per CTA, and the CTA that writes its last piece
//                   merges them by LSE (an atomic count per group), so there
//                   is no further launch and no per-block partial.
//
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
// Every wait is bounded; on a timeout the CTA raises MSA_STATUS_TIMEOUT,
// drains its copies and MMAs, frees tensor memory and exits.
//
// Source: the interface page, sparse_decode_atten_func and
// SparseDecodePagedAttentionWrapper (paged KV, seqused_k, uniform query
// length, split KV merged by LSE); the test page, the paged dense decode
// reference (running max and sum, lse = m + log l, -inf for empty rows) and
// its page-table addressing (logical block j of sequence b is page
// page_table[b][j]).
#pragma once
#include "attn_mma.cuh"
#include "tc.cuh"

namespace msa {

struct DecodeParams {
    const int32_t *q2k;         // [B][Hkv][Sq][topk]; null: every block of the sequence (dense)
    const int32_t *seqused;     // [B]
    const int32_t *page_table;  // [B][max_pages]
    const uint8_t *k8, *v8;     // e4m3 pools (FP8 instance)
    __nv_bfloat16 *o;           // [B*Sq][Hq][128]
    float *lse;                 // [B*Sq][Hq], or null
    // the plan (workspace)
    int32_t *nunits;     // [G] union size of each group
    int32_t *merge_cnt;  // [G] pieces of a cut group written so far
    int32_t *ublk;       // [G][maxu] union block ids, ascending
    int32_t *upage;      // [G][maxu] their pages (-1: invalid page-table entry)
    uint32_t *umask;     // [G][maxu][wq] the group's queries that selected the block
    float *slot_o;       // [grid][2][128][128] normalised O of a cut group's piece
    float *slot_lse;     // [grid][2][128] its LSE
    uint32_t *status;
    int B, Sq, Hq, Hkv, qpk, topk, max_pages, num_pages, causal;
    int qc, qgroups, G, maxu, wq;
    float scale, scale_log2;
    // a row's accumulated O is rescaled to a new reference max only when a
    // block's max exceeds the reference by more than this (log2 units)
    float p_bound;
    // 1: no plan kernel ran; CTA c < G plans group c itself and holds it whole
    // (the host sets this only when every group can have a CTA of its own and
    // no union is long: G <= grid and maxu <= 2 * kMinShare)
    int local_plan;
};

struct DGroup {
    int b, h, q0, nq;
};

// group g = (b * Hkv + h) * qgroups + query group
__device__ __forceinline__ DGroup dgroup(const DecodeParams &p, int g) {
    DGroup x;
    const int per_b = p.Hkv * p.qgroups;
    x.b = g / per_b;
    const int rem = g - x.b * per_b;
    x.h = rem / p.qgroups;
    x.q0 = (rem - x.h * p.qgroups) * p.qc;
    x.nq = min(p.qc, p.Sq - x.q0);
    return x;
}

// Loads of the plan, which an earlier kernel wrote: L2, not the
// non-coherent path.
__device__ __forceinline__ int ld_plan(const int32_t *p) { return __ldcg(p); }
__device__ __forceinline__ uint32_t ld_plan(const uint32_t *p) { return __ldcg(p); }

namespace pdk {

constexpr int kNKV = 3;  // K/V ring stages
// 12 warps (three per SM sub-partition: 168 registers a thread); TMEM lane
// quarter = warp % 4, so each warpgroup covers all 128 rows.
constexpr int kWarps = 12, kThreads = kWarps * 32;
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpDequant = 2, kWarpSoftmax0 = 4;
constexpr int kMaxGroups = 49152;  // the partition's prefix lives in the K/V ring before the pipeline starts
constexpr int kMinShare = 8;       // fewest units of a CTA's share in the balanced partition

// Shared memory: K [3] | V [3] | Q | mbarriers | TMEM slot | abort flag |
// walk start | merge flag.
struct Layout {
    static constexpr uint32_t K = 0, V = kNKV * 32768u, Q = 2 * kNKV * 32768u, BAR = Q + 32768u;
    enum : int {
        KV_FULL = 0,
        KV_EMPTY = kNKV,
        Q_FULL = 2 * kNKV,
        Q_EMPTY,
        S_FULL,
        P_FULL = S_FULL + 2,
        O_FULL = P_FULL + 2,
        PV_DONE = O_FULL + 2,
        DRAIN,
        NBAR
    };
    static constexpr uint32_t TSLOT = BAR + 8 * NBAR, ABORT = TSLOT + 4, WALK = ABORT + 4, MERGE = WALK + 48,
                              BYTES = MERGE + 4;
    static_assert(BYTES <= 232448, "shared memory budget");
};

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, 0, 1);

// Where a CTA's run of units starts (in shared memory, written once).
struct WalkStart {
    int valid, aligned, g0, off0, n0, j0, ue, grid;
    long long total;
};

// A role's position in the CTA's run: group g (its first global unit off,
// n units), unit j of it, the run's units of g are [j0, jend).
struct Walk {
    int g, off, n, j, j0, jend, ue;
    bool aligned;
};

__device__ __forceinline__ bool walk_begin(Walk &w, const WalkStart &s) {
    w.g = s.g0;
    w.off = s.off0;
    w.n = s.n0;
    w.j = w.j0 = s.j0;
    w.ue = s.ue;
    w.jend = min(w.n, w.ue - w.off);
    w.aligned = s.aligned != 0;
    return s.valid != 0;
}

// Next unit; false at the end of the run.  Groups with no units are skipped.
__device__ __forceinline__ bool walk_next(Walk &w, const DecodeParams &p) {
    if (++w.j < w.jend) return true;
    if (w.aligned) return false;
    w.off += w.n;
    while (w.off < w.ue) {
        ++w.g;
        w.n = ld_plan(p.nunits + w.g);
        if (w.n > 0) break;
    }
    if (w.off >= w.ue) return false;
    w.j = w.j0 = 0;
    w.jend = min(w.n, w.ue - w.off);
    return true;
}

// CTA holding global unit u of the balanced partition (units [total c /
// grid, total (c + 1) / grid) go to CTA c)
__device__ __forceinline__ int cta_of(long long u, long long total, int grid) {
    return (int)(((u + 1) * grid - 1) / total);
}

// AND of `pred` over the `count` threads of named barrier `id` (all of them
// wait for each other).
__device__ __forceinline__ bool bar_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

constexpr int kRowUpFront = 1024;  // page-table rows loaded whole by the plan

// Plan of group g by all NT threads of the CTA (every thread calls it alike;
// it ends at a CTA barrier), for the plan kernel (256 threads, one group per
// CTA) and the decode kernel's local-plan mode (its 384 threads).  Every global load is issued up front (the
// sequence length, its whole page-table row and the group's selections), so
// the plan waits on one round trip.  Scratch (32-bit words, in the K/V ring):
// page-table row [max_pages] | bitmap [nw] | per-word prefix [nw] | slots
// [qc topk] | kept [qc topk] | union [maxu] | masks [maxu][wq] | warp sums
// [kWarps] | sequence length | union size, nw = ceil(max_pages / 32).
template <int NT>
__device__ __noinline__ void plan_group(const DecodeParams &p, int g, uint32_t *scr) {
    const int nwords = (p.max_pages + 31) >> 5;
    const int nslot_max = p.q2k ? p.qc * p.topk : 0;
    int32_t *ptab = reinterpret_cast<int32_t *>(scr);
    uint32_t *bitmap = scr + p.max_pages;
    int32_t *wpre = reinterpret_cast<int32_t *>(bitmap + nwords);
    int32_t *sel = wpre + nwords;
    int32_t *kept = sel + nslot_max;
    int32_t *ul = kept + nslot_max;
    uint32_t *msk = reinterpret_cast<uint32_t *>(ul + p.maxu);
    int32_t *warp_tot = reinterpret_cast<int32_t *>(msk + p.maxu * p.wq);
    int32_t *s_kv = warp_tot + kWarps;  // (kWarps >= NW words reserved)
    int32_t *s_nu = s_kv + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const DGroup x = dgroup(p, g);
    const int nslots = p.q2k ? x.nq * p.topk : 0;
    // ---- loads (one round trip) and zeroed tables
    if (tid == 0) *s_kv = __ldg(p.seqused + x.b);
    // a short page-table row is loaded whole, with the selections; a long one
    // (many groups would each read it) only up to the sequence's length
    const bool row_up_front = p.max_pages <= kRowUpFront;
    if (row_up_front)
        for (int i = tid; i < p.max_pages; i += NT) ptab[i] = __ldg(p.page_table + (int64_t)x.b * p.max_pages + i);
    if (p.q2k) {
        const int32_t *src = p.q2k + (((int64_t)x.b * p.Hkv + x.h) * p.Sq + x.q0) * p.topk;
        for (int i = tid; i < nslots; i += NT) sel[i] = __ldg(src + i);
        for (int i = tid; i < nwords; i += NT) bitmap[i] = 0u;
        for (int i = tid; i < p.maxu * p.wq; i += NT) msk[i] = 0u;
    }
    __syncthreads();
    const int kv = *s_kv;
    const int nvalid = kv <= 0 ? 0 : (int)min(ceil_div(kv, kBlk), (int64_t)p.max_pages);
    if (!row_up_front)  // (read after the barriers below)
        for (int i = tid; i < nvalid; i += NT) ptab[i] = __ldg(p.page_table + (int64_t)x.b * p.max_pages + i);
    int nu;
    if (p.q2k) {
        // a slot is kept when its id is a valid block and no earlier slot of
        // its query holds the same id
        for (int i = tid; i < nslots; i += NT) {
            const int t = i % p.topk;
            const int j = sel[i];
            int keep = -1;
            if (j >= nvalid) {
                set_status(p.status, MSA_STATUS_INDEX_RANGE);
            } else if (j >= 0) {
                bool dup = false;
                for (int u = 1; u <= t; ++u) dup |= sel[i - u] == j;
                if (dup) {
                    set_status(p.status, MSA_STATUS_DUPLICATE);
                } else {
                    keep = j;
                    atomicOr(&bitmap[j >> 5], 1u << (j & 31));
                }
            }
            kept[i] = keep;
        }
        __syncthreads();
        // the union in ascending block order: each word's exclusive prefix
        // of set bits, and the union list
        const int per = (nwords + NT - 1) / NT;
        const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
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
            wpre[w] = pos;
            uint32_t m = bitmap[w];
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                ul[pos++] = w * 32 + bit;
            }
        }
        if (tid == NT - 1) *s_nu = pos;
        __syncthreads();
        nu = *s_nu;
        // the queries of each union block: a kept id's union position is its
        // word's prefix plus the set bits below it
        for (int i = tid; i < nslots; i += NT) {
            const int j = kept[i];
            if (j < 0) continue;
            const int qi = i / p.topk;
            const int e = wpre[j >> 5] + __popc(bitmap[j >> 5] & ((1u << (j & 31)) - 1u));
            atomicOr(&msk[e * p.wq + (qi >> 5)], 1u << (qi & 31));
        }
        __syncthreads();
    } else {
        nu = nvalid;  // dense: every block of the sequence, every query
        if (tid == 0) *s_nu = nu;
    }
    const int64_t gbase = (int64_t)g * p.maxu;
    for (int e = tid; e < nu; e += NT) {
        const int j = p.q2k ? ul[e] : e;
        int pg = ptab[j];
        if (pg < 0 || pg >= p.num_pages) {
            set_status(p.status, MSA_STATUS_PAGE_RANGE);
            pg = -1;  // the decode skips the block
        }
        p.ublk[gbase + e] = j;
        p.upage[gbase + e] = pg;
        for (int w = 0; w < p.wq; ++w) {
            uint32_t m;
            if (p.q2k) {
                m = msk[e * p.wq + w];
            } else {
                const int nb = min(32, x.nq - 32 * w);
                m = nb <= 0 ? 0u : (nb == 32 ? 0xffffffffu : (1u << nb) - 1u);
            }
            p.umask[(gbase + e) * p.wq + w] = m;
        }
    }
    if (tid == 0) {
        p.nunits[g] = nu;
        p.merge_cnt[g] = 0;
    }
    if (nu == 0) {
        // no visible key for any row of the group: O = 0, LSE = -inf
        const int rows = x.nq * p.qpk;
        for (int i = tid; i < rows * 16; i += NT) {
            const int r = i >> 4, c = i & 15;
            const int64_t row = ((int64_t)x.b * p.Sq + x.q0 + r / p.qpk) * p.Hq + x.h * p.qpk + r % p.qpk;
            reinterpret_cast<uint4 *>(p.o + row * kD)[c] = make_uint4(0, 0, 0, 0);
            if (c == 0 && p.lse) p.lse[row] = -INFINITY;
        }
    }
    __syncthreads();  // the scratch is reused by the next group
}

// Scratch words plan_group uses; its last word is the union size.
__host__ __device__ inline size_t plan_scratch_words(int max_pages, bool sparse, int qc, int topk, int maxu, int wq) {
    return (size_t)max_pages + 2 * (size_t)((max_pages + 31) / 32) + (sparse ? 2 * (size_t)qc * topk : 0) +
           (size_t)maxu * (1 + wq) + kWarps + 2;
}

}  // namespace pdk

// ---------------------------------------------------------------------------
// decode: persistent, one CTA per SM, 12 warps
// ---------------------------------------------------------------------------
template <int KV_FORMAT>
__global__ void __launch_bounds__(pdk::kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, DecodeParams p) {
    using namespace pdk;
    using L = Layout;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *const gbase = smem_raw;
    if (base & 1023u) {  // 128-byte swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_status(p.status, MSA_STATUS_LAUNCH);
        return;
    }
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + L::ABORT);
    WalkStart *ws = reinterpret_cast<WalkStart *>(gbase + L::WALK);
    volatile int *merge_flag = reinterpret_cast<volatile int *>(gbase + L::MERGE);
    auto bar = [&](int i) -> uint32_t { return base + L::BAR + 8u * (uint32_t)i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < kNKV; ++i) {
            // arrivals: the producer's copy (bf16), or the staging warp's 32 lanes (e4m3)
            tc::mbar_init(bar(L::KV_FULL + i), KV_FORMAT == MSA_KV_BF16 ? 1 : 32);
            tc::mbar_init(bar(L::KV_EMPTY + i), 1);
        }
        tc::mbar_init(bar(L::Q_FULL), 1);
        tc::mbar_init(bar(L::Q_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(L::S_FULL + i), 1);
            tc::mbar_init(bar(L::P_FULL + i), 256);  // both softmax warpgroups
            tc::mbar_init(bar(L::O_FULL + i), 1);
        }
        tc::mbar_init(bar(L::PV_DONE), 1);
        tc::mbar_init(bar(L::DRAIN), 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(base + L::TSLOT, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::tma_prefetch_desc(&tm_q);
        if (KV_FORMAT == MSA_KV_BF16) {
            tc::tma_prefetch_desc(&tm_k);
            tc::tma_prefetch_desc(&tm_v);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + L::TSLOT);
    grid_dependency_wait();  // the plan (local plan: the previous call, which may still read the workspace)
    grid_dependents_launch();

    if (p.local_plan) {
        // ------------------------------------------------------------ local plan
        // This CTA's own group, planned into the workspace (the K/V ring is
        // the scratch); the CTA holds it whole.
        if ((int)blockIdx.x < p.G) plan_group<kThreads>(p, blockIdx.x, reinterpret_cast<uint32_t *>(gbase));
        if (tid == 0) {
            // the union size: the plan scratch's last word
            const size_t last = plan_scratch_words(p.max_pages, p.q2k != nullptr, p.qc, p.topk, p.maxu, p.wq) - 1;
            const int n = (int)blockIdx.x < p.G ? reinterpret_cast<const int32_t *>(gbase)[last] : 0;
            WalkStart st{};
            st.aligned = 1;
            st.g0 = blockIdx.x;
            st.n0 = n;
            st.ue = n;
            st.valid = n > 0;
            st.grid = gridDim.x;
            st.total = n;
            *ws = st;
        }
        __syncthreads();
    }
    // ---------------------------------------------------------------- partition
    // Exclusive prefix of the union sizes in the K/V ring (free until the
    // pipeline starts), then this CTA's run of units.  The producer meanwhile
    // loads the page of unit 0 of group blockIdx.x, where a whole-group run
    // starts (used only if the run starts there).
    int page_guess = -1;
    if (KV_FORMAT == MSA_KV_BF16 && warp == kWarpLoad && lane == 0 && (int)blockIdx.x < p.G)
        page_guess = ld_plan(p.upage + (int64_t)blockIdx.x * p.maxu);
    if (!p.local_plan) {
        int *scr = reinterpret_cast<int *>(gbase);  // [G + 1] prefix | [kWarps] warp sums | [kWarps] maxima
        int *wsum = scr + p.G + 1, *wmax = wsum + kWarps;
        const int per = (p.G + kThreads - 1) / kThreads;
        const int g0 = min(tid * per, p.G), g1 = min(g0 + per, p.G);
        int s = 0, mx = 0;
        for (int g = g0; g < g1; ++g) {
            const int n = ld_plan(p.nunits + g);
            scr[g] = n;
            s += n;
            mx = max(mx, n);
        }
        int v = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 31) wsum[warp] = v;
        if (lane == 0) wmax[warp] = mx;
        __syncthreads();
        int run = v - s;
        for (int w = 0; w < warp; ++w) run += wsum[w];
        for (int g = g0; g < g1; ++g) {
            const int n = scr[g];
            scr[g] = run;
            run += n;
        }
        if (tid == kThreads - 1) scr[p.G] = run;
        __syncthreads();
        if (tid == 0) {
            int maxn = 0;
            for (int w = 0; w < kWarps; ++w) maxn = max(maxn, wmax[w]);
            const long long total = scr[p.G];
            const int c = (int)blockIdx.x;
            // CTAs of the balanced partition: every one holds at least
            // kMinShare units (so each CTA in a cut group's range holds one of
            // its pieces)
            const int grid = (int)max(1LL, min((long long)gridDim.x, total / kMinShare));
            WalkStart st{};
            st.total = total;
            st.grid = grid;
            // a whole group per CTA when the groups fit the grid and none is
            // much longer than an equal share (shares below kMinShare units
            // count as kMinShare)
            const long long share = max((total + gridDim.x - 1) / gridDim.x, (long long)kMinShare);
            st.aligned = p.G <= (int)gridDim.x && maxn <= share + share / 4;
            if (st.aligned) {
                if (c < p.G) {
                    st.g0 = c;
                    st.off0 = scr[c];
                    st.n0 = scr[c + 1] - scr[c];
                    st.j0 = 0;
                    st.ue = st.off0 + st.n0;
                    st.valid = st.n0 > 0;
                }
            } else if (total > 0 && c < grid) {
                const long long ub = total * c / grid, ue = total * (c + 1) / grid;
                if (ub < ue) {
                    int lo = 0, hi = p.G - 1;  // the last group starting at or before ub
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (scr[mid] <= ub) lo = mid;
                        else hi = mid - 1;
                    }
                    st.g0 = lo;
                    st.off0 = scr[lo];
                    st.n0 = scr[lo + 1] - scr[lo];
                    st.j0 = (int)(ub - st.off0);
                    st.ue = (int)ue;
                    st.valid = 1;
                }
            }
            *ws = st;
        }
        __syncthreads();
    }
    const WalkStart wstart = *ws;

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            Walk w;
            bool more = walk_begin(w, wstart);
            int k = 0, pc = -1;
            int kv_armed[kNKV], q_armed = -1;  // phase parity of each stage's last copy, -1: none
            for (int i = 0; i < kNKV; ++i) kv_armed[i] = -1;
            bool ok = true;
            DGroup x{};
            int page_next = 0;
            if (more && KV_FORMAT == MSA_KV_BF16)
                page_next = (w.g == (int)blockIdx.x && w.j == 0) ? page_guess
                                                                   : ld_plan(p.upage + (int64_t)w.g * p.maxu + w.j);
            while (more && ok) {
                const bool first = w.j == w.j0;
                if (first) {
                    ++pc;
                    x = dgroup(p, w.g);
                }
                const int page = page_next;
                const int s = k % kNKV;
                more = walk_next(w, p);
                if (KV_FORMAT == MSA_KV_BF16 && more) page_next = ld_plan(p.upage + (int64_t)w.g * p.maxu + w.j);
                if (KV_FORMAT == MSA_KV_BF16) {
                    if (k >= kNKV)
                        ok = tc::mbar_wait(bar(L::KV_EMPTY + s), ((k / kNKV) - 1) & 1, abort_flag, p.status,
                                           MSA_STATUS_TIMEOUT);
                    if (!ok) break;
                    if (page >= 0) {
                        tc::mbar_arrive_expect_tx(bar(L::KV_FULL + s), 65536u);
                        tc::tma_load_4d(base + L::K + s * 32768, &tm_k, bar(L::KV_FULL + s), 0, page * kBlk, 0, x.h);
                        tc::tma_load_4d(base + L::V + s * 32768, &tm_v, bar(L::KV_FULL + s), 0, page * kBlk, 0, x.h);
                    } else {
                        tc::mbar_arrive(bar(L::KV_FULL + s));  // invalid page: no copy, the rows are masked
                    }
                    kv_armed[s] = (k / kNKV) & 1;
                }
                if (first) {
                    // a new group's Q rows (after its first K/V, which does not
                    // wait for them), once the previous group's last S has read the tile
                    if (pc > 0)
                        ok = tc::mbar_wait(bar(L::Q_EMPTY), (pc - 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT);
                    if (!ok) break;
                    tc::mbar_arrive_expect_tx(bar(L::Q_FULL), 32768u);
                    const int row0 = x.b * p.Sq + x.q0;
                    tc::tma_load_3d(base + L::Q, &tm_q, bar(L::Q_FULL), 0, x.h * p.qpk, row0);
                    tc::tma_load_3d(base + L::Q + 16384, &tm_q, bar(L::Q_FULL), 64, x.h * p.qpk, row0);
                    q_armed = pc & 1;
                }
                ++k;
            }
            // drain the copies in flight before the CTA can exit
            volatile int dummy = 0;
            for (int i = 0; i < kNKV; ++i)
                if (kv_armed[i] >= 0) tc::mbar_wait(bar(L::KV_FULL + i), (uint32_t)kv_armed[i], &dummy, p.status, 0);
            if (q_armed >= 0) tc::mbar_wait(bar(L::Q_FULL), (uint32_t)q_armed, &dummy, p.status, 0);
        }
        __syncwarp();
    } else if (warp == kWarpDequant) {
        // ------------------------------------------------------------------ e4m3 K/V staging
        if (KV_FORMAT == MSA_KV_FP8) {
            Walk w;
            bool more = walk_begin(w, wstart);
            int k = 0, h = 0;
            bool ok = true;
            while (more && ok) {
                if (w.j == w.j0) h = dgroup(p, w.g).h;
                const int page = ld_plan(p.upage + (int64_t)w.g * p.maxu + w.j);
                const int s = k % kNKV;
                if (k >= kNKV)
                    ok = tc::mbar_wait(bar(L::KV_EMPTY + s), ((k / kNKV) - 1) & 1, abort_flag, p.status,
                                       MSA_STATUS_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // the page's 128 token rows of head h (an invalid page: zeros, its rows are masked)
                const int nrows = page >= 0 ? kBlk : 0;
                const int64_t first = page >= 0 ? ((int64_t)page * kBlk * p.Hkv + h) * 128 : 0;
                e4m3_rows_to_tile(base + L::K + s * 32768, p.k8 + first, (int64_t)p.Hkv * 128, nrows, lane);
                e4m3_rows_to_tile(base + L::V + s * 32768, p.v8 + first, (int64_t)p.Hkv * 128, nrows, lane);
                tc::fence_proxy_async();
                tc::mbar_arrive(bar(L::KV_FULL + s));
                more = walk_next(w, p);
                ++k;
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        // Per unit k two MMA groups are due: S_k = Q K_k^T (needs the unit's K
        // and the group's Q) and O += P_{k-1} V_{k-1} (needs P_{k-1} and, on a
        // group's first unit, a free O buffer).  The issuer polls both and
        // issues whichever becomes ready first.
        if (lane == 0) {
            Walk w;
            bool more = walk_begin(w, wstart);
            int k = 0, pc = -1;
            bool ok = true;
            int pv_k = -1, pv_s = 0, pv_pc = 0;
            bool pv_first = false, pv_last = false;
            // (a group's first PV overwrites the O buffer of group pc - 2, which
            // the softmax warps have read before they wrote this P)
            auto pv_ready = [&]() -> bool { return tc::mbar_test(bar(L::P_FULL + (pv_k & 1)), (pv_k >> 1) & 1); };
            auto issue_pv = [&]() {
                tc::fence_after_sync();
                const uint32_t vs = base + L::V + pv_s * 32768, ob = tmem + 256 + (pv_pc & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    // P of keys 16 kk .. 16 kk + 15: packed columns of key half kk / 4 (at 0 and 64)
                    tc::mma_ts(ob, tmem + (pv_k & 1) * 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                               tc::sdesc_sw128(vs + kk * 2048, 16384, 1024), kIdescPV, (kk > 0 || !pv_first) ? 1u : 0u);
                tc::mma_commit(bar(L::KV_EMPTY + pv_s));
                tc::mma_commit(bar(L::PV_DONE));
                if (pv_last) tc::mma_commit(bar(L::O_FULL + (pv_pc & 1)));
            };
            auto issue_s = [&](int kj, int s, bool last) {
                tc::fence_after_sync();
                const uint32_t qt = base + L::Q, ks = base + L::K + s * 32768;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    tc::mma_ss(tmem + (kj & 1) * 128, tc::sdesc_sw128(qt + off, 16, 1024),
                               tc::sdesc_sw128(ks + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(bar(L::S_FULL + (kj & 1)));
                if (last) tc::mma_commit(bar(L::Q_EMPTY));
            };
            // polls until S_kj (kj >= 0) and the pending PV are both issued
            auto drive = [&](int kj, int s, int q_par, bool last) -> bool {
                bool s_done = kj < 0, pv_done = pv_k < 0, kv_ok = kj < 0;
                const uint64_t t0 = tc::global_ns();
                for (uint32_t i = 0;; ++i) {
                    if (i > 0) __nanosleep(32);
                    if (!s_done) {
                        if (!kv_ok) kv_ok = tc::mbar_test(bar(L::KV_FULL + s), (kj / kNKV) & 1);
                        if (kv_ok && tc::mbar_test(bar(L::Q_FULL), (uint32_t)q_par)) {
                            issue_s(kj, s, last);
                            s_done = true;
                        }
                    }
                    if (!pv_done && pv_ready()) {
                        issue_pv();
                        pv_done = true;
                    }
                    if (s_done && pv_done) return true;
                    if ((i & 63u) == 63u) {
                        if (*abort_flag) return false;
                        if (tc::global_ns() - t0 > tc::kWaitLimitNs) break;
                    }
                }
                *abort_flag = 1;
                set_status(p.status, MSA_STATUS_TIMEOUT);
                return false;
            };
            while (more && ok) {
                const bool first = w.j == w.j0, last = w.j == w.jend - 1;
                if (first) ++pc;
                const int s = k % kNKV;
                ok = drive(k, s, pc & 1, last);
                pv_k = k;
                pv_s = s;
                pv_pc = pc;
                pv_first = first;
                pv_last = last;
                more = walk_next(w, p);
                ++k;
            }
            if (ok && pv_k >= 0) drive(-1, 0, 0, false);
            // all issued MMAs complete before tensor memory is released
            tc::mma_commit(bar(L::DRAIN));
            volatile int dummy = 0;
            tc::mbar_wait(bar(L::DRAIN), 0, &dummy, p.status, MSA_STATUS_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= kWarpSoftmax0) {
        // ------------------------------------------------------------------ softmax
        // Two warpgroups split each S row: warps 4-7 keys 0-63, warps 8-11
        // keys 64-127 of the same rows (TMEM lanes).  The two warps of a row
        // quarter exchange their half maxima through the unit's K tile, which
        // S has read and which is not reloaded before this unit's P is
        // complete, and agree on one reference max per row.
        const int hs = (warp - kWarpSoftmax0) >> 2;  // key half
        const int q4 = warp & 3;
        const int R = 32 * q4 + lane;  // row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int qi = R / p.qpk;
        Walk w;
        bool more = walk_begin(w, wstart);
        int k = 0, pc = -1;
        bool ok = true;
        DGroup x{};
        int kv = 0;
        int pg = 0, pj0 = 0, pj1 = 0, pof = 0, pn = 0;  // the group: id, this CTA's units [pj0, pj1), first unit, units
        // per row, over the group: reference max (raw score, the same in both
        // halves), this half's sum of P and of the rounded P
        float m_ref = -INFINITY, l_acc = 0.f, lr_acc = 0.f;
        // the unit's block and its selecting queries, loaded one unit ahead
        int64_t ui = more ? (int64_t)w.g * p.maxu + w.j : 0;
        int blk_n = more ? ld_plan(p.ublk + ui) : 0, page_n = more ? ld_plan(p.upage + ui) : 0;
        uint32_t mw_n = more ? ld_plan(p.umask + ui * p.wq + (qi >> 5)) : 0u;
        // (the loop is left only at a barrier of all eight warps)
        while (more) {
            const bool first = w.j == w.j0, last = w.j == w.jend - 1;
            if (first) {
                ++pc;
                x = dgroup(p, w.g);
                kv = __ldg(p.seqused + x.b);
                m_ref = -INFINITY;
                l_acc = lr_acc = 0.f;
                pg = w.g;
                pj0 = w.j0;
                pj1 = w.jend;
                pof = w.off;
                pn = w.n;
            }
            const int blk = blk_n, page = page_n;
            const uint32_t mw = mw_n;
            more = walk_next(w, p);
            if (more) {
                ui = (int64_t)w.g * p.maxu + w.j;
                blk_n = ld_plan(p.ublk + ui);
                page_n = ld_plan(p.upage + ui);
                mw_n = ld_plan(p.umask + ui * p.wq + (qi >> 5));
            }
            const int b = k & 1;
            // this half's 64 S columns; its packed P goes to the first 32 of them
            const uint32_t s_addr = tmem + lane_base + b * 128 + hs * 64;
            const uint32_t o_addr = tmem + lane_base + 256 + (pc & 1) * 128 + hs * 64;
            float *xch = reinterpret_cast<float *>(gbase + L::K + (k % kNKV) * 32768);
            // keys of the block visible to this row's query (0: not selected)
            int nvis = 0;
            if (qi < x.nq && ((mw >> (qi & 31)) & 1u) && page >= 0) {
                int limit = kv - 1;
                if (p.causal) limit = min(limit, kv - p.Sq + x.q0 + qi);  // bottom-right causal
                nvis = min(max(limit - blk * kBlk + 1, 0), kBlk);
            }
            const int nh = nvis - 64 * hs;  // visible keys of this half (may be <= 0 or > 64)
            ok = ok && tc::mbar_wait(bar(L::S_FULL + b), (k >> 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            tc::fence_after_sync();
            uint32_t pr[64];
            // (the same in both warps of the pair: nvis depends on the row only)
            const bool active = __any_sync(0xffffffffu, nvis > 0);
            // Every named barrier is reached by all the warps it names or by
            // none: the one per unit spans both warpgroups and carries their
            // `ok`, so all eight leave together when one has given up; after
            // it nothing leaves the loop before the next one.
            float mhalf = -INFINITY;
            if (active && ok) {
#define MSA_LOAD_S_HALF()                                                                    \
    do {                                                                                     \
        tc::tmem_ld64(s_addr, pr);                                                           \
        tc::tmem_ld_wait();                                                                  \
        if (nh < 64) {                                                                       \
            _Pragma("unroll") for (int j = 0; j < 64; ++j) if (j >= nh) pr[j] = 0xff800000u; \
        }                                                                                    \
    } while (0)
                MSA_LOAD_S_HALF();
                float mm[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) mm[a] = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
#pragma unroll
                    for (int a = 0; a < 4; ++a)
                        mm[a] = fmax3(mm[a], __uint_as_float(pr[j + 2 * a]), __uint_as_float(pr[j + 2 * a + 1]));
                }
                mhalf = fmax3(fmax3(mm[0], mm[1], mm[2]), mm[3], -INFINITY);
                xch[hs * 128 + R] = mhalf;
            }
            ok = pdk::bar_and(1, 256, ok);
            if (!ok) break;
            if (active) {
                const float mh = fmaxf(mhalf, xch[(1 - hs) * 128 + R]);
                // a row whose block max exceeds its reference by more than the
                // bound (rare): its O row and sums are rescaled to the new max
                // once the group's previous PV has completed (the next PV waits
                // for this unit's P); both halves decide alike
                const bool grow = nvis > 0 && m_ref != -INFINITY && (mh - m_ref) * p.scale_log2 > p.p_bound;
                if (__any_sync(0xffffffffu, grow)) {
                    bool okp = true;
                    if (!first) {
                        // (both warps of the pair take this path alike: grow
                        // follows from the shared maximum and reference)
                        okp = tc::mbar_wait(bar(L::PV_DONE), (k - 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT);
                        okp = pdk::bar_and(2 + q4, 64, __all_sync(0xffffffffu, okp));
                        ok = okp;  // on an abort, the next unit's barrier ends the loop
                    }
                    if (!first && okp) {
                        tc::fence_after_sync();
                        const float f = grow ? ex2_approx((m_ref - mh) * p.scale_log2) : 1.f;
#pragma unroll 1
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t po[32];
                            tc::tmem_ld32(o_addr + 32 * hf, po);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; ++j) po[j] = __float_as_uint(__uint_as_float(po[j]) * f);
                            tc::tmem_st32(o_addr + 32 * hf, po);
                        }
                        tc::tmem_st_wait();
                        if (grow) {
                            l_acc *= f;
                            lr_acc *= f;
                        }
                        MSA_LOAD_S_HALF();
                    }
                    if (grow) m_ref = mh;
                }
#undef MSA_LOAD_S_HALF
                if (nvis > 0 && m_ref == -INFINITY) m_ref = mh;  // the group's first visible keys of the row
                // P = exp2((S - m_ref) scale_log2) packed to bf16 in place (pr[j]
                // <- keys 2j, 2j+1 of the half); sums of P and of the rounded P
                // that PV uses
                const float mc = (m_ref == -INFINITY) ? 0.f : m_ref * p.scale_log2;
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-mc, -mc);
                float2 ll = make_float2(0.f, 0.f), lr = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float2 e = __ffma2_rn(make_float2(__uint_as_float(pr[2 * j]), __uint_as_float(pr[2 * j + 1])),
                                          sc2, nm2);
                    e.x = ex2_approx(e.x);
                    e.y = ex2_approx(e.y);
                    ll = __fadd2_rn(ll, e);
                    pr[j] = pack_bf16x2(e.x, e.y);
                    lr = __fadd2_rn(lr, make_float2(bf16_lo(pr[j]), bf16_hi(pr[j])));
                }
                l_acc += ll.x + ll.y;
                lr_acc += lr.x + lr.y;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) pr[j] = 0u;  // no row of the warp selects the block: P = 0
            }
            tc::tmem_st32(s_addr, pr);
            tc::tmem_st_wait();
            float2 tot = make_float2(0.f, 0.f);
            if (last) {
                // the group's sums over both halves (through the K tile, before
                // this unit's P lets the tile be reloaded)
                float2 *x2 = reinterpret_cast<float2 *>(xch + 256);
                x2[hs * 128 + R] = make_float2(l_acc, lr_acc);
                tc::named_bar_sync(2 + q4, 64);
                const float2 o2 = x2[(1 - hs) * 128 + R];
                tot = make_float2(l_acc + o2.x, lr_acc + o2.y);
            }
            tc::fence_proxy_async();  // generic writes to the K tile before its next TMA load
            tc::fence_before_sync();
            tc::mbar_arrive(bar(L::P_FULL + b));
            ++k;
            if (!last) continue;
            // -------- the group's end: once its last PV has completed, this
            // half's 64 columns of O / (sum of the rounded P) go to the output
            // (a group the CTA holds whole) or to the piece's slot (a cut
            // group).  The O buffer is read before any P of the group after
            // next exists, so the MMA needs no other signal to reuse it.
            const int pp = pc & 1;
            ok = ok && tc::mbar_wait(bar(L::O_FULL + pp), (pc >> 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT);
            // both warpgroups leave together on an abort (named barriers follow)
            ok = pdk::bar_and(1, 256, __all_sync(0xffffffffu, ok));
            if (!ok) break;
            tc::fence_after_sync();
            const float lse_row = tot.x > 0.f ? m_ref * p.scale + __logf(tot.x) : -INFINITY;
            const float inv = tot.y > 0.f ? 1.f / tot.y : 0.f;
            const bool cut = !wstart.aligned && (pj0 > 0 || pj1 < pn);
            const int64_t orow = ((int64_t)x.b * p.Sq + x.q0 + qi) * p.Hq + x.h * p.qpk + R % p.qpk;
            const int slot = pc == 0 ? 0 : 1;  // a cut group's piece: the CTA's first in slot 0, its last in slot 1
            const int64_t sb = ((int64_t)blockIdx.x * 2 + slot) * 128;
            {
                uint32_t o[64];
                tc::tmem_ld64(tmem + lane_base + 256 + pp * 128 + 64 * hs, o);
                tc::tmem_ld_wait();
                if (!cut && !more) {
                    // The CTA's last group: the K/V ring is idle (its last PV has
                    // run and nothing more is loaded), so each warp stages its 32
                    // rows' half (128 B a row, 16-byte chunks XOR-swizzled by
                    // row) in K stage 0 and stores them back transposed, eight
                    // lanes a row: whole 128-byte lines per store instruction.
                    const uint32_t wrow = (uint32_t)(warp - kWarpSoftmax0) * 4096u;
                    uint4 *stg = reinterpret_cast<uint4 *>(gbase + L::K + wrow);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        stg[lane * 8 + (c ^ (lane & 7))] =
                            make_uint4(pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                       pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                       pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                       pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
                    __syncwarp();
                    const int cc = lane & 7;
#pragma unroll
                    for (int k2 = 0; k2 < 8; ++k2) {
                        const int rw = 4 * k2 + (lane >> 3);  // row of the warp this lane stores
                        const int Rr = 32 * q4 + rw, qr = Rr / p.qpk;
                        if (qr < x.nq) {
                            const int64_t orr = ((int64_t)x.b * p.Sq + x.q0 + qr) * p.Hq + x.h * p.qpk + Rr % p.qpk;
                            reinterpret_cast<uint4 *>(p.o + orr * kD)[8 * hs + cc] = stg[rw * 8 + (cc ^ (rw & 7))];
                        }
                    }
                    if (hs == 0 && p.lse && qi < x.nq) p.lse[orow] = lse_row;
                } else if (!cut) {
                    if (qi < x.nq) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow * kD) + 8 * hs;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            dst[c] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
                        if (hs == 0 && p.lse) p.lse[orow] = lse_row;
                    }
                } else {
                    float4 *so = reinterpret_cast<float4 *>(p.slot_o + (sb + R) * kD) + 16 * hs;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        __stcg(so + c, make_float4(__uint_as_float(o[4 * c + 0]) * inv, __uint_as_float(o[4 * c + 1]) * inv,
                                                   __uint_as_float(o[4 * c + 2]) * inv, __uint_as_float(o[4 * c + 3]) * inv));
                    if (hs == 0) __stcg(p.slot_lse + sb + R, lse_row);
                }
            }
            if (cut) {
                // the CTA that writes the group's last piece merges all of them
                const long long total = wstart.total;
                const int grid = wstart.grid;
                const int c_first = cta_of(pof, total, grid), c_last = cta_of((long long)pof + pn - 1, total, grid);
                const int et = tid - kWarpSoftmax0 * 32;  // 0..255
                __threadfence();  // this thread's part of the piece is visible before the count says so
                tc::named_bar_sync(1, 256);
                if (et == 0) {
                    __threadfence();
                    const int prev = atomicAdd(p.merge_cnt + pg, 1);
                    __threadfence();
                    *merge_flag = prev == c_last - c_first;
                }
                tc::named_bar_sync(1, 256);
                if (*merge_flag) {
                    // Warp-cooperative: each of the eight warps merges 16 rows,
                    // eight at a time, lane l holding dims 4l .. 4l + 3; the
                    // pieces are folded in one pass with a running max.
                    const int npc = c_last - c_first + 1;
                    for (int r0 = (et >> 5) * 16; r0 < (et >> 5) * 16 + 16; r0 += 4) {
                        float mr[4], den[4];
                        float4 acc[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            mr[i] = -INFINITY;
                            den[i] = 0.f;
                            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        for (int k2 = 0; k2 < npc; ++k2) {
                            const int cc = c_first + k2;
                            const int sl = (cc > c_first || (long long)pof == total * cc / grid) ? 0 : 1;
                            const int64_t rb = ((int64_t)cc * 2 + sl) * 128 + r0;
                            float lv[4];
                            float4 ov[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                lv[i] = __ldcg(p.slot_lse + rb + i);
                                ov[i] = __ldcg(reinterpret_cast<const float4 *>(p.slot_o + (rb + i) * kD) + lane);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float mn = fmaxf(mr[i], lv[i]);
                                if (mn != -INFINITY) {  // the same for every lane (one row)
                                    const float a = __expf(mr[i] - mn), bw = __expf(lv[i] - mn);
                                    acc[i] = make_float4(acc[i].x * a + ov[i].x * bw, acc[i].y * a + ov[i].y * bw,
                                                         acc[i].z * a + ov[i].z * bw, acc[i].w * a + ov[i].w * bw);
                                    den[i] = den[i] * a + bw;
                                    mr[i] = mn;
                                }
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = r0 + i, rq = r / p.qpk;
                            if (rq >= x.nq) continue;
                            const float dinv = den[i] > 0.f ? 1.f / den[i] : 0.f;
                            const int64_t orr = ((int64_t)x.b * p.Sq + x.q0 + rq) * p.Hq + x.h * p.qpk + r % p.qpk;
                            reinterpret_cast<uint2 *>(p.o + orr * kD)[lane] =
                                make_uint2(pack_bf16x2(acc[i].x * dinv, acc[i].y * dinv),
                                           pack_bf16x2(acc[i].z * dinv, acc[i].w * dinv));
                            if (p.lse && lane == 0) p.lse[orr] = den[i] > 0.f ? mr[i] + __logf(den[i]) : -INFINITY;
                        }
                    }
                }
                // the merge flag is read by all before the next group's count
                // may change it (at the next cut group's first barrier)
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// The launch of the decode kernel instance for a K/V format; each instance is
// compiled in a translation unit of its own (paged_decode_*.cu).
#define MSA_DECODE_INSTANCE(NAME)                                                                                     \
    int NAME(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const DecodeParams &p, int grid, \
             cudaStream_t stream)
MSA_DECODE_INSTANCE(launch_paged_decode_bf16);
MSA_DECODE_INSTANCE(launch_paged_decode_fp8);

template <int KV_FORMAT>
int launch_paged_decode(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const DecodeParams &p,
                        int grid, cudaStream_t stream) {
    const size_t smem = pdk::Layout::BYTES;
    MSA_CUDA_TRY(
        cudaFuncSetAttribute(paged_decode_kernel<KV_FORMAT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    MSA_CUDA_TRY(launch_pdl(paged_decode_kernel<KV_FORMAT>, dim3(grid), dim3(pdk::kThreads), smem, stream, mk, mv, mq,
                            p));
    return MSA_OK;
}

}  // namespace msa
