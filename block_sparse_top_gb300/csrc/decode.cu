// decode.cu -- block-sparse paged decode by per-group block unions, the
// kernel behind msa_sparse_attn_paged_fwd_noalloc (its scratch is small
// enough for a static device array; msa_sparse_attn_paged_fwd runs the
// prefill tile pipeline over logical blocks instead, see attn.cu).
//
// A group is (sequence b, KV head h, 128/qhead_per_kv consecutive queries):
// 128 query-head rows that share the KV head.  Three launches:
//   1. union:  per group, the sorted union of the blocks its queries selected
//              (ids >= ceil(seqused/page) and repeats are dropped), with a
//              bitmask of the queries that selected each block; groups whose
//              union is empty write O = 0, LSE = -inf at once.
//   2. scan:   exclusive prefix of the union sizes -> one global block list.
//   3. main:   persistent, one CTA per SM; CTA c takes an equal slice of the
//              global list.  A producer warp streams each block's K and V
//              (logical block j of sequence b = physical page page_table[b][j];
//              token rows of Hkv*D bf16) by TMA through a 3-stage ring with
//              full/empty mbarriers; eight compute warps (16 rows each, warp
//              MMA) run an online softmax over the blocks their queries
//              selected, each at its own pace.  A group inside one slice is
//              written directly; a group cut by slice boundaries leaves one
//              partial per slice, merged by the warp that finishes last
//              (atomic counter over warps, no waiting).
//
// Source: interface.py sparse_decode_atten_func and
// SparseDecodePagedAttentionWrapper (paged KV, seqused_k, uniform seqlen_q,
// split-KV partials merged by LSE); test_sparse_atten.py
// _decode_paged_dense_reference (running max/sum, lse = m + log l, -inf for
// empty rows) and _decode_paged_kv_chunk (page-table addressing).
#include <algorithm>
#include <cstring>

#include "attn_mma.cuh"
#include "tc.cuh"

namespace msa {
namespace {

constexpr int kMaxPagesDecode = 8192;  // union bitmap bound (1M tokens per sequence)
constexpr int kDecStages = 3;
constexpr int kDecWarps = 9;           // warps 0-7 compute, warp 8 produces
constexpr int kDecThreads = kDecWarps * 32;
constexpr uint32_t kDecSmQ = kDecStages * 65536;          // 8 warps x 16 rows x 256 B
constexpr uint32_t kDecSmBar = kDecSmQ + 8 * 4096;
constexpr uint32_t kDecSmInfo = kDecSmBar + 8 * 2 * kDecStages;
constexpr uint32_t kDecSmMisc = kDecSmInfo + 16 * kDecStages;
constexpr uint32_t kDecSmBytes = kDecSmMisc + 16;
constexpr uint32_t kDecSmAlloc = kDecSmBytes + 1024;

struct DecParams {
    const __nv_bfloat16 *q;
    const int32_t *page_table, *seqused, *q2k;
    __nv_bfloat16 *o;
    float *lse;
    int32_t *ulist;      // [groups][maxu] union block ids (ascending)
    uint32_t *umask;     // [groups][maxu][wq] queries of the group that selected the block
    int32_t *off;        // [groups + 1] union sizes, then their exclusive prefix
    int32_t *counters;   // [groups] pieces of a cut group already written
    float *o_part;       // [grid][2][128][D] normalised partial O
    float *lse_part;     // [grid][2][128]
    uint32_t *status;
    int B, Sq, Hq, Hkv, qpk, topk, num_pages, max_pages, causal, qgroups, groups, maxu, wq, grid;
    float scale, scale_log2;
};

struct GroupInfo {
    int b, h, q0, nq, seqused;
};

__device__ __forceinline__ GroupInfo group_info(const DecParams &p, int g) {
    GroupInfo gi;
    const int qg = 128 / p.qpk;
    gi.b = g / (p.Hkv * p.qgroups);
    const int rem = g % (p.Hkv * p.qgroups);
    gi.h = rem / p.qgroups;
    gi.q0 = (rem % p.qgroups) * qg;
    gi.nq = min(qg, p.Sq - gi.q0);
    gi.seqused = p.seqused[gi.b];
    return gi;
}

// ---------------------------------------------------------------- 1. unions
__global__ void __launch_bounds__(256) decode_union_kernel(DecParams p) {
    extern __shared__ uint32_t dsm[];
    uint32_t *bitmap = dsm;                                                 // kMaxPagesDecode / 32
    int32_t *ul = reinterpret_cast<int32_t *>(dsm + kMaxPagesDecode / 32);  // maxu
    uint32_t *mk = reinterpret_cast<uint32_t *>(ul + p.maxu);              // maxu * wq
    __shared__ int32_t warp_tot[8];
    __shared__ int32_t s_nu;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupInfo gi = group_info(p, g);
    const int qg = 128 / p.qpk;
    const int nvalid = (int)min((int64_t)ceil_div((int64_t)max(gi.seqused, 0), kBlk), (int64_t)p.max_pages);
    const int nwords = (nvalid + 31) / 32;
    for (int i = tid; i < nwords; i += blockDim.x) bitmap[i] = 0u;
    for (int i = tid; i < p.maxu * p.wq; i += blockDim.x) mk[i] = 0u;
    __syncthreads();
    // dense mode (no q2k): every block below the used length, every query
    for (int j = tid; !p.q2k && j < nvalid; j += blockDim.x) atomicOr(&bitmap[j >> 5], 1u << (j & 31));
    for (int i = tid; p.q2k && i < gi.nq * p.topk; i += blockDim.x) {
        const int qi = i / p.topk, t = i % p.topk;
        const int32_t *sel = p.q2k + (((int64_t)gi.b * p.Hkv + gi.h) * p.Sq + gi.q0 + qi) * p.topk;
        int j = sel[t];
        if (j < 0) continue;
        if (j >= nvalid) {
            set_status(p.status, MSA_STATUS_INDEX_RANGE);
            continue;
        }
        bool dup = false;
        for (int u = 0; u < t; ++u) dup |= (sel[u] == j);
        if (dup) {
            set_status(p.status, MSA_STATUS_DUPLICATE);
            continue;
        }
        atomicOr(&bitmap[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    // compact in ascending block order
    {
        const int per = (nwords + blockDim.x - 1) / blockDim.x;
        const int w0 = tid * per, w1 = min(w0 + per, nwords);
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
        int pos = x - cnt;
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
    // selection masks: every query of the group (dense), or the position of
    // each selected block by binary search
    for (int i = tid; !p.q2k && i < nu * p.wq; i += blockDim.x) {
        const int w = i % p.wq, n = min(32, gi.nq - 32 * w);
        mk[i] = n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : ((1u << n) - 1u));
    }
    for (int i = tid; p.q2k && i < gi.nq * p.topk; i += blockDim.x) {
        const int qi = i / p.topk;
        const int32_t *sel = p.q2k + (((int64_t)gi.b * p.Hkv + gi.h) * p.Sq + gi.q0 + qi) * p.topk;
        const int j = sel[i % p.topk];
        if (j < 0 || j >= nvalid) continue;
        int lo = 0, hi = nu;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (ul[mid] < j) lo = mid + 1;
            else hi = mid;
        }
        atomicOr(&mk[lo * p.wq + (qi >> 5)], 1u << (qi & 31));
    }
    __syncthreads();
    for (int e = tid; e < nu; e += blockDim.x) p.ulist[(int64_t)g * p.maxu + e] = ul[e];
    for (int i = tid; i < nu * p.wq; i += blockDim.x) p.umask[(int64_t)g * p.maxu * p.wq + i] = mk[i];
    if (tid == 0) p.off[g] = nu;
    if (nu == 0) {
        // no block at all: O = 0, LSE = -inf for every row of the group
        for (int i = tid; i < qg * p.qpk * 16; i += blockDim.x) {
            const int R = i >> 4, ch = i & 15, qi = R / p.qpk;
            if (qi >= gi.nq) continue;
            const int64_t gq = (int64_t)gi.b * p.Sq + gi.q0 + qi;
            const int hq = gi.h * p.qpk + R % p.qpk;
            reinterpret_cast<uint4 *>(p.o + (gq * p.Hq + hq) * kD)[ch] = make_uint4(0, 0, 0, 0);
            if (ch == 0 && p.lse) p.lse[gq * p.Hq + hq] = -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- 2. scan
// In place: off[0..groups) sizes -> exclusive prefix, off[groups] = total.
__global__ void __launch_bounds__(1024) decode_scan_kernel(int32_t *off, int n) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int32_t v = (i < n) ? off[i] : 0;
        int32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int32_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry_s;
        if (i < n) off[i] = incl - v;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry_s = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) off[n] = carry_s;
}

// ---------------------------------------------------------------- 3. main
__device__ __forceinline__ int64_t slice_lo(int c, int64_t E, int G) { return (int64_t)c * E / G; }

// CTA whose slice holds entry e.
__device__ __forceinline__ int cta_of(int64_t e, int64_t E, int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (slice_lo(mid, E, G) <= e) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Slices that hold a part of [g_lo, g_hi): the non-empty slices between the
// owners of its first and last entry (small problems leave empty slices).
__device__ __forceinline__ int pieces_of(int64_t g_lo, int64_t g_hi, int64_t E, int G) {
    const int c_first = cta_of(g_lo, E, G), c_last = cta_of(g_hi - 1, E, G);
    int n = 0;
    for (int cc = c_first; cc <= c_last; ++cc) n += slice_lo(cc + 1, E, G) > slice_lo(cc, E, G) ? 1 : 0;
    return n;
}

// Group holding entry e (largest g with off[g] <= e).
__device__ __forceinline__ int group_of(const int32_t *off, int groups, int64_t e) {
    int lo = 0, hi = groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= e) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Last warp of a cut group: LSE-merges the partials of every slice that
// holds a part of the group and writes the group's O and LSE.  One warp; each
// lane handles 8 of the 256 (row, half of the dims) items.
__device__ __noinline__ void merge_pieces(const DecParams &p, const GroupInfo &gi, int64_t g_lo, int64_t g_hi,
                                          int64_t E, int G, int lane) {
    const int c_first = cta_of(g_lo, E, G), c_last = cta_of(g_hi - 1, E, G);
    for (int it = lane; it < 256; it += 32) {
        const int R = it >> 1, half = it & 1, qi = R / p.qpk;
        float mx = -INFINITY;
        for (int cc = c_first; cc <= c_last; ++cc) {
            if (slice_lo(cc + 1, E, G) <= slice_lo(cc, E, G)) continue;  // empty slice
            const int sl = (g_lo < slice_lo(cc, E, G)) ? 0 : 1;
            mx = fmaxf(mx, __ldcg(p.lse_part + ((int64_t)cc * 2 + sl) * 128 + R));
        }
        float den = 0.f, acc[64];
#pragma unroll
        for (int d = 0; d < 64; ++d) acc[d] = 0.f;
        for (int cc = c_first; cc <= c_last; ++cc) {
            if (slice_lo(cc + 1, E, G) <= slice_lo(cc, E, G)) continue;  // empty slice
            const int sl = (g_lo < slice_lo(cc, E, G)) ? 0 : 1;
            const float ls = __ldcg(p.lse_part + ((int64_t)cc * 2 + sl) * 128 + R);
            if (!(ls > -INFINITY) || !(mx > -INFINITY)) continue;
            const float w = __expf(ls - mx);
            den += w;
            const float4 *src =
                reinterpret_cast<const float4 *>(p.o_part + (((int64_t)cc * 2 + sl) * 128 + R) * kD + half * 64);
#pragma unroll
            for (int d4 = 0; d4 < 16; ++d4) {
                const float4 v = __ldcg(src + d4);
                acc[4 * d4] += w * v.x;
                acc[4 * d4 + 1] += w * v.y;
                acc[4 * d4 + 2] += w * v.z;
                acc[4 * d4 + 3] += w * v.w;
            }
        }
        if (qi < gi.nq) {
            const int64_t gq = (int64_t)gi.b * p.Sq + gi.q0 + qi;
            const int hq = gi.h * p.qpk + R % p.qpk;
            const float inv = den > 0.f ? 1.f / den : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + (gq * p.Hq + hq) * kD + half * 64);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                dst[cc] = make_uint4(pack_bf16x2(acc[8 * cc] * inv, acc[8 * cc + 1] * inv),
                                     pack_bf16x2(acc[8 * cc + 2] * inv, acc[8 * cc + 3] * inv),
                                     pack_bf16x2(acc[8 * cc + 4] * inv, acc[8 * cc + 5] * inv),
                                     pack_bf16x2(acc[8 * cc + 6] * inv, acc[8 * cc + 7] * inv));
            if (half == 0 && p.lse) p.lse[gq * p.Hq + hq] = den > 0.f ? mx + logf(den) : -INFINITY;
        }
    }
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_main_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       DecParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - smem_u32(smem_raw));
    int4 *info = reinterpret_cast<int4 *>(gbase + kDecSmInfo);                 // per stage: {g, local e, j, ok}
    volatile int *misc = reinterpret_cast<volatile int *>(gbase + kDecSmMisc);  // [0] abort, [1] last piece
    auto full = [&](int s) -> uint32_t { return base + kDecSmBar + 8u * s; };
    auto empty = [&](int s) -> uint32_t { return base + kDecSmBar + 8u * (kDecStages + s); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int64_t E = p.off[p.groups];
    const int64_t e_lo = slice_lo(c, E, G), e_hi = slice_lo(c + 1, E, G);
    const int n = (int)(e_hi - e_lo);

    if (tid == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            tc::mbar_init(full(s), 1);
            tc::mbar_init(empty(s), 8);
        }
        misc[0] = 0;
        tc::mbar_fence_init();
        tc::tma_prefetch_desc(&tm_k);
        tc::tma_prefetch_desc(&tm_v);
    }
    __syncthreads();

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            int armed[kDecStages];
            for (int s = 0; s < kDecStages; ++s) armed[s] = -1;
            int g = group_of(p.off, p.groups, e_lo);
            for (int k = 0; k < n; ++k) {
                const int64_t e = e_lo + k;
                const int s = k % kDecStages;
                if (k >= kDecStages &&
                    !tc::mbar_wait(empty(s), ((k / kDecStages) - 1) & 1, misc, p.status, MSA_STATUS_TIMEOUT))
                    break;
                while (p.off[g + 1] <= e) ++g;
                const GroupInfo gi = group_info(p, g);
                const int le = (int)(e - p.off[g]);
                const int j = p.ulist[(int64_t)g * p.maxu + le];
                const int page = p.page_table[(int64_t)gi.b * p.max_pages + j];
                const int ok = (page >= 0 && page < p.num_pages) ? 1 : 0;
                info[s] = make_int4(g, le, j, ok);
                if (ok) {
                    const uint32_t st = base + s * 65536;
                    tc::mbar_arrive_expect_tx(full(s), 65536);
                    tc::tma_load_4d(st, &tm_k, full(s), 0, page * kBlk, 0, gi.h);
                    tc::tma_load_4d(st + 32768, &tm_v, full(s), 0, page * kBlk, 0, gi.h);
                } else {
                    set_status(p.status, MSA_STATUS_PAGE_RANGE);
                    tc::mbar_arrive(full(s));
                }
                armed[s] = (k / kDecStages) & 1;
            }
            volatile int dummy = 0;
            for (int s = 0; s < kDecStages; ++s)
                if (armed[s] >= 0) tc::mbar_wait(full(s), (uint32_t)armed[s], &dummy, p.status, 0);
        }
        __syncwarp();
    } else if (n > 0) {
        // ------------------------------------------------------------ compute warps
        const int g_row = lane >> 2, t = lane & 3;
        const int row0 = warp * 16;
        const int qpk = p.qpk;
        int cur_g = -1;
        GroupInfo gi{};
        const uint32_t q_s = base + kDecSmQ + warp * 4096;  // this warp's 16 query rows
        float m[2], l[2], o[16][4];
        int qi_row[2], limit_row[2];
        bool ok = true;

        auto begin_group = [&](int g) {
            cur_g = g;
            gi = group_info(p, g);
            m[0] = m[1] = -INFINITY;
            l[0] = l[1] = 0.f;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int R = row0 + g_row + 8 * hr;
                qi_row[hr] = R / qpk;
                const int pos = gi.seqused - p.Sq + gi.q0 + qi_row[hr];
                limit_row[hr] = p.causal ? min(pos, gi.seqused - 1) : gi.seqused - 1;
            }
            // the warp's 16 query rows into its swizzled shared tile (zero rows past nq)
            __syncwarp();
#pragma unroll
            for (int i = lane; i < 16 * 16; i += 32) {
                const int r = i >> 4, ch = i & 15, R = row0 + r, qi = R / qpk;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (qi < gi.nq)
                    v = *reinterpret_cast<const uint4 *>(
                        p.q + (((int64_t)gi.b * p.Sq + gi.q0 + qi) * p.Hq + gi.h * qpk + R % qpk) * kD + ch * 8);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_s + swz_off(r, ch)), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w));
            }
            __syncwarp();
        };

        // writes the group's rows: final output when the whole group is in this
        // slice, else this slice's partial and, for the last piece, the merge.
        auto end_group = [&]() {
            const int64_t g_lo = p.off[cur_g], g_hi = p.off[cur_g + 1];
            const bool whole = (g_lo >= e_lo && g_hi <= e_hi);
            const int slot = (g_lo < e_lo) ? 0 : 1;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int R = row0 + g_row + 8 * hr;
                const float inv = l[hr] > 0.f ? 1.f / l[hr] : 0.f;
                const float lse_v = l[hr] > 0.f ? m[hr] * p.scale + logf(l[hr]) : -INFINITY;
                if (whole) {
                    if (qi_row[hr] >= gi.nq) continue;
                    const int64_t gq = (int64_t)gi.b * p.Sq + gi.q0 + qi_row[hr];
                    const int hq = gi.h * qpk + R % qpk;
                    __nv_bfloat16 *orow = p.o + (gq * p.Hq + hq) * kD;
#pragma unroll
                    for (int nt = 0; nt < 16; ++nt)
                        *reinterpret_cast<uint32_t *>(orow + nt * 8 + 2 * t) =
                            pack_bf16x2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
                    if (t == 0 && p.lse) p.lse[gq * p.Hq + hq] = lse_v;
                } else {
                    float *orow = p.o_part + (((int64_t)c * 2 + slot) * 128 + R) * kD;
#pragma unroll
                    for (int nt = 0; nt < 16; ++nt)
                        *reinterpret_cast<float2 *>(orow + nt * 8 + 2 * t) =
                            make_float2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
                    if (t == 0) p.lse_part[((int64_t)c * 2 + slot) * 128 + R] = lse_v;
                }
            }
            if (whole) return;
            // cut group: every warp of every piece counts itself once its rows
            // are written; the warp that arrives last merges (no CTA barrier)
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                const int prev = atomicAdd(&p.counters[cur_g], 1);
                last = (prev == pieces_of(g_lo, g_hi, E, G) * 8 - 1) ? 1 : 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!last) return;
            __threadfence();
            merge_pieces(p, gi, g_lo, g_hi, E, G, lane);
            if (lane == 0) p.counters[cur_g] = 0;  // ready for the next call
        };

        for (int k = 0; k < n; ++k) {
            const int s = k % kDecStages;
            ok = tc::mbar_wait(full(s), (k / kDecStages) & 1, misc, p.status, MSA_STATUS_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int4 in = info[s];
            if (in.x != cur_g) {
                if (cur_g >= 0) end_group();
                begin_group(in.x);
            }
            // does any query of this warp select the block?
            const uint32_t *mask = p.umask + ((int64_t)cur_g * p.maxu + in.y) * p.wq;
            const int wq0 = row0 / qpk, wq1 = (row0 + 15) / qpk;
            bool sel_row[2];
            bool any = false;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int qi = qi_row[hr];
                sel_row[hr] = qi < gi.nq && ((mask[qi >> 5] >> (qi & 31)) & 1u);
            }
            for (int qi = wq0; qi <= wq1 && qi < gi.nq; ++qi) any |= ((mask[qi >> 5] >> (qi & 31)) & 1u) != 0;
            if (in.w && any) {
                const uint32_t st = base + s * 65536;
                int nvis[2];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    nvis[hr] = sel_row[hr] ? max(0, min(128, limit_row[hr] - in.z * kBlk + 1)) : 0;
                // two halves of 64 keys, online softmax across them
#pragma unroll 1
                for (int kh = 0; kh < 2; ++kh) {
                    const bool none = __all_sync(0xffffffffu, nvis[0] <= kh * 64 && nvis[1] <= kh * 64);
                    if (none) break;  // no row of the warp sees a key of this half
                    float sc[8][4];
                    warp_qk_qs_tma_half(q_s, st, kh, sc);
                    float mnew[2] = {m[0], m[1]};
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                        for (int ee = 0; ee < 4; ++ee) {
                            const int hr = ee >> 1;
                            const int key = kh * 64 + nt * 8 + 2 * t + (ee & 1);
                            if (key >= nvis[hr]) sc[nt][ee] = -INFINITY;
                            mnew[hr] = fmaxf(mnew[hr], sc[nt][ee]);
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
                    uint32_t pk[8][2];
                    float lsum[2] = {0.f, 0.f};
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        float pe[4];
#pragma unroll
                        for (int ee = 0; ee < 4; ++ee) {
                            const int hr = ee >> 1;
                            const float x =
                                (m[hr] == -INFINITY) ? 0.f : ex2_approx((sc[nt][ee] - m[hr]) * p.scale_log2);
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
                    warp_pv_tma_half(st + 32768, kh, pk, o);
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(empty(s));
        }
        if (ok && cur_g >= 0) end_group();
    }
    __syncthreads();
}

struct DecWorkspace {
    size_t ulist, umask, off, counters, lse_part, o_part, bytes;
};

int decode_num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
        cached[dev] = n;
    }
    return cached[dev];
}

struct DecShape {
    int qgroups, groups, maxu, wq, grid;
};

DecShape dec_shape(int B, int Sq, int Hkv, int qpk, int topk, int max_pages) {
    DecShape d;
    const int qg = 128 / qpk;
    d.qgroups = (int)ceil_div(Sq, qg);
    d.groups = B * Hkv * d.qgroups;
    d.maxu = std::min(std::min(Sq, qg) * topk, max_pages);
    d.wq = (qg + 31) / 32;
    d.grid = decode_num_sms();
    return d;
}

DecWorkspace dec_workspace_layout(const DecShape &d) {
    DecWorkspace w;
    size_t o = 0;
    w.ulist = o;
    o = align_up(o + sizeof(int32_t) * (size_t)d.groups * d.maxu, 256);
    w.umask = o;
    o = align_up(o + sizeof(uint32_t) * (size_t)d.groups * d.maxu * d.wq, 256);
    w.off = o;
    o = align_up(o + sizeof(int32_t) * ((size_t)d.groups + 1), 256);
    w.counters = o;
    o = align_up(o + sizeof(int32_t) * (size_t)d.groups, 256);
    w.lse_part = o;
    o = align_up(o + sizeof(float) * (size_t)d.grid * 2 * 128, 256);
    w.o_part = o;
    o = align_up(o + sizeof(float) * (size_t)d.grid * 2 * 128 * kD, 256);
    w.bytes = o;
    return w;
}

}  // namespace

// Scratch bytes of union_paged_fwd for a shape (0: unsupported).
size_t union_paged_fwd_scratch(int B, int Sq, int Hq, int Hkv, int D, int topk, int max_pages) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || D != kD || topk <= 0 || max_pages <= 0 || Hq % Hkv) return 0;
    const int qpk = Hq / Hkv;
    if (!supported_qpk(qpk)) return 0;
    return dec_workspace_layout(dec_shape(B, Sq, Hkv, qpk, topk, max_pages)).bytes;
}

// Paged decode by per-group block unions (union, scan and main kernels
// above), in the scratch it is given.
int union_paged_fwd(const void *q, const void *k_pool, const void *v_pool, int num_pages, const int32_t *page_table,
                    int max_pages, const int32_t *seqused_k, const int32_t *q2k, int B, int Sq, int Hq, int Hkv,
                    int D, int page_size, int topk, int causal, float softmax_scale, void *o, float *lse,
                    void *workspace, size_t ws_bytes, uint32_t *status_dev, cudaStream_t stream) {
    // q2k == NULL: dense mode, every block of the sequence (topk is then unused)
    if (!q2k) topk = max_pages;
    if (!q || !k_pool || !v_pool || !page_table || !seqused_k || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pages <= 0 || topk <= 0 || Hq % Hkv)
        return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || page_size != kBlk || (q2k && !supported_topk(topk)) || !supported_qpk(qpk))
        return MSA_ERR_UNSUPPORTED;
    if (max_pages > kMaxPagesDecode || (int64_t)B * Sq >= (1 << 24)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)num_pages * kBlk >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o, 16))
        return MSA_ERR_INVALID_ARG;
    const DecShape d = dec_shape(B, Sq, Hkv, qpk, topk, max_pages);
    const DecWorkspace w = dec_workspace_layout(d);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);

    DecParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.page_table = page_table;
    p.seqused = seqused_k;
    p.q2k = q2k;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.ulist = reinterpret_cast<int32_t *>(ws + w.ulist);
    p.umask = reinterpret_cast<uint32_t *>(ws + w.umask);
    p.off = reinterpret_cast<int32_t *>(ws + w.off);
    p.counters = reinterpret_cast<int32_t *>(ws + w.counters);
    p.lse_part = reinterpret_cast<float *>(ws + w.lse_part);
    p.o_part = reinterpret_cast<float *>(ws + w.o_part);
    p.status = status_dev;
    p.B = B; p.Sq = Sq; p.Hq = Hq; p.Hkv = Hkv; p.qpk = qpk; p.topk = topk;
    p.num_pages = num_pages; p.max_pages = max_pages; p.causal = causal ? 1 : 0;
    p.qgroups = d.qgroups; p.groups = d.groups; p.maxu = d.maxu; p.wq = d.wq; p.grid = d.grid;
    p.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    p.scale_log2 = p.scale * 1.4426950408889634f;

    CUtensorMap mk, mv;
    if (!make_kv_map(&mk, k_pool, Hkv, (int64_t)num_pages * kBlk) ||
        !make_kv_map(&mv, v_pool, Hkv, (int64_t)num_pages * kBlk))
        return MSA_ERR_CUDA;

    MSA_CUDA_TRY(cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * (size_t)d.groups, stream));
    const size_t usmem = sizeof(uint32_t) * (kMaxPagesDecode / 32) + sizeof(int32_t) * (size_t)d.maxu +
                         sizeof(uint32_t) * (size_t)d.maxu * d.wq;
    if (usmem > 227 * 1024) return MSA_ERR_UNSUPPORTED;
    MSA_CUDA_TRY(cudaFuncSetAttribute(decode_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)std::max<size_t>(usmem, sizeof(uint32_t) * (kMaxPagesDecode / 32 + 128 * 32 * 5))));
    MSA_CUDA_TRY(cudaFuncSetAttribute(decode_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kDecSmAlloc));
    decode_union_kernel<<<d.groups, 256, usmem, stream>>>(p);
    MSA_LAUNCH_CHECK();
    decode_scan_kernel<<<1, 1024, 0, stream>>>(p.off, d.groups);
    MSA_LAUNCH_CHECK();
    decode_main_kernel<<<d.grid, kDecThreads, kDecSmAlloc, stream>>>(mk, mv, p);
    MSA_LAUNCH_CHECK();
    return MSA_OK;
}

}  // namespace msa

// ---------------------------------------------------------------------------
// Paged decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: a serving loop whose memory is fixed at start-up, or code that
// must not call cudaMalloc while other work is queued.  This variant runs the
// per-group union decode (whose scratch is small) and keeps that scratch
// (block unions, split counters and partials) in one file-scope device array of
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
    // the argument and support checks of the allocating entry point come
    // first, so that a bad argument is reported as such whatever its size
    if (!q || !k_pool || !v_pool || !page_table || !seqused_k || !q2k || !o) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pages <= 0 || topk <= 0 || Hq % Hkv)
        return MSA_ERR_INVALID_ARG;
    if (D != msa::kD || page_size != msa::kBlk || !msa::supported_topk(topk) || !msa::supported_qpk(Hq / Hkv))
        return MSA_ERR_UNSUPPORTED;
    if (max_pages > msa::kMaxPagesDecode || (int64_t)B * Sq >= (1 << 24)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)num_pages * msa::kBlk >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
    if (!msa::aligned(q, 16) || !msa::aligned(k_pool, 16) || !msa::aligned(v_pool, 16) || !msa::aligned(o, 16))
        return MSA_ERR_INVALID_ARG;
    const size_t need = msa::union_paged_fwd_scratch(B, Sq, Hq, Hkv, D, topk, max_pages);
    if (need == 0) return MSA_ERR_UNSUPPORTED;
    if (need > msa::kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // shape needs more than the static scratch
    void *scratch = msa::paged_scratch_for_current_device();
    if (!scratch) return MSA_ERR_CUDA;
    return msa::union_paged_fwd(q, k_pool, v_pool, num_pages, page_table, max_pages, seqused_k, q2k, B, Sq, Hq, Hkv,
                                D, page_size, topk, causal, softmax_scale, o, lse, scratch,
                                msa::kNoAllocScratchBytes, status_dev, stream);
}
