// attn_tc.cuh -- the tcgen05 (5th-gen tensor core) block-sparse prefill tile
// kernel: persistent, one CTA per SM, warp-specialised.
//
//   warps 0-3   loader: per work unit the K and V block by TMA (bf16; 128-byte
//               swizzle) or, for NVFP4, by plain loads dequantised into the
//               same swizzled layout; per chunk the 128 gathered Q rows
//               (128/qhead_per_kv queries x all heads of the GQA group) by
//               16-byte cp.async into a 3-stage ring.
//   warp 12     MMA issuer (one thread): S_i = Q_i K^T into tensor memory,
//               then O_{i-1} = P_{i-1} V with P read from tensor memory.
//   warps 4-7,  softmax + epilogue for even / odd chunks: each thread owns one
//   warps 8-11  S row (TMEM lane), applies the bottom-right causal limit,
//               writes P = exp(S - m) as bf16 over S, then scales O by 1/l and
//               stores the split partial (bf16) and its lse.
//
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
// Every wait is bounded; on a timeout the CTA raises MSA_STATUS_TIMEOUT,
// drains its copies and MMAs, frees tensor memory and exits.
#pragma once
#include "attn_mma.cuh"
#include "tc.cuh"

namespace msa {

struct TcParams {
    const __nv_bfloat16 *q;
    const uint8_t *k_packed, *v_packed;   // NVFP4 only
    const uint8_t *k_scales, *v_scales;   // NVFP4 only
    const int32_t *qsplit;
    const PlanHeader *plan;
    const PlanUnit *units;
    __nv_bfloat16 *o_part;                // [B*Sq][topk][Hq][D]
    float *lse_part;                      // [B*Sq][topk][Hq]
    uint32_t *status;
    int B, Sq, Skv, Hq, Hkv, qpk, topk, nblk, causal;
    int64_t cap;
    float scale, scale_log2;
};

namespace tck {

constexpr int kNQ = 3;
constexpr int kThreads = 13 * 32;
constexpr uint32_t kSmK = 0, kSmV = 65536, kSmQ = 131072;
constexpr uint32_t kSmBar = kSmQ + kNQ * 32768;
enum : int {
    KV_FULL = 0,
    KV_EMPTY = 2,
    Q_FULL = 4,
    Q_EMPTY = 4 + kNQ,
    S_FULL = 4 + 2 * kNQ,
    P_FULL = S_FULL + 2,
    O_FULL = P_FULL + 2,
    O_EMPTY = O_FULL + 2,
    DRAIN = O_EMPTY + 2,
    NBAR = DRAIN + 1
};
constexpr uint32_t kSmTslot = kSmBar + 8 * NBAR;
constexpr uint32_t kSmAbort = kSmTslot + 4;
constexpr uint32_t kSmRowq = (kSmAbort + 8 + 15) & ~15u;
constexpr uint32_t kSmBytes = kSmRowq + 128 * 4;
constexpr uint32_t kSmAlloc = kSmBytes + 1024;  // slack for 1024-byte alignment
static_assert(kSmAlloc <= 232448, "shared memory budget");

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, 0, 1);
constexpr uint32_t MSA_STATUS_TIMEOUT_BIT = MSA_STATUS_TIMEOUT;

struct Unit {
    int h, b, tok0, start, count, nch;
};

__device__ __forceinline__ Unit load_unit(const TcParams &p, int u) {
    PlanUnit pu = p.units[u];
    Unit x;
    x.h = pu.head;
    x.b = pu.row / p.nblk;
    x.tok0 = (pu.row % p.nblk) * kBlk;
    x.start = pu.start;
    x.count = pu.count;
    int qc = 128 / p.qpk;
    x.nch = (pu.count + qc - 1) / qc;
    return x;
}

}  // namespace tck

template <int KV_FORMAT>
__global__ void __launch_bounds__(tck::kThreads, 1)
    sparse_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         TcParams p) {
    using namespace tck;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - smem_u32(smem_raw));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kSmAbort);
    int32_t *rowq = reinterpret_cast<int32_t *>(gbase + kSmRowq);
    auto bar = [&](int i) -> uint32_t { return base + kSmBar + 8u * (uint32_t)i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qc = 128 / p.qpk;
    const int work = p.plan->work_count;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(KV_FULL + i), KV_FORMAT == MSA_KV_BF16 ? 1 : 128);
            tc::mbar_init(bar(KV_EMPTY + i), 1);
            tc::mbar_init(bar(S_FULL + i), 1);
            tc::mbar_init(bar(P_FULL + i), 128);
            tc::mbar_init(bar(O_FULL + i), 1);
            tc::mbar_init(bar(O_EMPTY + i), 128);
        }
        for (int i = 0; i < kNQ; ++i) {
            tc::mbar_init(bar(Q_FULL + i), 128);
            tc::mbar_init(bar(Q_EMPTY + i), 1);
        }
        tc::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == 12) {
        tc::tmem_alloc(base + kSmTslot, 512);
        tc::tmem_relinquish();
    }
    if (KV_FORMAT == MSA_KV_BF16 && tid == 0) {
        tc::tma_prefetch_desc(&tm_k);
        tc::tma_prefetch_desc(&tm_v);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + kSmTslot);

    if (warp < 4) {
        // ------------------------------------------------------------------ loader
        // Loader threads leave together: a failed wait is published in
        // loader_stop between two named barriers and read by all after them.
        volatile int *loader_stop = reinterpret_cast<volatile int *>(gbase + kSmAbort + 4);
        if (tid == 0) *loader_stop = 0;
        tc::named_bar_sync(1, 128);
        int ci = 0, ui = 0;
        int kv_armed[2] = {-1, -1};
        bool stopped = false;
        for (int u = blockIdx.x; u < work && !stopped; u += gridDim.x, ++ui) {
            const Unit x = load_unit(p, u);
            const int kb = ui & 1;
            for (int c = 0; c < x.nch; ++c, ++ci) {
                const int qs = ci % kNQ;
                bool mine = true;
                if (c == 0 && ci >= 1) {
                    // Publish the previous chunk before any wait on the K/V
                    // buffer: that wait can depend (through the MMA issue
                    // order) on the previous chunk's S MMA.
                    cp_async_wait<0>();
                    tc::fence_proxy_async();
                    tc::mbar_arrive(bar(Q_FULL + (ci - 1) % kNQ));
                }
                if (c == 0) {
                    if (KV_FORMAT == MSA_KV_BF16) {
                        if (tid == 0) {
                            if (ui >= 2)
                                mine = tc::mbar_wait(bar(KV_EMPTY + kb), ((ui >> 1) - 1) & 1, abort_flag, p.status,
                                                     MSA_STATUS_TIMEOUT_BIT);
                            if (mine) {
                                tc::mbar_arrive_expect_tx(bar(KV_FULL + kb), 65536);
                                const int row = x.b * p.Skv + x.tok0;
                                const uint32_t ks = base + kSmK + kb * 32768, vs = base + kSmV + kb * 32768;
                                tc::tma_load_3d(ks, &tm_k, bar(KV_FULL + kb), 0, x.h, row);
                                tc::tma_load_3d(ks + 16384, &tm_k, bar(KV_FULL + kb), 64, x.h, row);
                                tc::tma_load_3d(vs, &tm_v, bar(KV_FULL + kb), 0, x.h, row);
                                tc::tma_load_3d(vs + 16384, &tm_v, bar(KV_FULL + kb), 64, x.h, row);
                                kv_armed[kb] = (ui >> 1) & 1;
                            }
                        }
                    } else if (ui >= 2) {
                        mine = tc::mbar_wait(bar(KV_EMPTY + kb), ((ui >> 1) - 1) & 1, abort_flag, p.status,
                                             MSA_STATUS_TIMEOUT_BIT);
                    }
                }
                if (mine && ci >= kNQ)
                    mine = tc::mbar_wait(bar(Q_EMPTY + qs), ((ci / kNQ) - 1) & 1, abort_flag, p.status,
                                         MSA_STATUS_TIMEOUT_BIT);
                tc::named_bar_sync(1, 128);
                if (!mine) {
                    *loader_stop = 1;
                } else {
                    const int qi = tid / p.qpk, idx = c * qc + qi;
                    rowq[tid] = idx < x.count ? (p.qsplit[(int64_t)x.h * p.cap + x.start + idx] & 0xFFFFFF) : -1;
                }
                tc::named_bar_sync(1, 128);
                if (*loader_stop) {
                    stopped = true;
                    break;
                }
                if (KV_FORMAT == MSA_KV_NVFP4 && c == 0) {
                    // 128 tokens x 8 groups of 16 values, for K and for V
                    for (int it = tid; it < 2 * 128 * 8; it += 128) {
                        const int isv = it >> 10, r = (it >> 3) & 127, g = it & 7;
                        const int t = x.tok0 + r;
                        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                        if (t < p.Skv) {
                            const int64_t rr = ((int64_t)x.b * p.Skv + t) * p.Hkv + x.h;
                            const uint8_t *pk = isv ? p.v_packed : p.k_packed;
                            const uint8_t *sc = isv ? p.v_scales : p.k_scales;
                            uint2 w = *reinterpret_cast<const uint2 *>(pk + rr * 64 + g * 8);
                            nvfp4_group_to_bf16(w, sc[rr * 8 + g], lo, hi);
                        }
                        const uint32_t tile = base + (isv ? kSmV : kSmK) + kb * 32768 + (g >> 2) * 16384;
                        const int cch = (g & 3) * 2;
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(tile + tc::sw128_off(r, cch)),
                                     "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w));
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                                         tile + tc::sw128_off(r, cch + 1)),
                                     "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w));
                    }
                    tc::fence_proxy_async();
                    tc::mbar_arrive(bar(KV_FULL + kb));
                }
                const uint32_t qt = base + kSmQ + qs * 32768;
#pragma unroll 4
                for (int k = 0; k < 16; ++k) {
                    const int i = tid + 128 * k, R = i >> 4, ch = i & 15;
                    const int gq = rowq[R];
                    const int hq = x.h * p.qpk + (R % p.qpk);
                    const __nv_bfloat16 *src = p.q + ((int64_t)(gq < 0 ? 0 : gq) * p.Hq + hq) * kD + ch * 8;
                    cp_async16(qt + (ch >> 3) * 16384 + tc::sw128_off(R, ch & 7), src, gq >= 0);
                }
                cp_async_commit();
                if (c >= 1) {
                    cp_async_wait<1>();
                    tc::fence_proxy_async();
                    tc::mbar_arrive(bar(Q_FULL + (ci - 1) % kNQ));
                }
            }
        }
        cp_async_wait<0>();
        if (!stopped && ci >= 1) {
            tc::fence_proxy_async();
            tc::mbar_arrive(bar(Q_FULL + (ci - 1) % kNQ));
        }
        // drain outstanding TMA loads before the CTA can exit
        if (KV_FORMAT == MSA_KV_BF16 && tid == 0)
            for (int i = 0; i < 2; ++i)
                if (kv_armed[i] >= 0) {
                    volatile int dummy = 0;
                    tc::mbar_wait(bar(KV_FULL + i), (uint32_t)kv_armed[i], &dummy, p.status, MSA_STATUS_TIMEOUT_BIT);
                }
    } else if (warp == 12) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int ci = 0, ui = 0;
            bool ok = true;
            int pv_ci = -1, pv_kb = 0, pv_last = 0;
            auto issue_pv = [&](int cj, int kbj, int last) -> bool {
                const int b = cj & 1;
                if (!tc::mbar_wait(bar(P_FULL + b), (cj >> 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT_BIT))
                    return false;
                if (cj >= 2 && !tc::mbar_wait(bar(O_EMPTY + b), ((cj >> 1) - 1) & 1, abort_flag, p.status,
                                              MSA_STATUS_TIMEOUT_BIT))
                    return false;
                tc::fence_after_sync();
                const uint32_t vs = base + kSmV + kbj * 32768;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_ts(tmem + 256 + b * 128, tmem + b * 128 + kk * 8,
                               tc::sdesc_sw128(vs + kk * 2048, 16384, 1024), kIdescPV, kk > 0);
                tc::mma_commit(bar(O_FULL + b));
                if (last) tc::mma_commit(bar(KV_EMPTY + kbj));
                return true;
            };
            for (int u = blockIdx.x; u < work && ok; u += gridDim.x, ++ui) {
                const Unit x = load_unit(p, u);
                const int kb = ui & 1;
                ok = tc::mbar_wait(bar(KV_FULL + kb), (ui >> 1) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT_BIT);
                const uint32_t ks = base + kSmK + kb * 32768;
                for (int c = 0; c < x.nch && ok; ++c, ++ci) {
                    const int b = ci & 1, qs = ci % kNQ;
                    ok = tc::mbar_wait(bar(Q_FULL + qs), (ci / kNQ) & 1, abort_flag, p.status,
                                       MSA_STATUS_TIMEOUT_BIT);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t qt = base + kSmQ + qs * 32768;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        tc::mma_ss(tmem + b * 128, tc::sdesc_sw128(qt + off, 16, 1024),
                                   tc::sdesc_sw128(ks + off, 16, 1024), kIdescS, kk > 0);
                    }
                    tc::mma_commit(bar(S_FULL + b));
                    tc::mma_commit(bar(Q_EMPTY + qs));
                    if (pv_ci >= 0) ok = issue_pv(pv_ci, pv_kb, pv_last);
                    pv_ci = ci;
                    pv_kb = kb;
                    pv_last = (c == x.nch - 1);
                }
            }
            if (ok && pv_ci >= 0) issue_pv(pv_ci, pv_kb, pv_last);
            // all issued MMAs complete before tensor memory is released
            tc::mma_commit(bar(DRAIN));
            volatile int dummy = 0;
            tc::mbar_wait(bar(DRAIN), 0, &dummy, p.status, MSA_STATUS_TIMEOUT_BIT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax + epilogue
        const int wg = (warp - 4) >> 2;           // 0: even chunks, 1: odd chunks
        const int lt = tid - 128 - 128 * wg;      // row of the 128-row chunk = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t s_addr = tmem + lane_base + wg * 128;
        const uint32_t o_addr = tmem + lane_base + 256 + wg * 128;
        int ci = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < work && ok; u += gridDim.x) {
            const Unit x = load_unit(p, u);
            for (int c = 0; c < x.nch && ok; ++c, ++ci) {
                if ((ci & 1) != wg) continue;
                const uint32_t par = (ci >> 1) & 1;
                const int qi = lt / p.qpk, idx = c * qc + qi;
                const bool valid = idx < x.count;
                int gq = 0, split = 0, nvis = 0;
                if (valid) {
                    const int packed = p.qsplit[(int64_t)x.h * p.cap + x.start + idx];
                    gq = packed & 0xFFFFFF;
                    split = (packed >> 24) & 0xFF;
                    const int sq = gq % p.Sq;
                    int64_t limit = (int64_t)p.Skv - 1;
                    if (p.causal) limit = min(limit, (int64_t)sq + (int64_t)(p.Skv - p.Sq));
                    const int64_t nv = limit - x.tok0 + 1;
                    nvis = (int)(nv < 0 ? 0 : (nv > 128 ? 128 : nv));
                }
                ok = tc::mbar_wait(bar(S_FULL + wg), par, abort_flag, p.status, MSA_STATUS_TIMEOUT_BIT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::fence_after_sync();
                // pass 1: row max over visible keys
                float m = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[32];
                    tc::tmem_ld32(s_addr + cc * 32, r);
                    tc::tmem_ld_wait();
                    if (nvis >= cc * 32 + 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) m = fmaxf(m, __uint_as_float(r[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (cc * 32 + j < nvis) m = fmaxf(m, __uint_as_float(r[j]));
                    }
                }
                // pass 2: P = exp(S - m) (bf16, written over S), row sum
                const float mc = (m == -INFINITY) ? 0.f : m * p.scale_log2;
                float l = 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[32], w[16];
                    tc::tmem_ld32(s_addr + cc * 32, r);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int k0 = cc * 32 + 2 * j;
                        float x0 = (k0 < nvis) ? ex2_approx(fmaf(__uint_as_float(r[2 * j]), p.scale_log2, -mc)) : 0.f;
                        float x1 =
                            (k0 + 1 < nvis) ? ex2_approx(fmaf(__uint_as_float(r[2 * j + 1]), p.scale_log2, -mc)) : 0.f;
                        l += x0 + x1;
                        w[j] = pack_bf16x2(x0, x1);
                    }
                    tc::tmem_st16(s_addr + cc * 16, w);
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();
                tc::mbar_arrive(bar(P_FULL + wg));
                // epilogue: O / l -> bf16 partial, lse
                ok = tc::mbar_wait(bar(O_FULL + wg), par, abort_flag, p.status, MSA_STATUS_TIMEOUT_BIT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::fence_after_sync();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int hq = x.h * p.qpk + (lt % p.qpk);
                const int64_t slot = ((int64_t)gq * p.topk + split) * p.Hq + hq;
                uint4 *dst = reinterpret_cast<uint4 *>(p.o_part + slot * kD);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[32];
                    tc::tmem_ld32(o_addr + cc * 32, r);
                    tc::tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 o4;
                            o4.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
                            o4.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
                            o4.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
                            o4.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
                            dst[cc * 4 + v4] = o4;
                        }
                    }
                }
                tc::fence_before_sync();
                tc::mbar_arrive(bar(O_EMPTY + wg));
                if (valid) p.lse_part[slot] = (l > 0.f) ? (m * p.scale + logf(l)) : -INFINITY;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 12) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace msa
