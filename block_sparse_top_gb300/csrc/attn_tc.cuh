// attn_tc.cuh -- the tcgen05 (5th-gen tensor core) block-sparse attention tile
// kernel of the prefill forward: persistent, one CTA per SM,
// warp-specialised, 16 warps.
//
//   warp 11     feed: walks the CTA's chunks in plan order and copies each
//               chunk's plan unit, page and query ids into a 4-entry shared
//               memory ring with cp.async (the copies arrive on the slot's
//               barrier as they land), so no global load sits on the
//               loader's issue path.
//   warp 0      loader: per work unit the K and V block by TMA (bf16, 128-byte
//               swizzle, one 4D copy each, one issuing lane); per chunk the
//               128 gathered Q rows (128/qhead_per_kv queries x all heads of
//               the GQA group) by TMA into the Q ring: one 5D box per query
//               (its whole group) when qhead_per_kv >= 8, four rows per
//               tile::gather4 copy otherwise.  Requests are kept few and
//               large, and each lane issues one of them, so that one
//               instruction issues a chunk's copies.
//   warp 1      NVFP4 only: dequantises the K and V block into the same
//               swizzled bf16 layout (exact products).
//   warp 2      MMA issuer (one lane): S_i = Q_i K^T into tensor memory, then
//               O_{i-1} = P_{i-1} V with P read from tensor memory.
//   warps 3-6,  softmax for even / odd chunks: each thread owns one S row
//   warps 7-10  (TMEM lane), reads it in quarters of 32 columns, applies the
//               bottom-right causal limit, writes P = exp(S - m) as bf16 over
//               S and stores the split's statistics (m * scale, l = sum P);
//               the split partial is kept unnormalised so that the combine
//               applies each split's weight and 1/l in one product.  Packed
//               f32x2 FMA/add and three-input max halve the per-element
//               instruction count of the row pass.
//   warps 12-15 epilogue: once PV has run, each chunk's O = P V (TMEM lanes
//               of the warp) -> split partial, so the softmax warps never
//               wait for PV.
//
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
// Every wait is bounded; on a timeout the CTA raises MSA_STATUS_TIMEOUT,
// drains its copies and MMAs, frees tensor memory and exits.
#pragma once
#include "attn_mma.cuh"
#include "combine.cuh"
#include "tc.cuh"

namespace msa {

struct TcParams {
    const uint8_t *k_packed, *v_packed;   // NVFP4 only
    const uint8_t *k_scales, *v_scales;   // NVFP4 only
    const int32_t *qsplit;
    const PlanHeader *plan;
    const PlanUnit *units;
    void *o_part;                         // split partials (part_dtype), layout in combine.cuh
    float2 *stat_part;                    // split statistics, layout in combine.cuh
    float2 *stat_temp;                    // temperature statistics (OPTS instances, temp_on), same layout
    int part_dtype;                       // MSA_PARTIAL_*: storage of the split partials (OPTS instances)
    int temp_on;                          // 1: keep the temperature statistics (OPTS instances)
    float inv_temp;                       // 1 / lse_temperature_scale
    // ragged batches: cu_seqlens of the queries and keys [B+1]; null for a
    // uniform batch (sequence b holds queries b*Sq.. and keys b*Skv..)
    const int32_t *cu_q, *cu_k;
    uint32_t *status;
    int B, Sq, Skv, Hq, Hkv, qpk, topk, nblk, causal;
    int64_t cap;
    int64_t kv_rows;  // token rows of the K/V arrays (bound of the dequant loads)
    int64_t total_q;  // query rows of Q (all sequences)
    float scale, scale_log2;
};

namespace tck {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpLoad = 0, kWarpDequant = 1, kWarpMma = 2, kWarpSoftmax0 = 3, kWarpFeed = 11, kWarpEpi0 = 12;
// Chunk ring between the feed warp and the loader: per chunk its plan unit
// (16 B), its sequence's first key row (ragged batches, at byte 20), and up
// to 128 query ids (qsplit entries, from byte 32).
constexpr int kRing = 4;
constexpr uint32_t kRingEntry = 32 + 128 * 4;

// Shared memory of a kernel with NKV K/V stages and NQ Q stages of KS / QS
// bytes (bf16 K and Q tiles 32 KB, e4m3 ones 16 KB; V tiles are bf16, 32 KB):
// K [NKV] | V [NKV] | Q [NQ] | mbarriers | TMEM slot | abort flag | chunk ring.
template <int NKV, int NQ, uint32_t KS = 32768u, uint32_t QS = 32768u>
struct Layout {
    static constexpr uint32_t K = 0, V = NKV * KS, Q = V + NKV * 32768u, BAR = Q + NQ * QS;
    enum : int {
        KV_FULL = 0,
        KV_EMPTY = NKV,
        Q_FULL = 2 * NKV,
        Q_EMPTY = 2 * NKV + NQ,
        S_FULL = 2 * NKV + 2 * NQ,
        P_FULL = S_FULL + 2,
        O_FULL = P_FULL + 2,
        O_EMPTY = O_FULL + 2,
        RING_FULL = O_EMPTY + 2,
        RING_EMPTY = RING_FULL + kRing,
        DRAIN = RING_EMPTY + kRing,
        NBAR = DRAIN + 1
    };
    static constexpr uint32_t TSLOT = BAR + 8 * NBAR, ABORT = TSLOT + 4, RING = (ABORT + 4 + 15) & ~15u,
                              BYTES = RING + kRing * kRingEntry;
    // The dynamic shared memory base is 1024-byte aligned (no static shared
    // memory); the kernel checks this instead of reserving slack.
    static_assert(BYTES <= 232448, "shared memory budget");
};

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescS8 = tc::idesc_e4m3_f32(128, 128);

// K/V format of the instance that keeps Q and K in e4m3 (S = Q K^T as an fp8
// MMA) and stages V to bf16 (not a value of the public kv_format argument)
constexpr int kKvQk8 = 3;
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, 0, 1);

struct Unit {
    int h, b, tok0, start, count, nch;
};

__device__ __forceinline__ Unit load_unit(const TcParams &p, int u) {
    PlanUnit pu = p.units[u];
    Unit x;
    x.h = pu.head;
    x.b = pu.seq;
    x.tok0 = pu.blk * kBlk;
    x.start = pu.start;
    x.count = pu.count;
    const int qc_sh = 7 - (31 - __clz(p.qpk));  // log2(128 / qhead_per_kv): qhead_per_kv is a power of two
    x.nch = (pu.count + (1 << qc_sh) - 1) >> qc_sh;
    return x;
}

}  // namespace tck

// NKV, NQ: K/V and Q stages (32 KB tiles; 2 and 3 fill the shared memory).
// OPTS: the instance that serves the forward's options at run
// time -- the partials' storage type (bf16, fp16 or fp32) and, with temp_on,
// the row sum of 2^(x / T), x = (S - m) scale_log2, with its statistics (m
// scale / T, that sum) for the temperature LSE.  Without OPTS the epilogue
// stores bf16 and nothing else: the run-time type switch alone cost the
// 32K causal workload's tiles a tenth of their time.
template <int KV_FORMAT, int NKV, int NQ, bool OPTS>
__global__ void __launch_bounds__(tck::kThreads, 1)
    sparse_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qh,
                         TcParams p) {
    using namespace tck;
    constexpr bool QK8 = KV_FORMAT == kKvQk8;
    constexpr uint32_t KS = QK8 ? 16384u : 32768u, QS = QK8 ? 16384u : 32768u;  // K and Q stage bytes
    using L = Layout<NKV, NQ, KS, QS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *const gbase = smem_raw;
    if (base & 1023u) {  // 128-byte swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_status(p.status, MSA_STATUS_LAUNCH);
        return;
    }
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + L::ABORT);
    auto bar = [&](int i) -> uint32_t { return base + L::BAR + 8u * (uint32_t)i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // qhead_per_kv is a power of two: row R of a chunk is query R >> qpk_sh,
    // head R & (qhead_per_kv - 1)
    const int qpk_sh = 31 - __clz(p.qpk), qc_sh = 7 - qpk_sh;
    const int qc = 128 >> qpk_sh;

    if (tid == 0) {
        for (int i = 0; i < NKV; ++i) {
            // arrivals: the loader's copy (bf16 K and V; e4m3 K), the
            // dequantising warp's 32 lanes (NVFP4 / FP8 K and V; e4m3 V)
            tc::mbar_init(bar(L::KV_FULL + i), KV_FORMAT == MSA_KV_BF16 ? 1 : (QK8 ? 33 : 32));
            tc::mbar_init(bar(L::KV_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(L::S_FULL + i), 1);
            tc::mbar_init(bar(L::P_FULL + i), 128);
            tc::mbar_init(bar(L::O_FULL + i), 1);
            tc::mbar_init(bar(L::O_EMPTY + i), 128);
        }
        for (int i = 0; i < NQ; ++i) {
            tc::mbar_init(bar(L::Q_FULL + i), 1);
            tc::mbar_init(bar(L::Q_EMPTY + i), 1);
        }
        for (int i = 0; i < kRing; ++i) {
            tc::mbar_init(bar(L::RING_FULL + i), 32);  // one cp.async arrival per feed lane
            tc::mbar_init(bar(L::RING_EMPTY + i), 1);
        }
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
        if (QK8) tc::tma_prefetch_desc(&tm_k);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbase + L::TSLOT);
    // the plan comes from the previous kernel
    grid_dependency_wait();
    grid_dependents_launch();
    const int work = p.plan->work_count;
    // The CTA's units: every gridDim.x-th of the plan (consecutive units read
    // the same K/V head close together in time).  Every role walks the same
    // sequence.
    const int u_begin = (int)blockIdx.x, u_end = work, u_step = (int)gridDim.x;

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------------ loader
        // Walks the CTA's chunks in plan order, taking each chunk's unit and
        // query ids from the feed warp's ring (shared memory), so no global
        // load sits on its issue path; issues the unit's K/V on its first
        // chunk and the chunk's Q rows.
        int ci = 0, ui = 0, c = 0;
        int qn = 0;  // Q tiles loaded
        int kv_armed[NKV], q_armed[NQ];  // phase parity of each stage's last copy, -1: none
        for (int i = 0; i < NKV; ++i) kv_armed[i] = -1;
        for (int i = 0; i < NQ; ++i) q_armed[i] = -1;
        bool ok = true;
        const uint64_t keep = tc::l2_policy_evict_last();  // gather4 Q rows
        for (int u = u_begin; u < u_end && ok;) {
            const int slot = ci % kRing;
            ok = tc::mbar_wait(bar(L::RING_FULL + slot), (ci / kRing) & 1, abort_flag, p.status, MSA_STATUS_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int *e = reinterpret_cast<const int *>(gbase + L::RING + slot * kRingEntry);
            Unit x;
            x.h = e[0] & 0xFFFF;
            x.tok0 = (e[0] >> 16) * kBlk;
            x.b = e[1];
            x.start = e[2];
            x.count = e[3];
            x.nch = (x.count + qc - 1) >> qc_sh;
            const int seq_k0 = e[5];  // ragged: first key row of the sequence
            int ids[4];
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int qi = s4 * 32 + lane;
                ids[s4] = (qi < qc && c * qc + qi < x.count) ? (e[8 + qi] & 0xFFFFFF) : -1;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(L::RING_EMPTY + slot));
            const int kb = ui % NKV;
            if (c == 0 && (KV_FORMAT == MSA_KV_BF16 || QK8)) {
                if (lane == 0 && ui >= NKV)
                    ok = tc::mbar_wait(bar(L::KV_EMPTY + kb), ((ui / NKV) - 1) & 1, abort_flag, p.status,
                                       MSA_STATUS_TIMEOUT);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                // token row: the sequence's keys of a ragged batch, or dense [B][Skv]
                const int row = (p.cu_k ? seq_k0 : x.b * p.Skv) + x.tok0;
#ifdef MSA_TEST_DROP_KV_ARRIVAL
                // test build only: CTA 0 never signals its first unit's K/V, so
                // the MMA warp's bounded wait runs out and the CTA aborts
                const bool drop = blockIdx.x == 0 && ui == 0;
#else
                constexpr bool drop = false;
#endif
                if (lane == 0 && !drop) {
                    tc::mbar_arrive_expect_tx(bar(L::KV_FULL + kb), QK8 ? 16384u : 65536u);
                    kv_armed[kb] = (ui / NKV) & 1;
                }
                __syncwarp();
                if constexpr (QK8) {
                    // e4m3 K by TMA (V is staged to bf16 by the dequantising warp)
                    if (lane == 0 && !drop)
                        tc::tma_load_3d(base + L::K + kb * KS, &tm_k, bar(L::KV_FULL + kb), 0, row, x.h);
                } else {
                    // lane 0 copies K, lane 1 V, in one instruction
                    if (lane < 2 && !drop)
                        tc::tma_load_4d(base + (lane ? L::V : L::K) + kb * 32768, lane ? &tm_v : &tm_k,
                                        bar(L::KV_FULL + kb), 0, row, 0, x.h);
                }
            }
            const int first = __shfl_sync(0xffffffffu, ids[0], 0);  // always valid (count > c*qc)
            const int qs = qn % NQ;
            if (lane == 0 && qn >= NQ)
                ok = tc::mbar_wait(bar(L::Q_EMPTY + qs), ((qn / NQ) - 1) & 1, abort_flag, p.status,
                                   MSA_STATUS_TIMEOUT);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            q_armed[qs] = (qn / NQ) & 1;
            ++qn;
            // The chunk's 128 Q rows (row R = query R / qpk of the chunk, head
            // R % qpk of the group), 128-byte swizzled K-major.  qpk >= 8: one
            // 5D box per query holds its whole group (row octets 2048 bytes
            // apart, column halves 1024 apart); qpk < 8: four arbitrary rows
            // per tile::gather4 copy (rows 128 bytes apart, halves 16384).
            // qpk >= 8 loads only the chunk's real queries (padding rows keep
            // stale data; their keys are all masked, so they give P = 0);
            // gather4 rows of padding repeat the chunk's first query.
            const uint32_t qt = base + L::Q + qs * QS;
            const int nq = min(qc, x.count - c * qc);
            if (lane == 0)
                tc::mbar_arrive_expect_tx(bar(L::Q_FULL + qs),
                                          p.qpk >= 8 ? (uint32_t)(nq * p.qpk * (QK8 ? 128 : 256)) : QS);
            if (QK8) {
                // e4m3 rows of 128 bytes: one 4D box per query (qpk >= 8: its
                // row octets 1024 bytes apart), or four rows per gather4
                if (p.qpk >= 8) {
                    if (lane < nq)
                        tc::tma_load_4d(qt + (uint32_t)(lane * p.qpk * 128), &tm_q, bar(L::Q_FULL + qs), 0, 0, 0,
                                        ids[0] * p.Hkv + x.h);
                } else {
                    int r[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int R = 4 * lane + t, qi = R >> qpk_sh;
                        const int g0 = __shfl_sync(0xffffffffu, ids[0], qi & 31);
                        const int g1 = __shfl_sync(0xffffffffu, ids[1], qi & 31);
                        const int g2 = __shfl_sync(0xffffffffu, ids[2], qi & 31);
                        const int g3 = __shfl_sync(0xffffffffu, ids[3], qi & 31);
                        const int sl = qi >> 5;
                        int gq = sl == 0 ? g0 : sl == 1 ? g1 : sl == 2 ? g2 : g3;
                        if (gq < 0) gq = first;
                        r[t] = gq * p.Hq + x.h * p.qpk + (R & (p.qpk - 1));
                    }
                    tc::tma_gather4_hint(qt + lane * 512, &tm_q, bar(L::Q_FULL + qs), 0, r[0], r[1], r[2], r[3], keep);
                }
            } else if (p.qpk >= 8) {
                // lane l issues query slot l's box: one instruction issues them all
                if (lane < nq)
                    tc::tma_load_5d(qt + (uint32_t)(lane * p.qpk * 256), &tm_q, bar(L::Q_FULL + qs), 0, 0, 0, 0,
                                    ids[0] * p.Hkv + x.h);
            } else if (__all_sync(0xffffffffu, (lane >= nq || ids[0] == first + lane) &&
                                                   (32 + lane >= nq || ids[1] == first + 32 + lane) &&
                                                   (64 + lane >= nq || ids[2] == first + 64 + lane) &&
                                                   (96 + lane >= nq || ids[3] == first + 96 + lane)) &&
                       nq == qc) {
                // consecutive query positions (a sink or diagonal block's
                // queries): the chunk's rows are one box of (positions x heads
                // x 64 columns) per column half, rows in the gather's order
                if (lane < 2)
                    tc::tma_load_3d(qt + lane * 16384u, &tm_qh, bar(L::Q_FULL + qs), lane * 64, x.h * p.qpk, first);
            } else {
                // lane j issues the gather4 pair of rows 4j .. 4j+3
                int r[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int R = 4 * lane + t, qi = R >> qpk_sh;
                    const int g0 = __shfl_sync(0xffffffffu, ids[0], qi & 31);
                    const int g1 = __shfl_sync(0xffffffffu, ids[1], qi & 31);
                    const int g2 = __shfl_sync(0xffffffffu, ids[2], qi & 31);
                    const int g3 = __shfl_sync(0xffffffffu, ids[3], qi & 31);
                    const int sl = qi >> 5;
                    int gq = sl == 0 ? g0 : sl == 1 ? g1 : sl == 2 ? g2 : g3;
                    if (gq < 0) gq = first;
                    r[t] = gq * p.Hq + x.h * p.qpk + (R & (p.qpk - 1));
                }
                tc::tma_gather4_hint(qt + lane * 512, &tm_q, bar(L::Q_FULL + qs), 0, r[0], r[1], r[2], r[3], keep);
                tc::tma_gather4_hint(qt + 16384 + lane * 512, &tm_q, bar(L::Q_FULL + qs), 64, r[0], r[1], r[2], r[3],
                                     keep);
            }
            ++ci;
            if (++c == x.nch) {
                c = 0;
                ++ui;
                u += u_step;
            }
        }
        // drain outstanding copies (K/V and Q) before the CTA can exit: after
        // an abort, copies may still be landing in shared memory
        if (lane == 0) {
            volatile int dummy = 0;
            for (int i = 0; i < NKV; ++i)
                if (kv_armed[i] >= 0) tc::mbar_wait(bar(L::KV_FULL + i), (uint32_t)kv_armed[i], &dummy, p.status, 0);
            for (int i = 0; i < NQ; ++i)
                if (q_armed[i] >= 0) tc::mbar_wait(bar(L::Q_FULL + i), (uint32_t)q_armed[i], &dummy, p.status, 0);
        }
        __syncwarp();
    } else if (warp == kWarpFeed) {
        // ------------------------------------------------------------------ feed
        // Walks the same chunk sequence and copies each chunk's plan unit, page
        // and query ids into the ring with cp.async; every lane's copies arrive
        // on the slot's barrier as they land, so this warp never waits on a
        // global load and runs up to kRing chunks ahead of the loader.
        int k = 0;
        bool ok = true;
        for (int u = u_begin + lane * u_step; u < u_end; u += 32 * u_step) {
            tc::prefetch_l2(p.units + u);
        }
        Unit xn{};
        if (u_begin < u_end) xn = load_unit(p, u_begin);
        for (int u = u_begin; u < u_end && ok; u += u_step) {
            const Unit x = xn;  // loaded one unit ahead
            if (u + u_step < u_end) xn = load_unit(p, u + u_step);
            for (int c = 0; c < x.nch; ++c, ++k) {
                const int slot = k % kRing;
                if (lane == 0 && k >= kRing)
                    ok = tc::mbar_wait(bar(L::RING_EMPTY + slot), ((k / kRing) - 1) & 1, abort_flag, p.status,
                                       MSA_STATUS_TIMEOUT);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t e = base + L::RING + slot * kRingEntry;
                if (lane == 0) {
                    cp_async16(e, p.units + u);
                    if (p.cu_k) cp_async4(e + 20, p.cu_k + x.b);
                }
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int qi = s4 * 32 + lane, idx = c * qc + qi;
                    if (qi < qc && idx < x.count) cp_async4(e + 32 + qi * 4, p.qsplit + (int64_t)x.h * p.cap + x.start + idx);
                }
                tc::cp_async_mbar_arrive(bar(L::RING_FULL + slot));
            }
        }
        cp_async_wait<0>();
        __syncwarp();
    } else if (warp == kWarpDequant) {
        // ------------------------------------------------------------------ NVFP4 / FP8 K/V producer
        if (KV_FORMAT != MSA_KV_BF16) {  // NVFP4 / FP8: K and V; QK8: V
            int ui = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; u += u_step, ++ui) {
                const Unit x = load_unit(p, u);
                const int kb = ui % NKV;
                if (ui >= NKV)
                    ok = tc::mbar_wait(bar(L::KV_EMPTY + kb), ((ui / NKV) - 1) & 1, abort_flag, p.status,
                                       MSA_STATUS_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if constexpr (KV_FORMAT == MSA_KV_FP8 || QK8) {
                // 128 tokens of e4m3 K (not QK8: that K is copied by TMA) and V
                const int64_t k0row = (p.cu_k ? (int64_t)__ldg(p.cu_k + x.b) : (int64_t)x.b * p.Skv) + x.tok0;
                const int64_t klen =
                    (p.cu_k ? (int64_t)__ldg(p.cu_k + x.b + 1) - __ldg(p.cu_k + x.b) : (int64_t)p.Skv) - x.tok0;
                const int nrows = (int)max((int64_t)0, min(min(klen, (int64_t)kBlk), p.kv_rows - k0row));
                const int64_t first = nrows > 0 ? (k0row * p.Hkv + x.h) * 128 : 0;
                if constexpr (!QK8)
                    e4m3_rows_to_tile(base + L::K + kb * KS, p.k_packed + first, (int64_t)p.Hkv * 128, nrows, lane);
                e4m3_rows_to_tile(base + L::V + kb * 32768, p.v_packed + first, (int64_t)p.Hkv * 128, nrows, lane);
                } else {
                // 128 tokens x 4 pieces of 32 values (16 packed bytes, two
                // scales), for K and then for V.  Lane l converts piece l % 4
                // of tokens l / 4 + 8 i: lanes 4i..4i+3 read one token's 64
                // bytes.  Eight 16-byte loads are in flight before any is used.
                const int pc = lane & 3, r0 = lane >> 2;
                // the sequence's first key row and key count
                const int64_t k0row = p.cu_k ? (int64_t)__ldg(p.cu_k + x.b) : (int64_t)x.b * p.Skv;
                const int64_t klen = p.cu_k ? (int64_t)__ldg(p.cu_k + x.b + 1) - k0row : (int64_t)p.Skv;
#pragma unroll 1
                for (int k0 = 0; k0 < 32; k0 += 8) {
                    const int isv = k0 >> 4, rb = r0 + 8 * (k0 & 15);
                    const uint8_t *pbase = isv ? p.v_packed : p.k_packed;
                    const uint8_t *sbase = isv ? p.v_scales : p.k_scales;
                    const int64_t row0 = (k0row + x.tok0 + rb) * p.Hkv + x.h;
                    uint4 pk[8];
                    uint32_t sc2[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t rr = row0 + (int64_t)(8 * i) * p.Hkv;
                        const int64_t t = x.tok0 + rb + 8 * i;
                        const bool in = t < klen && k0row + t < p.kv_rows;
                        pk[i] = in ? __ldg(reinterpret_cast<const uint4 *>(pbase + rr * 64) + pc) : make_uint4(0, 0, 0, 0);
                        sc2[i] = in ? __ldg(reinterpret_cast<const uint16_t *>(sbase + rr * 8) + pc) : 0u;
                    }
                    // values 32 pc .. 32 pc + 31: column half pc / 2, chunks 4 (pc % 2) ..
                    const uint32_t tile = base + (isv ? L::V : L::K) + kb * 32768 + (pc >> 1) * 16384;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4 o4[4];
                        nvfp4_piece_to_bf16(pk[i], sc2[i], o4);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                                             tile + tc::sw128_off(rb + 8 * i, (pc & 1) * 4 + c)),
                                         "r"(o4[c].x), "r"(o4[c].y), "r"(o4[c].z), "r"(o4[c].w));
                    }
                }
                }
                tc::fence_proxy_async();
                tc::mbar_arrive(bar(L::KV_FULL + kb));
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        // Per chunk ci two MMA groups are due: S_ci = Q_ci K^T (needs Q_ci, and the
        // unit's K/V on its first chunk) and O_{ci-1} = P_{ci-1} V (needs P_{ci-1}
        // and a free O buffer).  Neither depends on the other, so the issuer polls
        // all their barriers and issues whichever becomes ready first.
        if (lane == 0) {
            int ci = 0, ui = 0;
            bool ok = true;
            int pv_ci = -1, pv_kb = 0, pv_last = 0;
            // Q tile geometry (see the loader): octet stride and half offset
            const uint32_t q_sbo = (p.qpk >= 8 && !QK8) ? 2048u : 1024u, q_half = p.qpk >= 8 ? 1024u : 16384u;
            auto pv_ready = [&](int cj) -> bool {
                const int b = cj & 1;
                return tc::mbar_test(bar(L::P_FULL + b), (cj >> 1) & 1) &&
                       (cj < 2 || tc::mbar_test(bar(L::O_EMPTY + b), ((cj >> 1) - 1) & 1));
            };
            auto issue_pv = [&](int cj, int kbj, int last) {
                const int b = cj & 1;
                tc::fence_after_sync();
                // step kk: P columns 8 kk.., V rows 16 kk.. (2048 bytes, 128
                // descriptor units, further on)
                const uint64_t vd = tc::sdesc_sw128(base + L::V + kbj * 32768, 16384, 1024);
                uint32_t pa[8];
                uint64_t vb[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    pa[kk] = tmem + b * 128 + kk * 8;
                    vb[kk] = vd + (uint64_t)(kk * 128);
                }
                tc::mma_ts8(tmem + 256 + b * 128, pa, vb, kIdescPV);
                tc::mma_commit(bar(L::O_FULL + b));
                if (last) tc::mma_commit(bar(L::KV_EMPTY + kbj));
            };
            // S_cj reads the Q tile in stage qs and frees the stage when
            // release_q (the tile's last chunk)
            auto issue_s = [&](int cj, int kbj, int qs, bool release_q) {
                const int b = cj & 1;
                tc::fence_after_sync();
                const uint32_t qt = base + L::Q + qs * QS, ks = base + L::K + kbj * KS;
                if constexpr (QK8) {
                    // e4m3: a 128-byte row holds all 128 dims, 32 per MMA
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ss_f8(tmem + b * 128, tc::sdesc_sw128(qt + kk * 32, 16, 1024),
                                      tc::sdesc_sw128(ks + kk * 32, 16, 1024), kIdescS8, kk > 0);
                } else {
                    // step kk: 32 bytes (2 descriptor units) into the row, the
                    // second 64-column half from kk = 4 (the stage bases are
                    // 1024-byte aligned, so base + offset never carries out of
                    // the address field)
                    const uint64_t qd = tc::sdesc_sw128(qt, 16, q_sbo), kd = tc::sdesc_sw128(ks, 16, 1024);
                    const uint64_t qd_h = qd + (q_half >> 4), kd_h = kd + (16384u >> 4);
                    uint64_t qa[8], kb8[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        qa[kk] = (kk < 4 ? qd : qd_h) + (uint64_t)((kk & 3) * 2);
                        kb8[kk] = (kk < 4 ? kd : kd_h) + (uint64_t)((kk & 3) * 2);
                    }
                    tc::mma_ss8(tmem + b * 128, qa, kb8, kIdescS);
                }
                tc::mma_commit(bar(L::S_FULL + b));
                if (release_q) tc::mma_commit(bar(L::Q_EMPTY + qs));
            };
            // polls until S_ci (if s_cj >= 0) and the pending PV are both issued
            auto drive = [&](int s_cj, int kbj, bool need_kv, int kv_par, int qs, uint32_t q_par, bool release_q) -> bool {
                bool s_done = s_cj < 0, pv_done = pv_ci < 0, kv_ok = !need_kv;
                const uint64_t t0 = tc::global_ns();
                for (uint32_t i = 0;; ++i) {
                    // back off between polls: a spinning lane would take issue
                    // slots from the softmax warps sharing its sub-partition
                    if (i > 0) __nanosleep(32);
                    if (!s_done) {
                        if (!kv_ok) kv_ok = tc::mbar_test(bar(L::KV_FULL + kbj), (uint32_t)kv_par);
                        if (kv_ok && tc::mbar_test(bar(L::Q_FULL + qs), q_par)) {
                            issue_s(s_cj, kbj, qs, release_q);
                            s_done = true;
                        }
                    }
                    if (!pv_done && pv_ready(pv_ci)) {
                        issue_pv(pv_ci, pv_kb, pv_last);
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
            // Q tiles as the loader issues them: one per chunk
            int q_stage = 0;  // stage and phase parity of the next Q tile
            uint32_t q_par = 0;
            Unit xnext{};
            if (u_begin < u_end) xnext = load_unit(p, u_begin);
            for (int u = u_begin; u < u_end && ok; u += u_step, ++ui) {
                const Unit x = xnext;
                if (u + u_step < u_end) xnext = load_unit(p, u + u_step);
                const int kb = ui % NKV;
                for (int c = 0; c < x.nch && ok; ++c, ++ci) {
                    ok = drive(ci, kb, c == 0, (ui / NKV) & 1, q_stage, q_par, true);
                    if (++q_stage == NQ) {
                        q_stage = 0;
                        q_par ^= 1u;
                    }
                    pv_ci = ci;
                    pv_kb = kb;
                    pv_last = (c == x.nch - 1);
                }
            }
            if (ok && pv_ci >= 0) drive(-1, 0, false, 0, 0, 0u, false);
            // all issued MMAs complete before tensor memory is released
            tc::mma_commit(bar(L::DRAIN));
            volatile int dummy = 0;
            tc::mbar_wait(bar(L::DRAIN), 0, &dummy, p.status, MSA_STATUS_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= kWarpEpi0) {
        // ------------------------------------------------------------------ epilogue
        // Chunk ci's O (TMEM lanes of this warp, buffer ci % 2) -> bf16 split
        // partial, once PV has run; frees the O buffer for the chunk two later.
        // The softmax warps store the statistics, so they never wait for PV.
        const int R = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int j_of_row = R & (p.qpk - 1), qi = R >> qpk_sh;
        int ci = 0;
        bool ok = true;
        Unit xnext{};
        if (u_begin < u_end) xnext = load_unit(p, u_begin);
        for (int u = u_begin; u < u_end && ok; u += u_step) {
            const Unit x = xnext;
            if (u + u_step < u_end) xnext = load_unit(p, u + u_step);
            for (int c = 0; c < x.nch && ok; ++c, ++ci) {
                const int b = ci & 1;
                const uint32_t par = (ci >> 1) & 1;
                const uint32_t o_addr = tmem + lane_base + 256 + b * 128;
                const int idx = c * qc + qi;
                const bool valid = idx < x.count;
                const int packed = valid ? p.qsplit[(int64_t)x.h * p.cap + x.start + idx] : 0;
                ok = tc::mbar_wait(bar(L::O_FULL + b), par, abort_flag, p.status, MSA_STATUS_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::fence_after_sync();
                if (__all_sync(0xffffffffu, !valid)) {  // padding rows only: nothing to store
                    tc::fence_before_sync();
                    tc::mbar_arrive(bar(L::O_EMPTY + b));
                    continue;
                }
                // grouped layout: for a fixed (split, c) the heads of one group are
                // contiguous, so each store instruction writes whole runs
                const int gq = packed & 0xFFFFFF, split = (packed >> 24) & 0xFF;
                const int64_t grp = (int64_t)gq * p.Hkv + x.h;
                // piece (8 values) of chunk c at byte (index + c * qpk) * piece bytes
                const int pb = part_piece_bytes(p.part_dtype);
                char *dst = static_cast<char *>(p.o_part) + part_o_index(grp, p.topk, p.qpk, split, 0, j_of_row) * pb;
                const int64_t cstride = (int64_t)p.qpk * pb;
                uint32_t r[32];
#pragma unroll 1
                for (int qq = 0; qq < 4; ++qq) {  // quarters of 32 columns: 4 pieces each
                    tc::tmem_ld32(o_addr + 32 * qq, r);
                    tc::tmem_ld_wait();
                    if (qq == 3) {
                        tc::fence_before_sync();
                        tc::mbar_arrive(bar(L::O_EMPTY + b));  // O is read: the next PV may start
                    }
                    if (!valid) continue;
                    // streaming stores: evict first from L2
                    if (OPTS && p.part_dtype == MSA_PARTIAL_FP32) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            float4 *d = reinterpret_cast<float4 *>(dst + (4 * qq + v4) * cstride);
                            __stcs(d, make_float4(__uint_as_float(r[8 * v4 + 0]), __uint_as_float(r[8 * v4 + 1]),
                                                  __uint_as_float(r[8 * v4 + 2]), __uint_as_float(r[8 * v4 + 3])));
                            __stcs(d + 1, make_float4(__uint_as_float(r[8 * v4 + 4]), __uint_as_float(r[8 * v4 + 5]),
                                                      __uint_as_float(r[8 * v4 + 6]), __uint_as_float(r[8 * v4 + 7])));
                        }
                    } else if (OPTS && p.part_dtype == MSA_PARTIAL_FP16) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 o4;
                            o4.x = pack_f16x2(__uint_as_float(r[8 * v4 + 0]), __uint_as_float(r[8 * v4 + 1]));
                            o4.y = pack_f16x2(__uint_as_float(r[8 * v4 + 2]), __uint_as_float(r[8 * v4 + 3]));
                            o4.z = pack_f16x2(__uint_as_float(r[8 * v4 + 4]), __uint_as_float(r[8 * v4 + 5]));
                            o4.w = pack_f16x2(__uint_as_float(r[8 * v4 + 6]), __uint_as_float(r[8 * v4 + 7]));
                            __stcs(reinterpret_cast<uint4 *>(dst + (4 * qq + v4) * cstride), o4);
                        }
                    } else {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 o4;
                            o4.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]), __uint_as_float(r[8 * v4 + 1]));
                            o4.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]), __uint_as_float(r[8 * v4 + 3]));
                            o4.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]), __uint_as_float(r[8 * v4 + 5]));
                            o4.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]), __uint_as_float(r[8 * v4 + 7]));
                            __stcs(reinterpret_cast<uint4 *>(dst + (4 * qq + v4) * cstride), o4);
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax
        const int wg = (warp - kWarpSoftmax0) >> 2;  // 0: even chunks, 1: odd chunks
        const int R = 32 * (warp & 3) + lane;        // chunk row = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t s_addr = tmem + lane_base + wg * 128;
        const int j_of_row = R & (p.qpk - 1);  // query head of the group this row holds
        int ci = 0;
        bool ok = true;
        // the unit and, loaded one unit ahead, its sequence's key count kv
        // (ragged: from cu_seqlens_k) and cb = kv - (first query + query
        // count) of the sequence: global query gq sees keys up to min(kv - 1,
        // gq + cb) (bottom-right causal: local query s sees keys up to s + kv
        // - Sq)
        auto seq_of = [&](const Unit &y) -> int2 {
            if (p.cu_k) {
                const int kv = __ldg(p.cu_k + y.b + 1) - __ldg(p.cu_k + y.b);
                return make_int2(kv, kv - __ldg(p.cu_q + y.b + 1));
            }
            return make_int2(p.Skv, p.Skv - (y.b + 1) * p.Sq);
        };
        Unit xnext{};
        int2 seqnext = make_int2(p.Skv, 0);
        if (u_begin < u_end) {
            xnext = load_unit(p, u_begin);
            seqnext = seq_of(xnext);
        }
        for (int u = u_begin; u < u_end && ok; u += u_step) {
            const Unit x = xnext;
            const int kv_len = seqnext.x, seq_cb = seqnext.y;
            if (u + u_step < u_end) {
                xnext = load_unit(p, u + u_step);
                seqnext = seq_of(xnext);
            }
            for (int c = 0; c < x.nch && ok; ++c, ++ci) {
                if ((ci & 1) != wg) continue;
                const uint32_t par = (ci >> 1) & 1;
                const int qi = R >> qpk_sh, idx = c * qc + qi;
                const bool in_chunk = idx < x.count;
                const int packed = in_chunk ? p.qsplit[(int64_t)x.h * p.cap + x.start + idx] : 0;
                const bool valid = in_chunk;
                ok = tc::mbar_wait(bar(L::S_FULL + wg), par, abort_flag, p.status, MSA_STATUS_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (__all_sync(0xffffffffu, !valid)) {
                    // no row of this warp holds a query (padding of a short
                    // chunk): its P and O rows are never stored, so skip them;
                    // the barrier protocol (arrive after each wait) stays
                    tc::fence_after_sync();
                    tc::fence_before_sync();
                    tc::mbar_arrive(bar(L::P_FULL + wg));
                    continue;
                }
                {
                    tc::fence_after_sync();
                    // The S row is read 32 keys at a time in rolled loops: one pass
                    // for the max, one for P.
                    uint32_t r[32];
                    tc::tmem_ld32(s_addr, r);
                    // row info while the load is in flight
                    const int gq = packed & 0xFFFFFF;
                    const int split = (packed >> 24) & 0xFF;
                    int nvis = 0;
                    if (valid) {
                        // keys of the block visible to query gq
                        int limit = kv_len - 1;
                        if (p.causal) limit = min(limit, gq + seq_cb);
                        const int nv = limit - x.tok0 + 1;
                        nvis = nv < 0 ? 0 : (nv > 128 ? 128 : nv);
                    }
                    // keys past the causal limit (diagonal block rows) become -inf
                    auto mask_q = [&](int qq) {
                        const int lim = nvis - 32 * qq;
                        if (lim < 32) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j >= lim) r[j] = 0xff800000u;
                        }
                    };
                    // row max: three-input max, four independent chains
                    float mm[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) mm[a] = -INFINITY;
                    bool masked = false;
#pragma unroll 1
                    for (int qq = 0; qq < 4; ++qq) {
                        if (qq > 0) tc::tmem_ld32(s_addr + 32 * qq, r);
                        tc::tmem_ld_wait();
                        // keys past the causal limit: -inf here and, stored back,
                        // for the P pass (the store is warp-wide: every lane
                        // writes its quarter, masked or not)
                        if (__any_sync(0xffffffffu, nvis - 32 * qq < 32)) {
                            mask_q(qq);
                            tc::tmem_st32(s_addr + 32 * qq, r);
                            masked = true;
                        }
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
#pragma unroll
                            for (int a = 0; a < 4; ++a)
                                mm[a] = fmax3(mm[a], __uint_as_float(r[j + 2 * a]), __uint_as_float(r[j + 2 * a + 1]));
                        }
                    }
                    const float m = fmax3(fmax3(mm[0], mm[1], mm[2]), mm[3], -INFINITY);
                    if (masked) tc::tmem_st_wait();  // the masked keys are in tensor memory
                    // P = exp2(S * scale_log2 - m * scale_log2): each quarter is
                    // read again, packed to bf16 pairs in place (r[j] <- keys 2j,
                    // 2j+1 of the quarter) and stored over columns already read;
                    // row sum in packed f32x2 adds (TEMP: also of 2^(x / T)), in the
                    // same order as over whole halves
                    const float mc = (m == -INFINITY) ? 0.f : m * p.scale_log2;
                    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nm2 = make_float2(-mc, -mc);
                    float2 ll[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 lt = make_float2(0.f, 0.f);
#pragma unroll 1
                    for (int qq = 0; qq < 4; ++qq) {
                        tc::tmem_ld32(s_addr + 32 * qq, r);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float2 e =
                                __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), sc2, nm2);
                            if (OPTS && p.temp_on) {
                                const float2 t = __fmul2_rn(e, make_float2(p.inv_temp, p.inv_temp));
                                lt = __fadd2_rn(lt, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                            }
                            e.x = ex2_approx(e.x);
                            e.y = ex2_approx(e.y);
                            ll[j & 1] = __fadd2_rn(ll[j & 1], e);
                            r[j] = pack_bf16x2(e.x, e.y);
                        }
                        tc::tmem_st16(s_addr + 16 * qq, r);
                    }
                    const float l = (ll[0].x + ll[0].y) + (ll[1].x + ll[1].y);
                    tc::tmem_st_wait();
                    tc::fence_before_sync();
                    tc::mbar_arrive(bar(L::P_FULL + wg));
                    // the split statistics (m * scale, l); the epilogue warpgroup
                    // stores the unnormalised O once PV has run
                    if (valid) {
                        const int64_t grp = (int64_t)gq * p.Hkv + x.h;
                        const int64_t si = part_stat_index(grp, p.topk, p.qpk, split, j_of_row);
                        const float2 st = make_float2(l > 0.f ? m * p.scale : -INFINITY, l);
                        __stcs(p.stat_part + si, st);
                        if (OPTS && p.temp_on) {
                            const float ltt = lt.x + lt.y;
                            __stcs(p.stat_temp + si, make_float2(ltt > 0.f ? m * p.scale * p.inv_temp : -INFINITY, ltt));
                        }
                    }
                }
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

}  // namespace msa
