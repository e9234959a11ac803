// attn.cu -- block-sparse prefill forward over the k->q CSR: per work unit
// (KV head h, KV block j of sequence b, a run of the queries that selected
// j) the K/V block is staged once in shared memory and every chunk of
// 128/qhead_per_kv queries (128 query-head rows, gathered from all heads of
// the GQA group) computes S = scale Q K^T, the single-block softmax
// (bottom-right causal mask on the diagonal block), the unnormalised
// U_p = P V and its (scale m, l = sum P); the result goes to the query's split
// slot.  The LSE combine then merges the splits of every (query, head).
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
#include "combine.cuh"
#include "tiles.h"

namespace msa {

// Split partials: topk slots per query head.
FwdWorkspace fwd_workspace_layout(int64_t total_q, int Hq, int topk, int D, int part_dtype, bool temp) {
    FwdWorkspace w;
    const size_t rows = (size_t)total_q * topk * Hq;
    const size_t elem = part_dtype == MSA_PARTIAL_FP32 ? 4 : 2;
    w.o_part = 0;
    w.stat_part = align_up(rows * D * elem, 256);
    w.stat_temp = align_up(w.stat_part + rows * sizeof(float2), 256);
    w.bytes = temp ? align_up(w.stat_temp + rows * sizeof(float2), 256) : w.stat_temp;
    return w;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

// Builds the tensor maps (Q rows; K and V over kv_tokens token rows) and
// launches the tile kernel for t, one CTA per SM, at most `capacity` CTAs
// (the plan's unit capacity).
int tiles_launch(const TcParams &t, int64_t capacity, const void *q, const void *k, const void *v, int64_t kv_tokens,
                 int kv_format, bool opts, cudaStream_t stream, bool qk_fp8) {
    int grid = (int)std::min<int64_t>(capacity, (int64_t)num_sms());
    if (grid < 1) grid = 1;
    CUtensorMap mk, mv, mq, mqh;
    memset(&mk, 0, sizeof mk);
    memset(&mv, 0, sizeof mv);
    memset(&mqh, 0, sizeof mqh);
    if (qk_fp8) {
        // e4m3 Q and K by TMA, e4m3 V staged by the dequantising warp
        if (!make_q8_map(&mq, q, t.total_q * t.Hq, t.qpk) || !make_k8_map(&mk, k, t.Hkv, kv_tokens))
            return MSA_ERR_CUDA;
        return opts ? launch_tiles_qk8_opts(mk, mv, mq, mqh, t, grid, stream)
                    : launch_tiles_qk8(mk, mv, mq, mqh, t, grid, stream);
    }
    // qpk < 8: rows gathered four at a time, or, for a chunk of consecutive
    // query positions, one (positions x heads) box per column half
    const bool q_ok = t.qpk >= 8 ? make_q_group_map(&mq, q, t.total_q * t.Hkv, t.qpk)
                                 : make_q_map(&mq, q, t.total_q * t.Hq, 1) &&
                                       make_q_heads_map(&mqh, q, t.total_q, t.Hq, t.qpk);
    if (!q_ok) return MSA_ERR_CUDA;
    if (kv_format == MSA_KV_BF16) {
        if (!make_kv_map(&mk, k, t.Hkv, kv_tokens) || !make_kv_map(&mv, v, t.Hkv, kv_tokens)) return MSA_ERR_CUDA;
        // two K/V stages and three Q stages
        return opts ? launch_tiles_bf16_opts(mk, mv, mq, mqh, t, grid, stream)
                    : launch_tiles_bf16(mk, mv, mq, mqh, t, grid, stream);
    }
    // NVFP4 / FP8: the dequantising warp reads K and V itself (no K/V maps)
    if (kv_format == MSA_KV_FP8) {
        return opts ? launch_tiles_fp8_opts(mk, mv, mq, mqh, t, grid, stream)
                    : launch_tiles_fp8(mk, mv, mq, mqh, t, grid, stream);
    }
    return opts ? launch_tiles_nvfp4_opts(mk, mv, mq, mqh, t, grid, stream)
                : launch_tiles_nvfp4(mk, mv, mq, mqh, t, grid, stream);
}

namespace {

// Standalone LSE combine: one thread per output piece (group, 8-dim chunk c,
// head j of the group), in the partials' own order, so for each split the
// threads of a warp read contiguous pieces.  The thread of chunk 0 also
// writes the LSE and, with temperature statistics, the temperature LSE.
template <int MAXS, int PD>
__global__ void __launch_bounds__(256, 2) combine_kernel(const void *__restrict__ o_part,
                                                         const float2 *__restrict__ stat_part,
                                                         const float2 *__restrict__ stat_temp,
                                                         const int32_t *__restrict__ split_counts, int64_t groups,
                                                         int qpk, int topk, uint4 *__restrict__ o,
                                                         float *__restrict__ lse, float *__restrict__ lse_temp) {
    grid_dependency_wait();  // the partials come from the previous kernel
    grid_dependents_launch();
    const int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int per_g = 16 * qpk;
    if (item >= groups * per_g) return;
    const int64_t grp = item / per_g;
    const int rem = (int)(item % per_g);
    const int c = rem / qpk, j = rem % qpk;
    int n = split_counts[grp];
    n = n < topk ? n : topk;
    uint4 out;
    float l;
    combine_piece<MAXS, PD, PD == MSA_PARTIAL_FP32 ? 8 : 16>(o_part, stat_part, grp, n, topk, qpk, c, j, out, l);
    // o [B*Sq][Hq][D]: group grp = gq*Hkv + h holds query heads h*qpk .. h*qpk+qpk-1
    const int64_t orow = grp * qpk + j;  // == gq*Hq + h*qpk + j
    o[orow * 16 + c] = out;
    if (c == 0 && lse) lse[orow] = l;
    if (c == 0 && lse_temp) lse_temp[orow] = combine_lse_temp(stat_temp, grp, n, topk, qpk, j);
}

// The combine for 16-byte pieces (bf16 / fp16 partials) and topk <= 16: a
// ring buffer holds a run of NG = 16 / qhead_per_kv consecutive groups (256
// pieces: one per merging thread); one persistent CTA per SM walks the runs
// blockIdx.x, + gridDim.x, ..., in three roles that meet only at mbarriers
// (no CTA barrier per run):
//   warp 12 (copies): copies each group's split partials (n x qpk x 256 B,
//     contiguous) and the run's statistics into a ring of kRingBufs
//     shared-memory buffers with bulk copies, kRingBufs runs ahead;
//   warps 8-11 (weights), once a run's copy has landed: lane (row r = group
//     r / qpk, head r % qpk; split s), two passes of two rows per warp, the
//     split's weight w = exp(a_s - A_r), with A_r the max over the group's
//     splits and den_r = sum w l_s (16-lane shuffles), into the buffer's
//     weight table; lane s = 0 writes the LSE A_r + ln den_r; then the
//     buffer is READY;
//   warps 0-7 (merge, thread = (group, 8-dim chunk c, head j), head
//     fastest): once READY, fold O = sum_s w_s U_s / den over their pieces
//     in packed f32x2 FMAs, store it, and release the buffer (one arrival
//     per warp),
// so each weight is computed once, not once per piece, and the merging warps
// never wait for one another.
constexpr int kRingBufs = 3;
constexpr int kCombineThreads = 416;
__host__ __device__ constexpr uint32_t ring_buf_bytes(int topk) { return (uint32_t)topk * (4096u + 128u); }
template <int PD, int QPK>
__global__ void __launch_bounds__(kCombineThreads, 1) combine_ring_kernel(const uint4 *__restrict__ o_part,
                                                                          const float2 *__restrict__ stat_part,
                                                                          const float2 *__restrict__ stat_temp,
                                                                          const int32_t *__restrict__ split_counts,
                                                                          int64_t groups, int topk,
                                                                          uint4 *__restrict__ o,
                                                                          float *__restrict__ lse,
                                                                          float *__restrict__ lse_temp,
                                                                          uint32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t base = smem_u32(smem), bb = ring_buf_bytes(topk);
    const uint32_t bars = base + kRingBufs * bb;  // FULL[kRingBufs], EMPTY[kRingBufs], READY[kRingBufs]
    auto full = [&](int b) { return bars + 8u * b; };
    auto empty = [&](int b) { return bars + 8u * (kRingBufs + b); };
    auto ready = [&](int b) { return bars + 8u * (2 * kRingBufs + b); };
    __shared__ int abort_flag_s;
    __shared__ float wts[kRingBufs][16][17];  // [buffer][row = group * qpk + head][split] weights
    __shared__ float inv_den[kRingBufs][16];
    __shared__ int nsplit[kRingBufs][16];     // [buffer][group of the run]
    volatile int *abort_flag = &abort_flag_s;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    constexpr int qpk = QPK;
    constexpr int ng = 16 / qpk;  // groups per run
    const int64_t runs = (groups + ng - 1) / ng;
    const uint32_t gbytes = (uint32_t)topk * (uint32_t)qpk * 256u;  // a group's partial slots
    if (t == 0) {
        for (int b = 0; b < kRingBufs; ++b) {
            tc::mbar_init(full(b), 1);
            tc::mbar_init(empty(b), 8);    // one arrival per merging warp
            tc::mbar_init(ready(b), 128);  // every weights thread (each releases its own table writes)
        }
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    grid_dependency_wait();  // the partials come from the previous kernel
    grid_dependents_launch();
    __syncthreads();
    const int64_t G = gridDim.x;
    if (warp == 12) {
        // ------------------------------------------------------------ copies
        if (lane != 0) return;
        int64_t k = 0;
        for (; blockIdx.x + k * G < runs; ++k) {
            const int64_t run = blockIdx.x + k * G, grp0 = run * ng;
            const int b = (int)(k % kRingBufs);
            if (k >= kRingBufs &&
                !tc::mbar_wait(empty(b), (uint32_t)(((k / kRingBufs) - 1) & 1), abort_flag, status,
                               MSA_STATUS_TIMEOUT))
                break;
            const int nr = (int)min((int64_t)ng, groups - grp0);  // groups of this run
            uint32_t bytes = 0;
            for (int g = 0; g < nr; ++g) {
                int n = split_counts[grp0 + g];
                n = n < topk ? n : topk;
                nsplit[b][g] = n;
                bytes += (uint32_t)n * (uint32_t)qpk * 256u;
            }
            for (int g = nr; g < ng; ++g) nsplit[b][g] = 0;
            // the run's statistics, every split slot of its groups (topk qpk 8 B
            // a group: a multiple of 16 bytes)
            const uint32_t sbytes = (uint32_t)nr * (uint32_t)topk * (uint32_t)qpk * 8u;
            tc::mbar_arrive_expect_tx(full(b), bytes + sbytes);
            for (int g = 0; g < nr; ++g)
                if (nsplit[b][g] > 0)
                    tc::bulk_load(base + b * bb + g * gbytes, o_part + (grp0 + g) * topk * 16 * qpk,
                                  (uint32_t)nsplit[b][g] * (uint32_t)qpk * 256u, full(b));
            tc::bulk_load(base + b * bb + topk * 4096u, stat_part + grp0 * topk * qpk, sbytes, full(b));
        }
        // the last kRingBufs copies land before the CTA can exit (after an
        // abort nobody else waits for them)
        volatile int dummy = 0;
        for (int64_t kk = k > kRingBufs ? k - kRingBufs : 0; kk < k; ++kk)
            tc::mbar_wait(full((int)(kk % kRingBufs)), (uint32_t)((kk / kRingBufs) & 1), &dummy, status, 0);
        return;
    }
    if (warp >= 8) {
        // ------------------------------------------------------------ weights
        const int sw = lane & 15;
        for (int64_t k = 0; blockIdx.x + k * G < runs; ++k) {
            const int64_t grp0 = (blockIdx.x + k * G) * ng;
            const int b = (int)(k % kRingBufs);
            const bool ok =
                tc::mbar_wait(full(b), (uint32_t)((k / kRingBufs) & 1), abort_flag, status, MSA_STATUS_TIMEOUT);
            if (!__all_sync(0xffffffffu, ok)) break;
            const float2 *stp = reinterpret_cast<const float2 *>(smem + b * bb + topk * 4096);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = 4 * (warp - 8) + 2 * i + (lane >> 4);  // row: group r / qpk, head r % qpk
                const int g = ng == 1 ? 0 : r / qpk, j = r - g * qpk;
                const int n = nsplit[b][g];
                const float2 st = sw < n ? stp[(g * topk + sw) * qpk + j] : make_float2(-INFINITY, 0.f);
                const float a = isfinite(st.x) ? st.x : -INFINITY;
                float A = a;
#pragma unroll
                for (int o2 = 8; o2 > 0; o2 >>= 1) A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, o2));
                const float w = (a == -INFINITY) ? 0.f : __expf(a - A);
                float den = w * st.y;
#pragma unroll
                for (int o2 = 8; o2 > 0; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
                wts[b][r][sw] = w;
                if (sw == 0) {
                    inv_den[b][r] = den > 0.f ? 1.f / den : 0.f;
                    const int64_t grp = grp0 + g;
                    if (grp < groups) {
                        const int64_t orow = grp * qpk + j;
                        if (lse) lse[orow] = den > 0.f ? A + logf(den) : -INFINITY;
                        if (lse_temp) lse_temp[orow] = combine_lse_temp(stat_temp, grp, n, topk, qpk, j);
                    }
                }
            }
            tc::mbar_arrive(ready(b));
        }
        return;
    }
    // ---------------------------------------------------------------- mergers
    const int j = t % qpk, c = (t / qpk) & 15, g = ng == 1 ? 0 : t / (16 * qpk), r = g * qpk + j;
    for (int64_t k = 0; blockIdx.x + k * G < runs; ++k) {
        const int64_t grp = (blockIdx.x + k * G) * ng + g;
        const int b = (int)(k % kRingBufs);
        const bool ok = tc::mbar_wait(ready(b), (uint32_t)((k / kRingBufs) & 1), abort_flag, status,
                                      MSA_STATUS_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int n = nsplit[b][g];
        const uint4 *up = reinterpret_cast<const uint4 *>(smem + b * bb + g * gbytes);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int sp = 0; sp < 16; ++sp) {
            if (sp >= n) break;
            const uint4 u = up[(sp * 16 + c) * qpk + j];
            const float w = wts[b][r][sp];
            const float2 w2 = make_float2(w, w);
            const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 v;
                if (PD == MSA_PARTIAL_FP16) {
                    v = __half22float2(*reinterpret_cast<const __half2 *>(&words[i]));
                } else {
                    v = make_float2(bf16_lo(words[i]), bf16_hi(words[i]));
                }
                acc[i] = __ffma2_rn(v, w2, acc[i]);
            }
        }
        const float inv = inv_den[b][r];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty(b));  // this warp is done with the buffer and its table
        if (grp < groups) {
            uint4 out;
            out.x = pack_bf16x2(acc[0].x * inv, acc[0].y * inv);
            out.y = pack_bf16x2(acc[1].x * inv, acc[1].y * inv);
            out.z = pack_bf16x2(acc[2].x * inv, acc[2].y * inv);
            out.w = pack_bf16x2(acc[3].x * inv, acc[3].y * inv);
            o[(grp * qpk + j) * 16 + c] = out;
        }
    }
}

template <int PD>
int combine_generic(const void *op, const float2 *sp, const float2 *tp, const int32_t *split_counts, int64_t groups,
                    int qpk, int topk, uint4 *ob, float *lse, float *lse_temp, cudaStream_t stream) {
    const int64_t blocks = ceil_div(groups * 16 * qpk, 256);
    if (topk <= 16)
        MSA_CUDA_TRY(launch_pdl(combine_kernel<16, PD>, dim3((unsigned)blocks), dim3(256), 0, stream, op, sp, tp,
                                split_counts, groups, qpk, topk, ob, lse, lse_temp));
    else
        MSA_CUDA_TRY(launch_pdl(combine_kernel<32, PD>, dim3((unsigned)blocks), dim3(256), 0, stream, op, sp, tp,
                                split_counts, groups, qpk, topk, ob, lse, lse_temp));
    return MSA_OK;
}

template <int PD, int QPK>
int combine_ring_q(const void *op, const float2 *sp, const float2 *tp, const int32_t *split_counts, int64_t groups,
                   int topk, uint4 *ob, float *lse, float *lse_temp, cudaStream_t stream) {
    const size_t smem = kRingBufs * ring_buf_bytes(topk) + 24u * kRingBufs;
    MSA_CUDA_TRY(
        cudaFuncSetAttribute(combine_ring_kernel<PD, QPK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const int64_t runs = (groups + 16 / QPK - 1) / (16 / QPK);
    const int grid = (int)std::min<int64_t>(runs, (int64_t)num_sms());
    MSA_CUDA_TRY(launch_pdl(combine_ring_kernel<PD, QPK>, dim3(grid), dim3(kCombineThreads), smem, stream,
                            static_cast<const uint4 *>(op), sp, tp, split_counts, groups, topk, ob, lse, lse_temp,
                            (uint32_t *)nullptr));
    return MSA_OK;
}

template <int PD>
int combine_ring(const void *op, const float2 *sp, const float2 *tp, const int32_t *split_counts, int64_t groups,
                 int qpk, int topk, uint4 *ob, float *lse, float *lse_temp, cudaStream_t stream) {
    switch (qpk) {
        case 1: return combine_ring_q<PD, 1>(op, sp, tp, split_counts, groups, topk, ob, lse, lse_temp, stream);
        case 2: return combine_ring_q<PD, 2>(op, sp, tp, split_counts, groups, topk, ob, lse, lse_temp, stream);
        case 4: return combine_ring_q<PD, 4>(op, sp, tp, split_counts, groups, topk, ob, lse, lse_temp, stream);
        case 8: return combine_ring_q<PD, 8>(op, sp, tp, split_counts, groups, topk, ob, lse, lse_temp, stream);
        default: return combine_ring_q<PD, 16>(op, sp, tp, split_counts, groups, topk, ob, lse, lse_temp, stream);
    }
}

}  // namespace

int combine_launch(const int32_t *split_counts, int64_t groups, int qpk, int topk, void *o, float *lse,
                   float *lse_temp, const char *ws, const FwdWorkspace &w, int part_dtype, cudaStream_t stream) {
    const void *op = ws + w.o_part;
    const float2 *sp = reinterpret_cast<const float2 *>(ws + w.stat_part);
    const float2 *tp = lse_temp ? reinterpret_cast<const float2 *>(ws + w.stat_temp) : nullptr;
    uint4 *ob = static_cast<uint4 *>(o);
    // 16-byte pieces and topk <= 16: staged through a shared-memory ring
    if (topk <= 16 && part_dtype == MSA_PARTIAL_BF16)
        return combine_ring<MSA_PARTIAL_BF16>(op, sp, tp, split_counts, groups, qpk, topk, ob, lse, lse_temp, stream);
    if (topk <= 16 && part_dtype == MSA_PARTIAL_FP16)
        return combine_ring<MSA_PARTIAL_FP16>(op, sp, tp, split_counts, groups, qpk, topk, ob, lse, lse_temp, stream);
    if (part_dtype == MSA_PARTIAL_FP32)
        return combine_generic<MSA_PARTIAL_FP32>(op, sp, tp, split_counts, groups, qpk, topk, ob, lse, lse_temp,
                                                 stream);
    if (part_dtype == MSA_PARTIAL_FP16)
        return combine_generic<MSA_PARTIAL_FP16>(op, sp, tp, split_counts, groups, qpk, topk, ob, lse, lse_temp,
                                                 stream);
    return combine_generic<MSA_PARTIAL_BF16>(op, sp, tp, split_counts, groups, qpk, topk, ob, lse, lse_temp, stream);
}

namespace {

// TcParams of a prefill forward (uniform or ragged; the caller sets the
// batch-specific fields).
TcParams prefill_params(const void *k, const void *v, const void *k_scales, const void *v_scales,
                        const int32_t *qsplit, const void *plan, char *ws, const FwdWorkspace &w, int Hq, int Hkv,
                        int D, int topk, int causal, float softmax_scale, uint32_t *status_dev) {
    TcParams t;
    memset(&t, 0, sizeof t);
    t.k_packed = static_cast<const uint8_t *>(k);
    t.v_packed = static_cast<const uint8_t *>(v);
    t.k_scales = static_cast<const uint8_t *>(k_scales);
    t.v_scales = static_cast<const uint8_t *>(v_scales);
    t.qsplit = qsplit;
    t.plan = static_cast<const PlanHeader *>(plan);
    t.units = reinterpret_cast<const PlanUnit *>(t.plan + 1);
    t.o_part = ws + w.o_part;
    t.stat_part = reinterpret_cast<float2 *>(ws + w.stat_part);
    t.stat_temp = reinterpret_cast<float2 *>(ws + w.stat_temp);
    t.part_dtype = MSA_PARTIAL_BF16;
    t.inv_temp = 1.f;
    t.cu_q = t.cu_k = nullptr;
    t.status = status_dev;
    t.Hq = Hq; t.Hkv = Hkv; t.qpk = Hq / Hkv; t.topk = topk;
    t.causal = causal ? 1 : 0;
    t.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    t.scale_log2 = t.scale * 1.4426950408889634f;
    return t;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_attn_fwd_workspace_size(int B, int Sq, int Hq, int topk, int D) {
    if (B <= 0 || Sq <= 0 || Hq <= 0 || topk <= 0 || D != kD) return 0;
    return fwd_workspace_layout((int64_t)B * Sq, Hq, topk, D).bytes;
}

extern "C" int msa_sparse_attn_fwd_partial(const void *q, const void *k, const void *v, int kv_format,
                                           const void *k_scales, const void *v_scales, const int32_t *q_indices,
                                           const int32_t *qsplit, const void *plan, int B, int Sq, int Skv, int Hq,
                                           int Hkv, int D, int blk_kv, int topk, int causal, float softmax_scale,
                                           void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                           cudaStream_t stream) {
    if (!q || !k || !v || !q_indices || !qsplit || !plan || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Skv <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv) return MSA_ERR_INVALID_ARG;
    if (Hkv > kMaxHkv || ceil_div(Skv, kBlk) > kMaxNblk) return MSA_ERR_UNSUPPORTED;
    if (kv_format != MSA_KV_BF16 && kv_format != MSA_KV_NVFP4 && kv_format != MSA_KV_FP8) return MSA_ERR_INVALID_ARG;
    if (kv_format == MSA_KV_NVFP4 && (!k_scales || !v_scales)) return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || blk_kv != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if ((int64_t)B * Sq >= (1 << 24)) return MSA_ERR_UNSUPPORTED;
    const FwdWorkspace w = fwd_workspace_layout((int64_t)B * Sq, Hq, topk, D);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(plan, 16)) return MSA_ERR_INVALID_ARG;

    TcParams t = prefill_params(k, v, k_scales, v_scales, qsplit, plan, static_cast<char *>(workspace), w, Hq, Hkv,
                                D, topk, causal, softmax_scale, status_dev);
    t.B = B; t.Sq = Sq; t.Skv = Skv;
    t.nblk = (int)ceil_div(Skv, kBlk);
    t.cap = (int64_t)B * Sq * topk;
    t.kv_rows = (int64_t)B * Skv;
    t.total_q = (int64_t)B * Sq;
    const int64_t cap = plan_capacity((int64_t)B * t.nblk, (int64_t)B * Sq, Hkv, topk, qpk);
    return tiles_launch(t, cap, q, k, v, (int64_t)B * Skv, kv_format, false, stream);
}

extern "C" int msa_sparse_attn_combine(const int32_t *split_counts, int B, int Sq, int Hq, int Hkv, int D, int topk,
                                       void *o, float *lse, const void *workspace, size_t ws_bytes,
                                       cudaStream_t stream) {
    if (!split_counts || !o || !workspace) return MSA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv) return MSA_ERR_INVALID_ARG;
    if (D != kD || !supported_topk(topk)) return MSA_ERR_UNSUPPORTED;
    const FwdWorkspace w = fwd_workspace_layout((int64_t)B * Sq, Hq, topk, D);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (!aligned(o, 16)) return MSA_ERR_INVALID_ARG;
    return combine_launch(split_counts, (int64_t)B * Sq * Hkv, Hq / Hkv, topk, o, lse, nullptr,
                          static_cast<const char *>(workspace), w, MSA_PARTIAL_BF16, stream);
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

// Options of a ragged-batch forward: 0, or MSA_ERR_* for a value outside the supported set.
static int check_options(const msa_fwd_options *opts) {
    if (!opts) return MSA_OK;
    if (opts->partial_dtype != MSA_PARTIAL_BF16 && opts->partial_dtype != MSA_PARTIAL_FP16 &&
        opts->partial_dtype != MSA_PARTIAL_FP32)
        return MSA_ERR_UNSUPPORTED;
    if (opts->lse_temperature &&
        !(opts->lse_temperature_scale > 0.f && opts->lse_temperature_scale < INFINITY))
        return MSA_ERR_INVALID_ARG;
    return MSA_OK;
}

extern "C" size_t msa_sparse_attn_fwd_varlen_workspace_size(int total_q, int Hq, int topk, int D,
                                                          const msa_fwd_options *opts) {
    if (total_q <= 0 || Hq <= 0 || topk <= 0 || D != kD || check_options(opts) != MSA_OK) return 0;
    return fwd_workspace_layout(total_q, Hq, topk, D, opts ? opts->partial_dtype : MSA_PARTIAL_BF16,
                                opts && opts->lse_temperature)
        .bytes;
}

extern "C" int msa_sparse_attn_fwd_varlen(const void *q, const void *k, const void *v, int kv_format,
                                          const void *k_scales, const void *v_scales, const int32_t *q_indices,
                                          const int32_t *qsplit, const int32_t *split_counts, const void *plan,
                                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B,
                                          int total_q, int total_k, int Hq, int Hkv, int D, int blk_kv, int topk,
                                          int causal, float softmax_scale, const msa_fwd_options *opts, void *o,
                                          float *lse, void *workspace, size_t ws_bytes, uint32_t *status_dev,
                                          cudaStream_t stream) {
    if (!q || !k || !v || !q_indices || !qsplit || !split_counts || !plan || !cu_seqlens_q || !cu_seqlens_k ||
        !o || !workspace)
        return MSA_ERR_INVALID_ARG;
    if (B <= 0 || total_q <= 0 || total_k <= 0 || Hq <= 0 || Hkv <= 0 || topk <= 0 || Hq % Hkv)
        return MSA_ERR_INVALID_ARG;
    if (kv_format != MSA_KV_BF16 && kv_format != MSA_KV_NVFP4 && kv_format != MSA_KV_FP8) return MSA_ERR_INVALID_ARG;
    if (kv_format == MSA_KV_NVFP4 && (!k_scales || !v_scales)) return MSA_ERR_INVALID_ARG;
    const int qpk = Hq / Hkv;
    if (D != kD || blk_kv != kBlk || !supported_topk(topk) || !supported_qpk(qpk)) return MSA_ERR_UNSUPPORTED;
    if (total_q >= (1 << 24) || Hkv > kMaxHkv) return MSA_ERR_UNSUPPORTED;
    const int orc = check_options(opts);
    if (orc != MSA_OK) return orc;
    const bool qk_fp8 = opts && opts->qk_fp8;
    if (qk_fp8 && kv_format != MSA_KV_FP8) return MSA_ERR_INVALID_ARG;
    const int part_dtype = opts ? opts->partial_dtype : MSA_PARTIAL_BF16;
    float *lse_temp = opts ? opts->lse_temperature : nullptr;
    const FwdWorkspace w = fwd_workspace_layout(total_q, Hq, topk, D, part_dtype, lse_temp != nullptr);
    if (ws_bytes < w.bytes || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(plan, 16) || !aligned(o, 16))
        return MSA_ERR_INVALID_ARG;

    TcParams t = prefill_params(k, v, k_scales, v_scales, qsplit, plan, static_cast<char *>(workspace), w, Hq, Hkv,
                                D, topk, causal, softmax_scale, status_dev);
    t.cu_q = cu_seqlens_q;
    t.cu_k = cu_seqlens_k;
    // per-sequence sizes come from cu_seqlens; Sq / Skv / nblk are unused
    t.B = B; t.Sq = 1; t.Skv = 1; t.nblk = 1;
    t.cap = (int64_t)total_q * topk;
    t.kv_rows = total_k;
    t.total_q = total_q;
    t.part_dtype = part_dtype;
    if (lse_temp) {
        t.temp_on = 1;
        t.inv_temp = 1.f / opts->lse_temperature_scale;
    }
    const bool use_opts = lse_temp != nullptr || part_dtype != MSA_PARTIAL_BF16;
    int rc = tiles_launch(t, (int64_t)num_sms(), q, k, v, total_k, kv_format, use_opts, stream, qk_fp8);
    if (rc != MSA_OK) return rc;
    // the combine's groups are (query, KV head) pairs over all sequences
    return combine_launch(split_counts, (int64_t)total_q * Hkv, qpk, topk, o, lse, lse_temp,
                          static_cast<const char *>(workspace), w, part_dtype, stream);
}
