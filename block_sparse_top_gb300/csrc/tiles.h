// tiles.h -- host-side pieces of the prefill attention tile pipeline
// (attn.cu, the tiles_*.cu instances).
#pragma once
#include "attn_tc.cuh"

namespace msa {

// Split partials of a forward: topk slots per query head (layout in
// combine.cuh), of the partial type; with `temp` also the temperature
// statistics.
struct FwdWorkspace {
    size_t o_part, stat_part, stat_temp, bytes;
};
FwdWorkspace fwd_workspace_layout(int64_t total_q, int Hq, int topk, int D, int part_dtype = MSA_PARTIAL_BF16,
                                  bool temp = false);

// Multiprocessor count of the current device.
int num_sms();

// Launches the tile kernel for the plan in t (grid: at most one CTA per SM and
// at most `capacity` CTAs); K and V are viewed as kv_tokens token rows; opts
// selects the instance that serves t's options (partial type, temperature).
int tiles_launch(const TcParams &t, int64_t capacity, const void *q, const void *k, const void *v, int64_t kv_tokens,
                 int kv_format, bool opts, cudaStream_t stream, bool qk_fp8 = false);

// LSE combine of a forward's split partials (workspace ws laid out as w) over
// `groups` (query, KV head) pairs into o, lse (may be null) and, when the
// workspace holds temperature statistics, lse_temp.
int combine_launch(const int32_t *split_counts, int64_t groups, int qpk, int topk, void *o, float *lse,
                   float *lse_temp, const char *ws, const FwdWorkspace &w, int part_dtype, cudaStream_t stream);

// One launch function per tile-kernel instance, each compiled in a
// translation unit of its own (tiles_*.cu) so that the build runs them in
// parallel.
#define MSA_TILE_INSTANCE(NAME)                                                                             \
    int NAME(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const CUtensorMap &mqh, \
             const TcParams &t, int grid, cudaStream_t stream)
MSA_TILE_INSTANCE(launch_tiles_bf16);
MSA_TILE_INSTANCE(launch_tiles_bf16_opts);
MSA_TILE_INSTANCE(launch_tiles_nvfp4);
MSA_TILE_INSTANCE(launch_tiles_nvfp4_opts);
MSA_TILE_INSTANCE(launch_tiles_fp8);
MSA_TILE_INSTANCE(launch_tiles_fp8_opts);
MSA_TILE_INSTANCE(launch_tiles_qk8);
MSA_TILE_INSTANCE(launch_tiles_qk8_opts);

// The launch of instance <KV_FORMAT, NKV, NQ, OPTS> (used by tiles_*.cu).
template <int KV_FORMAT, int NKV, int NQ, bool OPTS>
int launch_tiles(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mq, const CUtensorMap &mqh,
                 const TcParams &t, int grid, cudaStream_t stream) {
    constexpr uint32_t S = KV_FORMAT == tck::kKvQk8 ? 16384u : 32768u;  // K and Q stage bytes
    const size_t smem = tck::Layout<NKV, NQ, S, S>::BYTES;
    MSA_CUDA_TRY(cudaFuncSetAttribute(sparse_fwd_tc_kernel<KV_FORMAT, NKV, NQ, OPTS>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    MSA_CUDA_TRY(launch_pdl(sparse_fwd_tc_kernel<KV_FORMAT, NKV, NQ, OPTS>, dim3(grid),
                            dim3(tck::kThreads), smem, stream, mk, mv, mq, mqh, t));
    return MSA_OK;
}

}  // namespace msa
