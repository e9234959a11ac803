// tiles.h -- host-side pieces of the attention tile pipeline shared by the
// prefill (attn.cu) and the paged decode (paged.cu).
#pragma once
#include "attn_tc.cuh"

namespace msa {

// Split partials of a forward: topk slots per query head (layout in combine.cuh).
struct FwdWorkspace {
    size_t o_part, stat_part, bytes;
};
FwdWorkspace fwd_workspace_layout(int B, int Sq, int Hq, int topk, int D);

// Multiprocessor count of the current device.
int num_sms();

// Launches the tile kernel for the plan in t (grid: at most one CTA per SM and
// at most `capacity` CTAs); K and V are viewed as kv_tokens token rows.
int tiles_launch(const TcParams &t, int64_t capacity, const void *q, const void *k, const void *v, int64_t kv_tokens,
                 int kv_format, cudaStream_t stream);

}  // namespace msa
