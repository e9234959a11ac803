// paged_decode_fp8.cu -- paged decode kernel instance: e4m3 K/V pools staged to bf16.
#include "paged_tc.cuh"

namespace msa {
MSA_DECODE_INSTANCE(launch_paged_decode_fp8) { return launch_paged_decode<MSA_KV_FP8>(mk, mv, mq, p, grid, stream); }
}  // namespace msa
