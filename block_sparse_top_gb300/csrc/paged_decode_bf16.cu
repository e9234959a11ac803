// paged_decode_bf16.cu -- paged decode kernel instance: bf16 K/V pools (TMA).
#include "paged_tc.cuh"

namespace msa {
MSA_DECODE_INSTANCE(launch_paged_decode_bf16) { return launch_paged_decode<MSA_KV_BF16>(mk, mv, mq, p, grid, stream); }
}  // namespace msa
