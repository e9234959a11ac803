// tiles_paged_fp8.cu -- tile-kernel instance: paged decode over an e4m3 K/V pool staged to bf16 on load.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_paged_fp8) { return launch_tiles<MSA_KV_FP8, 3, 1, true, false>(mk, mv, mq, t, grid, stream); }
}  // namespace msa
