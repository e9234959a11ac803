// tiles_fp8.cu -- tile-kernel instance: e4m3 K/V staged to bf16 on load, prefill.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_fp8) {
    return launch_tiles<MSA_KV_FP8, 2, 3, false>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
