// tiles_nvfp4.cu -- tile-kernel instance: NVFP4 K/V dequantised on load, prefill.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_nvfp4) {
    return launch_tiles<MSA_KV_NVFP4, 2, 3, false>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
