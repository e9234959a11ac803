// tiles_nvfp4_temp.cu -- tile-kernel instance: NVFP4 K/V dequantised on load, prefill with the temperature statistics.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_nvfp4_temp) { return launch_tiles<MSA_KV_NVFP4, 2, 3, false, true>(mk, mv, mq, t, grid, stream); }
}  // namespace msa
