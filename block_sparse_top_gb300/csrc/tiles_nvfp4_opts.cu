// tiles_nvfp4_opts.cu -- tile-kernel instance: NVFP4 K/V dequantised on load, prefill serving the forward's options (partial type, temperature statistics).
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_nvfp4_opts) {
    return launch_tiles<MSA_KV_NVFP4, 2, 3, true>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
