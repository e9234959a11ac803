// tiles_bf16.cu -- tile-kernel instance: bf16 K/V, prefill.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_bf16) {
    return launch_tiles<MSA_KV_BF16, 2, 3, false>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
