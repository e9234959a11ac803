// tiles_bf16_opts.cu -- tile-kernel instance: bf16 K/V, prefill serving the forward's options (partial type, temperature statistics).
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_bf16_opts) {
    return launch_tiles<MSA_KV_BF16, 2, 3, true>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
