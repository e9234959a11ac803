// tiles_fp8_opts.cu -- tile-kernel instance: e4m3 K/V staged to bf16 on load, prefill serving the forward's options (partial type, temperature statistics).
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_fp8_opts) {
    return launch_tiles<MSA_KV_FP8, 2, 3, true>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
