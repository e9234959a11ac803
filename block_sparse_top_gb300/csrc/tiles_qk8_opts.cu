// tiles_qk8_opts.cu -- tile-kernel instance: e4m3 Q and K (S = Q K^T as an fp8 MMA), e4m3 V staged to bf16 for PV,
// serving the forward's options (partial type, temperature statistics).
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_qk8_opts) {
    return launch_tiles<tck::kKvQk8, 3, 4, true>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
