// tiles_qk8.cu -- tile-kernel instance: e4m3 Q and K (S = Q K^T as an fp8 MMA), e4m3 V staged to bf16 for PV.
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_qk8) {
    return launch_tiles<tck::kKvQk8, 3, 4, false>(mk, mv, mq, mqh, t, grid, stream);
}
}  // namespace msa
