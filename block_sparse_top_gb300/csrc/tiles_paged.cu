// tiles_paged.cu -- tile-kernel instance: paged decode (three K/V stages, one Q stage, whole-row softmax).
#include "tiles.h"

namespace msa {
MSA_TILE_INSTANCE(launch_tiles_paged) { return launch_tiles<MSA_KV_BF16, 3, 1, true, false>(mk, mv, mq, t, grid, stream); }
}  // namespace msa
