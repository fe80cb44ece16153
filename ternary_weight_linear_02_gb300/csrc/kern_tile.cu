// kern_tile.cu -- large-M tile path (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
#include "kernels.h"

namespace tl {
bool tile_supported(int64_t, int64_t, int64_t) { return false; }
cudaError_t launch_tile(const TileArgs &, bool, bool, int, int, cudaStream_t, bool) {
    return cudaErrorNotSupported;
}
}  // namespace tl
