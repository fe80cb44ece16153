// kern_tile.cu -- large-M ternary linear on the tensor cores: support check and
// the plain-output entry point.  The kernel itself is in tile.cuh.
#include "tile.cuh"

namespace tl {

bool tile_supported(int64_t M, int64_t N, int64_t K) {
    // grid y = ceil(M / BN) with BN = 256 above M = 128
    return M >= 1 && N >= 1 && K >= 64 && K % 64 == 0 && M <= 65535ll * 256 &&
           encode_fn() != nullptr;
}

cudaError_t launch_tile(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                        cudaStream_t st, bool pdl) {
    return launch_tile_any<false>(a, bf, group, out_dtype, sm_count, st, pdl);
}

}  // namespace tl
