// kern_tile_silu.cu -- large-M fused gate/up projection with the SiLU-gated
// product, out[m, j] = silu(g[m, j]) * u[m, j]; the kernel in tile.cuh with
// SILU = true (64 gate rows and the matching 64 up rows per CTA).
#include "tile_persist.cuh"

namespace tl {

bool use_persist(const TileArgs &a, bool silu, int sm_count);

cudaError_t launch_tile_silu(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                             cudaStream_t st, bool pdl) {
    if (use_persist(a, true, sm_count))
        return launch_persist<true>(a, bf, group, out_dtype, sm_count, st, pdl);
    return launch_tile_any<true>(a, bf, group, out_dtype, 0, st, pdl);  // no split K
}

}  // namespace tl
