// kern_tile_silu.cu -- large-M fused gate/up projection with the SiLU-gated
// product, out[m, j] = silu(g[m, j]) * u[m, j]; the kernel in tile.cuh with
// SILU = true (64 gate rows and the matching 64 up rows per CTA).
#include "tile_persist.cuh"

namespace tl {

int persist_form(const TileArgs &a, bool silu, bool group, int sm_count);

cudaError_t launch_tile_silu(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                             cudaStream_t st, bool pdl) {
    const int form = persist_form(a, true, group, sm_count);
    if (form > 0) return launch_persist<true>(a, bf, group, out_dtype, sm_count, st, pdl, form);
    return launch_tile_any<true>(a, bf, group, out_dtype, 0, st, pdl);  // no split K
}

}  // namespace tl
