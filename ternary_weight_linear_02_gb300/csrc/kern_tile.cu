// kern_tile.cu -- large-M ternary linear on the tensor cores: support check and
// the plain-output entry point.  The kernel itself is in tile.cuh.
#include "tile_persist.cuh"

namespace tl {

bool tile_supported(int64_t M, int64_t N, int64_t K) {
    // grid y = ceil(M / BN) with BN = 256 above M = 128
    return M >= 1 && N >= 1 && K >= 64 && K % 64 == 0 && M <= 65535ll * 256 &&
           encode_fn() != nullptr;
}

// The persistent form takes large-M calls whose tiles it spreads more evenly over
// the SMs, or whose per-tile fixed time it hides, than one tile per CTA does.
// Costs in 64-k chunk times of a 256-token tile (fitted to the 7B shapes at
// M = 2048): one tile per CTA = waves x (chunks + 18) (+8 per split-K exchange,
// +6 for the gated epilogue); persistent = busiest CTA's tiles x (chunks + 2) x
// P192 + 18, P192 the measured time of a 192-token chunk relative to a 256-token one;
// with per-channel scales also the 256-token persistent form (persist_cost).
// Returns 0 (one tile per CTA) or the persistent form's tile width.
int persist_form(const TileArgs &a, bool silu, bool group, int sm_count) {
    if (a.persist >= 0) return a.persist == 0 ? 0 : (a.persist == 2 && !group ? 256 : 192);
    if (a.M <= 256 || sm_count <= 0) return 0;
    const int64_t rb = silu ? (a.nh + 63) / 64 : (a.N + 127) / 128;
    const int nch = a.K / 64;
    double classic = 0.0;
    const int64_t tiles256 = rb * ((a.M + 255) / 256);
    for (int sk = 1; sk <= (silu ? 1 : 2); ++sk) {
        const int64_t waves = (tiles256 * sk + sm_count - 1) / sm_count;
        const double c = (double)waves * ((nch + sk - 1) / sk + 18.0 + (sk > 1 ? 8.0 : 0.0) + (silu ? 6.0 : 0.0));
        if (classic == 0.0 || c < classic) classic = c;
    }
    int form = 0;
    double best = classic;
    const double p192 = persist_cost(a, silu, sm_count, 192);
    if (p192 < best) {
        best = p192;
        form = 192;
    }
    if (!group && persist_cost(a, silu, sm_count, 256) < best) form = 256;
    return form;
}

cudaError_t launch_tile(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                        cudaStream_t st, bool pdl) {
    const int form = persist_form(a, false, group, sm_count);
    if (form > 0) return launch_persist<false>(a, bf, group, out_dtype, sm_count, st, pdl, form);
    return launch_tile_any<false>(a, bf, group, out_dtype, sm_count, st, pdl);
}

}  // namespace tl
