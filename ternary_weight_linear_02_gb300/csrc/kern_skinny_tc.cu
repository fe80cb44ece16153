// kern_skinny_tc.cu -- decode-shaped ternary linear (M <= 32 tokens) on the
// tensor cores: the plan (row tiles, split K) and the plain-output entry point.
// The kernel itself is in skinny_tc.cuh.
#include "skinny_tc.cuh"

namespace tl {

SkinnyTcPlan plan_skinny_tc(int64_t M, int64_t N, int64_t K, int sm_count, int force_sk,
                            int ctas_per_sm) {
    SkinnyTcPlan p{};
    p.ok = M >= 1 && M <= 32 && N >= 1 && K >= 64 && K % 64 == 0 && encode_fn() != nullptr;
    if (!p.ok) return p;
    p.nt = M <= 16 ? 16 : 32;
    p.row_tiles = (int)((N + 127) / 128);
    const int units = (int)((K + 127) / 128);
    // K is split (a thread-block cluster per row block) until the CTAs fill the
    // ctas_per_sm resident slots of every SM -- but never beyond them: a second,
    // partial wave costs a whole CTA's latency.  Clusters of 5 or 7 CTAs pack
    // poorly into the GPCs (measured: 40 row blocks x 7 ran 1.6x slower than x 6),
    // so those sizes step down to 4 and 6.
    const int64_t target = (int64_t)sm_count * (ctas_per_sm > 0 ? ctas_per_sm : 2);
    int sk = force_sk > 0 ? force_sk : (int)(target / p.row_tiles);
    if (sk < 1) sk = 1;
    if (sk > 8) sk = 8;
    if (sk > units) sk = units;
    if (force_sk <= 0 && (sk == 5 || sk == 7)) --sk;
    const int upc = (units + sk - 1) / sk;  // units per CTA
    p.kc = upc * 128;
    p.sk = (int)((K + p.kc - 1) / p.kc);
    return p;
}

cudaError_t launch_skinny_tc(const SkinnyTcArgs &a, bool bf, bool group, int out_dtype,
                             const SkinnyTcPlan &p, cudaStream_t st, bool pdl) {
    if (p.nt == 16) return launch_nt<16, false>(a, bf, group, out_dtype, p, st, pdl);
    return launch_nt<32, false>(a, bf, group, out_dtype, p, st, pdl);
}

}  // namespace tl
