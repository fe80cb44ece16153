// kern_gemv.cu -- decode-shaped ternary linear (M <= 16 tokens): the plan (rows
// per CTA, split K, ring depth) and the plain-output entry point.  The kernel
// itself is in gemv.cuh.
#include "gemv.cuh"

namespace tl {

// Rows per CTA (16 * rg) and the K split are chosen to spread the weights
// evenly over the SMs: the cost of a plan is the busiest warp's work (rows x
// 64-k columns) times the number of CTA waves, plus a small charge for the
// epilogue and for a cluster reduction.  K ranges are multiples of 256 k (one
// TMA stage) so no CTA loads bytes it does not use.
GemvPlan plan_gemv(int64_t M, int64_t rows, int64_t K, int sm_count, bool gated, int force_sk) {
    GemvPlan p{};
    p.ok = M >= 1 && M <= kGemvMaxM && rows >= 1 && K >= 64 && K % 64 == 0 && sm_count > 0 &&
           (!gated || rows % 2 == 0) && gemv::encode_fn() != nullptr;
    if (!p.ok) return p;
    p.nt8 = M <= 8 ? 1 : 2;
    const int rgmax = p.nt8 == 1 ? gemv::Cfg<1>::RGMAX : gemv::Cfg<2>::RGMAX;
    const int rgmin = p.nt8 == 1 ? 4 : 2;
    const int64_t units = (K + gemv::kStageK - 1) / gemv::kStageK;
    double best = 1e300;
    int64_t best_ctas = 0;
    for (int rg = rgmin; rg <= rgmax; ++rg) {
        const int64_t RB = 16 * rg;
        const int64_t tiles = gated ? (rows / 2 + RB / 2 - 1) / (RB / 2) : (rows + RB - 1) / RB;
        for (int sk = 1; sk <= 8; ++sk) {
            if (force_sk > 0 && sk != force_sk) continue;
            if (sk > units) break;
            const int64_t spc = (units + sk - 1) / sk;  // stages per CTA
            const int64_t skr = (units + spc - 1) / spc;
            if (skr != sk && force_sk <= 0) continue;  // the same split as a smaller sk
            const int64_t ctas = tiles * skr;
            const int64_t waves = (ctas + sm_count - 1) / sm_count;
            const double busiest = (double)RB * (double)((spc + 1) / 2);
            const double over = 0.25 * RB + (skr > 1 ? 0.5 * RB : 0.0);
            const double cost = (double)waves * (busiest + over);
            if (cost < best * (1 - 1e-9) || (cost <= best * (1 + 1e-9) && ctas < best_ctas)) {
                best = cost;
                best_ctas = ctas;
                p.rg = rg;
                p.tiles = (int)tiles;
                p.sk = (int)skr;
                p.kc = (int)(spc * gemv::kStageK);
            }
        }
    }
    if (best >= 1e300) {
        p.ok = false;
        return p;
    }
    int ws = gemv::kRingBytes / (64 * 16 * p.rg);
    if (ws > gemv::kMaxStages) ws = gemv::kMaxStages;
    p.ws = ws;
    return p;
}

cudaError_t launch_gemv(const GemvArgs &a, bool bf, bool group, int out_dtype, const GemvPlan &p,
                        cudaStream_t st, bool pdl) {
    return bf ? gemv::launch_dtype<true, false>(a, group, out_dtype, p, st, pdl)
              : gemv::launch_dtype<false, false>(a, group, out_dtype, p, st, pdl);
}

}  // namespace tl
