// kern_gemv.cu -- decode-shaped ternary linear (M <= 16 tokens): the plan (rows
// per CTA, split K, ring depth) and the plain-output entry point.  The kernel
// itself is in gemv.cuh.
#include <map>
#include <mutex>
#include <utility>

#include "gemv.cuh"

namespace tl {

// A kernel with nothing to do, launched never: the occupancy query below asks how
// many clusters of a given size fit when each SM holds one CTA.
__global__ void cluster_capacity_probe() {}

// CTAs that clusters of sk CTAs can place one per SM in one wave.  A cluster
// must fit inside one GPC, so on parts whose GPCs do not hold a multiple of sk
// SMs some SMs are left out (measured on 152-SM parts: clusters of 4 use 144
// SMs, of 8 use 128).  The driver's occupancy query answers it exactly: a
// 150 KB shared-memory footprint allows one CTA per SM.
static int cluster_capacity(int sk, int sm_count) {
    if (sk <= 1) return sm_count;
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find({dev, sk});
    if (it != cache.end()) return it->second;
    int cap = sk <= 2 ? sm_count : 0;
    const int smem = 150 * 1024;
    if (cudaFuncSetAttribute(cluster_capacity_probe, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)sk * 64, 1);
        cfg.blockDim = dim3(32, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)sk;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, cluster_capacity_probe, &cfg) == cudaSuccess && n > 0)
            cap = n * sk;
    }
    cudaGetLastError();
    if (cap <= 0) cap = sm_count / 2;  // unknown: stay well inside one wave
    if (cap > sm_count) cap = sm_count;
    cache[{dev, sk}] = cap;
    return cap;
}

// Rows per CTA (RB = 32 * rgw) and the K split are chosen to spread the weights
// evenly over the SMs.  A warp's time for one 256-k stage is a fixed part (the
// barrier wait, the x fragments, the hand-back) plus one part per row group
// (two code words, the decode, the MMAs); the cost of a plan is the busiest
// warp's time times the number of CTA waves (CTAs beyond one per SM share
// SMs), plus the epilogue and, with split K, the cluster reduction.  K ranges
// are multiples of 256 k (one TMA stage), so no CTA loads bytes it does not use.
GemvPlan plan_gemv(int64_t M, int64_t rows, int64_t K, int sm_count, bool gated, bool group,
                   int force_sk) {
    GemvPlan p{};
    p.ok = M >= 1 && M <= kGemvMaxM && rows >= 1 && K >= 64 && K % 64 == 0 && sm_count > 0 &&
           (!gated || rows % 2 == 0) && gemv::encode_fn() != nullptr;
    if (!p.ok) return p;
    p.nt8 = M <= 8 ? 1 : 2;
    const int64_t units = (K + gemv::kStageK - 1) / gemv::kStageK;
    // measured (ns on a 2.07 GHz part): a stage costs ~250 plus ~90 per row group of a
    // warp (two token tiles: ~150); the epilogue ~1000, a cluster reduction ~1000 more
    const double stage_fixed = 250.0, per_rg = p.nt8 == 1 ? 90.0 : 150.0;
    double best = 1e300;
    int64_t best_ctas = 0;
    const int rgw_hi = gemv::rgw_max(p.nt8, group);
    for (int rgw = 1; rgw <= rgw_hi; ++rgw) {
        const int64_t RB = 32 * rgw;
        const int64_t tiles = gated ? (rows / 2 + RB / 2 - 1) / (RB / 2) : (rows + RB - 1) / RB;
        for (int sk = 1; sk <= 8; ++sk) {
            if (force_sk > 0 && sk != force_sk) continue;
            if (sk > units) break;
            const int64_t spc = (units + sk - 1) / sk;  // stages per CTA
            const int64_t skr = (units + spc - 1) / spc;
            if (skr != sk && force_sk <= 0) continue;  // the same split as a smaller sk
            const int64_t ctas = tiles * skr;
            const int64_t cap = cluster_capacity((int)skr, sm_count);
            // CTAs on the busiest SM over the call; two resident CTAs share an SM at
            // ~1.5x the throughput of one (measured), so n > 1 of them take ~2n/3 of
            // one CTA's time each
            const int64_t n = (ctas + cap - 1) / cap;
            const double waves = n <= 1 ? 1.0 : 0.667 * (double)n;
            const double busiest = (double)spc * (stage_fixed + per_rg * rgw);
            const double over = 1000.0 + (skr > 1 ? 1000.0 : 0.0);
            const double cost = waves * (busiest + over);
            if (cost < best * (1 - 1e-9) || (cost <= best * (1 + 1e-9) && ctas < best_ctas)) {
                best = cost;
                best_ctas = ctas;
                p.rg = 2 * rgw;
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
    int ws = gemv::kRingBytes / gemv::stage_stride(p.nt8, p.rg / 2);
    if (ws > gemv::kMaxStages) ws = gemv::kMaxStages;
    p.ws = ws;
    return p;
}

cudaError_t launch_gemv(const GemvArgs &a, bool bf, bool group, const GemvPlan &p, cudaStream_t st,
                        bool pdl) {
    return bf ? gemv::launch_dtype<true, false>(a, group, p, st, pdl)
              : gemv::launch_dtype<false, false>(a, group, p, st, pdl);
}

}  // namespace tl
