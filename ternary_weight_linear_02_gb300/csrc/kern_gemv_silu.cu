// kern_gemv_silu.cu -- decode-shaped fused gate/up projection with the
// SiLU-gated product, out[m, j] = silu(g[m, j]) * u[m, j]: the kernel of gemv.cuh
// with SILU = true.  A CTA stages RB/2 gate rows and the matching RB/2 up rows
// (two TMA boxes per stage), so each (gate, up) pair meets in one CTA's
// epilogue ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战" §3.2 on stacked
// shards; the product feeds the down projection).
#include "gemv.cuh"

namespace tl {

cudaError_t launch_gemv_silu(const GemvArgs &a, bool bf, bool group, const GemvPlan &p,
                             cudaStream_t st, bool pdl) {
    return bf ? gemv::launch_dtype<true, true>(a, group, p, st, pdl)
              : gemv::launch_dtype<false, true>(a, group, p, st, pdl);
}

}  // namespace tl
