// kern_skinny_silu.cu -- fused gate/up projection with the SiLU-gated product,
// out[m, j] = silu(g[m, j]) * u[m, j], for decode-shaped M.  g and u are the two
// shards of a stacked gate/up layer ("三元量化模型接入vLLM：从逆向加载到Kernel优化的
// 完整实战" §3.2 on stacked shards; the product feeds the down projection).  A CTA
// holds 64 gate rows and the matching 64 up rows, so the pair meets in one CTA's
// epilogue; the kernel is the one in skinny_tc.cuh with SILU = true.
#include "skinny_tc.cuh"

namespace tl {

cudaError_t launch_skinny_silu(const SkinnyTcArgs &a, bool bf, bool group, int out_dtype,
                               const SkinnyTcPlan &p, cudaStream_t st, bool pdl) {
    if (p.nt == 16) return launch_nt<16, true>(a, bf, group, out_dtype, p, st, pdl);
    return launch_nt<32, true>(a, bf, group, out_dtype, p, st, pdl);
}

}  // namespace tl
