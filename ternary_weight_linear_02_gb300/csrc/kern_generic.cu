// kern_generic.cu -- ternary linear for shapes the TMA-fed kernels do not take:
// K not a multiple of 64, so packed rows are not 16-byte pitched.  Any K is
// served: a row takes ceil(K/4) bytes and, when K % 4 != 0, the last byte's
// fields past K are padding that is never read as a weight (the Qwen2.5-7B
// ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §2.3: an export pads rows
// to whole bytes and the padding is cut off after unpacking).
//
// out[m,n] = sum_k t[n,k] x[m,k] scaled per output channel, or
// sum_g s[n,g] sum_{k in g} t[n,k] x[m,k] for groups of G = 32, 64, 128 or 256
// ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战" §1.1, §3.1, §4.2),
// t decoded with that page's code table (§3.1) as b0 - b1 of the code bits.
//
// CUDA cores, fp32: one warp per output row (gated: per gate/up row pair) and
// MT tokens; lane l takes the packed bytes l, l + 32, ... of the row (coalesced
// byte loads), decodes the four weights of each and accumulates t * x (times
// the group's scale in group mode) for each token; the lanes' partial sums are
// added with a fixed butterfly, so results are reproducible run to run.
#include "common.cuh"
#include "kernels.h"

namespace tl {

namespace {

constexpr int kGenWarps = 8;
constexpr int kGenTokens = 8;  // tokens per CTA

template <bool BF>
__device__ __forceinline__ float x_at(const uint16_t *x, int64_t i) {
    const uint16_t b = x[i];
    if constexpr (BF) return __uint_as_float((uint32_t)b << 16);
    else return __half2float(__ushort_as_half(b));
}

template <bool BF, bool GROUP>
__device__ __forceinline__ void row_dot(const GenArgs &a, int n, int m0, int mt,
                                        float (&acc)[kGenTokens]) {
    const int lane = threadIdx.x & 31;
    const int64_t Kq = (a.K + 3) >> 2;
    const uint8_t *prow = a.packed + (int64_t)n * Kq;
    const int ngk = GROUP ? a.K >> a.gshift : 0;
#pragma unroll
    for (int t = 0; t < kGenTokens; ++t) acc[t] = 0.f;
    for (int64_t b = lane; b < Kq; b += 32) {
        const uint32_t byte = prow[b];
        const float s = GROUP ? h2f(a.scale[(int64_t)n * ngk + ((4 * b) >> a.gshift)]) : 1.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t k = 4 * b + j;
            if (k >= a.K) break;  // padding fields of the last byte
            const uint32_t code = (byte >> (2 * j)) & 3u;
            const float w = (float)((int)(code & 1u) - (int)(code >> 1)) * s;
#pragma unroll
            for (int t = 0; t < kGenTokens; ++t)
                if (t < mt) acc[t] = fmaf(w, x_at<BF>(a.x, (int64_t)(m0 + t) * a.K + k), acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < kGenTokens; ++t)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    if constexpr (!GROUP) {
        const float s = h2f(a.scale[n]);
#pragma unroll
        for (int t = 0; t < kGenTokens; ++t) acc[t] *= s;
    }
}

__device__ __forceinline__ void store_any(int odt, void *base, int64_t idx, float v) {
    if (odt == 0) OutStore<0>::st(base, idx, v);
    else if (odt == 1) OutStore<1>::st(base, idx, v);
    else OutStore<2>::st(base, idx, v);
}

template <bool BF, bool GROUP, bool SILU>
__global__ void __launch_bounds__(32 * kGenWarps) generic_kernel(GenArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kGenWarps + warp;  // output column (gated: pair index)
    pdl_wait();  // x and out belong to the previous kernel until here
    if (row >= (SILU ? a.nh : a.N)) return;  // whole warps leave together
    for (int m0 = blockIdx.y * kGenTokens; m0 < a.M; m0 += gridDim.y * kGenTokens) {
        const int mt = min(kGenTokens, a.M - m0);
        float v = 0.f;
        if constexpr (SILU) {
            float g[kGenTokens], u[kGenTokens];
            row_dot<BF, GROUP>(a, row, m0, mt, g);
            row_dot<BF, GROUP>(a, a.nh + row, m0, mt, u);
#pragma unroll
            for (int t = 0; t < kGenTokens; ++t)
                if (t == lane) v = g[t] / (1.f + expf(-g[t])) * u[t];
            if (lane < mt) store_any(a.odt, a.out, (int64_t)(m0 + lane) * a.nh + row, v);
        } else {
            float acc[kGenTokens];
            row_dot<BF, GROUP>(a, row, m0, mt, acc);
#pragma unroll
            for (int t = 0; t < kGenTokens; ++t)
                if (t == lane) v = acc[t];
            if (lane < mt) store_any(a.odt, a.out, (int64_t)(m0 + lane) * a.N + row, v);
        }
    }
}

template <bool BF, bool GROUP, bool SILU>
cudaError_t launch_gen(const GenArgs &a, cudaStream_t st, bool pdl) {
    const int rows = SILU ? a.nh : a.N;
    cudaLaunchConfig_t cfg = {};
    const int mblocks = (a.M + kGenTokens - 1) / kGenTokens;
    cfg.gridDim = dim3((unsigned)((rows + kGenWarps - 1) / kGenWarps),
                       (unsigned)(mblocks < 65535 ? mblocks : 65535), 1);
    cfg.blockDim = dim3(32 * kGenWarps, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, generic_kernel<BF, GROUP, SILU>, a);
}

}  // namespace

cudaError_t launch_generic(const GenArgs &a, bool bf, bool group, bool silu, cudaStream_t st,
                           bool pdl) {
    if (silu)
        return bf ? (group ? launch_gen<true, true, true>(a, st, pdl) : launch_gen<true, false, true>(a, st, pdl))
                  : (group ? launch_gen<false, true, true>(a, st, pdl) : launch_gen<false, false, true>(a, st, pdl));
    return bf ? (group ? launch_gen<true, true, false>(a, st, pdl) : launch_gen<true, false, false>(a, st, pdl))
              : (group ? launch_gen<false, true, false>(a, st, pdl) : launch_gen<false, false, false>(a, st, pdl));
}

}  // namespace tl
