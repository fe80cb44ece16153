// kern_skinny.cu -- decode-shaped ternary linear (M <= 32 tokens).
//
// out[m,n] = sum_k t[n,k] x[m,k], scaled per output channel
// (Qwen2.5-7B ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or
// per 128-wide K group ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §3.1, §4.2), with t decoded from the packed 2-bit codes
// (same page §3.1).
//
// Design (memory-bound: every packed byte is read from HBM exactly once).
//  * The pages turn each +-1/0 product into add / subtract / skip on CUDA
//    cores.  On GB300 that costs >= M adds per weight and saturates the ALUs
//    long before HBM at M > 1, so here the decoded weight is fed to a warp MMA
//    instead: 2*t in {+-2, +-0} is exact in bf16 and fp16, each product
//    2*t*x is exact in the fp32 accumulator, so the MMA performs exactly the
//    same signed additions (zeros contribute +-0).  Decode cost is paid once
//    per weight, independent of M.
//  * Decode: two 2-bit codes -> one bf16x2/f16x2 register with one shift and
//    one AND (tl::pair2), after one XOR pass per 16 codes (tl::sign_nz).
//  * Operand mapping for mma.m16n8k16 (A row-major 16x16, B col-major 16x8):
//    A = 16 weight rows, B = x^T (8 tokens per n-tile).  Thread (g = lane/4,
//    t = lane%4) reads 8 bytes (32 codes) of rows g and g+8 in each 128-k group;
//    the four threads t of a row together cover the group, so one MMA never
//    mixes two scale groups.  The k-order inside the MMA is permuted (the
//    same permutation is applied to x when it is staged in shared memory), so
//    each A register is one pair2() result and each B fragment one 8-byte
//    shared load.
//  * Group scale: per-group fp32 partial in registers, folded into the total
//    with s[n,g] at the group boundary.  Channel scale: once in the epilogue.
//  * Split K across the CTAs of a thread-block cluster (<= 8); partial tiles
//    are summed through distributed shared memory in rank order 0..SK-1, so
//    the result is bit-identical run to run.  No global scratch.
//  * The CTA's packed rows are bulk-prefetched into L2 before
//    griddepcontrol.wait, so with programmatic dependent launch a layer's
//    weight stream starts while the previous kernel in the stream finishes.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace tl {

template <bool BF>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Slot of the staged x fragment for (group, word, step, n-tile, lane).  One
// slot = 8 bytes = the B fragment {b0, b1} of one lane; the 32 lanes of a
// (group, word, step, n-tile) read 256 contiguous bytes.
template <int NT8>
__device__ __forceinline__ int xslot(int grp, int w, int s, int nt, int t, int g) {
    return ((((grp * 2 + w) * 4 + s) * NT8 + nt) * 4 + t) * 8 + g;
}

template <int NT8, int MT, int D, bool BF, bool GROUP, int OUT>
__global__ void __launch_bounds__(kSkinnyThreads) skinny_mma_kernel(SkinnyArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int RT = 16 * MT * (kSkinnyThreads / 32);  // rows per CTA
    constexpr int MP = 8 * NT8;                          // padded tokens
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * RT;
    const int kb = blockIdx.y * a.kc;
    const int ke = min(a.K, kb + a.kc);
    const int klen = max(ke - kb, 0);
    const int ng = (klen + 127) >> 7;  // groups in this CTA (the last may be half)
    const int64_t Kq = a.K >> 2;       // bytes per packed row

    // 1. start this CTA's weight stream: bulk prefetch of its rows into L2
    if (klen > 0) {
        for (int r = threadIdx.x; r < RT; r += blockDim.x) {
            const int n = n0 + r;
            if (n < a.N) prefetch_l2_bulk(a.packed + (int64_t)n * Kq + (kb >> 2), klen >> 2);
        }
    }
    pdl_launch_dependents();
    pdl_wait();  // x / out may be produced / consumed by the previous kernel

    // 2. stage x[:, kb:ke) in fragment order
    uint2 *xs = reinterpret_cast<uint2 *>(smem);
    {
        const int units = MP * ng * 8;  // (token, group, t, word); 16 k each
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int w = u & 1, tt = (u >> 1) & 3, rest = u >> 3;
            const int grp = rest % ng, m = rest / ng;
            const int k = kb + grp * 128 + 32 * tt + 16 * w;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (m < a.M && k < ke) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)m * a.K + k);
                lo = src[0];
                hi = src[1];
            }
            const uint32_t W[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                // slot s holds x at in-group offsets {s, s+8} (b0) and {s+4, s+12} (b1)
                const uint32_t sel = (s & 1) ? 0x7632u : 0x5410u;
                const uint32_t b0 = __byte_perm(W[s >> 1], W[(s >> 1) + 4], sel);
                const uint32_t b1 = __byte_perm(W[(s >> 1) + 2], W[(s >> 1) + 6], sel);
                xs[xslot<NT8>(grp, w, s, m >> 3, tt, m & 7)] = make_uint2(b0, b1);
            }
        }
    }
    __syncthreads();

    // 3. main loop over the 128-k groups of this CTA
    float acc[MT][NT8][4];
    float accg[MT][NT8][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

    const uint8_t *rowp[MT][2];
    const uint16_t *srow[MT][2];
    bool rowok[MT][2];
    const int ngk = a.K >> 7;  // scale groups per row (group mode)
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + (warp * MT + i) * 16 + g + 8 * h;
            rowok[i][h] = n < a.N;
            const int nn = rowok[i][h] ? n : 0;
            rowp[i][h] = a.packed + (int64_t)nn * Kq + (kb >> 2) + 8 * t;
            srow[i][h] = a.scale + (GROUP ? (int64_t)nn * ngk + (kb >> 7) : 0);
        }

    uint2 ring[D][MT][2];
    uint16_t sring[D][MT][2];
    auto load_group = [&](int slot, int grp) {
        const bool kin = grp < ng && (grp * 128 + 32 * t) < klen;
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                ring[slot][i][h] = (kin && rowok[i][h]) ? ldg_nc_v2(rowp[i][h] + grp * 32)
                                                        : make_uint2(0, 0);
                if constexpr (GROUP)
                    sring[slot][i][h] = (grp < ng && rowok[i][h]) ? srow[i][h][grp] : (uint16_t)0;
            }
    };
#pragma unroll
    for (int d = 0; d < D; ++d) load_group(d, d);

    for (int g0 = 0; g0 < ng; g0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int grp = g0 + d;
            if (grp < ng) {
                uint2 cw[MT][2];
                float sc[MT][2];
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        cw[i][h] = ring[d][i][h];
                        if constexpr (GROUP) sc[i][h] = h2f(sring[d][i][h]);
                    }
                load_group(d, grp + D);
                if constexpr (GROUP) {
#pragma unroll
                    for (int i = 0; i < MT; ++i)
#pragma unroll
                        for (int j = 0; j < NT8; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) accg[i][j][e] = 0.f;
                }
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    uint32_t zg[MT], zh[MT];
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        zg[i] = sign_nz(w ? cw[i][0].y : cw[i][0].x);
                        zh[i] = sign_nz(w ? cw[i][1].y : cw[i][1].x);
                    }
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        uint2 b[NT8];
#pragma unroll
                        for (int j = 0; j < NT8; ++j) b[j] = xs[xslot<NT8>(grp, w, s, j, t, g)];
#pragma unroll
                        for (int i = 0; i < MT; ++i) {
                            const uint32_t a0 = pair2(zg[i], s), a1 = pair2(zh[i], s);
                            const uint32_t a2 = pair2(zg[i], s + 4), a3 = pair2(zh[i], s + 4);
#pragma unroll
                            for (int j = 0; j < NT8; ++j) {
                                if constexpr (GROUP)
                                    mma16816<BF>(accg[i][j], a0, a1, a2, a3, b[j].x, b[j].y);
                                else
                                    mma16816<BF>(acc[i][j], a0, a1, a2, a3, b[j].x, b[j].y);
                            }
                        }
                    }
                }
                if constexpr (GROUP) {
#pragma unroll
                    for (int i = 0; i < MT; ++i)
#pragma unroll
                        for (int j = 0; j < NT8; ++j) {
                            acc[i][j][0] = fmaf(sc[i][0], accg[i][j][0], acc[i][j][0]);
                            acc[i][j][1] = fmaf(sc[i][0], accg[i][j][1], acc[i][j][1]);
                            acc[i][j][2] = fmaf(sc[i][1], accg[i][j][2], acc[i][j][2]);
                            acc[i][j][3] = fmaf(sc[i][1], accg[i][j][3], acc[i][j][3]);
                        }
                }
            }
        }
    }

    // 4. partial tile -> shared memory, [RT rows][MP tokens] fp32
    __syncthreads();  // x fragments are no longer needed; reuse the space
    float *part = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
            const int r = (warp * MT + i) * 16 + g;
            *reinterpret_cast<float2 *>(&part[r * MP + j * 8 + 2 * t]) =
                make_float2(acc[i][j][0], acc[i][j][1]);
            *reinterpret_cast<float2 *>(&part[(r + 8) * MP + j * 8 + 2 * t]) =
                make_float2(acc[i][j][2], acc[i][j][3]);
        }

    // 5. split-K reduction across the cluster (rank order), scale, store
    const int SK = gridDim.y;
    int rank = 0;
    if (SK > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        rank = (int)cluster.block_rank();
    } else {
        __syncthreads();
    }
    const int r_begin = (RT * rank) / SK, r_end = (RT * (rank + 1)) / SK;
    const int rows_mine = r_end - r_begin;
    const int total = rows_mine * a.M;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int r = r_begin + idx % rows_mine;
        const int m = idx / rows_mine;
        const int n = n0 + r;
        if (n >= a.N) continue;
        float v = 0.f;
        if (SK > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            for (int q = 0; q < SK; ++q) v += cluster.map_shared_rank(part, q)[r * MP + m];
        } else {
            v = part[r * MP + m];
        }
        v *= 0.5f;  // the decoded operand is 2*t
        if constexpr (!GROUP) v *= h2f(a.scale[n]);
        OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, v);
    }
    if (SK > 1) cg::this_cluster().sync();  // keep our partials alive for readers
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int NT8, int MT, bool BF, bool GROUP, int OUT>
static cudaError_t launch_cfg(const SkinnyArgs &a, int rows_per_cta, int sk, size_t smem,
                              cudaStream_t st, bool pdl) {
    constexpr int D = (MT == 1) ? 4 : 2;
    auto kern = skinny_mma_kernel<NT8, MT, D, BF, GROUP, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + rows_per_cta - 1) / rows_per_cta), (unsigned)sk, 1);
    cfg.blockDim = dim3(kSkinnyThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (sk > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)sk;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int NT8, int MT, bool BF, bool GROUP>
static cudaError_t dispatch_out(const SkinnyArgs &a, int out_dtype, int rpc, int sk, size_t smem,
                                cudaStream_t st, bool pdl) {
    switch (out_dtype) {
    case 0: return launch_cfg<NT8, MT, BF, GROUP, 0>(a, rpc, sk, smem, st, pdl);
    case 1: return launch_cfg<NT8, MT, BF, GROUP, 1>(a, rpc, sk, smem, st, pdl);
    default: return launch_cfg<NT8, MT, BF, GROUP, 2>(a, rpc, sk, smem, st, pdl);
    }
}

template <int NT8, int MT>
static cudaError_t dispatch_types(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                                  int rpc, int sk, size_t smem, cudaStream_t st, bool pdl) {
    if (bf) {
        return group ? dispatch_out<NT8, MT, true, true>(a, out_dtype, rpc, sk, smem, st, pdl)
                     : dispatch_out<NT8, MT, true, false>(a, out_dtype, rpc, sk, smem, st, pdl);
    }
    return group ? dispatch_out<NT8, MT, false, true>(a, out_dtype, rpc, sk, smem, st, pdl)
                 : dispatch_out<NT8, MT, false, false>(a, out_dtype, rpc, sk, smem, st, pdl);
}

SkinnyPlan plan_skinny(int64_t M, int64_t N, int64_t K, int sm_count) {
    SkinnyPlan p{};
    p.nt8 = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
    p.mt = p.nt8 == 1 ? 1 : 2;
    p.rows_per_cta = 16 * p.mt * (kSkinnyThreads / 32);
    const int64_t row_tiles = (N + p.rows_per_cta - 1) / p.rows_per_cta;
    const int64_t ngk = (K + 127) / 128;  // 128-k groups (last may be half)
    const int64_t want_ctas = 2LL * sm_count;
    int64_t sk = (want_ctas + row_tiles - 1) / row_tiles;
    if (sk > kSkinnyMaxCluster) sk = kSkinnyMaxCluster;
    if (sk > ngk) sk = ngk;
    if (sk < 1) sk = 1;
    int64_t gpc = (ngk + sk - 1) / sk;  // groups per CTA
    // shared memory: x fragments (2048 B per group per n-tile) or the partial tile
    const int64_t per_group = 2048LL * p.nt8;
    while (gpc * per_group > kSkinnyMaxSmem && sk < kSkinnyMaxCluster) {
        ++sk;
        gpc = (ngk + sk - 1) / sk;
    }
    sk = (ngk + gpc - 1) / gpc;  // no CTA without work
    if (sk < 1) sk = 1;
    p.sk = (int)sk;
    p.kc = (int)(gpc * 128);
    const int64_t xbytes = gpc * per_group;
    const int64_t pbytes = (int64_t)p.rows_per_cta * 8 * p.nt8 * 4;
    p.smem = (size_t)(xbytes > pbytes ? xbytes : pbytes);
    p.ok = xbytes <= kSkinnyMaxSmem && M <= 32;
    return p;
}

cudaError_t launch_skinny(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                          const SkinnyPlan &p, cudaStream_t st, bool pdl) {
    SkinnyArgs b = a;
    b.kc = p.kc;
    switch (p.nt8) {
    case 1: return dispatch_types<1, 1>(b, bf, group, out_dtype, p.rows_per_cta, p.sk, p.smem, st, pdl);
    case 2: return dispatch_types<2, 2>(b, bf, group, out_dtype, p.rows_per_cta, p.sk, p.smem, st, pdl);
    default: return dispatch_types<4, 2>(b, bf, group, out_dtype, p.rows_per_cta, p.sk, p.smem, st, pdl);
    }
}

}  // namespace tl
