// kern_skinny.cu -- decode-shaped ternary linear on register-fed warp MMAs.
//
// Serves M <= 2 tokens by default (the tcgen05 kernel in kern_skinny_tc.cu
// takes M >= 3): its 16-row CTAs need no split K for most layers, which keeps
// each CTA's critical path short -- the quantity that decides the time of a
// single-token decode layer.  It can serve any M <= 32 when forced.
//
// out[m,n] = sum_k t[n,k] x[m,k], scaled per output channel
// (Qwen2.5-7B ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or
// per 128-wide K group ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §3.1, §4.2), with t decoded from the packed 2-bit codes
// (same page §3.1).
//
// Design (memory-bound: every packed byte is read from HBM exactly once).
//  * Work split: a CTA owns a block of RB = 16*TPC weight rows x KB of K
//    (KB a multiple of 128).  Its packed rows are fetched as 1-D bulk async
//    copies (one per row) into shared memory, all issued at kernel entry and
//    tracked by one mbarrier.  With TL_FLAG_STATIC_WEIGHTS they are issued
//    before griddepcontrol.wait, so under programmatic dependent launch a
//    layer's weight stream runs while the previous kernel finishes.
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
//  * 8 warps per CTA: 8/TPC warps share each 16-row tile and split its K
//    range; their partials are summed in a fixed order through shared memory.
//  * Group scale: per-group fp32 partial in registers, folded into the total
//    with s[n,g] at the group boundary.  Channel scale: once in the epilogue.
//  * Split K across the CTAs of a thread-block cluster (<= 8): each CTA pushes
//    its partial rows into the owning CTA's shared memory (distributed shared
//    memory stores), one cluster barrier publishes them, and the owner sums
//    them in rank order 0..SK-1, so the result is bit-identical run to run.
//    No global scratch.
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

// Slot of the staged x fragment for (group, word, step, n-tile, lane (g, t)).
// One slot = 8 bytes = the B fragment {b0, b1} of one lane.  ts is the token
// stride: 8, or M rounded up to a power of two when M < 8 (lanes of padding
// tokens read nothing), so the lanes of one (group, word, step, n-tile) read
// 32*ts contiguous bytes.
template <int NT8>
__device__ __forceinline__ int xslot(int grp, int w, int s, int nt, int t, int g, int ts) {
    return ((((grp * 2 + w) * 4 + s) * NT8 + nt) * 4 + t) * ts + g;
}

constexpr int kNW = kSkinnyWarps;

template <int NT8, int TPC, bool BF, bool GROUP, int OUT>
__global__ void __launch_bounds__(32 * kNW) skinny_mma_kernel(SkinnyArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RB = 16 * TPC;     // rows per CTA
    constexpr int KWS = kNW / TPC;   // warps per 16-row tile (split its K)
    constexpr int MP = 8 * NT8;      // padded tokens
    constexpr int NTH = 32 * kNW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * RB;
    const int kb = blockIdx.y * a.kc;
    const int ke = min(a.K, kb + a.kc);
    const int klen = max(ke - kb, 0);
    const int ng = (klen + 127) >> 7;  // 128-k groups of this CTA (the last may be half)
    const int64_t Kq = a.K >> 2;       // bytes per packed row
    const int SK = gridDim.y;
    const int valid_rows = max(0, min(RB, a.N - n0));

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint8_t *codes = smem + 16;                                   // [RB][row_stride]
    uint2 *xs = reinterpret_cast<uint2 *>(smem + a.x_off);        // fragment-ordered x
    float *wpart = reinterpret_cast<float *>(smem + a.red_off);   // [kNW][16][MP]
    float *recv = reinterpret_cast<float *>(smem + a.recv_off);   // [SK][rows_max][MP]

    if (SK > 1) cluster_arrive_relaxed();  // cluster phase 1: this CTA runs
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    // 1. weight stream: one bulk copy per packed row segment
    auto issue_weights = [&]() {
        if (warp == 0) {
            const uint32_t row_bytes = (uint32_t)(klen >> 2);
            if (lane == 0) mbar_arrive_expect_tx(bar, row_bytes * (uint32_t)valid_rows);
            __syncwarp();
            if (row_bytes > 0)
                for (int r = lane; r < valid_rows; r += 32)
                    bulk_g2s(codes + (size_t)r * a.row_stride,
                             a.packed + (int64_t)(n0 + r) * Kq + (kb >> 2), row_bytes, bar);
        }
    };
    const bool early_w = (a.flags & kSkinnyStaticWeights) != 0;
    if (early_w) issue_weights();
    if (!(a.flags & (kSkinnyTriggerLate | kSkinnyTriggerNever))) pdl_launch_dependents();
    pdl_wait();  // x / out may be produced / consumed by the previous kernel
    if (!early_w) issue_weights();

    // per-channel scales of the outputs this thread stores (loaded early)
    int rank = 0;
    if (SK > 1) rank = (int)cg::this_cluster().block_rank();
    const int r_begin = (RB * rank) / SK, r_end = (RB * (rank + 1)) / SK;
    const int rows_mine = r_end - r_begin;
    const int total = rows_mine * a.M;
    constexpr int EPT = (RB * 32 + NTH - 1) / NTH;  // outputs per thread (M <= 32)
    float osc[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int idx = threadIdx.x + e * NTH;
        const int n = n0 + r_begin + (idx < total ? idx % rows_mine : 0);
        osc[e] = (!GROUP && idx < total && n < a.N) ? h2f(a.scale[n]) : 1.f;
    }

    // 2. stage x[:M, kb:ke) in fragment order (padding tokens are never read:
    //    their lanes feed zero B fragments); one batch = one memory round trip
    {
        constexpr int UB = 4;
        const int upm = ng * 8;  // units per token: (group, t, word), 16 k each
        const int units = a.M * upm;
        for (int base = 0; base < units; base += UB * NTH) {
            uint4 lo[UB], hi[UB];
#pragma unroll
            for (int q = 0; q < UB; ++q) {
                const int u = base + q * NTH + threadIdx.x;
                lo[q] = make_uint4(0, 0, 0, 0);
                hi[q] = lo[q];
                if (u < units) {
                    const int m = u / upm, r = u - m * upm;
                    const int k = kb + (r >> 3) * 128 + 32 * ((r >> 1) & 3) + 16 * (r & 1);
                    if (k < ke) {
                        const uint4 *src =
                            reinterpret_cast<const uint4 *>(a.x + (int64_t)m * a.K + k);
                        lo[q] = src[0];
                        hi[q] = src[1];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < UB; ++q) {
                const int u = base + q * NTH + threadIdx.x;
                if (u < units) {
                    const int m = u / upm, r = u - m * upm;
                    const int grp = r >> 3, tt = (r >> 1) & 3, w = r & 1;
                    const uint32_t W[8] = {lo[q].x, lo[q].y, lo[q].z, lo[q].w,
                                           hi[q].x, hi[q].y, hi[q].z, hi[q].w};
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        // slot s holds x at in-group offsets {s, s+8} (b0), {s+4, s+12} (b1)
                        const uint32_t sel = (s & 1) ? 0x7632u : 0x5410u;
                        const uint32_t b0 = __byte_perm(W[s >> 1], W[(s >> 1) + 4], sel);
                        const uint32_t b1 = __byte_perm(W[(s >> 1) + 2], W[(s >> 1) + 6], sel);
                        xs[xslot<NT8>(grp, w, s, m >> 3, tt, m & 7, a.xts)] = make_uint2(b0, b1);
                    }
                }
            }
        }
    }
    __syncthreads();

    // 3. wait for this CTA's weights (bounded: a stuck copy sets the status
    //    word and the CTA skips its work after one more bounded wait)
    bool ok = mbar_wait_bounded(bar, 0);
    if (!ok) {
        if (a.status) atomicExch(a.status, kStatusTimeout);
        mbar_wait_bounded(bar, 0);
    }
    ok = __syncthreads_and(ok);

    // 4. main loop: warp -> (tile, K part); rows g and g+8 of the tile
    const int tile = warp / KWS, kpart = warp % KWS;
    const int gb = (ng * kpart) / KWS, ge = (ng * (kpart + 1)) / KWS;
    constexpr int NC = (NT8 == 1) ? 2 : 1;  // independent MMA chains
    float acc[NC][NT8][4];
    float accg[NC][NT8][4];
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[c][j][e] = 0.f;
    bool tok_ok[NT8];
#pragma unroll
    for (int j = 0; j < NT8; ++j) tok_ok[j] = (j * 8 + g) < a.M;
    const int row_g = tile * 16 + g;
    const uint8_t *cg0 = codes + (size_t)row_g * a.row_stride + 8 * t;
    const uint8_t *cg8 = cg0 + (size_t)8 * a.row_stride;
    const int ngk = a.K >> a.gshift;  // scale groups per row (group mode, G = 128 or 256)
    const bool ok0 = n0 + row_g < a.N, ok8 = n0 + row_g + 8 < a.N;
    const uint16_t *s0 = a.scale + (GROUP ? (int64_t)(ok0 ? n0 + row_g : 0) * ngk : 0);
    const uint16_t *s8 = a.scale + (GROUP ? (int64_t)(ok8 ? n0 + row_g + 8 : 0) * ngk : 0);
    // 128-k group grp of this warp's range belongs to scale group ((kb >> 7) + grp) >> gsh
    const int g0 = kb >> 7, gsh = a.gshift - 7;

    uint16_t sn0 = 0, sn8 = 0;  // next group's scales (group mode)
    if (GROUP && gb < ge) {
        sn0 = ok0 ? s0[(g0 + gb) >> gsh] : (uint16_t)0;
        sn8 = ok8 ? s8[(g0 + gb) >> gsh] : (uint16_t)0;
    }
    for (int grp = ok ? gb : ge; grp < ge; ++grp) {
        const uint2 w0 = *reinterpret_cast<const uint2 *>(cg0 + grp * 32);
        const uint2 w8 = *reinterpret_cast<const uint2 *>(cg8 + grp * 32);
        float sc0 = 0.f, sc8 = 0.f;
        if constexpr (GROUP) {
            sc0 = h2f(sn0);
            sc8 = h2f(sn8);
            if (grp + 1 < ge) {
                sn0 = ok0 ? s0[(g0 + grp + 1) >> gsh] : (uint16_t)0;
                sn8 = ok8 ? s8[(g0 + grp + 1) >> gsh] : (uint16_t)0;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int j = 0; j < NT8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) accg[c][j][e] = 0.f;
        }
        const uint2 *xg = xs + (size_t)grp * 32 * a.xts * NT8;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const uint32_t zg = sign_nz(w ? w0.y : w0.x);
            const uint32_t zh = sign_nz(w ? w8.y : w8.x);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint2 b[NT8];
#pragma unroll
                for (int j = 0; j < NT8; ++j)
                    b[j] = tok_ok[j] ? xg[xslot<NT8>(0, w, s, j, t, g, a.xts)] : make_uint2(0, 0);
                const uint32_t a0 = pair2(zg, s), a1 = pair2(zh, s);
                const uint32_t a2 = pair2(zg, s + 4), a3 = pair2(zh, s + 4);
#pragma unroll
                for (int j = 0; j < NT8; ++j) {
                    if constexpr (GROUP)
                        mma16816<BF>(accg[s % NC][j], a0, a1, a2, a3, b[j].x, b[j].y);
                    else
                        mma16816<BF>(acc[s % NC][j], a0, a1, a2, a3, b[j].x, b[j].y);
                }
            }
        }
        if constexpr (GROUP) {
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    p[e] = accg[0][j][e];
                    if constexpr (NC == 2) p[e] += accg[NC - 1][j][e];
                }
                acc[0][j][0] = fmaf(sc0, p[0], acc[0][j][0]);
                acc[0][j][1] = fmaf(sc0, p[1], acc[0][j][1]);
                acc[0][j][2] = fmaf(sc8, p[2], acc[0][j][2]);
                acc[0][j][3] = fmaf(sc8, p[3], acc[0][j][3]);
            }
        }
    }
    if (a.flags & kSkinnyTriggerLate) pdl_launch_dependents();
    if constexpr (!GROUP && NC == 2) {
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[0][j][e] += acc[NC - 1][j][e];
    }

    // 5. warp partials -> shared memory; the KWS warps of a tile are summed
    //    in a fixed order into the slot of the tile's first warp.  The CTA
    //    partial of row r then lives at part(r) below.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float *dst = wpart + ((size_t)warp * 16 + g + 8 * h) * MP;
#pragma unroll
        for (int j = 0; j < NT8; ++j)
            *reinterpret_cast<float2 *>(dst + j * 8 + 2 * t) =
                make_float2(acc[0][j][2 * h], acc[0][j][2 * h + 1]);
    }
    auto part = [&](int r) { return wpart + ((size_t)(r >> 4) * KWS * 16 + (r & 15)) * MP; };
    if constexpr (KWS > 1) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < RB * MP; idx += NTH) {
            const int r = idx / MP, m = idx - r * MP;
            const float *src = part(r) + m;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < KWS; ++w) v += src[(size_t)w * 16 * MP];
            part(r)[m] = v;  // element read and written by this thread only
        }
    }

    // 6. split-K across the cluster: push each row's CTA partial into slot
    //    `rank` of the owning CTA's receive buffer; one cluster barrier
    //    publishes them.  Rank q owns rows [RB*q/SK, RB*(q+1)/SK).
    const int rows_max = (RB + SK - 1) / SK;
    if (SK > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        if constexpr (KWS == 1) __syncthreads();
        cluster_wait();  // every CTA of the cluster has started
        for (int idx = threadIdx.x; idx < RB * MP; idx += NTH) {
            const int r = idx / MP, m = idx - r * MP;
            int o = (r * SK) / RB;
            while (o > 0 && r < (RB * o) / SK) --o;
            while (o + 1 < SK && r >= (RB * (o + 1)) / SK) ++o;
            cluster.map_shared_rank(recv, o)[((size_t)rank * rows_max + (r - (RB * o) / SK)) * MP + m] =
                part(r)[m];
        }
        cluster.sync();
    } else {
        __syncthreads();
    }

    // 7. sum the CTA partials in rank order, scale, convert, store
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int idx = threadIdx.x + e * NTH;
        if (idx >= total) break;
        const int rr = idx % rows_mine;
        const int m = idx / rows_mine;
        const int n = n0 + r_begin + rr;
        if (n >= a.N || !ok) continue;
        float v = 0.f;
        if (SK > 1) {
            for (int q = 0; q < SK; ++q) v += recv[((size_t)q * rows_max + rr) * MP + m];
        } else {
            v = part(rr)[m];
        }
        v *= 0.5f;  // the decoded operand is 2*t
        if constexpr (!GROUP) v *= osc[e];
        OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, v);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int NT8, int TPC, bool BF, bool GROUP, int OUT>
static cudaError_t launch_cfg(const SkinnyArgs &a, const SkinnyPlan &p, cudaStream_t st,
                              bool pdl) {
    auto kern = skinny_mma_kernel<NT8, TPC, BF, GROUP, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + p.rows_per_cta - 1) / p.rows_per_cta), (unsigned)p.sk, 1);
    cfg.blockDim = dim3(32 * kNW, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.sk > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)p.sk;
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

template <int NT8, int TPC, bool BF, bool GROUP>
static cudaError_t dispatch_out(const SkinnyArgs &a, int out_dtype, const SkinnyPlan &p,
                                cudaStream_t st, bool pdl) {
    switch (out_dtype) {
    case 0: return launch_cfg<NT8, TPC, BF, GROUP, 0>(a, p, st, pdl);
    case 1: return launch_cfg<NT8, TPC, BF, GROUP, 1>(a, p, st, pdl);
    default: return launch_cfg<NT8, TPC, BF, GROUP, 2>(a, p, st, pdl);
    }
}

template <int NT8, int TPC>
static cudaError_t dispatch_types(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                                  const SkinnyPlan &p, cudaStream_t st, bool pdl) {
    if (bf)
        return group ? dispatch_out<NT8, TPC, true, true>(a, out_dtype, p, st, pdl)
                     : dispatch_out<NT8, TPC, true, false>(a, out_dtype, p, st, pdl);
    return group ? dispatch_out<NT8, TPC, false, true>(a, out_dtype, p, st, pdl)
                 : dispatch_out<NT8, TPC, false, false>(a, out_dtype, p, st, pdl);
}

template <int NT8>
static cudaError_t dispatch_tpc(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                                const SkinnyPlan &p, cudaStream_t st, bool pdl) {
    switch (p.rows_per_cta / 16) {
    case 1: return dispatch_types<NT8, 1>(a, bf, group, out_dtype, p, st, pdl);
    case 2: return dispatch_types<NT8, 2>(a, bf, group, out_dtype, p, st, pdl);
    case 4: return dispatch_types<NT8, 4>(a, bf, group, out_dtype, p, st, pdl);
    default: return dispatch_types<NT8, 8>(a, bf, group, out_dtype, p, st, pdl);
    }
}

static SkinnyPlan make_plan(int64_t M, int64_t N, int64_t K, int64_t rb, int64_t sk) {
    SkinnyPlan p{};
    p.nt8 = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
    p.rows_per_cta = (int)rb;
    const int64_t G = (K + 127) / 128;  // 128-k groups (last may be half)
    if (sk > kSkinnyMaxCluster) sk = kSkinnyMaxCluster;
    if (sk > G) sk = G;
    if (sk < 1) sk = 1;
    const int64_t gpc = (G + sk - 1) / sk;  // groups per CTA
    sk = (G + gpc - 1) / gpc;               // no CTA without work
    const int64_t mp = 8LL * p.nt8;
    int64_t ts = 8;
    if (M < 8) ts = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    p.xts = (int)ts;
    const int64_t row_stride = 32 * (gpc | 1);  // odd multiple of 32 B: conflict-free reads
    const int64_t codes = rb * row_stride;
    const int64_t xbytes = gpc * 256LL * ts * p.nt8;  // 8 slots of 8 B per (word, step, t)
    const int64_t wbytes = (int64_t)kNW * 16 * mp * 4;
    const int64_t rows_max = (rb + sk - 1) / sk;
    const int64_t rbytes = sk > 1 ? sk * rows_max * mp * 4 : 0;
    p.sk = (int)sk;
    p.kc = (int)(gpc * 128);
    p.row_stride = (int)row_stride;
    p.x_off = (int)(16 + codes);
    p.red_off = (int)(16 + codes + xbytes);
    p.recv_off = (int)(16 + codes + xbytes + wbytes);
    p.smem = (size_t)(16 + codes + xbytes + wbytes + rbytes);
    p.ok = (int64_t)p.smem <= kSkinnyMaxSmem && M <= 32 && M >= 1;
    return p;
}

SkinnyPlan plan_skinny(int64_t M, int64_t N, int64_t K, int sm_count, int force_sk) {
    // Rows per CTA: large enough that the staged x slice (2*M bytes per k) is
    // small next to the weight slice (RB/4 bytes per k), capped at 128.
    int64_t rb = 16;
    while (rb < 128 && rb < 16 * M) rb *= 2;
    const int64_t G = (K + 127) / 128;
    auto choose_sk = [&](int64_t rbv) {
        const int64_t R = (N + rbv - 1) / rbv;
        int64_t sk = R >= sm_count ? 1 : (sm_count + R - 1) / R;
        if (force_sk > 0) sk = force_sk;
        return sk;
    };
    SkinnyPlan p = make_plan(M, N, K, rb, choose_sk(rb));
    // keep one CTA within the budget that lets two CTAs share an SM
    while (p.smem > (size_t)kSkinnyTargetSmem && p.sk < kSkinnyMaxCluster && p.sk < G)
        p = make_plan(M, N, K, rb, p.sk + 1);
    while ((!p.ok || p.smem > (size_t)kSkinnyTargetSmem) && rb > 16) {
        rb /= 2;
        p = make_plan(M, N, K, rb, choose_sk(rb));
        while (p.smem > (size_t)kSkinnyTargetSmem && p.sk < kSkinnyMaxCluster && p.sk < G)
            p = make_plan(M, N, K, rb, p.sk + 1);
    }
    return p;
}

cudaError_t launch_skinny(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                          const SkinnyPlan &p, cudaStream_t st, bool pdl) {
    SkinnyArgs b = a;
    b.kc = p.kc;
    b.row_stride = p.row_stride;
    b.x_off = p.x_off;
    b.red_off = p.red_off;
    b.recv_off = p.recv_off;
    b.xts = p.xts;
    if (p.nt8 == 1) return dispatch_tpc<1>(b, bf, group, out_dtype, p, st, pdl);
    if (p.nt8 == 2) return dispatch_tpc<2>(b, bf, group, out_dtype, p, st, pdl);
    return dispatch_tpc<4>(b, bf, group, out_dtype, p, st, pdl);
}

}  // namespace tl
