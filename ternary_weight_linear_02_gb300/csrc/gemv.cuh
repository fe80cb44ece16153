// gemv.cuh -- the decode-shaped kernel (M <= 16 tokens): fused unpack and
// accumulate on register-fed warp MMAs, packed weights staged by TMA.  Shared
// by kern_gemv.cu (plain output) and kern_gemv_silu.cu (SiLU-gated gate/up).
//
// out[m,n] = sum_k t[n,k] x[m,k], scaled per output channel (Qwen2.5-7B
// ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or per K group of
// G = 64, 128 or 256 weights ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §1.1, §3.1, §4.2; the "Bonsai 2 27B" port, §4.2, §5.2),
// t decoded with the code table of the first page's §3.1.
//
// Memory-bound design: every packed byte is read from HBM once and decoded
// once, in registers; the decoded +-1/0 weights are fed straight from
// registers to mma.sync (m16n8k16, fp32 accumulate), whose cost does not grow
// with the number of tokens.  Nothing is handed from one warp to another
// inside the main loop.
//
// Work split.  A CTA owns RB = 16*RG weight rows x a K range (a multiple of 256
// k); the K ranges of a row block are the CTAs of one thread-block cluster
// (split K <= 8).  The K range is cut into 64-k columns; warp w (of 8) takes
// the columns at offset 64*(w%4) of every other 256-k stage (stages of parity
// w/4), and for each of its columns runs every row group of the CTA through
// that column with the column's x fragments held in registers (loaded straight
// from global memory one column ahead, so x is never staged or re-read per
// row).  Warp 8 is the producer: one 2-D TMA per 256-k stage (64 B x RB rows,
// 64-byte swizzle) into a ring of shared-memory stages; with static weights
// the ring is filled before griddepcontrol.wait, so under programmatic
// dependent launch a layer's weights stream while the previous kernel ends.
//
// Operand mapping for mma.m16n8k16 (A = 16 weight rows, B = x^T, 8 tokens per
// n-tile).  Lane (g = lane/4, c = lane%4) reads the 32-bit word c (16 codes) of
// the column for rows g and g+8.  After sign_nz, pair2(z, i) holds codes i and
// i+8 as {2t, 2t} in one f16x2/bf16x2 register (exact: +-2 or +-0).  MMA i of
// the column (i = 0..3) takes pair2(z, i) as the k-slots (2c, 2c+1) and
// pair2(z, i+4) as (2c+8, 2c+9); the lane's B registers hold x at the same k
// (16c + i, +8) and (16c + i + 4, +12).  So one MMA covers 16 k of one 64-k
// column: a group scale (G >= 64) is constant over it.
//
// Scales: channel -> once in the epilogue (times 0.5: the operand is 2t);
// group -> each column's MMAs start from zero and are folded into the row's
// fp32 total with that group's scale.
//
// Reduction: the 8 warps' partial tiles are summed in warp order through the
// (then idle) ring; split K across the cluster pushes each CTA's partial rows
// into the owning CTA's shared memory (st.shared::cluster) and the owner sums
// them in rank order.  The same inputs give bit-identical outputs, and
// nothing is allocated.
//
// Every mbarrier wait is bounded (give-up time from the launch arguments).  A
// wait that gives up sets the device status word; the CTA stops, the producer
// still waits (with the long default limit) for its copies in flight, every CTA
// still joins its cluster barriers, and no output of the call is written.
#pragma once

#include <cuda.h>

#include "kernels.h"
#include "tc.cuh"

namespace tl {
namespace gemv {

constexpr int kWarps = 8;                   // consumer warps
constexpr int kThreads = 32 * (kWarps + 1); // + the producer warp
constexpr int kStageK = 256;                // k per weight stage: a 64-byte box per row
constexpr int kRingBytes = 96 * 1024;
constexpr int kMaxStages = 24;

template <int NT8>
struct Cfg {
    static constexpr int RGMAX = NT8 == 1 ? 8 : 4;  // row groups per CTA (16 rows each)
    static constexpr int MP = 8 * NT8;              // padded tokens
    static constexpr int RBMAX = 16 * RGMAX;
    // split-K receive rows: sk * ceil(RB / sk) <= RB + 8 (or gated: 2 * sk * ceil(RB/2 / sk))
    static constexpr int RECV_FLOATS = (RBMAX + 16) * MP;
    static constexpr int RECV_OFF = kRingBytes;
    static constexpr int FLAG_OFF = RECV_OFF + RECV_FLOATS * 4;       // 8 abort flags (one per rank)
    static constexpr int BAR_OFF = FLAG_OFF + 64;
    static constexpr int SMEM = BAR_OFF + (2 * kMaxStages + 2) * 8 + 16 + 1024;
    static_assert(kWarps * RBMAX * MP * 4 <= kRingBytes, "reduction tiles fit in the ring");
    static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
};

// ------------------------------------------------------------------ device helpers
template <bool BF>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// D = A * B (accumulator starts from zero)
template <bool BF>
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    }
}

__device__ __forceinline__ uint32_t cl_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cl_st_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

// x[n, k .. k+16) of token n as the four (b0, b1) pairs of MMA i = 0..3:
// b0 = (x[k+i], x[k+i+8]), b1 = (x[k+i+4], x[k+i+12])
__device__ __forceinline__ void x_frag(const uint4 &lo, const uint4 &hi, uint32_t (&b)[4][2]) {
    // lo = (x0 x1)(x2 x3)(x4 x5)(x6 x7), hi = (x8 x9)...(x14 x15)
    b[0][0] = __byte_perm(lo.x, hi.x, 0x5410);  // x0, x8
    b[1][0] = __byte_perm(lo.x, hi.x, 0x7632);  // x1, x9
    b[2][0] = __byte_perm(lo.y, hi.y, 0x5410);  // x2, x10
    b[3][0] = __byte_perm(lo.y, hi.y, 0x7632);  // x3, x11
    b[0][1] = __byte_perm(lo.z, hi.z, 0x5410);  // x4, x12
    b[1][1] = __byte_perm(lo.z, hi.z, 0x7632);  // x5, x13
    b[2][1] = __byte_perm(lo.w, hi.w, 0x5410);  // x6, x14
    b[3][1] = __byte_perm(lo.w, hi.w, 0x7632);  // x7, x15
}

template <int NT8, bool BF, bool GROUP, int OUT, bool SILU>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_kernel(const __grid_constant__ CUtensorMap tmw, GemvArgs a) {
    using C = Cfg<NT8>;
    constexpr int RGMAX = C::RGMAX, MP = C::MP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    float *recv = reinterpret_cast<float *>(smem + C::RECV_OFF);
    uint32_t *aflags = reinterpret_cast<uint32_t *>(smem + C::FLAG_OFF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + kMaxStages;
    uint64_t *never = empty + kMaxStages;  // nothing arrives on it (test stall)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(never + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int RG = a.rg, RB = 16 * RG, PH = RB / 2;
    const int rank = blockIdx.y, sk = gridDim.y;
    const int k0 = rank * a.kc, k1 = min(a.K, k0 + a.kc);
    const int nst = (k1 - k0 + kStageK - 1) / kStageK;
    const int stage_bytes = 64 * RB;
    // plain: rows [n0, n0 + RB); gated: gate rows [j0, j0 + PH) then up rows [nh + j0, ...)
    const int n0 = blockIdx.x * RB, j0 = blockIdx.x * PH;
    const long long lim = a.wait_limit;

    if (sk > 1) cl_arrive_relaxed();  // cluster phase 1: this CTA has started
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ws; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);  // the four warps that read a stage
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarps && lane == 0) tc::prefetch_tmap(&tmw);
    __syncthreads();
    pdl_launch_dependents();

    auto give_up = [&]() {
        *abort_flag = 1;
        if (a.status) atomicExch(a.status, kStatusTimeout);
    };

    float acc[RGMAX][NT8][4];
#pragma unroll
    for (int r = 0; r < RGMAX; ++r)
#pragma unroll
        for (int t = 0; t < NT8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][t][e] = 0.f;

    // weight row (global) of CTA row r, and whether it exists
    auto wrow = [&](int r) -> int {
        if constexpr (SILU) return r < PH ? j0 + r : a.nh + j0 + (r - PH);
        else return n0 + r;
    };

    if (warp == kWarps) {
        // ------------------------------------------------ producer: TMA of weight stages
        if (lane == 0) {
            if (!(a.flags & kGemvStaticWeights)) pdl_wait();
            int issued = 0;
            bool ok = true;
            for (int s = 0; s < nst; ++s) {
                const int slot = s % a.ws;
                if (s >= a.ws && (*abort_flag || !mbar_wait_bounded(&empty[slot], ((s / a.ws) - 1) & 1, lim))) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], (uint32_t)stage_bytes);
                uint8_t *dst = ring + (size_t)slot * stage_bytes;
                const int kb = (k0 >> 2) + s * 64;  // byte column of the stage
                if constexpr (SILU) {
                    tc::tma_load_2d(dst, &tmw, kb, j0, &full[slot]);
                    tc::tma_load_2d(dst + stage_bytes / 2, &tmw, kb, a.nh + j0, &full[slot]);
                } else {
                    tc::tma_load_2d(dst, &tmw, kb, n0, &full[slot]);
                }
                ++issued;
            }
            if (!ok) give_up();
            // drain: every copy still in flight lands before the ring is reused or the CTA exits
            for (int s = issued - a.ws < 0 ? 0 : issued - a.ws; s < issued; ++s)
                if (!mbar_wait_bounded(&full[s % a.ws], (s / a.ws) & 1)) give_up();
        }
    } else {
        // ------------------------------------------------ consumers
        pdl_wait();  // x (and out) belong to the previous kernel until here
        const int par = warp >> 2, cw = warp & 3;
        uint4 xr[NT8][2];
        uint32_t scn[RGMAX];  // next column's group scales: row g (low half), row g + 8 (high half)
        auto load_x = [&](int kcol) {
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                const int n = t * 8 + g;
                if (n < a.M && kcol < k1) {
                    const uint16_t *p = a.x + (int64_t)n * a.K + kcol + 16 * c;
                    xr[t][0] = ldg_nc_v4(p);
                    xr[t][1] = ldg_nc_v4(p + 8);
                } else {
                    xr[t][0] = make_uint4(0, 0, 0, 0);
                    xr[t][1] = xr[t][0];
                }
            }
        };
        auto load_sc = [&](int kcol) {
            if constexpr (GROUP) {
                const int ngk = a.K >> a.gshift, gi = kcol >> a.gshift;
#pragma unroll
                for (int r = 0; r < RGMAX; ++r) {
                    uint32_t v = 0;
                    if (r < RG && kcol < k1) {
                        const int lo = wrow(r * 16 + g), hi = wrow(r * 16 + g + 8);
                        const uint32_t slo = lo < a.N ? (uint32_t)a.scale[(int64_t)lo * ngk + gi] : 0u;
                        const uint32_t shi = hi < a.N ? (uint32_t)a.scale[(int64_t)hi * ngk + gi] : 0u;
                        v = slo | (shi << 16);
                    }
                    scn[r] = v;
                }
            }
        };
        int kcol = k0 + par * kStageK + cw * 64;
        load_x(kcol);
        load_sc(kcol);
        bool ok = true;
        if (a.flags & kGemvTestStall) {
            // testing aid: a wait on a barrier nothing arrives on runs out
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(never, 0, lim));
            if (!ok && lane == 0) give_up();
        }
        for (int s = par; ok && s < nst; s += 2) {
            const int slot = s % a.ws;
            const int kc_now = kcol;
            uint32_t b[NT8][4][2];
#pragma unroll
            for (int t = 0; t < NT8; ++t) x_frag(xr[t][0], xr[t][1], b[t]);
            uint32_t sc[RGMAX];
#pragma unroll
            for (int r = 0; r < RGMAX; ++r) sc[r] = GROUP ? scn[r] : 0u;
            kcol += 2 * kStageK;
            load_x(kcol);  // next column of this warp, in flight during this one
            load_sc(kcol);
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (s / a.ws) & 1, lim))) {
                if (lane == 0) give_up();
                ok = false;
                break;
            }
            if (*abort_flag) {
                ok = false;
                break;
            }
            if (kc_now < k1) {
                const uint8_t *st = ring + (size_t)slot * stage_bytes;
#pragma unroll
                for (int r = 0; r < RGMAX; ++r) {
                    if (r >= RG) break;
                    const int rlo = r * 16 + g, rhi = rlo + 8;
                    // 64-byte swizzle: 16-byte chunk j of row q sits at chunk j ^ ((q >> 1) & 3)
                    const uint32_t wlo = *reinterpret_cast<const uint32_t *>(
                        st + rlo * 64 + ((cw ^ ((rlo >> 1) & 3)) << 4) + 4 * c);
                    const uint32_t whi = *reinterpret_cast<const uint32_t *>(
                        st + rhi * 64 + ((cw ^ ((rhi >> 1) & 3)) << 4) + 4 * c);
                    const uint32_t zlo = sign_nz(wlo), zhi = sign_nz(whi);
                    if constexpr (GROUP) {
                        float d[NT8][4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t a0 = pair2(zlo, i), a1 = pair2(zhi, i);
                            const uint32_t a2 = pair2(zlo, i + 4), a3 = pair2(zhi, i + 4);
#pragma unroll
                            for (int t = 0; t < NT8; ++t) {
                                if (i == 0)
                                    mma16816_z<BF>(d[t], a0, a1, a2, a3, b[t][i][0], b[t][i][1]);
                                else
                                    mma16816<BF>(d[t], a0, a1, a2, a3, b[t][i][0], b[t][i][1]);
                            }
                        }
                        const float slo = h2f((uint16_t)(sc[r] & 0xffffu));
                        const float shi = h2f((uint16_t)(sc[r] >> 16));
#pragma unroll
                        for (int t = 0; t < NT8; ++t) {
                            acc[r][t][0] = fmaf(slo, d[t][0], acc[r][t][0]);
                            acc[r][t][1] = fmaf(slo, d[t][1], acc[r][t][1]);
                            acc[r][t][2] = fmaf(shi, d[t][2], acc[r][t][2]);
                            acc[r][t][3] = fmaf(shi, d[t][3], acc[r][t][3]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t a0 = pair2(zlo, i), a1 = pair2(zhi, i);
                            const uint32_t a2 = pair2(zlo, i + 4), a3 = pair2(zhi, i + 4);
#pragma unroll
                            for (int t = 0; t < NT8; ++t)
                                mma16816<BF>(acc[r][t], a0, a1, a2, a3, b[t][i][0], b[t][i][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    // ------------------------------------------------ reduction and epilogue
    __syncthreads();  // every stage consumed (or abandoned) and no copy in flight
    pdl_wait();       // (the producer warp stores below too)
    const bool aborted = *abort_flag != 0;
    float *red = reinterpret_cast<float *>(ring);  // [warp][RB][MP]
    if (warp < kWarps && !aborted) {
#pragma unroll
        for (int r = 0; r < RGMAX; ++r) {
            if (r >= RG) break;
            const int rlo = r * 16 + g;
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                float *p = red + ((size_t)warp * RB + rlo) * MP + t * 8 + 2 * c;
                *reinterpret_cast<float2 *>(p) = make_float2(acc[r][t][0], acc[r][t][1]);
                *reinterpret_cast<float2 *>(p + 8 * MP) = make_float2(acc[r][t][2], acc[r][t][3]);
            }
        }
    }
    __syncthreads();
    // the CTA's partial of row r, token m: the 8 warps summed in warp order
    auto part = [&](int r, int m) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[((size_t)w * RB + r) * MP + m];
        return v;
    };
    // final value (scaled) of stacked row r from its summed partial
    auto scaled = [&](int r, float v) {
        if constexpr (GROUP) {
            return 0.5f * v;  // group scales are folded in; the operand was 2t
        } else {
            const int n = wrow(r);
            return 0.5f * h2f(a.scale[n < a.N ? n : 0]) * v;
        }
    };

    if (sk == 1) {
        if (!aborted) {
            if constexpr (SILU) {
                for (int idx = threadIdx.x; idx < PH * a.M; idx += kThreads) {
                    const int m = idx / PH, p = idx - m * PH;
                    const int j = j0 + p;
                    if (j >= a.nh) continue;
                    const float gv = scaled(p, part(p, m)), uv = scaled(PH + p, part(PH + p, m));
                    OutStore<OUT>::st(a.out, (int64_t)m * a.nh + j, silu(gv) * uv);
                }
            } else {
                for (int idx = threadIdx.x; idx < RB * a.M; idx += kThreads) {
                    const int m = idx / RB, r = idx - m * RB;
                    const int n = n0 + r;
                    if (n >= a.N) continue;
                    OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, scaled(r, part(r, m)));
                }
            }
        }
        return;
    }

    // ------------------------------------------------ split K over the cluster
    // owner q holds rows [q*RB/sk, (q+1)*RB/sk) (gated: pairs [q*PH/sk, (q+1)*PH/sk))
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // phase 1: every peer runs
    const int span = SILU ? PH : RB;
    const int SL = (span + sk - 1) / sk;
    auto owner = [&](int p) {
        int q = (p * sk) / span;
        while (q + 1 < sk && ((q + 1) * span) / sk <= p) ++q;
        while ((q * span) / sk > p) --q;
        return q;
    };
    if (!aborted) {
        if constexpr (SILU) {
            for (int idx = threadIdx.x; idx < RB * a.M; idx += kThreads) {
                const int m = idx / RB, r = idx - m * RB;
                const int half = r >= PH ? 1 : 0, p = r - half * PH;
                const int q = owner(p), pp = p - (q * span) / sk;
                const float *slot = recv + ((size_t)(rank * 2 + half) * SL + pp) * MP + m;
                cl_st_f32(cl_map(smem_u32(slot), (uint32_t)q), part(r, m));
            }
        } else {
            for (int idx = threadIdx.x; idx < RB * a.M; idx += kThreads) {
                const int m = idx / RB, r = idx - m * RB;
                const int q = owner(r), rr = r - (q * span) / sk;
                const float *slot = recv + ((size_t)rank * SL + rr) * MP + m;
                cl_st_f32(cl_map(smem_u32(slot), (uint32_t)q), part(r, m));
            }
        }
    }
    if (threadIdx.x < (unsigned)sk)
        cl_st_u32(cl_map(smem_u32(aflags + rank), threadIdx.x), aborted ? 1u : 0u);
    cl_arrive_release();  // phase 2: every partial is in place
    cl_wait_acquire();
    bool any = false;
    for (int q = 0; q < sk; ++q) any = any || aflags[q] != 0;
    if (any) return;
    const int ps = (rank * span) / sk, plen = ((rank + 1) * span) / sk - ps;
    if constexpr (SILU) {
        for (int idx = threadIdx.x; idx < plen * a.M; idx += kThreads) {
            const int m = idx / plen, pp = idx - m * plen;
            const int p = ps + pp, j = j0 + p;
            if (j >= a.nh) continue;
            float gv = 0.f, uv = 0.f;
            for (int q = 0; q < sk; ++q) {
                gv += recv[((size_t)(q * 2) * SL + pp) * MP + m];
                uv += recv[((size_t)(q * 2 + 1) * SL + pp) * MP + m];
            }
            OutStore<OUT>::st(a.out, (int64_t)m * a.nh + j, silu(scaled(p, gv)) * scaled(PH + p, uv));
        }
    } else {
        for (int idx = threadIdx.x; idx < plen * a.M; idx += kThreads) {
            const int m = idx / plen, rr = idx - m * plen;
            const int r = ps + rr, n = n0 + r;
            if (n >= a.N) continue;
            float v = 0.f;
            for (int q = 0; q < sk; ++q) v += recv[((size_t)q * SL + rr) * MP + m];
            OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, scaled(r, v));
        }
    }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            p = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

template <int NT8, bool BF, bool GROUP, int OUT, bool SILU>
cudaError_t launch_one(const GemvArgs &a, const GemvPlan &p, cudaStream_t st, bool pdl) {
    using C = Cfg<NT8>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int RB = 16 * p.rg;
    // packed [N, K/4] bytes; box = 64 bytes (256 k) x RB rows (gated: RB/2 rows, loaded
    // twice per stage: gate rows and up rows); rows >= N and bytes >= K/4 read as zero
    CUtensorMap mw;
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 4), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 4)};
    const cuuint32_t box[2] = {64u, (cuuint32_t)(SILU ? RB / 2 : RB)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = gemv_kernel<NT8, BF, GROUP, OUT, SILU>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    GemvArgs b = a;
    b.rg = p.rg;
    b.kc = p.kc;
    b.ws = p.ws;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.tiles, (unsigned)p.sk, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
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
    return cudaLaunchKernelEx(&cfg, kern, mw, b);
}

template <int NT8, bool BF, bool GROUP, bool SILU>
cudaError_t launch_out(const GemvArgs &a, int out_dtype, const GemvPlan &p, cudaStream_t st,
                       bool pdl) {
    switch (out_dtype) {
    case 0: return launch_one<NT8, BF, GROUP, 0, SILU>(a, p, st, pdl);
    case 1: return launch_one<NT8, BF, GROUP, 1, SILU>(a, p, st, pdl);
    default: return launch_one<NT8, BF, GROUP, 2, SILU>(a, p, st, pdl);
    }
}

template <bool BF, bool SILU>
cudaError_t launch_dtype(const GemvArgs &a, bool group, int out_dtype, const GemvPlan &p,
                         cudaStream_t st, bool pdl) {
    if (p.nt8 == 1)
        return group ? launch_out<1, BF, true, SILU>(a, out_dtype, p, st, pdl)
                     : launch_out<1, BF, false, SILU>(a, out_dtype, p, st, pdl);
    return group ? launch_out<2, BF, true, SILU>(a, out_dtype, p, st, pdl)
                 : launch_out<2, BF, false, SILU>(a, out_dtype, p, st, pdl);
}

}  // namespace gemv
}  // namespace tl
