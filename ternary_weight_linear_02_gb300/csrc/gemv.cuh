// gemv.cuh -- the decode-shaped kernel (M <= 16 tokens): fused unpack and
// accumulate on register-fed warp MMAs, packed weights and x staged by TMA.
// Shared by kern_gemv.cu (plain output) and kern_gemv_silu.cu (SiLU-gated
// gate/up).
//
// out[m,n] = sum_k t[n,k] x[m,k], scaled per output channel (Qwen2.5-7B
// ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or per K group of
// G = 64, 128 or 256 weights ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §1.1, §3.1, §4.2; the "Bonsai 2 27B" port, §4.2, §5.2),
// t decoded with the code table of the first page's §3.1.
//
// Memory-bound design: every packed byte is read from HBM once and decoded
// once, in registers; the decoded +-1/0 weights go straight from registers to
// mma.sync (m16n8k16, fp32 accumulate), whose cost does not grow with the
// number of tokens.  Nothing is handed from one warp to another inside the
// main loop.
//
// Work split.  A CTA owns RB = 32*RGW weight rows x a K range (a multiple of
// 256 k); the K ranges of a row block are the CTAs of one thread-block cluster
// (split K).  Warp 8 is the producer: per 256-k stage one 2-D TMA of the packed
// weights (64 B x RB rows, 64-byte swizzle) and one 3-D TMA of x (four 64-k
// chunks x 8*NT8 token rows, 128-byte swizzle; token rows >= M and chunks past
// K read as zero), into a ring of shared-memory stages.  With static weights
// the weight half of the first stages is requested before griddepcontrol.wait,
// so under programmatic dependent launch a layer's weights stream in while the
// previous kernel ends; x follows after the wait.  Warps 0-7: warp w reads
// 64-k column w%4 of every stage for the row half w/4 of the CTA (RGW row
// groups of 16 rows), so a warp keeps only RGW row groups of accumulators --
// few enough registers for the decode and the MMAs of all its row groups to
// overlap.
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
// Reduction: the four column warps of a row half are summed in column order
// through the (then idle) ring; split K across the cluster pushes each CTA's
// partial rows into the owning CTA's shared memory (st.shared::cluster) and the
// owner sums them in rank order.  The same inputs give bit-identical outputs,
// and nothing is allocated.
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

constexpr int kWarps = 8;                   // consumer warps: 4 columns x 2 row halves
constexpr int kThreads = 32 * (kWarps + 1); // + the producer warp
constexpr int kStageK = 256;                // k per stage: a 64-byte weight box per row
constexpr int kRingBytes = 96 * 1024;
constexpr int kMaxStages = 16;

// Row groups (16 rows) per warp the kernel is compiled for: 1..4 (RB = 32..128
// rows per CTA).  Four row groups of accumulators and code words per warp keep
// the decode and the MMAs of a column overlapping (measured: more row groups per
// warp serialise them).  The software pipeline holds two stages' code words and
// x in registers; the largest counts that compile without spilling at two CTAs
// per SM (96 registers) are below -- group scales also hold each column's
// partials and the next column's scales.
constexpr int kRgwMax = 4;
__host__ __device__ constexpr int rgw_max(int nt8, bool group) {
    return nt8 == 1 ? (group ? 2 : 4) : (group ? 1 : 3);
}

template <int NT8>
struct Cfg {
    static constexpr int MP = 8 * NT8;               // padded tokens
    static constexpr int RBMAX = 32 * kRgwMax;       // rows per CTA at most
    static constexpr int XSTAGE = 4 * MP * 128;      // x bytes per stage: 4 chunks x MP rows x 128 B
    // split-K receive rows: sk * ceil(RB / sk) <= RB + 8 (gated: 2 * sk * ceil(RB/2 / sk))
    static constexpr int RECV_FLOATS = (RBMAX + 16) * MP;
    static constexpr int RECV_OFF = kRingBytes;
    static constexpr int FLAG_OFF = RECV_OFF + RECV_FLOATS * 4;  // 8 abort flags (one per rank)
    static constexpr int BAR_OFF = FLAG_OFF + 64;
    static constexpr int SMEM = BAR_OFF + (2 * kMaxStages + 2) * 8 + 16 + 1024;
    static_assert(kWarps * (RBMAX / 2) * MP * 4 <= kRingBytes, "reduction tiles fit in the ring");
    static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
};

// bytes of one ring stage (x part first, 1024-aligned; then the weight part)
__host__ __device__ constexpr int stage_stride(int nt8, int rgw) {
    return 4 * 8 * nt8 * 128 + 64 * 32 * rgw;
}

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


__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

// fp32 -> out element: fp16 / bf16 (round to nearest even) or fp32
__device__ __forceinline__ void store_out(int odt, void *base, int64_t idx, float v) {
    if (odt == 0) OutStore<0>::st(base, idx, v);
    else if (odt == 1) OutStore<1>::st(base, idx, v);
    else OutStore<2>::st(base, idx, v);
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

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

template <int NT8, int RGW, bool BF, bool GROUP, bool SILU>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                GemvArgs a) {
    using C = Cfg<NT8>;
    constexpr int MP = C::MP;
    constexpr int RB = 32 * RGW, PH = RB / 2;   // rows per CTA; rows per half
    constexpr int XST = C::XSTAGE, WST = 64 * RB, STRIDE = XST + WST;
    static_assert(STRIDE == stage_stride(NT8, RGW), "stage layout");
    static_assert(RGW >= 1 && RGW <= kRgwMax, "row groups per warp");
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
    const int rank = blockIdx.y, sk = gridDim.y;
    const int k0 = rank * a.kc, k1 = min(a.K, k0 + a.kc);
    const int nst = (k1 - k0 + kStageK - 1) / kStageK;
    // plain: rows [n0, n0 + RB); gated: gate rows [j0, j0 + PH) then up rows [nh + j0, ...)
    const int n0 = blockIdx.x * RB, j0 = blockIdx.x * PH;
    const long long lim = a.wait_limit;

    if (sk > 1) cluster_arrive_relaxed();  // cluster phase 1: this CTA has started
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ws; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarps && lane == 0) {
        tc::prefetch_tmap(&tmw);
        tc::prefetch_tmap(&tmx);
    }
    __syncthreads();
    pdl_launch_dependents();

    auto give_up = [&]() {
        *abort_flag = 1;
        if (a.status) atomicExch(a.status, kStatusTimeout);
    };

    // weight row (global) of CTA row r
    auto wrow = [&](int r) -> int {
        if constexpr (SILU) return r < PH ? j0 + r : a.nh + j0 + (r - PH);
        else return n0 + r;
    };

    // Zero-block map (a.mask, optional): bit kb of word [rb][kb / 32] is set when
    // rows [128 rb, +128) x k [64 kb, +64) hold a non-zero weight.  A stage whose
    // blocks are all zero is neither loaded nor multiplied (producer and consumers
    // walk the same live stages, so ring slots follow the count of live stages);
    // a warp skips the decode and MMAs of a zero 64-k column.
    auto rows_live = [&](int r0, int r1, int kb0, int nkb) -> bool {
        if (r1 <= r0) return false;
        for (int rb = r0 >> 7; rb <= (r1 - 1) >> 7; ++rb)
            for (int kb = kb0; kb < kb0 + nkb; ++kb)
                if ((__ldg(a.mask + (int64_t)rb * a.mask_words + (kb >> 5)) >> (kb & 31)) & 1u) return true;
        return false;
    };
    // rows of the CTA's half h (gated: h = 0 gate rows, h = 1 up rows)
    auto half_rows = [&](int h, int &r0, int &r1) {
        if constexpr (SILU) {
            r0 = (h ? a.nh : 0) + j0;
            r1 = min(r0 + PH, (h ? 2 * a.nh : a.nh));
        } else {
            r0 = n0 + h * PH;
            r1 = min(r0 + PH, a.N);
        }
    };
    auto stage_live = [&](int s) -> bool {
        if (a.mask == nullptr) return true;
        const int kb0 = (k0 >> 6) + 4 * s;
        int r0, r1;
        half_rows(0, r0, r1);
        if (rows_live(r0, r1, kb0, 4)) return true;
        half_rows(1, r0, r1);
        return rows_live(r0, r1, kb0, 4);
    };
    auto next_live = [&](int s) {
        while (s < nst && !stage_live(s)) ++s;
        return s;
    };

    float acc[RGW][NT8][4];
#pragma unroll
    for (int r = 0; r < RGW; ++r)
#pragma unroll
        for (int t = 0; t < NT8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][t][e] = 0.f;

    if (warp == kWarps) {
        // ------------------------------------------------ producer: TMA of weight and x stages
        if (lane == 0) {
            const bool static_w = (a.flags & kGemvStaticWeights) != 0;
            if (!static_w) pdl_wait();
            auto issue_w = [&](int s, int slot) {
                uint8_t *dst = ring + (size_t)slot * STRIDE + XST;
                const int kb = (k0 >> 2) + s * 64;  // byte column of the stage
                if constexpr (SILU) {
                    tc::tma_load_2d(dst, &tmw, kb, j0, &full[slot]);
                    tc::tma_load_2d(dst + WST / 2, &tmw, kb, a.nh + j0, &full[slot]);
                } else {
                    tc::tma_load_2d(dst, &tmw, kb, n0, &full[slot]);
                }
            };
            auto issue_x = [&](int s, int slot) {
                uint8_t *dst = ring + (size_t)slot * STRIDE;
                tc::tma_load_3d(dst, &tmx, 0, 0, (k0 >> 6) + s * 4, &full[slot]);
            };
            // the first (up to ws) live stages: weights now (static weights: before
            // the wait), x after it
            int pre_s[kMaxStages];
            int issued = 0, s = next_live(0);
            for (; s < nst && issued < a.ws; s = next_live(s + 1)) {
                mbar_arrive_expect_tx(&full[issued], (uint32_t)STRIDE);
                issue_w(s, issued);
                pre_s[issued++] = s;
            }
            if (static_w) pdl_wait();  // x belongs to the previous kernel until here
            for (int i = 0; i < issued; ++i) issue_x(pre_s[i], i);
            bool ok = true;
            for (; s < nst; s = next_live(s + 1)) {
                const int slot = issued % a.ws;
                if (*abort_flag || !mbar_wait_bounded(&empty[slot], ((issued / a.ws) - 1) & 1, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], (uint32_t)STRIDE);
                issue_w(s, slot);
                issue_x(s, slot);
                ++issued;
            }
            if (!ok) give_up();
            // drain: every copy still in flight lands before the ring is reused or the CTA exits
            for (int s = issued - a.ws < 0 ? 0 : issued - a.ws; s < issued; ++s)
                if (!mbar_wait_bounded(&full[s % a.ws], (s / a.ws) & 1)) give_up();
        }
    } else {
        // ------------------------------------------------ consumers
        const int cw = warp & 3;     // 64-k column of every stage
        const int half = warp >> 2;  // rows [half * PH, half * PH + PH) of the CTA
        // this lane's offsets inside a stage: x (128-byte swizzle: 16-byte unit u of
        // token row n at u ^ (n & 7), and n & 7 == g) and weights (64-byte swizzle:
        // 16-byte chunk j of row q at j ^ ((q >> 1) & 3), and for every row this lane
        // reads, (q >> 1) & 3 == (g >> 1) & 3)
        const int xo_lo = (cw * MP + g) * 128 + (((2 * c) ^ g) << 4);
        const int xo_hi = (cw * MP + g) * 128 + (((2 * c + 1) ^ g) << 4);
        const int wo = XST + (half * PH + g) * 64 + ((cw ^ ((g >> 1) & 3)) << 4) + 4 * c;
        uint32_t scn[RGW];  // next column's group scales: row g (low half), row g + 8 (high half)
        auto load_sc = [&](int kcol) {
            if constexpr (GROUP) {
                const int ngk = a.K >> a.gshift, gi = kcol >> a.gshift;
#pragma unroll
                for (int r = 0; r < RGW; ++r) {
                    uint32_t v = 0;
                    if (kcol < k1) {
                        const int rlo = wrow(half * PH + r * 16 + g);
                        const int rhi = wrow(half * PH + r * 16 + g + 8);
                        const uint32_t slo = rlo < a.N ? (uint32_t)a.scale[(int64_t)rlo * ngk + gi] : 0u;
                        const uint32_t shi = rhi < a.N ? (uint32_t)a.scale[(int64_t)rhi * ngk + gi] : 0u;
                        v = slo | (shi << 16);
                    }
                    scn[r] = v;
                }
            }
        };
        bool ok = true;
        if (a.flags & kGemvTestStall) {
            // testing aid: a wait on a barrier nothing arrives on runs out
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(never, 0, lim));
            if (!ok && lane == 0) give_up();
        }
        // Software pipeline over stages: the next stage is waited for and moved into
        // registers (its code words and x) before this stage's decode and MMAs, and its
        // ring slot is handed back as soon as the loads are done, so shared-memory
        // latency and the barrier wait overlap the arithmetic.
        uint32_t wc[2 * RGW], wn[2 * RGW];  // code words (lo, hi per row group): current, next
        uint4 xc[NT8][2], xn[NT8][2];       // x (two 16-byte halves per token tile)
        // fetch live stage number L (the L-th stage the producer issued) into registers
        auto fetch = [&](int L, uint32_t (&w)[2 * RGW], uint4 (&x)[NT8][2]) -> bool {
            const int slot = L % a.ws;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (L / a.ws) & 1, lim))) {
                if (lane == 0) give_up();
                return false;
            }
            const uint8_t *st = ring + (size_t)slot * STRIDE;
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                x[t][0] = lds128(st + xo_lo + t * 8 * 128);
                x[t][1] = lds128(st + xo_hi + t * 8 * 128);
            }
#pragma unroll
            for (int r = 0; r < RGW; ++r) {
                w[2 * r] = *reinterpret_cast<const uint32_t *>(st + wo + r * 1024);
                w[2 * r + 1] = *reinterpret_cast<const uint32_t *>(st + wo + r * 1024 + 512);
            }
            // the values are in registers: the slot may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            return true;
        };
        int hr0, hr1;  // this warp's rows, for the column test of the zero-block map
        half_rows(half, hr0, hr1);
        int s = ok ? next_live(0) : nst, L = 0;
        if (s < nst) load_sc(k0 + s * kStageK + cw * 64);
        if (s < nst) ok = ok && fetch(0, wc, xc);
        for (; ok && s < nst; ++L) {
            const int kcol = k0 + s * kStageK + cw * 64;
            const int sn = next_live(s + 1);
            uint32_t sc[RGW];
#pragma unroll
            for (int r = 0; r < RGW; ++r) sc[r] = 0u;
            if constexpr (GROUP) {
#pragma unroll
                for (int r = 0; r < RGW; ++r) sc[r] = scn[r];
                if (sn < nst) load_sc(k0 + sn * kStageK + cw * 64);  // in flight during this stage
            }
            if (sn < nst && !fetch(L + 1, wn, xn)) {
                ok = false;
                break;
            }
            const bool col_live = a.mask == nullptr || rows_live(hr0, hr1, kcol >> 6, 1);
            if (kcol < k1 && col_live) {
                uint32_t b[NT8][4][2];
#pragma unroll
                for (int t = 0; t < NT8; ++t) x_frag(xc[t][0], xc[t][1], b[t]);
                uint32_t zlo[RGW], zhi[RGW];
#pragma unroll
                for (int r = 0; r < RGW; ++r) {
                    zlo[r] = sign_nz(wc[2 * r]);
                    zhi[r] = sign_nz(wc[2 * r + 1]);
                }
                if constexpr (GROUP) {
#pragma unroll
                    for (int r = 0; r < RGW; ++r) {
                        float d[NT8][4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t a0 = pair2(zlo[r], i), a1 = pair2(zhi[r], i);
                            const uint32_t a2 = pair2(zlo[r], i + 4), a3 = pair2(zhi[r], i + 4);
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
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int r = 0; r < RGW; ++r) {
                            const uint32_t a0 = pair2(zlo[r], i), a1 = pair2(zhi[r], i);
                            const uint32_t a2 = pair2(zlo[r], i + 4), a3 = pair2(zhi[r], i + 4);
#pragma unroll
                            for (int t = 0; t < NT8; ++t)
                                mma16816<BF>(acc[r][t], a0, a1, a2, a3, b[t][i][0], b[t][i][1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 2 * RGW; ++q) wc[q] = wn[q];
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                xc[t][0] = xn[t][0];
                xc[t][1] = xn[t][1];
            }
            s = sn;
        }
    }

    // ------------------------------------------------ reduction and epilogue
    __syncthreads();  // every stage consumed (or abandoned) and no copy in flight
    pdl_wait();       // out belongs to the previous kernel until here
    const bool aborted = *abort_flag != 0;
    float *red = reinterpret_cast<float *>(ring);  // [warp][PH][MP]: a warp's rows of its half
    if (warp < kWarps && !aborted) {
#pragma unroll
        for (int r = 0; r < RGW; ++r) {
            const int rl = r * 16 + g;
#pragma unroll
            for (int t = 0; t < NT8; ++t) {
                float *p = red + ((size_t)warp * PH + rl) * MP + t * 8 + 2 * c;
                *reinterpret_cast<float2 *>(p) = make_float2(acc[r][t][0], acc[r][t][1]);
                *reinterpret_cast<float2 *>(p + 8 * MP) = make_float2(acc[r][t][2], acc[r][t][3]);
            }
        }
    }
    __syncthreads();
    // the CTA's partial of row r, token m: its half's four column warps summed in order
    auto part = [&](int r, int m) {
        const int h = r >= PH ? 1 : 0, rl = r - h * PH;
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) v += red[((size_t)(h * 4 + q) * PH + rl) * MP + m];
        return v;
    };
    // final value (scaled) of stacked row r from its summed partial
    auto scaled = [&](int r, float v) {
        if constexpr (GROUP) {
            (void)r;
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
                    store_out(a.odt, a.out, (int64_t)m * a.nh + j, silu(gv) * uv);
                }
            } else {
                for (int idx = threadIdx.x; idx < RB * a.M; idx += kThreads) {
                    const int m = idx / RB, r = idx - m * RB;
                    const int n = n0 + r;
                    if (n >= a.N) continue;
                    store_out(a.odt, a.out, (int64_t)m * a.N + n, scaled(r, part(r, m)));
                }
            }
        }
        return;
    }

    // ------------------------------------------------ split K over the cluster
    // owner q holds rows [q*RB/sk, (q+1)*RB/sk) (gated: pairs [q*PH/sk, (q+1)*PH/sk))
    cluster_wait();  // phase 1: every peer runs
    constexpr int span = SILU ? PH : RB;
    const int SL = (span + sk - 1) / sk;
    auto owner = [&](int p) {
        int q = (p * sk) / span;
        while (q + 1 < sk && ((q + 1) * span) / sk <= p) ++q;
        while ((q * span) / sk > p) --q;
        return q;
    };
    if (!aborted) {
        for (int idx = threadIdx.x; idx < RB * a.M; idx += kThreads) {
            const int m = idx / RB, r = idx - m * RB;
            if constexpr (SILU) {
                const int hf = r >= PH ? 1 : 0, p = r - hf * PH;
                const int q = owner(p), pp = p - (q * span) / sk;
                const float *slot = recv + ((size_t)(rank * 2 + hf) * SL + pp) * MP + m;
                cl_st_f32(cl_map(smem_u32(slot), (uint32_t)q), part(r, m));
            } else {
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
            store_out(a.odt, a.out, (int64_t)m * a.nh + j, silu(scaled(p, gv)) * scaled(PH + p, uv));
        }
    } else {
        for (int idx = threadIdx.x; idx < plen * a.M; idx += kThreads) {
            const int m = idx / plen, rr = idx - m * plen;
            const int r = ps + rr, n = n0 + r;
            if (n >= a.N) continue;
            float v = 0.f;
            for (int q = 0; q < sk; ++q) v += recv[((size_t)q * SL + rr) * MP + m];
            store_out(a.odt, a.out, (int64_t)m * a.N + n, scaled(r, v));
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

template <int NT8, int RGW, bool BF, bool GROUP, bool SILU>
cudaError_t launch_one(const GemvArgs &a, const GemvPlan &p, cudaStream_t st, bool pdl) {
    using C = Cfg<NT8>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    constexpr int RB = 32 * RGW;
    // packed [N, K/4] bytes; box = 64 bytes (256 k) x RB rows (gated: RB/2 rows, loaded
    // twice per stage: gate rows and up rows); rows >= N and bytes >= K/4 read as zero
    CUtensorMap mw;
    const cuuint64_t wdims[2] = {(cuuint64_t)(a.K / 4), (cuuint64_t)a.N};
    const cuuint64_t wstrides[1] = {(cuuint64_t)(a.K / 4)};
    const cuuint32_t wbox[2] = {64u, (cuuint32_t)(SILU ? RB / 2 : RB)};
    const cuuint32_t estr2[2] = {1, 1};
    CUresult r = enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), wdims,
                     wstrides, wbox, estr2, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // x [M, K] 16-bit viewed as [K/64 chunks][M rows][64 k]: one box = 4 chunks x MP
    // token rows x 64 k (rows >= M and chunks past K read as zero)
    CUtensorMap mx;
    const cuuint64_t xdims[3] = {64u, (cuuint64_t)a.M, (cuuint64_t)(a.K / 64)};
    const cuuint64_t xstrides[2] = {(cuuint64_t)a.K * 2, 128u};
    const cuuint32_t xbox[3] = {64u, (cuuint32_t)C::MP, 4u};
    const cuuint32_t estr3[3] = {1, 1, 1};
    r = enc(&mx, BF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<uint16_t *>(a.x), xdims, xstrides, xbox, estr3, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = gemv_kernel<NT8, RGW, BF, GROUP, SILU>;
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
    return cudaLaunchKernelEx(&cfg, kern, mw, mx, b);
}

// one instantiation per row-group count per warp (GemvPlan::rg = 2 * RGW row groups per CTA)
template <int NT8, bool BF, bool GROUP, bool SILU>
cudaError_t launch_rgw(const GemvArgs &a, const GemvPlan &p, cudaStream_t st, bool pdl) {
    constexpr int hi = rgw_max(NT8, GROUP);
    switch (p.rg / 2) {
    case 1: return launch_one<NT8, 1, BF, GROUP, SILU>(a, p, st, pdl);
    case 2: if constexpr (hi >= 2) return launch_one<NT8, 2, BF, GROUP, SILU>(a, p, st, pdl); break;
    case 3: if constexpr (hi >= 3) return launch_one<NT8, 3, BF, GROUP, SILU>(a, p, st, pdl); break;
    case 4: if constexpr (hi >= 4) return launch_one<NT8, 4, BF, GROUP, SILU>(a, p, st, pdl); break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

template <bool BF, bool SILU>
cudaError_t launch_dtype(const GemvArgs &a, bool group, const GemvPlan &p, cudaStream_t st,
                         bool pdl) {
    if (p.rg % 2 != 0) return cudaErrorInvalidValue;
    if (p.nt8 == 1)
        return group ? launch_rgw<1, BF, true, SILU>(a, p, st, pdl)
                     : launch_rgw<1, BF, false, SILU>(a, p, st, pdl);
    return group ? launch_rgw<2, BF, true, SILU>(a, p, st, pdl)
                 : launch_rgw<2, BF, false, SILU>(a, p, st, pdl);
}

}  // namespace gemv
}  // namespace tl
