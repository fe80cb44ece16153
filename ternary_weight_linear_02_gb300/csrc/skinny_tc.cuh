// skinny_tc.cuh -- the decode-shaped tcgen05 kernel template and its launch
// helpers, shared by kern_skinny_tc.cu (plain output) and kern_skinny_silu.cu
// (SiLU-gated gate/up output).
//
// decode-shaped ternary linear (M <= 32 tokens) on the
// 5th-generation tensor cores.
//
// out[m,n] = sum_k t[n,k] x[m,k] with a per-channel scale (Qwen2.5-7B
// ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or a
// per-128-wide-K-group scale ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §3.1, §4.2); t decoded with the code table of that
// page's §3.1.
//
// Memory-bound design: every packed byte is read from HBM once, decoded once,
// and the +-1/0 "multiplications" run on the tensor cores, where the decode
// cost does not grow with the number of tokens.
//
// One CTA owns 128 weight rows (one TMEM lane each) x a K range (a multiple of
// 128).  The K ranges of a row block are the CTAs of one thread-block cluster
// (split K, <= 8).  Two CTAs fit on an SM, so the next layer's CTAs can start
// (programmatic dependent launch) while this one finishes.
//  * Warp 8 (producer): TMA of the packed weights, 128 rows x 128 B (512 k) per
//    stage, 128-byte swizzle, 3-stage ring; with static weights the first
//    stages are requested before griddepcontrol.wait.  After the wait, one
//    3-D TMA per 512-k x stage (8 chunks of 64 k x NT token rows; rows >= M
//    are zero-filled by the TMA unit).
//  * Warps 0-7 (two decoder sets; thread = weight row = TMEM lane): read 16 B
//    of codes per 64 k from the staged row (conflict-free thanks to the
//    swizzle), decode every 2-bit code into 2*t in {+-2, +-0} (exact in fp16
//    and bf16) with one shift + one AND per register (tl::pair2: codes j and
//    j+8 of a 16-code word share one f16x2/bf16x2 register) and store it
//    into a TMEM A stage with tcgen05.st.  Channel scales: one A stage per
//    64-k chunk h, decoded by set h mod 2.  Group scales: one A stage per 128-k
//    unit u (a scale group), decoded by set u mod 2.  Decoders never wait for x.
//  * Warp 9: permutes each 16-k block of every staged x row in place so that
//    MMA k-slot (2j, 2j+1) holds x[j], x[j+8] -- the order in which pair2
//    packs the weights -- then hands the stage to the MMA.
//  * Warps 10.. (NI MMA issuers): issuer i runs the tcgen05.mma (kind::f16,
//    M = 128 rows, N = NT tokens, A from TMEM, B from shared memory) of chunks
//    h = i mod NI (channel scales) or units u = i mod 2 (group scales) into its
//    own fp32 TMEM accumulator.  One warp issues a small-N MMA only every
//    ~120-260 cycles whatever N is, and issuers in different warps proceed in
//    parallel (measured on GB300), so issue is spread over NI warps: three at
//    M <= 16, two where the accumulators take more TMEM.
//  * Stage ownership.  The A-stage count NA is a multiple of 2 and of NI, so an
//    A stage is always filled by the same decoder set and drained by the same
//    issuer: each full/empty mbarrier pair then has one waiter that takes its
//    phases in order.  (With an odd count, consecutive uses of a stage alternate
//    between waiters, and a waiter one phase ahead can pass a parity wait on
//    the phase before -- a parity wait cannot tell the two apart.)
//  * Scales.  Channel: the issuers' accumulators are summed, reduced over
//    the split K, then multiplied by 0.5*s[n] (the 2 of the +-2 decode).
//    Group: each 128-k unit lands in its issuer's accumulator slot; the decoder
//    set that owns the unit reads it back (tcgen05.ld) and folds
//    acc += 0.5*s[n,g] * D_g in fp32 registers; the two sets' sums are added.
//  * Split K: every row's fp32 partial is stored into the shared memory of the
//    cluster CTA that owns the row (st.shared::cluster) and announced with a
//    remote mbarrier arrive; the owner sums senders 0..sk-1 in that fixed
//    order, so the result is bit-identical run to run and nothing is
//    allocated.
//  * SiLU-gated mode (SILU = true): a fused gate/up layer with gate rows [0, nh)
//    and up rows [nh, 2 nh); a CTA stages 64 gate rows and the same 64 up rows
//    (two 64-row weight boxes per stage), so lanes j and 64 + j hold one pair.
//    The owner of a pair writes out[m, j] = silu(g) * u with g, u scaled sums
//    (split K: owners hold slices of the 64 pairs).
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// word and the CTA stops issuing work, drains its copies and MMAs, still joins
// the cluster barrier, frees its TMEM and returns.
#pragma once

#include <cuda.h>

#include "kernels.h"
#include "tc.cuh"

namespace tl {

namespace {

constexpr uint32_t kTmemCols = 256;    // two CTAs per SM share the 512 columns
constexpr int kSmemFloor = 96 * 1024;  // keeps residency at <= two CTAs per SM

// warp roles
// warps 0-7: two decoder sets (set = warp / 4, lane quarter = warp % 4)
constexpr int kWarpProd = 8, kWarpPerm = 9, kWarpMma0 = 10;
constexpr int kUnitsPerW = 4;        // 128-k units per weight stage (512 k)
constexpr int kWStage = 128 * 128;   // packed bytes per weight stage (128 rows x 128 B)

template <int NT, bool GROUP>
struct SkCfg {
    // Channel scales: A stages of one 64-k chunk (32 TMEM columns) and NI issuers,
    // each with its own accumulator.  Group scales: A stages of one 128-k unit and
    // two issuers whose accumulator slots hold one unit at a time.
    static constexpr bool CH = !GROUP;
    static constexpr int NI = (CH && NT == 16) ? 3 : 2;     // MMA issuer warps
    static constexpr int ACOLS = CH ? 32 : 64;              // TMEM columns per A stage
    static constexpr int NA = CH ? 6 : 2;                   // A stages
    static constexpr int THREADS = (kWarpMma0 + NI) * 32;
    static constexpr int XB = NT == 16 ? 8 : 4;       // 64-k x boxes per x stage
    static constexpr int UPX = XB / 2;                // units per x stage
    static constexpr int XBOX = NT * 128;             // one box: NT rows x 128 B
    static constexpr int XSTAGE = XB * XBOX;
    static constexpr int XS = 2;                      // x stages
    static constexpr int WS = 3;                      // weight stages
    static constexpr int W_OFF = XS * XSTAGE;
    static constexpr int RECV_OFF = W_OFF + WS * kWStage;
    // split-K receive rows: sk * ceil(128/sk) <= 135, or (gated) sk * 2 * ceil(64/sk) <= 140
    static constexpr int RECV_BYTES = (128 + 16) * NT * 4;
    static constexpr int BAR_OFF = RECV_OFF + RECV_BYTES;
    static constexpr int NBARS = 3 * XS + 2 * WS + 2 * NA + 3 * NI + 2;
    static constexpr int USED = BAR_OFF + NBARS * 8 + 16;
    static constexpr int SMEM = (USED + 1024 > kSmemFloor) ? USED + 1024 : kSmemFloor;
    static_assert(NA * ACOLS + NI * NT <= (int)kTmemCols, "TMEM budget");
    static_assert(NA % 2 == 0 && NA % NI == 0, "each A stage has one decoder set and one issuer");
    static_assert(!CH || NA * ACOLS + 64 <= (int)kTmemCols, "two 32-column stores zero the accumulators");
    static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
};

// SiLU (x * sigmoid(x)) of the gated product, fp32 with CUDA's expf
__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Every lane of the warp waits (bounded) on the same phase; the result is made
// warp-uniform, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int /*lane*/) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

// bounded wait with cluster-scope acquire (the arrivals come from other CTAs)
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 255u && clock64() - t0 > (1ll << 30)) return false;
    }
}

__device__ __forceinline__ void cluster_arrive_aligned() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_aligned() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// arrive (release, cluster scope) on an mbarrier of another CTA of the cluster
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

template <int NT>
__device__ __forceinline__ void ld_d(uint32_t taddr, uint32_t (&d)[NT]) {
    if constexpr (NT == 16) {
        ld_32x32b_x16(taddr, d);
    } else {
        tc::ld_32x32b_x32(taddr, d);
    }
}

// One 16-byte chunk of packed codes (64 weights, 4 words of 16 codes) ->
// 32 registers; register 8q+j = {2 t[16q+j], 2 t[16q+j+8]}.
__device__ __forceinline__ void decode_chunk(const uint4 &c, uint32_t (&r)[32]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t z = sign_nz(w[q]);
#pragma unroll
        for (int j = 0; j < 8; ++j) r[8 * q + j] = pair2(z, j);
    }
}

template <int NT, bool BF, bool GROUP, int OUT, bool SILU>
__global__ void __launch_bounds__(SkCfg<NT, GROUP>::THREADS, 2)
    skinny_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                     SkinnyTcArgs a) {
    using C = SkCfg<NT, GROUP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *xring = smem;
    uint8_t *wring = smem + C::W_OFF;
    float *recv = reinterpret_cast<float *>(smem + C::RECV_OFF);  // [sk][NT][SL] split-K partials
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *tfull = bars, *bfull = bars + C::XS, *xempty = bars + 2 * C::XS;
    uint64_t *wfull = bars + 3 * C::XS, *wempty = wfull + C::WS;
    uint64_t *afull = wempty + C::WS, *aempty = afull + C::NA;
    uint64_t *dfull = aempty + C::NA, *dempty = dfull + C::NI, *mdone = dempty + C::NI;
    uint64_t *rbar = mdone + C::NI, *dzero = rbar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 128 weight rows per CTA.  SILU: 64 gate rows [j0, j0 + 64) in lanes 0..63 and
    // the matching up rows [nh + j0, nh + j0 + 64) in lanes 64..127
    const int j0 = blockIdx.x * 64;
    const int n0 = SILU ? j0 : blockIdx.x * 128;
    const int rank = blockIdx.y;   // cluster rank = K split index (cluster dims 1 x sk x 1)
    const int sk = gridDim.y;
    const int k0 = rank * a.kc;
    const int k1 = min(a.K, k0 + a.kc);
    const int nch = (k1 - k0) >> 6;  // 64-k chunks
    const int nun = (nch + 1) >> 1;  // 128-k units (A stages, scale groups)
    const int nws = (nun + kUnitsPerW - 1) / kUnitsPerW;  // weight stages
    const int nxs = (nch + C::XB - 1) / C::XB;             // x stages
    const int SL = (128 + sk - 1) / sk;                     // rows per split-K slice (max)
    const int rs = (rank * 128) / sk, slen = ((rank + 1) * 128) / sk - rs;  // this CTA's slice
    // SILU split K: slices of the 64 (gate, up) row pairs
    const int SLP = (64 + sk - 1) / sk;
    const int ps = (rank * 64) / sk, plen = ((rank + 1) * 64) / sk - ps;
    const bool static_w = (a.flags & kSkinnyStaticWeights) != 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::XS; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&bfull[i], 1);
            mbar_init(&xempty[i], C::NI);  // one commit per MMA issuer
        }
        for (int i = 0; i < C::WS; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], 8);  // one arrival per decoder warp (both sets)
        }
        for (int i = 0; i < C::NA; ++i) {
            mbar_init(&afull[i], 4);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < C::NI; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], 4);
            mbar_init(&mdone[i], 1);
        }
        // one arrival per (sender, row of this slice)
        mbar_init(rbar, (uint32_t)(SILU ? sk * 2 * plen : sk * slen));
        mbar_init(dzero, 4);  // decoder set 0 has zeroed the accumulators (channel scales)
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma0) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (sk > 1) cluster_arrive_aligned();  // this CTA's barriers are initialised
    const uint32_t tmem = *tmem_slot;
    const uint32_t dbase = tmem + (uint32_t)(C::NA * C::ACOLS);
    // dependents may start once every CTA of this grid holds its TMEM
    if (!(a.flags & (kSkinnyTriggerLate | kSkinnyTriggerNever))) pdl_launch_dependents();

    // Zero-block map (a.mask, optional; channel scales only): bit kb of word
    // [rb][kb / 32] is set when rows [128 rb, +128) x k [64 kb, +64) hold a
    // non-zero weight.  A chunk whose blocks are zero for this CTA's rows is
    // neither decoded nor multiplied; its codes are still staged (the weight
    // ring keeps its order) and every chunk keeps its decoder set, issuer and A
    // stage, so a masked call adds the same partial sums in the same order as
    // an unmasked one.
    auto rows_live = [&](int r0, int r1, int kb) -> bool {
        if (r1 <= r0) return false;
        for (int rb = r0 >> 7; rb <= (r1 - 1) >> 7; ++rb)
            if ((__ldg(a.mask + (int64_t)rb * a.mask_words + (kb >> 5)) >> (kb & 31)) & 1u) return true;
        return false;
    };
    auto chunk_live = [&](int h) -> bool {  // chunk h of this CTA's K range
        if (!C::CH || a.mask == nullptr) return true;
        const int kb = (k0 >> 6) + h;
        if constexpr (SILU)
            return rows_live(j0, min(j0 + 64, a.nh), kb) ||
                   rows_live(a.nh + j0, min(a.nh + j0 + 64, 2 * a.nh), kb);
        else
            return rows_live(n0, min(n0 + 128, a.N), kb);
    };

    auto give_up = [&]() {
        *abort_flag = 1;
        if (a.status) atomicExch(a.status, kStatusTimeout);
    };

    if (warp == kWarpProd) {
        // ------------------------------------------------ TMA producer: weights (512 k per
        // stage, may run ahead of griddepcontrol.wait) and x (XB chunks of 64 k per stage)
        if (lane == 0) {
            tc::prefetch_tmap(&tmw);
            tc::prefetch_tmap(&tmx);
        }
        if (!static_w) pdl_wait();
        int wi = 0;  // weight stages issued
        auto issue_w = [&](int upto) -> bool {
            for (; wi < upto; ++wi) {
                const int s = wi % C::WS;
                if (wi >= C::WS && !warp_wait(&wempty[s], ((wi / C::WS) - 1) & 1, lane)) return false;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&wfull[s], (uint32_t)kWStage);
                    if constexpr (SILU) {  // two 64-row boxes: gate rows, then up rows
                        tc::tma_load_2d(wring + (size_t)s * kWStage, &tmw, (k0 >> 2) + wi * 128, j0, &wfull[s]);
                        tc::tma_load_2d(wring + (size_t)s * kWStage + kWStage / 2, &tmw, (k0 >> 2) + wi * 128,
                                        a.nh + j0, &wfull[s]);
                    } else {
                        tc::tma_load_2d(wring + (size_t)s * kWStage, &tmw, (k0 >> 2) + wi * 128, n0, &wfull[s]);
                    }
                }
                __syncwarp();
            }
            return true;
        };
        bool ok = issue_w(min(nws, C::WS));
        pdl_wait();  // x may be produced by the previous kernel
        int xi = 0;  // x stages issued
        for (; ok && xi < nxs; ++xi) {
            const int s = xi % C::XS;
            if (xi >= C::XS && !warp_wait(&xempty[s], ((xi / C::XS) - 1) & 1, lane)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                // one 3-D box: XB chunks of 64 k x NT token rows (chunk-major in shared memory)
                mbar_arrive_expect_tx(&tfull[s], (uint32_t)C::XSTAGE);
                tc::tma_load_3d(xring + (size_t)s * C::XSTAGE, &tmx, 0, 0, (k0 >> 6) + xi * C::XB,
                                &tfull[s]);
            }
            __syncwarp();
            // keep the weight ring WS - 1 stages ahead of the x stage just issued
            ok = issue_w(min(nws, xi * C::XB / (2 * kUnitsPerW) + C::WS));
        }
        if (ok) ok = issue_w(nws);
        if (!ok && lane == 0) give_up();
        // drain: no copy may still be landing in shared memory when the CTA exits
        for (int w = wi - C::WS < 0 ? 0 : wi - C::WS; w < wi; ++w)
            if (!warp_wait(&wfull[w % C::WS], (w / C::WS) & 1, lane) && lane == 0) give_up();
        for (int i = xi - C::XS < 0 ? 0 : xi - C::XS; i < xi; ++i)
            if (!warp_wait(&tfull[i % C::XS], (i / C::XS) & 1, lane) && lane == 0) give_up();
    } else if (warp == kWarpPerm) {
        // ------------------------------------------------ x permuter
        // Within each 16-k block of a staged row: slot 2j <- x[j], 2j+1 <- x[j+8].
        const uint32_t magic = (65536u + (uint32_t)a.M - 1u) / (uint32_t)a.M;  // it/M for it < 256
        for (int i = 0; i < nxs; ++i) {
            const int s = i % C::XS;
            if (!warp_wait(&tfull[s], (i / C::XS) & 1, lane)) {
                if (lane == 0) give_up();
                break;
            }
            const int nb = min(C::XB, nch - i * C::XB);
            const int items = nb * a.M * 4;  // (box, token row, 16-k block)
            uint8_t *stage = xring + (size_t)s * C::XSTAGE;
            for (int base = lane; base < items; base += 128) {
                // up to 4 items per lane per pass: all loads first, then permute and store
                uint4 *p0[4], *p1[4];
                uint4 v0[4], v1[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int it = base + 32 * t;
                    const int itc = it < items ? it : base;  // clamp: a repeated item is rewritten identically
                    const uint32_t rj = (uint32_t)itc >> 2, b = (uint32_t)itc & 3u;
                    const uint32_t j = (rj * magic) >> 16, r = rj - j * (uint32_t)a.M;
                    uint8_t *rowp = stage + j * C::XBOX + (r >> 3) * 1024 + (r & 7) * 128;
                    p0[t] = reinterpret_cast<uint4 *>(rowp + (((2 * b) ^ (r & 7)) << 4));
                    p1[t] = reinterpret_cast<uint4 *>(rowp + (((2 * b + 1) ^ (r & 7)) << 4));
                    v0[t] = *p0[t];
                    v1[t] = *p1[t];
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    if (base + 32 * t >= items) continue;
                    uint4 o0, o1;
                    o0.x = __byte_perm(v0[t].x, v1[t].x, 0x5410);  // x0, x8
                    o0.y = __byte_perm(v0[t].x, v1[t].x, 0x7632);  // x1, x9
                    o0.z = __byte_perm(v0[t].y, v1[t].y, 0x5410);  // x2, x10
                    o0.w = __byte_perm(v0[t].y, v1[t].y, 0x7632);  // x3, x11
                    o1.x = __byte_perm(v0[t].z, v1[t].z, 0x5410);  // x4, x12
                    o1.y = __byte_perm(v0[t].z, v1[t].z, 0x7632);  // x5, x13
                    o1.z = __byte_perm(v0[t].w, v1[t].w, 0x5410);  // x6, x14
                    o1.w = __byte_perm(v0[t].w, v1[t].w, 0x7632);  // x7, x15
                    *p0[t] = o0;
                    *p1[t] = o1;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bfull[s]);
        }
    } else if (warp >= kWarpMma0 && C::CH) {
        // ------------------------------------------------ MMA issuers, channel scales:
        // issuer iss takes chunks h = iss mod NI (A stages iss, iss + NI, ...) into its
        // own slot: without a zero-block map every chunk, the first MMA overwriting
        // the slot; with one the live chunks only, into a slot decoder set 0 zeroed
        const int iss = warp - kWarpMma0;
        constexpr uint32_t idesc = tc::idesc_f16(NT, BF);
        const uint32_t d = dbase + (uint32_t)(iss * NT);
        bool ok = true;
        if (a.mask == nullptr) {
            bool first = true;
            for (int i = 0; i < nxs && ok; ++i) {
                const int s = i % C::XS;
                if (!warp_wait(&bfull[s], (i / C::XS) & 1, lane)) {
                    ok = false;
                    break;
                }
                const uint64_t xdesc = tc::desc_sw128(xring + (size_t)s * C::XSTAGE);
                const int hb = i * C::XB, he = min(nch, hb + C::XB);
                for (int h = hb + (iss - hb % C::NI + C::NI) % C::NI; h < he; h += C::NI) {
                    const int st = h % C::NA;
                    if (!warp_wait(&afull[st], (h / C::NA) & 1, lane)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tc::fence_after_sync();
                        const uint32_t acol = tmem + (uint32_t)(st * C::ACOLS);
                        const uint64_t b0 = xdesc + (uint64_t)(((h - hb) * C::XBOX) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ts(d, acol + kk * 8, b0 + (uint64_t)(kk * 2), idesc,
                                       (first && kk == 0) ? 0u : 1u);  // the first MMA overwrites the slot
                        tc::commit(&aempty[st]);
                    }
                    first = false;
                    __syncwarp();
                }
                if (lane == 0) tc::commit(&xempty[s]);
                __syncwarp();
            }
        } else {
            // zero-block map: live chunks only, accumulators zeroed by decoder set 0
            ok = warp_wait(dzero, 0, lane);
            uint32_t par = 0;  // bit st: uses of A stage st so far, mod 2 (its next afull phase)
            for (int i = 0; i < nxs && ok; ++i) {
                const int s = i % C::XS;
                if (!warp_wait(&bfull[s], (i / C::XS) & 1, lane)) {
                    ok = false;
                    break;
                }
                const uint64_t xdesc = tc::desc_sw128(xring + (size_t)s * C::XSTAGE);
                const int hb = i * C::XB, he = min(nch, hb + C::XB);
                for (int h = hb + (iss - hb % C::NI + C::NI) % C::NI; h < he; h += C::NI) {
                    if (!chunk_live(h)) continue;
                    const int st = h % C::NA;
                    if (!warp_wait(&afull[st], (par >> st) & 1u, lane)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tc::fence_after_sync();
                        const uint32_t acol = tmem + (uint32_t)(st * C::ACOLS);
                        const uint64_t b0 = xdesc + (uint64_t)(((h - hb) * C::XBOX) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ts(d, acol + kk * 8, b0 + (uint64_t)(kk * 2), idesc, 1u);
                        tc::commit(&aempty[st]);
                    }
                    par ^= 1u << st;
                    __syncwarp();
                }
                if (lane == 0) tc::commit(&xempty[s]);
                __syncwarp();
            }
        }
        if (lane == 0) {
            if (!ok) give_up();
            tc::commit(&dfull[iss]);
            // drain: every MMA of this issuer has completed before TMEM is released
            tc::commit(&mdone[iss]);
        }
        __syncwarp();
        if (!warp_wait(&mdone[iss], 0, lane) && lane == 0) give_up();
    } else if (warp >= kWarpMma0) {
        // ------------------------------------------------ MMA issuers, group scales:
        // issuer iss takes units u = iss mod 2, one unit per accumulator fill
        const int iss = warp - kWarpMma0;
        constexpr uint32_t idesc = tc::idesc_f16(NT, BF);
        const uint32_t d = dbase + (uint32_t)(iss * NT);
        bool ok = true;
        for (int i = 0; i < nxs && ok; ++i) {
            const int s = i % C::XS;
            if (!warp_wait(&bfull[s], (i / C::XS) & 1, lane)) {
                ok = false;
                break;
            }
            const uint64_t xdesc = tc::desc_sw128(xring + (size_t)s * C::XSTAGE);
            const int ub = i * C::UPX, ue = min(nun, ub + C::UPX);
            for (int u = ub + ((ub & 1) != iss ? 1 : 0); u < ue; u += 2) {
                const int st = u % C::NA;
                if (!warp_wait(&afull[st], (u / C::NA) & 1, lane) ||
                    (u >= 2 && !warp_wait(&dempty[iss], ((u >> 1) - 1) & 1, lane))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    tc::fence_after_sync();
                    const uint32_t acol = tmem + (uint32_t)(st * C::ACOLS);
                    const uint64_t b0 = xdesc + (uint64_t)((2 * (u - ub) * C::XBOX) >> 4);
                    constexpr bool fresh = true;  // every unit overwrites the slot
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ts(d, acol + kk * 8, b0 + (uint64_t)(kk * 2), idesc,
                                   (fresh && kk == 0) ? 0u : 1u);
                    if (2 * u + 1 < nch) {
                        const uint64_t b1 = b0 + (uint64_t)(C::XBOX >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ts(d, acol + 32 + kk * 8, b1 + (uint64_t)(kk * 2), idesc, 1u);
                    }
                    tc::commit(&aempty[st]);
                    tc::commit(&dfull[iss]);
                }
                __syncwarp();
            }
            if (lane == 0) tc::commit(&xempty[s]);
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) give_up();
            // drain: every MMA of this issuer has completed before TMEM is released
            tc::commit(&mdone[iss]);
        }
        __syncwarp();
        if (!warp_wait(&mdone[iss], 0, lane) && lane == 0) give_up();
    } else {
        // ------------------------------------------------ decoders (thread = weight row)
        // Set s = warp / 4 decodes the chunks (channel scales) or units (group
        // scales) of parity s; warp % 4 selects the TMEM lane quarter.
        const int set = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const int n = SILU ? (row < 64 ? j0 + row : a.nh + j0 + row - 64) : n0 + row;
        const bool rowok = SILU ? j0 + (row & 63) < a.nh : n < a.N;
        // group mode: unit v (128 k) of this CTA uses scale group ((k0 >> 7) + v) >> (gshift - 7)
        const uint16_t *srow = GROUP ? a.scale + (int64_t)(rowok ? n : 0) * (a.K >> a.gshift) : a.scale;
        const int g0 = k0 >> 7, gsh = a.gshift - 7;
        const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
        const uint8_t *wrow = wring + row * 128;
        const int sw = row & 7;  // 128-byte swizzle of this staged row
        float acc[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0.f;

        bool ok = true;
        if constexpr (C::CH) {
            // chunk h (64 k) -> A stage h mod NA, decoded by set h mod 2, multiplied
            // by issuer h mod NI.  Software pipeline: the next chunk is decoded
            // while this one's TMEM store is in flight (tcgen05.wait::st follows).
            if (a.mask == nullptr) {
                uint4 cw = make_uint4(0, 0, 0, 0);
                // codes of chunk h into cw; releases a weight stage after this set's
                // last chunk in it (the final stage is never refilled)
                auto load_chunk = [&](int h) -> bool {
                    const int w = h >> 3, ws = w % C::WS, uw = h & 7;
                    if (uw < 2 && !warp_wait(&wfull[ws], (w / C::WS) & 1, lane)) return false;
                    cw = *reinterpret_cast<const uint4 *>(wrow + (size_t)ws * kWStage + ((uw ^ sw) << 4));
                    if (uw >= 6 && w + 1 < nws) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&wempty[ws]);  // codes are in registers
                    }
                    return true;
                };
                uint32_t r[32];
                if (set < nch) {
                    ok = load_chunk(set);
                    decode_chunk(cw, r);
                }
                for (int h = set; h < nch && ok; h += 2) {
                    const int st = h % C::NA;
                    if (h >= C::NA && !warp_wait(&aempty[st], ((h / C::NA) - 1) & 1, lane)) {
                        ok = false;
                        break;
                    }
                    tc::st_32x32b_x32(tlane + (uint32_t)(st * C::ACOLS), r);
                    if (h + 2 < nch) {
                        if (!load_chunk(h + 2)) {
                            ok = false;
                            break;
                        }
                        decode_chunk(cw, r);  // overlaps the store above
                    }
                    tc::wait_st();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&afull[st]);
                }
            } else {
                // zero-block map: set 0 first zeroes the accumulators, then each set
                // decodes its live chunks; an A stage's phase is its count of uses
                if (set == 0) {
                    uint32_t z[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) z[i] = 0u;
                    tc::st_32x32b_x32(tlane + (uint32_t)(C::NA * C::ACOLS), z);
                    tc::st_32x32b_x32(tlane + (uint32_t)(C::NA * C::ACOLS + 32), z);
                    tc::wait_st();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dzero);
                }
                uint4 cw = make_uint4(0, 0, 0, 0);
                // The weight-ring bookkeeping of chunk h: this set waits for a stage at
                // its first chunk in it and releases it after its last (the final stage
                // is never refilled); load_chunk also reads the codes into cw.
                auto ring_wait = [&](int h) -> bool {
                    const int w = h >> 3;
                    return (h & 7) >= 2 || warp_wait(&wfull[w % C::WS], (w / C::WS) & 1, lane);
                };
                auto ring_release = [&](int h) {
                    const int w = h >> 3;
                    if ((h & 7) >= 6 && w + 1 < nws) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&wempty[w % C::WS]);
                    }
                };
                auto load_chunk = [&](int h) -> bool {
                    if (!ring_wait(h)) return false;
                    const int ws = (h >> 3) % C::WS, uw = h & 7;
                    cw = *reinterpret_cast<const uint4 *>(wrow + (size_t)ws * kWStage + ((uw ^ sw) << 4));
                    ring_release(h);  // codes are in registers
                    return true;
                };
                // this set's next live chunk at or after h (-1: a wait gave up)
                auto next_mine = [&](int h) -> int {
                    for (; h < nch; h += 2) {
                        if (chunk_live(h)) return h;
                        if (!ring_wait(h)) return -1;
                        ring_release(h);
                    }
                    return nch;
                };
                uint32_t r[32];
                uint32_t par = 0, used = 0;  // bit st: uses of A stage st so far mod 2, and any use
                int h = next_mine(set);
                if (h < 0) {
                    ok = false;
                } else if (h < nch) {
                    ok = load_chunk(h);
                    decode_chunk(cw, r);
                }
                while (ok && h < nch) {
                    const int st = h % C::NA;
                    if (((used >> st) & 1u) && !warp_wait(&aempty[st], ((par >> st) & 1u) ^ 1u, lane)) {
                        ok = false;
                        break;
                    }
                    tc::st_32x32b_x32(tlane + (uint32_t)(st * C::ACOLS), r);
                    const int hn = next_mine(h + 2);
                    if (hn < 0) {
                        ok = false;
                        break;
                    }
                    if (hn < nch) {
                        if (!load_chunk(hn)) {
                            ok = false;
                            break;
                        }
                        decode_chunk(cw, r);  // overlaps the store above
                    }
                    tc::wait_st();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&afull[st]);
                    par ^= 1u << st;
                    used |= 1u << st;
                    h = hn;
                }
            }
            if (ok && set == 0) {
                // sum of the issuers' accumulators, in issuer order: without a map,
                // of the issuers that ran (issuer j's first chunk is j); with one,
                // of all (zeroed first), which adds the same values
                const int nsum = (a.mask == nullptr && nch < C::NI) ? nch : C::NI;
                for (int j = 0; j < nsum && ok; ++j) {
                    ok = warp_wait(&dfull[j], 0, lane);
                    if (!ok) break;
                    tc::fence_after_sync();
                    uint32_t dv[NT];
                    ld_d<NT>(tlane + (uint32_t)(C::NA * C::ACOLS + j * NT), dv);
                    tc::wait_ld();
#pragma unroll
                    for (int m = 0; m < NT; ++m)
                        acc[m] = (j == 0) ? __uint_as_float(dv[m]) : acc[m] + __uint_as_float(dv[m]);
                }
            }
        } else {
            // fold unit v's accumulator slot (v mod 2 = set) into acc with the group scale sv
            auto fold = [&](int v, float sv) {
                const int slot = v & 1;
                ok = ok && warp_wait(&dfull[slot], (v >> 1) & 1, lane);
                if (!ok) return;
                tc::fence_after_sync();
#pragma unroll
                for (int h = 0; h < NT / 16; ++h) {  // 16 columns at a time keeps registers low
                    uint32_t dv[16];
                    ld_32x32b_x16(tlane + (uint32_t)(C::NA * C::ACOLS + slot * NT + 16 * h), dv);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[16 * h + j] = fmaf(sv, __uint_as_float(dv[j]), acc[16 * h + j]);
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[slot]);
            };

            // Software pipeline: the next unit's first chunk is decoded while this
            // unit's TMEM stores are in flight (tcgen05.wait::st comes after it).
            uint4 c0 = make_uint4(0, 0, 0, 0), c1 = make_uint4(0, 0, 0, 0);
            float su = 0.f, s_prev = 0.f;
            // codes (and group scale) of unit v into c0/c1/su; releases a weight stage
            // after this set's last unit in it (the final stage is never refilled)
            auto load_unit = [&](int v) -> bool {
                const int w = v / kUnitsPerW, ws = w % C::WS, uw = v % kUnitsPerW;
                if (uw < 2 && !warp_wait(&wfull[ws], (w / C::WS) & 1, lane)) return false;
                const uint8_t *stage = wrow + (size_t)ws * kWStage;
                c0 = *reinterpret_cast<const uint4 *>(stage + (((2 * uw) ^ sw) << 4));
                c1 = (2 * v + 1 < nch) ? *reinterpret_cast<const uint4 *>(stage + (((2 * uw + 1) ^ sw) << 4))
                                       : make_uint4(0, 0, 0, 0);
                su = (GROUP && rowok) ? 0.5f * h2f(srow[(g0 + v) >> gsh]) : 0.f;
                if (uw >= 2 && w + 1 < nws) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&wempty[ws]);  // codes are in registers
                }
                return true;
            };
            uint32_t r[32];
            if (set < nun) {
                ok = load_unit(set);
                decode_chunk(c0, r);
            }
            for (int u = set; u < nun && ok; u += 2) {
                const int st = u % C::NA;
                const bool two = 2 * u + 1 < nch;
                const float su_u = su;
                const uint4 c1_u = c1;
                if (u >= C::NA && !warp_wait(&aempty[st], ((u / C::NA) - 1) & 1, lane)) {
                    ok = false;
                    break;
                }
                tc::st_32x32b_x32(tlane + (uint32_t)(st * C::ACOLS), r);
                if (two) {
                    decode_chunk(c1_u, r);
                    tc::st_32x32b_x32(tlane + (uint32_t)(st * C::ACOLS + 32), r);
                }
                if (u + 2 < nun) {
                    if (!load_unit(u + 2)) {
                        ok = false;
                        break;
                    }
                    decode_chunk(c0, r);  // overlaps the stores above
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[st]);
                if (GROUP && u >= 2) {
                    fold(u - 2, s_prev);
                    if (!ok) break;
                }
                s_prev = su_u;
            }
            if (GROUP && ok && set < nun) fold(set + ((nun - 1 - set) / 2) * 2, s_prev);
        }
        if (!ok) give_up();
        if (GROUP) {
            // set 1's partial sums join set 0's through the (now idle) weight ring
            float *comb = reinterpret_cast<float *>(wring);
            named_bar(1, 256);
            if (set == 1) {
#pragma unroll
                for (int j = 0; j < NT; ++j) comb[j * 128 + row] = acc[j];
            }
            named_bar(1, 256);
            if (set == 0) {
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[j] += comb[j * 128 + row];
            }
        }
        if (set == 0 && sk == 1) {
            if constexpr (SILU) {
                // the up rows' values reach the gate lanes through shared memory;
                // out[m, j] = silu(gate) * up
                const float fs = (GROUP || !rowok) ? 1.f : 0.5f * h2f(a.scale[n]);
                if (row >= 64) {
#pragma unroll
                    for (int m = 0; m < NT; ++m) recv[m * 64 + (row - 64)] = acc[m] * fs;
                }
                named_bar(3, 128);
                if (row < 64 && rowok && !*abort_flag) {
                    pdl_wait();
#pragma unroll
                    for (int m = 0; m < NT; ++m)
                        if (m < a.M)
                            OutStore<OUT>::st(a.out, (int64_t)m * a.nh + j0 + row,
                                              silu_f(acc[m] * fs) * recv[m * 64 + row]);
                }
            } else if (rowok && !*abort_flag) {
                pdl_wait();
                const float fs = GROUP ? 1.f : 0.5f * h2f(a.scale[n]);
#pragma unroll
                for (int m = 0; m < NT; ++m)
                    if (m < a.M) OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, acc[m] * fs);
            }
        } else if (set == 0) {
            // ---------------- split K: push this row's partial to the CTA that owns the row
            cluster_wait_aligned();  // every CTA of the cluster has initialised its barriers
            if constexpr (SILU) {
                // owners hold slices of the 64 (gate, up) pairs: slot = half * SLP + pair offset
                const int pr = row & 63, half = row >> 6;
                int o = (pr * sk) >> 6;
                while (o + 1 < sk && ((o + 1) * 64) / sk <= pr) ++o;
                while ((o * 64) / sk > pr) --o;
                const int slot = half * SLP + pr - (o * 64) / sk;
                const uint32_t rbase = map_rank(smem_u32(recv), (uint32_t)o);
#pragma unroll
                for (int m = 0; m < NT; ++m)
                    if (m < a.M)
                        st_cluster_f32(rbase + (uint32_t)(((rank * NT + m) * 2 * SLP + slot) * 4), acc[m]);
                mbar_arrive_remote(map_rank(smem_u32(rbar), (uint32_t)o));
            } else {
                int o = (row * sk) >> 7;
                while (o + 1 < sk && ((o + 1) * 128) / sk <= row) ++o;
                while ((o * 128) / sk > row) --o;
                const int rr = row - (o * 128) / sk;
                const uint32_t rbase = map_rank(smem_u32(recv), (uint32_t)o);
#pragma unroll
                for (int m = 0; m < NT; ++m)
                    if (m < a.M) st_cluster_f32(rbase + (uint32_t)(((rank * NT + m) * SL + rr) * 4), acc[m]);
                mbar_arrive_remote(map_rank(smem_u32(rbar), (uint32_t)o));
            }
            // ---------------- owner: sum the slice over senders 0..sk-1 in order
            const bool got = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(rbar, 0));
            if (!got) give_up();
            if (got && !*abort_flag && SILU) {
                pdl_wait();
                const int pairs = a.M * plen;
                const uint32_t lmagic = (1u << 20) / (uint32_t)plen + 1u;  // p/plen for p < 4096
                for (int p = row; p < pairs; p += 128) {
                    const int m = (int)(((uint32_t)p * lmagic) >> 20), qq = p - m * plen;
                    const int j = j0 + ps + qq;
                    if (j >= a.nh) continue;
                    float g = 0.f, u = 0.f;
#pragma unroll
                    for (int src = 0; src < 8; ++src)
                        if (src < sk) {
                            g += recv[(src * NT + m) * 2 * SLP + qq];
                            u += recv[(src * NT + m) * 2 * SLP + SLP + qq];
                        }
                    const float gs = GROUP ? 1.f : 0.5f * h2f(a.scale[j]);
                    const float us = GROUP ? 1.f : 0.5f * h2f(a.scale[a.nh + j]);
                    OutStore<OUT>::st(a.out, (int64_t)m * a.nh + j, silu_f(g * gs) * (u * us));
                }
            } else if (got && !*abort_flag) {
                pdl_wait();
                const int pairs = a.M * slen;
                const uint32_t lmagic = (1u << 20) / (uint32_t)slen + 1u;  // p/slen for p < 4096
                for (int p = row; p < pairs; p += 128) {
                    const int m = (int)(((uint32_t)p * lmagic) >> 20), qq = p - m * slen;
                    const int nn = n0 + rs + qq;
                    if (nn >= a.N) continue;
                    float v = 0.f;
#pragma unroll
                    for (int src = 0; src < 8; ++src)
                        if (src < sk) v += recv[(src * NT + m) * SL + qq];
                    const float fs = GROUP ? 1.f : 0.5f * h2f(a.scale[nn]);
                    OutStore<OUT>::st(a.out, (int64_t)m * a.N + nn, v * fs);
                }
            }
        }
    }

    __syncwarp();
    if (a.flags & kSkinnyTriggerLate) pdl_launch_dependents();
    if (sk > 1 && warp >= 4) cluster_wait_aligned();  // set 1 and the helper warps
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kWarpMma0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

template <int NT, bool BF, bool GROUP, int OUT, bool SILU>
cudaError_t launch_one(const SkinnyTcArgs &a, const SkinnyTcPlan &p, cudaStream_t st, bool pdl) {
    using C = SkCfg<NT, GROUP>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[2] = {1, 1};
    // x [M, K] 16-bit viewed as [K/64 chunks][M rows][64 k]: one box = XB chunks x NT
    // token rows x 64 k (rows >= M and chunks past K read as zero)
    CUtensorMap mx;
    const cuuint64_t xdims[3] = {64u, (cuuint64_t)a.M, (cuuint64_t)(a.K / 64)};
    const cuuint64_t xstrides[2] = {(cuuint64_t)a.K * 2, 128u};
    const cuuint32_t xbox[3] = {64u, (cuuint32_t)NT, (cuuint32_t)C::XB};
    const cuuint32_t estr3[3] = {1, 1, 1};
    CUresult r = enc(&mx, BF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<uint16_t *>(a.x), xdims, xstrides, xbox, estr3,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // packed [N, K/4] bytes: boxes of 128 B (512 k) x 128 rows (rows >= N read as zero);
    // the gated call loads two 64-row boxes (gate rows, up rows) per stage
    CUtensorMap mw;
    const cuuint64_t wdims[2] = {(cuuint64_t)(a.K / 4), (cuuint64_t)a.N};
    const cuuint64_t wstrides[1] = {(cuuint64_t)(a.K / 4)};
    const cuuint32_t wbox[2] = {128u, SILU ? 64u : 128u};
    r = enc(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), wdims, wstrides,
            wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = skinny_tc_kernel<NT, BF, GROUP, OUT, SILU>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.row_tiles, (unsigned)p.sk, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
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
    SkinnyTcArgs b = a;
    b.kc = p.kc;
    return cudaLaunchKernelEx(&cfg, kern, mx, mw, b);
}

template <int NT, bool BF, bool GROUP, bool SILU>
cudaError_t launch_out(const SkinnyTcArgs &a, int out_dtype, const SkinnyTcPlan &p,
                       cudaStream_t st, bool pdl) {
    switch (out_dtype) {
    case 0: return launch_one<NT, BF, GROUP, 0, SILU>(a, p, st, pdl);
    case 1: return launch_one<NT, BF, GROUP, 1, SILU>(a, p, st, pdl);
    default: return launch_one<NT, BF, GROUP, 2, SILU>(a, p, st, pdl);
    }
}

template <int NT, bool SILU>
cudaError_t launch_nt(const SkinnyTcArgs &a, bool bf, bool group, int out_dtype,
                      const SkinnyTcPlan &p, cudaStream_t st, bool pdl) {
    if (bf)
        return group ? launch_out<NT, true, true, SILU>(a, out_dtype, p, st, pdl)
                     : launch_out<NT, true, false, SILU>(a, out_dtype, p, st, pdl);
    return group ? launch_out<NT, false, true, SILU>(a, out_dtype, p, st, pdl)
                 : launch_out<NT, false, false, SILU>(a, out_dtype, p, st, pdl);
}

}  // namespace

}  // namespace tl
