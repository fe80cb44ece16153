// tile.cuh -- the large-M tcgen05 tile kernel template and its launch helpers,
// shared by kern_tile.cu (plain output) and kern_tile_silu.cu (SiLU-gated
// gate/up output).
//
// large-M ternary linear on the 5th-generation tensor cores.
//
// out[m,n] = sum_k t[n,k] x[m,k] with a per-channel scale (Qwen2.5-7B
// ternary-in-vLLM write-up, m.nxbn.cn/news/169761, §3.2, §4.2) or a
// per-128-wide-K-group scale ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
// trdm.cn/news/729035, §3.1, §4.2) -- or 64-wide groups, the variant of the
// "Bonsai 2 27B" port (m.xxqk.cn/news/593501, §4.2, §5.2); codes decoded with
// the table of the first page's §3.1.  The scale is applied per 64-k chunk, so
// either group size is one chunk or two.
//
// One CTA computes a 128 (weight rows n) x BN (tokens m) output tile:
//   D[n, m] = sum_k A[n, k] B[k, m],  A = decoded weights, B = x^T.
//  * Warps 0-3 (one thread per weight row = one TMEM lane) read their row's
//    packed codes from global memory, decode 64 codes per chunk into 32
//    registers of bf16x2 / f16x2 and store them into a TMEM A stage with
//    tcgen05.st.  The decoded weights never touch shared memory.
//  * Warp 4 streams x tiles (BN x 64 k, natural K order) into a 4-stage
//    shared-memory ring with TMA (128-byte swizzle).
//  * Warp 5 allocates TMEM and issues tcgen05.mma (kind::f16, A from TMEM,
//    B from shared memory, fp32 accumulator D in TMEM), committing each chunk
//    to the barriers that free its A stage and x stage.
//  * Epilogue: warps 0-3 read D with tcgen05.ld, apply the scale, convert and
//    store; a warp's 32 lanes write 32 consecutive n of one token row.
// Weight decode: 2*t in {+-2, +-0}, exact in both 16-bit formats, so every
// product is exact and the fp32 accumulation performs the same signed sums as
// the add / subtract / skip formulation.  Scales:
//   per channel        -> out = 0.5 * s[n] * D
//   per group, fp16 x  -> A holds t*s[n,g] exactly (s is fp16)
//   per group, bf16 x  -> s = s_hi + s_lo with both parts exact in bf16; two
//                         MMAs per k step (A_hi and A_lo) into the same D.
//  * Split K (a.sk > 1, plain output only): a cluster of sk CTAs along grid z
//    shares one output tile; CTA r multiplies chunks [r cpc, (r + 1) cpc) into its
//    own D.  The tile's BN token columns are dealt out in sk slices; every CTA
//    sends slice q of its D to CTA q's shared memory (st.shared::cluster into
//    the x ring, idle once the cluster has passed a barrier that follows every
//    CTA's last MMA), and CTA q adds the sk partials of its slice in rank order
//    -- the sum is the same on every run -- then scales and stores.  Fills the
//    GPU when ceil(N/128) * ceil(M/BN) tiles alone would leave SMs idle.
//  * SiLU-gated mode (SILU = true, a stacked gate/up layer): the CTA's 128 rows
//    are 64 gate rows and the matching 64 up rows; in the epilogue every lane
//    writes its scaled row to shared memory (the x ring, idle once D is
//    complete), and after one barrier the 128 threads split the (pair, token)
//    outputs out[m, j] = silu(g) * u between them.
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// word, the CTA stops issuing work, frees its TMEM and returns.
#pragma once

#include <cuda.h>
#include <stdio.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "tc.cuh"

namespace tl {

namespace {

constexpr int kKC = 64;   // k per pipeline chunk = one 128-byte row of x
constexpr int kThreads = 192;

enum { kChannel = 0, kFold = 1, kSplit = 2 };

__host__ __device__ constexpr uint32_t pow2ceil(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

template <int BN, int SMODE>
struct TileCfg {
    // A pipeline stage holds CPS consecutive live 64-k chunks: one round of
    // barrier waits and commits per stage.  Measured: the hand-offs of a round,
    // not the MMA rate, bounded the loop at one chunk per round (twice the MMAs per
    // round cost 1.37x the time), so stages take two chunks -- except for split
    // scales on the smaller tiles, whose 64-column chunks would leave one A stage
    // in the 256 columns of a two-CTA-per-SM allocation.
    static constexpr int CPS = (BN == 256 || SMODE != kSplit) ? 2 : 1;
    static constexpr int ACOLS = (SMODE == kSplit) ? 64 : 32;  // TMEM columns per chunk of A
    // A stages: at BN = 256 they fill the 256 TMEM columns next to D; smaller tiles
    // keep the allocation at 256 columns (two CTAs per SM)
    static constexpr int NA = (BN == 256) ? 256 / (ACOLS * CPS)
                              : (CPS == 2) ? (BN == 128 ? 2 : 3)
                                           : (SMODE == kSplit ? 3 : 4);
    static constexpr uint32_t TMEM_COLS = pow2ceil(NA * ACOLS * CPS + BN);
    static constexpr int NS = (BN == 256 || (BN == 128 && CPS == 2)) ? 3 : 4;  // x stages
    static constexpr int XCHUNK = BN * 128;                    // bytes of x per 64-k chunk
    static constexpr int XSTAGE = CPS * XCHUNK;                // bytes per x stage
    static_assert(NS * XSTAGE >= 4 * XCHUNK, "x ring holds the epilogue exchanges (512 * BN bytes)");
    // shared memory: [x stages][barriers][tmem slot, abort flag] + 1 KB alignment slack
    static constexpr int BAR_OFF = NS * XSTAGE;
    static constexpr int NBARS = 2 * NS + 2 * NA + 1;
    // [tmem slot, abort flag, four epilogue flags, -, -, eight split-K rank flags]
    // after the barriers
    static constexpr int SMEM = BAR_OFF + NBARS * 8 + 64 + 1024;
    // Shared memory requested per CTA: at least enough that an SM holds no more CTAs
    // than its 512 tensor-memory columns serve.  A CTA resident beyond that would wait
    // in tcgen05.alloc; with split-K clusters its peers would wait on it at the
    // cluster barrier while holding the columns it needs.
    static constexpr int TMEM_CPS = (int)(512 / TMEM_COLS);
    static constexpr int SMEM_FLOOR = TMEM_CPS >= 2 ? 80 * 1024 : 116 * 1024;
    static constexpr int SMEM_REQ = SMEM > SMEM_FLOOR ? SMEM : SMEM_FLOOR;
    static_assert(TMEM_CPS >= 1 && TMEM_CPS <= 2, "tensor memory budget");
    static_assert((TMEM_CPS + 1) * (SMEM_REQ + 1024) > 228 * 1024, "residency <= tensor memory");
    static_assert(TMEM_CPS * (SMEM_REQ + 1024) <= 228 * 1024, "shared memory");
};

// Adjacent-pair decode of one 32-bit word of 16 codes (k = 0..15 of the word)
// into 8 registers, register p = {2*t[2p], 2*t[2p+1]} (low half = lower k):
// after sign_nz, nibble p holds the two codes as (b1, nz) pairs; isolating the
// nibble and multiplying by 2^(14-4p) + 2^(28-4p) places code 2p at bits
// 15:14 and code 2p+1 at bits 31:30 (the two partial products do not overlap).
__device__ __forceinline__ void decode_word_adjacent(uint32_t w, uint32_t *r) {
    const uint32_t z = sign_nz(w);
    const uint32_t zh = z >> 16;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t mul = (1u << (14 - 4 * p)) + (1u << (28 - 4 * p));
        r[p] = ((z & (0xFu << (4 * p))) * mul) & 0xC000C000u;
        r[p + 4] = ((zh & (0xFu << (4 * p))) * mul) & 0xC000C000u;
    }
}

__device__ __forceinline__ void tile_named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// SiLU (x * sigmoid(x)) of the gated product, fp32 with CUDA's expf
__device__ __forceinline__ float tile_silu(float v) { return v / (1.f + expf(-v)); }

template <int BN, bool BF, int SMODE, int OUT, bool SILU>
__global__ void __launch_bounds__(kThreads, 1)
    tile_tc_kernel(const __grid_constant__ CUtensorMap tmx, TileArgs a) {
    using C = TileCfg<BN, SMODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *xfull = bars, *xempty = bars + C::NS;
    uint64_t *afull = bars + 2 * C::NS, *aempty = afull + C::NA;
    uint64_t *dfull = aempty + C::NA;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // SILU: gate rows [j0, j0 + 64) in lanes 0..63, up rows [nh + j0, ...) in lanes 64..127
    const int j0 = blockIdx.x * 64;
    const int n0 = SILU ? j0 : blockIdx.x * 128, m0 = blockIdx.y * BN;
    const int nchunks = a.K / kKC;
    // split K: this CTA's chunks [cb, ce) (the whole K when a.sk == 1)
    const int krank = a.sk > 1 ? (int)cluster_ctarank() : 0;
    const int cb = min(nchunks, krank * a.cpc), ce = a.sk > 1 ? min(nchunks, cb + a.cpc) : nchunks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < C::NA; ++i) {
            mbar_init(&afull[i], 4);  // one arrival per decoder warp
            mbar_init(&aempty[i], 1);
        }
        mbar_init(dfull, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t dcol = tmem + (uint32_t)(C::NA * C::CPS * C::ACOLS);

    pdl_launch_dependents();
    pdl_wait();  // x / packed / out may be produced / consumed by the previous kernel

    auto give_up = [&]() {
        *abort_flag = 1;
        if (a.status) atomicExch(a.status, kStatusTimeout);
    };

    // Split K: the producer and MMA warps only join the cluster's two phases.
    auto split_phases_idle = [&]() {
        __syncwarp();
        cl_arrive_release();  // phase 1: this CTA's work is issued and its D final
        cl_wait_acquire();
        cl_arrive_release();  // phase 2: partials exchanged
        cl_wait_acquire();
    };
    // Split K, decoder / epilogue warps: exchange the partial D slices through the
    // x rings, then add the slice this CTA owns in rank order, scale and store.
    auto split_epilogue = [&](bool ready, bool ok, int lc, int row, int n, bool rowok) {
        volatile int *wready = reinterpret_cast<volatile int *>(tmem_slot + 2);   // per epilogue warp
        volatile int *rank_ok = reinterpret_cast<volatile int *>(tmem_slot + 8);  // per cluster rank
        if (lane == 0) wready[warp] = ready ? 1 : 0;
        if (!ready && ok) give_up();
        __syncwarp();
        cl_arrive_release();  // phase 1: every CTA's D is final (or given up), its x ring idle
        cl_wait_acquire();
        const bool cta_ok = !*abort_flag && wready[0] && wready[1] && wready[2] && wready[3];
        const int sk = a.sk, slice = BN / sk, lsl = 31 - __clz(slice), g4 = slice >> 2;
        // receive buffer [source rank][slice column / 4][128 rows][4] fp32 = 512 * BN
        // bytes, the size of the x ring: one 16-byte store per 4 columns, lanes write
        // consecutive rows (no bank conflicts)
        const float4 *recv = reinterpret_cast<const float4 *>(smem);
        const uint32_t recv_u32 = smem_u32(smem);
        if (cta_ok) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
                uint32_t d[32];
                tc::ld_32x32b_x32(dcol + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * 32), d);
                tc::wait_ld();
                if (lc == 0) {  // no live chunk in this CTA's range: D was never written
#pragma unroll
                    for (int i = 0; i < 32; ++i) d[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int q = j * 32 + i;  // token column of the tile (slice holds whole 4s)
                    const uint32_t off =
                        ((uint32_t)(krank * g4 + ((q & (slice - 1)) >> 2)) * 128u + (uint32_t)row) * 16u;
                    cl_st_v4_f32(cl_map(recv_u32 + off, (uint32_t)(q >> lsl)), __uint_as_float(d[i]),
                                 __uint_as_float(d[i + 1]), __uint_as_float(d[i + 2]), __uint_as_float(d[i + 3]));
                }
            }
        }
        if (threadIdx.x == 0)
            for (int r = 0; r < sk; ++r)
                cl_st_u32(cl_map(smem_u32((const void *)(rank_ok + krank)), (uint32_t)r), cta_ok ? 1u : 0u);
        __syncwarp();
        cl_arrive_release();  // phase 2: every slice's partials and every rank's flag in place
        cl_wait_acquire();
        bool all_ok = true;
        for (int r = 0; r < sk; ++r) all_ok = all_ok && rank_ok[r] != 0;
        if (!all_ok || !rowok) return;
        // channel mode: A held 2*t, so D = 2*sum(t x); group modes: A held t*s
        float sc = 1.f;
        if constexpr (SMODE == kChannel) sc = 0.5f * h2f(a.scale[n]);
        const int mb = m0 + krank * slice;
        for (int c4 = 0; c4 < g4 && mb + 4 * c4 < a.M; ++c4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < sk; ++r) {
                const float4 p = recv[(r * g4 + c4) * 128 + row];
                v.x += p.x;
                v.y += p.y;
                v.z += p.z;
                v.w += p.w;
            }
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (mb + 4 * c4 + e < a.M) OutStore<OUT>::st(a.out, (int64_t)(mb + 4 * c4 + e) * a.N + n, vv[e] * sc);
        }
    };

    // Zero-block map (a.mask, optional; bit kb of word [rb][kb / 32] set when rows
    // [128 rb, +128) x k [64 kb, +64) hold a non-zero weight): a 64-k chunk whose
    // blocks are zero for this CTA's rows is neither loaded nor multiplied.  All
    // three roles walk the same live chunks; stage indices and the MMA's
    // accumulate flag follow the count of live chunks.
    auto rows_live = [&](int r0, int r1, int kb) -> bool {
        if (r1 <= r0) return false;
        for (int rb = r0 >> 7; rb <= (r1 - 1) >> 7; ++rb)
            if ((__ldg(a.mask + (int64_t)rb * a.mask_words + (kb >> 5)) >> (kb & 31)) & 1u) return true;
        return false;
    };
    auto chunk_live = [&](int c) -> bool {
        if (a.mask == nullptr) return true;
        if constexpr (SILU)
            return rows_live(j0, min(j0 + 64, a.nh), c) || rows_live(a.nh + j0, min(a.nh + j0 + 64, 2 * a.nh), c);
        else
            return rows_live(n0, min(n0 + 128, a.N), c);
    };
    auto next_live = [&](int c) {
        while (c < ce && !chunk_live(c)) ++c;
        return c;
    };

    if (warp == 4) {
        // ---------------- TMA producer: x tiles
        if (lane == 0) {
            tc::prefetch_tmap(&tmx);
            int lc = 0;  // live chunks issued
            for (int c = next_live(cb); c < ce && !*abort_flag; ++lc) {
                const int cn = next_live(c + 1);
                const int st = lc / C::CPS, h = lc % C::CPS, s = st % C::NS;
                if (h == 0) {
                    if (st >= C::NS && !mbar_wait_bounded(&xempty[s], ((st / C::NS) - 1) & 1)) {
                        give_up();
                        break;
                    }
                    // one arrival per stage, expecting every chunk the stage will hold
                    const int nch = (C::CPS == 2 && cn < ce) ? 2 : 1;
                    mbar_arrive_expect_tx(&xfull[s], (uint32_t)(nch * C::XCHUNK));
                }
                tc::tma_load_2d(smem + (size_t)s * C::XSTAGE + (size_t)h * C::XCHUNK, &tmx, c * kKC, m0,
                                &xfull[s]);
                c = cn;
            }
        }
        if (a.sk > 1) split_phases_idle();
    } else if (warp == 5) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16(BN, BF);
            int lc = 0;  // live chunks multiplied
            for (int c = next_live(cb), st = 0; c < ce; ++st) {
                const int s = st % C::NA, xs = st % C::NS;
                if (*abort_flag || !mbar_wait_bounded(&afull[s], (st / C::NA) & 1) ||
                    !mbar_wait_bounded(&xfull[xs], (st / C::NS) & 1)) {
                    give_up();
                    break;
                }
                tc::fence_after_sync();
                for (int h = 0; h < C::CPS && c < ce; ++h, ++lc, c = next_live(c + 1)) {
                    const uint64_t bdesc = tc::desc_sw128(smem + (size_t)xs * C::XSTAGE + (size_t)h * C::XCHUNK);
                    const uint32_t acol = tmem + (uint32_t)((s * C::CPS + h) * C::ACOLS);
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk) {
                        const uint64_t b = bdesc + (uint64_t)(kk * 2);  // +32 B per 16 elements
                        tc::mma_ts(dcol, acol + kk * 8, b, idesc, (lc | kk) != 0);
                        if constexpr (SMODE == kSplit) tc::mma_ts(dcol, acol + 32 + kk * 8, b, idesc, 1);
                    }
                }
                tc::commit(&aempty[s]);
                tc::commit(&xempty[xs]);
            }
            tc::commit(dfull);
        }
        if (a.sk > 1) split_phases_idle();
    } else {
        // ---------------- decoders / epilogue: thread = weight row = TMEM lane
        const int row = warp * 32 + lane;
        const int n = SILU ? (row < 64 ? j0 + row : a.nh + j0 + row - 64) : n0 + row;
        const bool rowok = SILU ? j0 + (row & 63) < a.nh : n < a.N;
        const int64_t Kq = a.K >> 2;
        const uint8_t *prow = a.packed + (int64_t)(rowok ? n : 0) * Kq;
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        const int ngk = a.K >> a.gshift;  // scale groups per row (G = 32, 64, 128 or 256)
        const uint16_t *srow = a.scale + (SMODE == kChannel ? 0 : (int64_t)(rowok ? n : 0) * ngk);

        // live chunks c (current), c1 and c2 (codes loaded one and two chunks ahead)
        int c = next_live(cb);
        int c1 = c < ce ? next_live(c + 1) : ce;
        uint4 cur = rowok && c < ce ? *reinterpret_cast<const uint4 *>(prow + (size_t)c * 16)
                                    : make_uint4(0, 0, 0, 0);
        uint4 nxt = rowok && c1 < ce ? *reinterpret_cast<const uint4 *>(prow + (size_t)c1 * 16)
                                     : make_uint4(0, 0, 0, 0);
        bool ok = true;
        int lc = 0;  // live chunks decoded
        for (; c < ce; ++lc) {
            // stage st = lc / CPS holds this chunk in half h; the A ring is waited for
            // at a stage's first chunk and handed to the issuer after its last
            const int st = lc / C::CPS, h = lc % C::CPS, s = st % C::NA;
            const bool stage_end = (h == C::CPS - 1) || c1 >= ce;
            const uint4 codes = cur;
            cur = nxt;
            const int c2 = c1 < ce ? next_live(c1 + 1) : ce;
            if (rowok && c2 < ce)
                nxt = *reinterpret_cast<const uint4 *>(prow + (size_t)c2 * 16);
            uint32_t r[32];
            decode_word_adjacent(codes.x, r + 0);
            decode_word_adjacent(codes.y, r + 8);
            decode_word_adjacent(codes.z, r + 16);
            decode_word_adjacent(codes.w, r + 24);
            uint32_t rl[32];
            if constexpr (SMODE != kChannel) {
                // registers 0-15 hold k 0-31 of the chunk, 16-31 hold k 32-63: with
                // 32-wide groups the two halves have their own scales (the same one
                // for wider groups); an adjacent pair never straddles a group
                const uint16_t sb0 = rowok ? srow[(c * kKC) >> a.gshift] : (uint16_t)0;
                const uint16_t sb1 = rowok ? srow[(c * kKC + 32) >> a.gshift] : (uint16_t)0;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float sf = h2f(hf ? sb1 : sb0);
                    if constexpr (SMODE == kFold) {
                        // fp16: (+-2) * (s/2) = +-s exactly
                        const __half2 h2 = __half2half2(__float2half_rn(0.5f * sf));
#pragma unroll
                        for (int i = 16 * hf; i < 16 * hf + 16; ++i) {
                            __half2 v = *reinterpret_cast<__half2 *>(&r[i]);
                            v = __hmul2(v, h2);
                            r[i] = *reinterpret_cast<uint32_t *>(&v);
                        }
                    } else {
                        // bf16: s = s_hi + s_lo, both exact in bf16
                        const __nv_bfloat16 hi = __float2bfloat16_rn(sf);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(sf - __bfloat162float(hi));
                        const __nv_bfloat162 h2 =
                            __bfloat162bfloat162(__float2bfloat16_rn(0.5f * __bfloat162float(hi)));
                        const __nv_bfloat162 l2 =
                            __bfloat162bfloat162(__float2bfloat16_rn(0.5f * __bfloat162float(lo)));
#pragma unroll
                        for (int i = 16 * hf; i < 16 * hf + 16; ++i) {
                            __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r[i]);
                            __nv_bfloat162 vh = __hmul2(v, h2), vl = __hmul2(v, l2);
                            r[i] = *reinterpret_cast<uint32_t *>(&vh);
                            rl[i] = *reinterpret_cast<uint32_t *>(&vl);
                        }
                    }
                }
            }
            // wait results are made warp-uniform: tcgen05.st below is warp-collective
            if (h == 0 && st >= C::NA)
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&aempty[s], ((st / C::NA) - 1) & 1));
            if (!ok) give_up();
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t acol = tlane + (uint32_t)((s * C::CPS + h) * C::ACOLS);
            tc::st_32x32b_x32(acol, r);
            if constexpr (SMODE == kSplit) tc::st_32x32b_x32(acol + 32, rl);
            if (stage_end) {
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[s]);
            }
            c = c1;
            c1 = c2;
        }
        // ---------------- epilogue
        ok = __all_sync(0xffffffffu, ok);
        bool ready = ok && __all_sync(0xffffffffu, mbar_wait_bounded(dfull, 0));
        if (a.sk > 1) {
            split_epilogue(ready, ok, lc, row, n, rowok);
        } else {
            if constexpr (SILU) {
                // the four epilogue warps exchange values below: decide together
                volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 2);
                if (lane == 0) flags[warp] = ready ? 1 : 0;
                tile_named_bar(1, 128);
                ready = flags[0] && flags[1] && flags[2] && flags[3];
                if (!ready && ok) give_up();
                ok = ok && ready;
            }
            if (ready) {
                tc::fence_after_sync();
                // channel mode: A held 2*t, so D = 2*sum(t x); group modes: A held t*s
                float sc = 1.f;
                if constexpr (SMODE == kChannel) sc = 0.5f * (rowok ? h2f(a.scale[n]) : 0.f);
                if constexpr (SILU) {
                    // every row's scaled values go to shared memory (the idle x ring,
                    // [token][128 rows] fp32 = 512 * BN bytes); after one barrier thread
                    // t writes pair p = t % 64 for half t / 64 of the tokens:
                    // out[m, j0 + p] = silu(gate) * up
                    float *ex = reinterpret_cast<float *>(smem);
#pragma unroll 1
                    for (int j = 0; j < BN / 32; ++j) {
                        uint32_t d[32];
                        tc::ld_32x32b_x32(dcol + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * 32), d);
                        tc::wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q)  // lc == 0: every chunk a zero block, D never written
                            ex[(j * 32 + q) * 128 + row] = lc == 0 ? 0.f : __uint_as_float(d[q]) * sc;
                    }
                    tile_named_bar(1, 128);
                    const int p = row & 63, q0 = (row >> 6) * (BN / 2);
                    if (j0 + p < a.nh) {
#pragma unroll 4
                        for (int q = q0; q < q0 + BN / 2 && m0 + q < a.M; ++q)
                            OutStore<OUT>::st(a.out, (int64_t)(m0 + q) * a.nh + j0 + p,
                                              tile_silu(ex[q * 128 + p]) * ex[q * 128 + 64 + p]);
                    }
                } else {
#pragma unroll 1
                    for (int j = 0; j < BN / 32; ++j) {
                        uint32_t d[32];
                        tc::ld_32x32b_x32(dcol + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * 32), d);
                        tc::wait_ld();
                        if (lc == 0) {  // every chunk of this CTA's rows is a zero block: D was never written
#pragma unroll
                            for (int q = 0; q < 32; ++q) d[q] = 0u;
                        }
                        if (rowok) {
#pragma unroll
                            for (int q = 0; q < 32; ++q) {
                                const int m = m0 + j * 32 + q;
                                if (m < a.M)
                                    OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, __uint_as_float(d[q]) * sc);
                            }
                        }
                    }
                }
            } else if (ok) {
                give_up();
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 5) tc::tmem_dealloc(tmem, C::TMEM_COLS);
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

// CTAs of one kernel instantiation that a cluster size of sk can keep resident at
// once.  CTAs per SM come from the kernel's resources -- shared memory (228 KB per
// SM, 1 KB reserved per CTA), threads, registers and the 512 TMEM columns: the
// occupancy query assumes the default split of L1 and shared memory and reports
// one CTA per SM for tiles that measurably run two.  The cluster query adds the
// GPC placement limit and is scaled by the ratio of the two per-SM counts.
// Cached per device, instantiation and sk.
template <typename Kern>
int tile_capacity(Kern kern, int smem, uint32_t tmem_cols, int sk, int sm_count) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, reinterpret_cast<const void *>(kern), sk);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int per_sm = (int)(512 / tmem_cols);
    const int by_smem = (228 * 1024) / (smem + 1024), by_threads = 2048 / kThreads;
    per_sm = by_smem < per_sm ? by_smem : per_sm;
    per_sm = by_threads < per_sm ? by_threads : per_sm;
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs > 0) {
        const int warp_regs = ((fa.numRegs * 32 + 255) / 256) * 256;  // allocated per warp
        const int by_regs = 65536 / (warp_regs * (kThreads / 32));
        per_sm = by_regs < per_sm ? by_regs : per_sm;
    }
    per_sm = per_sm < 1 ? 1 : per_sm;
    int api_per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&api_per_sm, kern, kThreads, smem) != cudaSuccess ||
        api_per_sm < 1)
        api_per_sm = 1;
    int cap = sm_count * per_sm;
    if (sk > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, (unsigned)sk);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)sk;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
            const int64_t ctas = (int64_t)n * sk * per_sm / api_per_sm;
            cap = (int)(ctas < cap ? ctas : cap);
        } else {
            cap = 0;  // cluster size not placeable
        }
    }
    cudaGetLastError();
    cache[key] = cap;
    return cap;
}

// Split K for the plain-output tile kernel (TERNARY_PLAN_LOG in the environment
// prints every candidate to stderr).  Cost of a plan, in 64-k chunk times of one
// CTA (fitted to per-layer timings of the 7B stack's shapes at M = 64, 256 and
// 2048):  waves * (chunks per CTA + O + E [split]) * sharing, where O is a CTA's
// fixed time (set-up, pipeline fill, epilogue: ~18 chunks at BN = 256, ~12 at
// BN <= 128), E the cluster exchange (~8 at BN = 256, ~3 at BN = 64), waves come
// from the occupancy query, and an SM running two CTAs at once takes ~1.4x as long
// as one.
template <typename Kern>
void plan_tile_split(Kern kern, int smem, uint32_t tmem_cols, int bn, TileArgs &a, int sm_count) {
    const int nchunks = a.K / kKC;
    a.sk = 1;
    a.cpc = nchunks;
    static const int force = [] {
        const char *e = getenv("TERNARY_TILE_SK");
        return e ? atoi(e) : 0;
    }();
    const int64_t tiles = (int64_t)((a.N + 127) / 128) * ((a.M + bn - 1) / bn);
    const int cap1 = tile_capacity(kern, smem, tmem_cols, 1, sm_count);
    const int per_sm = cap1 >= sm_count && sm_count > 0 ? cap1 / sm_count : 1;  // CTAs per SM
    const double O = bn >= 256 ? 18.0 : 12.0;
    const double E = 3.0 + 5.0 * (bn - 64) / 192.0;
    static const bool log = getenv("TERNARY_PLAN_LOG") != nullptr;
    double best = 0.0;
    for (int sk = 1; sk <= 8; sk *= 2) {
        if (sk > nchunks || bn / sk < 8) break;
        if (force && sk != force) continue;
        const int cap = tile_capacity(kern, smem, tmem_cols, sk, sm_count);
        if (cap < sk) continue;
        const int cpc = (nchunks + sk - 1) / sk;
        const int64_t total = tiles * sk;
        const int64_t waves = (total + cap - 1) / cap;
        const int64_t sms = cap / per_sm;  // SMs the clusters reach
        const int64_t in_wave = total < cap ? total : cap;
        const int64_t load = (in_wave + sms - 1) / sms;  // CTAs on the busiest SM
        const double share = 1.0 + 0.4 * (double)(load - 1);
        const double cost = (double)waves * (cpc + O + (sk > 1 ? E : 0.0)) * share;
        if (log)
            fprintf(stderr, "tile plan M=%d N=%d K=%d BN=%d: sk=%d capacity=%d CTAs (%d per SM) waves=%lld cost=%.1f\n",
                    a.M, a.N, a.K, bn, sk, cap, per_sm, (long long)waves, cost);
        if (best == 0.0 || cost < best * 0.97) {
            best = cost;
            a.sk = sk;
            a.cpc = cpc;
        }
    }
}

template <int BN, bool BF, int SMODE, int OUT, bool SILU>
cudaError_t launch_one(const TileArgs &a_in, int sm_count, cudaStream_t st, bool pdl) {
    using C = TileCfg<BN, SMODE>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TileArgs a = a_in;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&map, BF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<uint16_t *>(a.x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = tile_tc_kernel<BN, BF, SMODE, OUT, SILU>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_REQ);
    if (e != cudaSuccess) return e;
    a.sk = 1;
    a.cpc = a.K / kKC;
    if constexpr (!SILU) plan_tile_split(kern, C::SMEM_REQ, C::TMEM_COLS, BN, a, sm_count);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.N + 127) / 128), (unsigned)((a.M + BN - 1) / BN), (unsigned)a.sk);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_REQ;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.sk > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)a.sk;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

template <int BN, bool BF, int SMODE, bool SILU>
cudaError_t launch_out(const TileArgs &a, int out_dtype, int sm_count, cudaStream_t st, bool pdl) {
    switch (out_dtype) {
    case 0: return launch_one<BN, BF, SMODE, 0, SILU>(a, sm_count, st, pdl);
    case 1: return launch_one<BN, BF, SMODE, 1, SILU>(a, sm_count, st, pdl);
    default: return launch_one<BN, BF, SMODE, 2, SILU>(a, sm_count, st, pdl);
    }
}

template <int BN, bool SILU>
cudaError_t launch_bn(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                      cudaStream_t st, bool pdl) {
    if (!group)
        return bf ? launch_out<BN, true, kChannel, SILU>(a, out_dtype, sm_count, st, pdl)
                  : launch_out<BN, false, kChannel, SILU>(a, out_dtype, sm_count, st, pdl);
    return bf ? launch_out<BN, true, kSplit, SILU>(a, out_dtype, sm_count, st, pdl)
              : launch_out<BN, false, kFold, SILU>(a, out_dtype, sm_count, st, pdl);
}

inline int tile_bn_for(int64_t M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

template <bool SILU>
cudaError_t launch_tile_any(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                            cudaStream_t st, bool pdl) {
    switch (tile_bn_for(a.M)) {
    case 64: return launch_bn<64, SILU>(a, bf, group, out_dtype, sm_count, st, pdl);
    case 128: return launch_bn<128, SILU>(a, bf, group, out_dtype, sm_count, st, pdl);
    default: return launch_bn<256, SILU>(a, bf, group, out_dtype, sm_count, st, pdl);
    }
}

}  // namespace

}  // namespace tl
