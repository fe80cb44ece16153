// tile_persist.cuh -- the persistent variant of the tile kernel (tile.cuh) for
// many output tiles: one CTA per SM walks a list of 128-row x PBN-token tiles,
// so set-up and pipeline fill are paid once.  PBN = 192: two TMEM accumulators,
// the epilogue of one tile overlapping the main loop of the next.  PBN = 256
// (per-channel scales): one accumulator and four A stages; the issuer waits for
// the epilogue to read the accumulator out, but each MMA instruction carries a
// third more work -- one warp issues tcgen05.mma at a fixed rate whatever N is,
// and that rate bounds the 192-token form.
//
// Same arithmetic as the tile kernel (ternary codes of "三元量化模型接入vLLM：
// 从逆向加载到Kernel优化的完整实战" §3.1 decoded to 2t in 16-bit registers,
// tcgen05.mma kind::f16 with fp32 accumulation, per-channel scale of the
// Qwen2.5-7B ternary-in-vLLM write-up §3.2 in the epilogue or group scales
// folded into A), with these roles:
//  * warps 0-3, decoders: thread = weight row = TMEM lane; they walk the CTA's
//    (tile, live chunk) sequence without a break between tiles, loading each
//    chunk's 16 code bytes four items ahead and storing the decoded chunk into
//    a TMEM A stage (a stage holds two chunks of one tile: one round of barrier
//    waits and commits per stage);
//  * warp 8, producer: TMA of x tiles (PBN tokens x 64 k per chunk) into a ring
//    of stages that also runs across tiles;
//  * warp 9: TMEM allocation and the MMA issuer; tile i accumulates into TMEM
//    buffer i % NB (NB accumulators of PBN columns + the A stages = 512 columns);
//  * warps 4-7, epilogue: read buffer i % NB with tcgen05.ld, hand it back to
//    the issuer as soon as the last columns are in registers, scale, convert
//    and store -- with two buffers, while the issuer already fills the other.  The gated
//    variant (64 gate + 64 up rows per tile) exchanges rows through a 16 KB
//    shared-memory buffer, 32 tokens at a time.
// Tiles are numbered with the token tile fastest, so the CTAs running at the
// same time share the weight rows of a few row blocks and all of x in L2.
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// word and the CTA stops, frees its TMEM and returns.
#pragma once

#include <type_traits>

#include "tile.cuh"

namespace tl {

namespace {

constexpr int kPWarps = 10;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kPWarpEpi0 = 4, kPWarpProd = 8, kPWarpMma = 9;

template <int SMODE, int PBN>
struct PCfg {
    // A pipeline stage holds up to CPS consecutive live chunks of one tile (one
    // round of waits and commits per stage: the rounds, not the MMA rate, bound
    // the loop at one chunk per round); the A stages and the NB accumulators
    // fill the 512 TMEM columns.
    static_assert(PBN == 192 || (PBN == 256 && SMODE == kChannel), "tile widths");
    static constexpr int NB = PBN == 256 ? 1 : 2;             // accumulators
    static constexpr int CPS = (SMODE == kSplit) ? 1 : 2;
    static constexpr int ACOLS = (SMODE == kSplit) ? 64 : 32;  // TMEM columns per chunk of A
    static constexpr int NA = (512 - NB * PBN) / (ACOLS * CPS);  // A stages
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int DCOL0 = NA * CPS * ACOLS;             // accumulators at DCOL0 + b * PBN
    static_assert(NA >= 2 && DCOL0 + NB * PBN <= 512, "tensor memory budget");
    static constexpr int NS = (CPS == 2) ? 3 : 4;              // x stages
    static constexpr int XCHUNK = PBN * 128;                   // x of one chunk: PBN rows x 128 B
    static constexpr int XSTAGE = CPS * XCHUNK;
    static constexpr int EX_OFF = NS * XSTAGE;                 // gated exchange [32 tokens][128 rows]
    static constexpr int EX_BYTES = 32 * 128 * 4;
    static constexpr int BAR_OFF = EX_OFF + EX_BYTES;
    static constexpr int NBARS = 2 * NS + 2 * NA + 4;
    // [tmem slot, abort flag, -, -, eight epilogue flags (two parities x four warps)]
    static constexpr int SMEM = BAR_OFF + NBARS * 8 + 64 + 1024;
    // one CTA per SM: it holds all 512 TMEM columns, so no second CTA may become
    // resident and wait in tcgen05.alloc
    static constexpr int SMEM_REQ = SMEM > 116 * 1024 ? SMEM : 116 * 1024;
    static_assert(2 * (SMEM_REQ + 1024) > 228 * 1024, "one CTA per SM");
    static_assert(SMEM_REQ + 1024 <= 228 * 1024, "shared memory");
};

template <bool BF, int SMODE, int OUT, bool SILU, int PBN>
__global__ void __launch_bounds__(kPThreads, 1)
    tile_persist_kernel(const __grid_constant__ CUtensorMap tmx, TileArgs a) {
    using C = PCfg<SMODE, PBN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *xfull = bars, *xempty = bars + C::NS;
    uint64_t *afull = bars + 2 * C::NS, *aempty = afull + C::NA;
    uint64_t *dfull = aempty + C::NA, *dempty = dfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *epi_flags = reinterpret_cast<volatile int *>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nchunks = a.K / kKC;
    const int RB = SILU ? (a.nh + 63) / 64 : (a.N + 127) / 128;  // row blocks
    const int MB = (a.M + PBN - 1) / PBN;                         // token tiles
    const int T = RB * MB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < C::NA; ++i) {
            mbar_init(&afull[i], 4);  // one arrival per decoder warp
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], 4);  // one arrival per epilogue warp
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kPWarpMma) tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    pdl_launch_dependents();
    pdl_wait();  // x / out may be produced / consumed by the previous kernel

    auto give_up = [&]() {
        *abort_flag = 1;
        if (a.status) atomicExch(a.status, kStatusTimeout);
    };
    // tile t: token tile t % MB (fastest), row block t / MB
    auto tile_m0 = [&](int t) { return (t % MB) * PBN; };
    auto tile_rb = [&](int t) { return t / MB; };
    // weight row of TMEM lane r in tile t, and whether it exists
    auto row_of = [&](int t, int r, bool &ok) -> int {
        if constexpr (SILU) {
            const int j0 = tile_rb(t) * 64;
            ok = j0 + (r & 63) < a.nh;
            return r < 64 ? j0 + r : a.nh + j0 + r - 64;
        } else {
            const int n = tile_rb(t) * 128 + r;
            ok = n < a.N;
            return n;
        }
    };
    // Zero-block map: a chunk whose blocks are all zero for the tile's rows is
    // neither loaded nor multiplied; every role walks the same live chunks.
    auto rows_live = [&](int r0, int r1, int kb) -> bool {
        if (r1 <= r0) return false;
        for (int rb = r0 >> 7; rb <= (r1 - 1) >> 7; ++rb)
            if ((__ldg(a.mask + (int64_t)rb * a.mask_words + (kb >> 5)) >> (kb & 31)) & 1u) return true;
        return false;
    };
    auto next_live = [&](int t, int c) {
        if (a.mask == nullptr) return c;
        for (; c < nchunks; ++c) {
            bool live;
            if constexpr (SILU) {
                const int j0 = tile_rb(t) * 64;
                live = rows_live(j0, min(j0 + 64, a.nh), c) ||
                       rows_live(a.nh + j0, min(a.nh + j0 + 64, 2 * a.nh), c);
            } else {
                const int n0 = tile_rb(t) * 128;
                live = rows_live(n0, min(n0 + 128, a.N), c);
            }
            if (live) break;
        }
        return c;
    };

    if (warp == kPWarpProd) {
        // ---------------- TMA producer: x tiles, one ring across all tiles
        if (lane == 0) {
            tc::prefetch_tmap(&tmx);
            int st = 0;  // stages issued
            bool ok = true;
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x) {
                const int m0 = tile_m0(t);
                int h = 0;  // chunk of the current stage
                for (int c = next_live(t, 0); c < nchunks;) {
                    const int cn = next_live(t, c + 1);
                    const int s = st % C::NS;
                    if (h == 0) {
                        if (*abort_flag || (st >= C::NS && !mbar_wait_bounded(&xempty[s], ((st / C::NS) - 1) & 1))) {
                            if (!*abort_flag) give_up();
                            ok = false;
                            break;
                        }
                        // one arrival per stage, expecting every chunk the stage will hold
                        const int nch = (C::CPS == 2 && cn < nchunks) ? 2 : 1;
                        mbar_arrive_expect_tx(&xfull[s], (uint32_t)(nch * C::XCHUNK));
                    }
                    tc::tma_load_2d(smem + (size_t)s * C::XSTAGE + (size_t)h * C::XCHUNK, &tmx, c * kKC, m0,
                                    &xfull[s]);
                    if (++h == C::CPS || cn >= nchunks) {
                        h = 0;
                        ++st;
                    }
                    c = cn;
                }
            }
        }
    } else if (warp == kPWarpMma) {
        // ---------------- MMA issuer: tile i into accumulator i % NB
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16(PBN, BF);
            int st = 0, i = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x, ++i) {
                const int buf = i % C::NB;
                if (i >= C::NB && !mbar_wait_bounded(&dempty[buf], ((i / C::NB) - 1) & 1)) {
                    give_up();
                    break;
                }
                tc::fence_after_sync();
                const uint32_t dcol = tmem + (uint32_t)(C::DCOL0 + buf * PBN);
                int tlc = 0;  // live chunks of this tile
                for (int c = next_live(t, 0); c < nchunks; ++st) {
                    const int s = st % C::NA, xs = st % C::NS;
                    if (*abort_flag || !mbar_wait_bounded(&afull[s], (st / C::NA) & 1) ||
                        !mbar_wait_bounded(&xfull[xs], (st / C::NS) & 1)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    for (int h = 0; h < C::CPS && c < nchunks; ++h, ++tlc, c = next_live(t, c + 1)) {
                        const uint64_t bdesc =
                            tc::desc_sw128(smem + (size_t)xs * C::XSTAGE + (size_t)h * C::XCHUNK);
                        const uint32_t acol = tmem + (uint32_t)((s * C::CPS + h) * C::ACOLS);
#pragma unroll
                        for (int kk = 0; kk < kKC / 16; ++kk) {
                            const uint64_t b = bdesc + (uint64_t)(kk * 2);  // +32 B per 16 elements
                            tc::mma_ts(dcol, acol + kk * 8, b, idesc, (tlc | kk) != 0);
                            if constexpr (SMODE == kSplit) tc::mma_ts(dcol, acol + 32 + kk * 8, b, idesc, 1);
                        }
                    }
                    tc::commit(&aempty[s]);
                    tc::commit(&xempty[xs]);
                }
                if (ok) tc::commit(&dfull[buf]);
            }
        }
    } else if (warp < 4) {
        // ---------------- decoders: thread = weight row = TMEM lane
        const int row = warp * 32 + lane;
        const int64_t Kq = a.K >> 2;
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        const int ngk = a.K >> a.gshift;  // scale groups per row (G = 32, 64, 128 or 256)
        // A cursor walks the CTA's (tile, live chunk) sequence (tile t >= T marks its
        // end) and keeps this row's code address for its tile, so the division by
        // the token-tile count happens once per tile.
        int ct = blockIdx.x, cc = -1;
        const uint8_t *crow = nullptr;
        auto set_row = [&]() {
            bool ok;
            const int n = row_of(ct, row, ok);
            crow = ok ? a.packed + (int64_t)n * Kq : nullptr;
        };
        auto next = [&]() {
            cc = next_live(ct, cc + 1);
            while (cc >= nchunks) {
                ct += (int)gridDim.x;
                if (ct >= T) return;
                set_row();
                cc = next_live(ct, 0);
            }
        };
        auto load = [&]() -> uint4 {
            return (ct < T && crow != nullptr) ? *reinterpret_cast<const uint4 *>(crow + (size_t)cc * 16)
                                               : make_uint4(0, 0, 0, 0);
        };
        if (ct < T) {
            set_row();
            next();
        }
        // queue of the next kPF items: tile, chunk and codes (loads in flight), so a
        // load has kPF chunk times to arrive
        constexpr int kPF = 4;
        int it[kPF], ic[kPF];
        uint4 q[kPF];
#pragma unroll
        for (int k = 0; k < kPF; ++k) {
            it[k] = ct;
            ic[k] = cc;
            q[k] = load();
            if (ct < T) next();
        }
        // the decoded item's tile and, for group scales, its row's scale array
        int dt = -1;
        const uint16_t *srow = a.scale;
        bool drowok = false;
        int st = 0, h = 0;  // stage, and this chunk's place in it (stages do not span tiles)
        while (it[0] < T) {
            const int s = st % C::NA;
            const int t0 = it[0], c0 = ic[0];
            const uint4 codes = q[0];
#pragma unroll
            for (int k = 0; k + 1 < kPF; ++k) {
                it[k] = it[k + 1];
                ic[k] = ic[k + 1];
                q[k] = q[k + 1];
            }
            it[kPF - 1] = ct;
            ic[kPF - 1] = cc;
            q[kPF - 1] = load();
            if (ct < T) next();
            if constexpr (SMODE != kChannel) {
                if (t0 != dt) {
                    dt = t0;
                    const int n = row_of(t0, row, drowok);
                    srow = a.scale + (int64_t)(drowok ? n : 0) * ngk;
                }
            }
            uint32_t r[32];
            decode_word_adjacent(codes.x, r + 0);
            decode_word_adjacent(codes.y, r + 8);
            decode_word_adjacent(codes.z, r + 16);
            decode_word_adjacent(codes.w, r + 24);
            uint32_t rl[32];
            if constexpr (SMODE != kChannel) {
                // registers 0-15 hold k 0-31 of the chunk, 16-31 hold k 32-63 (one
                // scale each for 32-wide groups, the same one for wider groups)
                const uint16_t sb0 = drowok ? srow[(c0 * kKC) >> a.gshift] : (uint16_t)0;
                const uint16_t sb1 = drowok ? srow[(c0 * kKC + 32) >> a.gshift] : (uint16_t)0;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float sf = h2f(hf ? sb1 : sb0);
                    if constexpr (SMODE == kFold) {
                        const __half2 h2 = __half2half2(__float2half_rn(0.5f * sf));
#pragma unroll
                        for (int q = 16 * hf; q < 16 * hf + 16; ++q) {
                            __half2 v = *reinterpret_cast<__half2 *>(&r[q]);
                            v = __hmul2(v, h2);
                            r[q] = *reinterpret_cast<uint32_t *>(&v);
                        }
                    } else {
                        const __nv_bfloat16 hi = __float2bfloat16_rn(sf);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(sf - __bfloat162float(hi));
                        const __nv_bfloat162 h2 =
                            __bfloat162bfloat162(__float2bfloat16_rn(0.5f * __bfloat162float(hi)));
                        const __nv_bfloat162 l2 =
                            __bfloat162bfloat162(__float2bfloat16_rn(0.5f * __bfloat162float(lo)));
#pragma unroll
                        for (int q = 16 * hf; q < 16 * hf + 16; ++q) {
                            __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&r[q]);
                            __nv_bfloat162 vh = __hmul2(v, h2), vl = __hmul2(v, l2);
                            r[q] = *reinterpret_cast<uint32_t *>(&vh);
                            rl[q] = *reinterpret_cast<uint32_t *>(&vl);
                        }
                    }
                }
            }
            // wait results are made warp-uniform: tcgen05.st below is warp-collective
            bool ok = true;
            if (h == 0 && st >= C::NA)
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&aempty[s], ((st / C::NA) - 1) & 1));
            if (!ok) give_up();
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            const uint32_t acol = tlane + (uint32_t)((s * C::CPS + h) * C::ACOLS);
            tc::st_32x32b_x32(acol, r);
            if constexpr (SMODE == kSplit) tc::st_32x32b_x32(acol + 32, rl);
            // it[0] is now the next item: the stage ends with this chunk when it is
            // full or the next chunk belongs to another tile
            if (++h == C::CPS || it[0] != t0) {
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[s]);
                h = 0;
                ++st;
            }
        }
    } else {
        // ---------------- epilogue warps 4-7 (TMEM lane quarter warp % 4)
        const int e = warp - kPWarpEpi0, row = e * 32 + lane;
        float *ex = reinterpret_cast<float *>(smem + C::EX_OFF);  // [32 tokens][128 rows]
        int i = 0;
        for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
            const int buf = i % C::NB;
            bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&dfull[buf], (i / C::NB) & 1));
            if (!got) give_up();
            got = got && !*abort_flag;
            if constexpr (SILU) {
                // the four warps meet at barriers below: decide together (flags of
                // two parities, so a fast warp never overwrites one still being read)
                if (lane == 0) epi_flags[(i & 1) * 4 + e] = got ? 1 : 0;
                tile_named_bar(1, 128);
                got = epi_flags[(i & 1) * 4 + 0] && epi_flags[(i & 1) * 4 + 1] &&
                      epi_flags[(i & 1) * 4 + 2] && epi_flags[(i & 1) * 4 + 3];
            }
            if (!got) break;
            tc::fence_after_sync();
            bool rowok;
            const int n = row_of(t, row, rowok);
            const int m0 = tile_m0(t);
            const bool empty = next_live(t, 0) >= nchunks;  // no live chunk: D never written
            float sc = 1.f;  // channel mode: A held 2*t, so D = 2*sum(t x); group modes: A held t*s
            if constexpr (SMODE == kChannel) sc = 0.5f * (rowok ? h2f(a.scale[n]) : 0.f);
            const uint32_t dbase = tmem + (uint32_t)(C::DCOL0 + buf * PBN) + ((uint32_t)(e * 32) << 16);
#pragma unroll 1
            for (int j = 0; j < PBN / 32; ++j) {
                uint32_t d[32];
                tc::ld_32x32b_x32(dbase + (uint32_t)(j * 32), d);
                tc::wait_ld();
                if (j == PBN / 32 - 1) {  // every column is in registers: the issuer may reuse the buffer
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dempty[buf]);
                }
                if (empty) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) d[q] = 0u;
                }
                if constexpr (SILU) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) ex[q * 128 + row] = __uint_as_float(d[q]) * sc;
                    tile_named_bar(1, 128);
                    // thread: pair p = row % 64, tokens [16 h, 16 h + 16) of the 32, h = row / 64
                    const int p = row & 63, q0 = (row >> 6) * 16, j0 = tile_rb(t) * 64;
                    if (j0 + p < a.nh) {
#pragma unroll 4
                        for (int q = q0; q < q0 + 16; ++q) {
                            const int m = m0 + j * 32 + q;
                            if (m < a.M)
                                OutStore<OUT>::st(a.out, (int64_t)m * a.nh + j0 + p,
                                                  tile_silu(ex[q * 128 + p]) * ex[q * 128 + 64 + p]);
                        }
                    }
                    tile_named_bar(1, 128);
                } else if (rowok) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int m = m0 + j * 32 + q;
                        if (m < a.M) OutStore<OUT>::st(a.out, (int64_t)m * a.N + n, __uint_as_float(d[q]) * sc);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kPWarpMma) tc::tmem_dealloc(tmem, C::TMEM_COLS);
}

// Time of a 192-token chunk in the persistent kernel relative to a 256-token chunk
// in the one-tile-per-CTA kernel (measured on the 7B gate/up at M = 2048: 767 vs
// 882 cycles).
constexpr double kP192 = 0.87;

// Cost, in 64-k chunk times of a 256-token tile, of running `a` on the persistent
// kernel with PBN-token tiles: the busiest CTA's tiles x (chunks + a per-tile
// part), plus one CTA's fixed set-up.  With one accumulator (PBN = 256) the
// per-tile part holds the epilogue's read-out, which the issuer waits for: ~4
// chunk times for a plain output, ~25 for the gated one, whose 32-token
// exchange rounds all sit on that path (fitted to the 7B shapes at M = 1024 and
// 2048: q/k/v 28.0 / 51.9 us against 31.3 / 60.3 one tile per CTA; gate/up
// 568 us against 478 with 192-token tiles).
inline double persist_cost(const TileArgs &a, bool silu, int sm_count, int pbn = 192) {
    const int64_t rb = silu ? (a.nh + 63) / 64 : (a.N + 127) / 128;
    const int64_t tiles = rb * ((a.M + pbn - 1) / pbn);
    const int64_t ctas = tiles < sm_count ? tiles : sm_count;
    const int64_t per_cta = (tiles + ctas - 1) / ctas;
    if (pbn == 256) return (double)per_cta * (a.K / kKC + (silu ? 25.0 : 4.0)) + 12.0;
    return (double)per_cta * (a.K / kKC + 2.0) * kP192 + 18.0;
}

template <bool BF, int SMODE, int OUT, bool SILU, int PBN>
cudaError_t launch_persist_one(const TileArgs &a, int sm_count, cudaStream_t st, bool pdl) {
    using C = PCfg<SMODE, PBN>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)PBN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&map, BF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<uint16_t *>(a.x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = tile_persist_kernel<BF, SMODE, OUT, SILU, PBN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_REQ);
    if (e != cudaSuccess) return e;
    const int64_t rb = SILU ? (a.nh + 63) / 64 : (a.N + 127) / 128;
    const int64_t tiles = rb * ((a.M + PBN - 1) / PBN);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < sm_count ? tiles : sm_count), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_REQ;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    TileArgs b = a;
    b.sk = 1;
    b.cpc = a.K / kKC;
    return cudaLaunchKernelEx(&cfg, kern, map, b);
}

// pbn: 192 or 256 (256 with per-channel scales only; group scales take 192)
template <bool SILU>
cudaError_t launch_persist(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                           cudaStream_t st, bool pdl, int pbn = 192) {
    auto go = [&](auto bfc, auto smc) -> cudaError_t {
        constexpr bool B = decltype(bfc)::value;
        constexpr int S = decltype(smc)::value;
        if constexpr (S == kChannel) {
            if (pbn == 256) {
                switch (out_dtype) {
                case 0: return launch_persist_one<B, S, 0, SILU, 256>(a, sm_count, st, pdl);
                case 1: return launch_persist_one<B, S, 1, SILU, 256>(a, sm_count, st, pdl);
                default: return launch_persist_one<B, S, 2, SILU, 256>(a, sm_count, st, pdl);
                }
            }
        }
        switch (out_dtype) {
        case 0: return launch_persist_one<B, S, 0, SILU, 192>(a, sm_count, st, pdl);
        case 1: return launch_persist_one<B, S, 1, SILU, 192>(a, sm_count, st, pdl);
        default: return launch_persist_one<B, S, 2, SILU, 192>(a, sm_count, st, pdl);
        }
    };
    using T_ = std::true_type;
    using F_ = std::false_type;
    if (!group) return bf ? go(T_{}, std::integral_constant<int, kChannel>{})
                          : go(F_{}, std::integral_constant<int, kChannel>{});
    return bf ? go(T_{}, std::integral_constant<int, kSplit>{}) : go(F_{}, std::integral_constant<int, kFold>{});
}

}  // namespace

}  // namespace tl
