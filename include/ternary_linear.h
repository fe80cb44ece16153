/*
 * ternary_linear.h -- C ABI of libternary_gb300.so, a ternary-weight linear
 * layer for NVIDIA GB300 (sm_103a).
 *
 * Format (all calls): a weight matrix W[N,K] with entries in {-1,0,+1} is
 * stored packed as uint8 [N, ceil(K/4)], row-major, K contiguous (written
 * [N, K/4] below: the two agree when K % 4 == 0).  Weight k of row n is the
 * 2-bit field (packed[n, k/4] >> 2*(k%4)) & 3 -- four weights per byte,
 * little-endian, first weight in the lowest two bits -- with the code table
 * 00 -> 0, 01 -> +1, 10 -> -1, 11 -> reserved, read as 0.  When K % 4 != 0 the
 * last byte of a row holds K % 4 weights and 4 - K % 4 padding fields, which no
 * call reads as weights (pack writes them 00).
 *   Source: "三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战"
 *   (trdm.cn/news/729035) §2.2, §3.1; the Qwen2.5-7B ternary-in-vLLM write-up
 *   (m.nxbn.cn/news/169761) §2.1, §2.2, and §2.3 for the padding (an export
 *   pads rows to whole bytes; the padding is cut off after unpacking).
 *
 * Conventions shared by every entry point:
 *   - Pointers named in the signature are DEVICE pointers (cudaMalloc'd or
 *     otherwise device-accessible) unless stated otherwise.  The caller owns
 *     every buffer; the library allocates nothing on these paths except one
 *     4-byte device status word per device, created on the first call to
 *     ternary_linear on that device (make that first call before any stream
 *     capture).
 *   - Arrays are dense row-major with no padding; pointers must be 16-byte
 *     aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued asynchronously on it; no call synchronises.
 *   - Argument errors are detected on the host before anything is enqueued; the
 *     call then returns the error code and writes nothing.
 *   - Launch failures return TL_ERR_CUDA (the CUDA error is cleared).
 */
#ifndef TERNARY_LINEAR_H
#define TERNARY_LINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TL_OK = 0,
    TL_ERR_NULL = 1,        /* a required pointer is NULL                        */
    TL_ERR_SHAPE = 2,       /* negative size, K not a multiple of the
                               group size, or a size beyond the supported range  */
    TL_ERR_DTYPE = 3,       /* unknown dtype code or unsupported group size      */
    TL_ERR_ALIGN = 4,       /* pointer not 16-byte aligned                      */
    TL_ERR_VALUE = 5,       /* reserved for callers mapping a non-zero invalid /
                               reserved count to an error                        */
    TL_ERR_CUDA = 6,        /* a CUDA runtime call or a kernel launch failed     */
    TL_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (see
                               ternary_device_status)                            */
    TL_ERR_UNSUPPORTED = 8  /* no sm_103 device current, or a path that cannot
                               serve the arguments was forced                    */
} tl_status;

typedef enum { TL_F16 = 0, TL_BF16 = 1, TL_F32 = 2 } tl_dtype;

/* Kernel path selection for ternary_linear_path. */
typedef enum {
    TL_PATH_AUTO = 0,    /* skinny path for M <= ternary_skinny_max_m(), else tile */
    TL_PATH_SKINNY = 1,  /* fused decode + register-fed MMA GEMV / skinny GEMM     */
    TL_PATH_TILE = 2,    /* TMA + tcgen05 + TMEM tile GEMM                          */
    TL_PATH_GENERIC = 3  /* CUDA-core kernel for any K (the one TL_PATH_AUTO
                            uses when K % 64 != 0); SKINNY and TILE need K % 64 == 0 */
} tl_path;

/*
 * ternary_pack -- t [N,K] int8 in {-1,0,+1}  ->  packed [N,K/4] uint8.
 *   Writes 00 for 0, 01 for +1, 10 for -1; never writes the reserved code 11.
 *   ("三元量化模型接入vLLM…完整实战" §3.1.)
 *   An entry outside {-1,0,+1} is written as 00 and counted.
 *   invalid_count: device int64, may be NULL.  When non-NULL the library sets
 *   it to zero on `stream` and then adds the number of invalid entries; read it
 *   after synchronising `stream`.
 *   Any K >= 0 (padding fields of a K % 4 != 0 row are written 00).  N == 0 or
 *   K == 0 enqueues only the count reset.
 */
tl_status ternary_pack(const int8_t *t, uint8_t *packed, int64_t N, int64_t K,
                       int64_t *invalid_count, void *stream);

/*
 * ternary_unpack -- packed [N,K/4] uint8  ->  t [N,K] int8 in {-1,0,+1}.
 *   Bit-exact decode with the code table above; 11 decodes to 0 and is counted.
 *   ("三元量化模型接入vLLM…完整实战" §3.1; Qwen2.5-7B write-up §2.2.)
 *   reserved_count: device int64, may be NULL; reset to zero on `stream`, then
 *   the number of 11 fields is added.
 *   Any K >= 0: padding fields of a K % 4 != 0 row are neither decoded nor
 *   counted.
 */
tl_status ternary_unpack(const uint8_t *packed, int8_t *t, int64_t N, int64_t K,
                         int64_t *reserved_count, void *stream);

/*
 * ternary_linear -- out[M,N] = x[M,K] * W^T with W = t * scale.
 *   group_size == 0   : per-output-channel scale, scale is fp16 [N]
 *                       out[m,n] = scale[n] * sum_k t[n,k] x[m,k]
 *                       (Qwen2.5-7B write-up §3.2, §4.2)
 *   group_size == 128 : per-(row, 128-wide K group) scale, scale is fp16 [N, K/128]
 *                       out[m,n] = sum_g scale[n,g] * sum_{k in group g} t[n,k] x[m,k]
 *                       ("三元量化模型接入vLLM…完整实战" §1.1, §3.1, §4.2)
 *   group_size == 64  : the same with 64-wide groups, scale fp16 [N, K/64]
 *                       ("Bonsai 2 27B" port §4.2, §5.2); the skinny path
 *                       serves it for M <= 16, the tile kernel above
 *   group_size == 32  : the same with 32-wide groups, scale fp16 [N, K/32]
 *                       (the finer per-group choice of "第13章 量化：精度与速度的
 *                       工程平衡" §13.3.3); served by the tile kernel at every M
 *   group_size == 256 : the same with 256-wide groups, scale fp16 [N, K/256]
 *                       (the coarser per-group choice of "第13章 量化：精度与速度的
 *                       工程平衡" §13.3.3); every path serves it
 *   Any other group_size returns TL_ERR_DTYPE.
 *   x_dtype  : TL_F16 or TL_BF16.  scale is always fp16.
 *   out_dtype: TL_F16, TL_BF16 or TL_F32.  Accumulation is fp32; a 16-bit
 *              output is rounded to nearest even from fp32.
 *   Sizes: M, N >= 0; K >= 0 (a multiple of the group size in group mode, so
 *   K % 4 != 0 is per-channel only).  M == 0 or N == 0 is a no-op; K == 0 writes zeros.
 *   K % 64 != 0 (packed rows not 16-byte pitched: the Qwen2.5-7B write-up §2.3
 *   notes input widths that do not fit the packing neatly) runs on the generic
 *   CUDA-core kernel, whose reads need no alignment beyond the element's; the
 *   16-byte pointer rule above still applies to every call.
 *   Fused layers (QKV, gate/up) are one call over the stacked rows: shard i
 *   occupies rows [off_i, off_i + N_i) of packed and of scale, and columns
 *   [off_i, off_i + N_i) of out.
 *   Non-finite x is outside the contract.
 */
tl_status ternary_linear(const void *x, int32_t x_dtype, const uint8_t *packed,
                         const void *scale, int32_t group_size, void *out,
                         int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                         void *stream);

/* Flags for ternary_linear_ex. */
typedef enum {
    /* packed and scale (and, for the masked calls, the zero-block map) are not
     * written by any work still running on `stream` when this call's kernel
     * starts (true for model weights loaded once).  Lets the kernel read them
     * before its stream predecessor has finished (programmatic dependent
     * launch), overlapping consecutive layers. */
    TL_FLAG_STATIC_WEIGHTS = 1
} tl_flags;

/* ternary_linear with an explicit kernel path (tl_path) and tl_flags bits.
 * Returns TL_ERR_UNSUPPORTED if the forced path cannot serve the arguments
 * (the skinny path serves M <= 32 with groups of 64 only for M <= 16 and no
 * 32-wide groups; SKINNY and TILE need K % 64 == 0), TL_ERR_DTYPE for an
 * unknown path or flag bit.  ternary_linear(...) == ternary_linear_ex(..., TL_PATH_AUTO, 0, stream). */
tl_status ternary_linear_ex(const void *x, int32_t x_dtype, const uint8_t *packed,
                            const void *scale, int32_t group_size, void *out,
                            int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                            int32_t path, uint32_t flags, void *stream);

/*
 * ternary_linear_silu_mul -- a fused gate/up layer followed by the SiLU-gated
 * product that feeds the down projection:
 *   g = ternary_linear over rows [0, N)  of packed / scale  (gate shard)
 *   u = ternary_linear over rows [N, 2N) of packed / scale  (up shard)
 *   out[m, j] = silu(g[m, j]) * u[m, j],  silu(v) = v / (1 + exp(-v)),  j < N
 * The stacked layout is the fused gate/up layer of ternary_linear (shards at
 * row offsets 0 and N; "三元量化模型接入vLLM…完整实战" §3.2).
 *   packed: [2N, K/4]; scale: fp16 [2N] (group_size 0) or [2N, K/G] (G = 32,
 *   64, 128 or 256); out: [M, N] in out_dtype; g and u are fp32 (scaled) and the
 *   product is computed in fp32, then rounded to out_dtype.
 *   flags: TL_FLAG_STATIC_WEIGHTS or 0.
 * Decode shapes run on the decode kernel, the rest on the tile kernel (K % 64
 * != 0: the generic kernel), each with the product in its epilogue.
 * Argument errors as ternary_linear (with 2N rows).  N == 0 or M == 0 is a
 * no-op; K == 0 writes zeros.  Asynchronous on stream.
 */
tl_status ternary_linear_silu_mul(const void *x, int32_t x_dtype, const uint8_t *packed,
                                  const void *scale, int32_t group_size, void *out,
                                  int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                                  uint32_t flags, void *stream);

/*
 * Zero-block map -- skipping all-zero weight blocks ("三元量化模型接入vLLM…完整实战"
 * §6: ternary weights often come with sparse structure; a mask of zero blocks
 * lets the kernel skip them).
 *
 * ternary_block_mask -- build the map of packed [N, K/4]: block (rb, kb) covers
 *   rows [128*rb, 128*rb + 128) and weights k in [64*kb, 64*kb + 64), clipped to
 *   the matrix; its bit (bit kb%32 of word mask[rb * W + kb/32], W =
 *   ceil(ceil(K/64) / 32)) is 1 when any weight in it decodes to a non-zero value
 *   (a block of 00 and 11 codes is a zero block).  mask: device uint32
 *   [ternary_block_mask_words(N, K)], written entirely.  zero_blocks: device
 *   int64, may be NULL; reset on `stream`, then the number of zero blocks is
 *   added.  Any K >= 0 (padding fields never light a block); reads the
 *   packed matrix once (HBM-bound).
 *   Errors: TL_ERR_SHAPE, TL_ERR_NULL, TL_ERR_ALIGN (mask not 4-byte or count
 *   not 8-byte aligned), TL_ERR_CUDA.  Asynchronous on stream.
 */
int64_t ternary_block_mask_words(int64_t N, int64_t K);  /* -1 for invalid sizes */
tl_status ternary_block_mask(const uint8_t *packed, int64_t N, int64_t K, uint32_t *mask,
                             int64_t *zero_blocks, void *stream);

/*
 * ternary_linear_masked / ternary_linear_silu_mul_masked -- ternary_linear and
 * ternary_linear_silu_mul (same arguments, TL_PATH_AUTO) that read the zero-block
 * map `mask` of the same packed matrix (for the gated call: of all 2N stacked
 * rows) and neither load nor multiply blocks whose bit is 0 (a zero bit is the
 * caller's promise that the block's weights are zero).  With per-channel scales
 * and with 64-wide groups the masked call runs on the kernel the unmasked call
 * runs on; with 128- and 256-wide groups the tcgen05 skinny kernel reads no map,
 * so masked calls at M <= 32 run on the decode kernel (M <= 16) or the tile
 * kernel.  With the map that ternary_block_mask built, the result equals the
 * unmasked call's bit for bit whenever both run on the same kernel (up to the
 * sign of an exact zero), and agrees within the stated tolerance otherwise.
 * mask: device, 4-byte aligned, NULL only when nothing is computed.
 */
tl_status ternary_linear_masked(const void *x, int32_t x_dtype, const uint8_t *packed,
                                const void *scale, int32_t group_size, const uint32_t *mask,
                                void *out, int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                                uint32_t flags, void *stream);
tl_status ternary_linear_silu_mul_masked(const void *x, int32_t x_dtype, const uint8_t *packed,
                                         const void *scale, int32_t group_size,
                                         const uint32_t *mask, void *out, int32_t out_dtype,
                                         int64_t M, int64_t N, int64_t K, uint32_t flags,
                                         void *stream);

/* Kernels by M (TL_PATH_AUTO, K % 64 == 0): M <= 16 -> the decode kernel
 * (register-fed warp MMAs, TMA-staged weights) or, for 9 <= M and for plain
 * layers of 2049..4608 rows at M <= 8, the tcgen05 skinny kernel (groups 0 /
 * 128 / 256; a zero-block map only with per-channel scales: whichever was
 * measured faster on the 7B and 27B shapes); 17 <= M <= 32 -> the tcgen05
 * skinny kernel (64-wide groups: tile kernel); larger M -> the tcgen05 tile
 * kernel.  32-wide groups run on the tile
 * kernel at every M; K % 64 != 0 runs on the generic kernel at every M, which
 * reads no zero-block map (the masked calls then equal the unmasked ones
 * trivially). */

/* Largest M the automatic dispatch sends to the skinny path (default 32,
 * overridable with the environment variable TERNARY_SKINNY_MAX_M, read once). */
int32_t ternary_skinny_max_m(void);

/*
 * ternary_device_status -- read (and optionally clear) the current device's
 * status word.  Kernels whose waits are bounded write a non-zero code there
 * when a wait gives up; *code receives TL_OK or TL_ERR_TIMEOUT.  Synchronous:
 * call after the work in question has completed (e.g. after a stream sync).
 */
tl_status ternary_device_status(int32_t *code, int32_t clear);

/*
 * ternary_device_status_async -- enqueue on `stream` a copy of the current
 * device's status word into *dst (device memory or pinned host memory, 4-byte
 * aligned; the raw word: 0 = OK, 7 = a bounded wait gave up), then, if clear is
 * non-zero, reset the word.  The copy is ordered after the work already on
 * `stream`, so a non-zero value read after synchronising `stream` was set by
 * that work or by work on another stream that ran before it.  Asynchronous.
 * Errors: TL_ERR_NULL (dst NULL), TL_ERR_ALIGN, TL_ERR_CUDA,
 * TL_ERR_UNSUPPORTED (no sm_103 device).
 */
tl_status ternary_device_status_async(int32_t *dst, int32_t clear, void *stream);

/* Human-readable name of a tl_status value (static storage, never NULL). */
const char *ternary_status_string(int32_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t ternary_version(void);

/* Testing aid (host only): the next n calls that pass argument validation
 * return TL_ERR_CUDA without touching CUDA, as a failed launch would.  Lets
 * error handling above the ABI be exercised without a GPU fault. */
void ternary_test_inject_launch_failures(int32_t n);

/* Testing aid: the give-up time, in SM clock cycles, of the decode kernel's
 * main-loop waits for every later launch (cycles <= 0 restores the default of
 * about 2^30 cycles, ~0.5 s).  stall != 0 additionally makes each of those
 * launches first wait on a barrier that nothing arrives on, so the wait runs
 * out: the call then writes no output and sets the device status word to
 * TL_ERR_TIMEOUT, while every copy in flight still lands before the kernel
 * exits (those waits keep the default limit).  Lets the give-up path be tested
 * without a fault or a hang. */
void ternary_test_set_wait_limit(int64_t cycles, int32_t stall);

/* Testing aid: the form of the tile kernel for every later call that runs on
 * it: 0 = chosen per call by the library (default), 1 = one output tile per
 * CTA (with split K where planned), 2 = persistent CTAs (one per SM, each
 * walking a list of 128-row x 192-token tiles, two accumulators), 3 = persistent
 * CTAs with 128-row x 256-token tiles and one accumulator (per-channel scales;
 * group scales take 2).  All forms compute the same sums; any other value
 * restores 0.  Lets tests cover every form on any shape. */
void ternary_test_set_tile_mode(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* TERNARY_LINEAR_H */
