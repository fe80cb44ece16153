// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tl {

// ------------------------------------------------------------ pack / unpack
cudaError_t launch_unpack(const uint8_t *packed, int8_t *t, int64_t nbytes,
                          unsigned long long *reserved, int sm_count, cudaStream_t st);
cudaError_t launch_pack(const int8_t *t, uint8_t *packed, int64_t nbytes,
                        unsigned long long *invalid, int sm_count, cudaStream_t st);
// K % 4 != 0: rows of ceil(K/4) bytes, padding fields 00 on pack, skipped on unpack
cudaError_t launch_unpack_rows(const uint8_t *packed, int8_t *t, int64_t N, int64_t K,
                               unsigned long long *reserved, int sm_count, cudaStream_t st);
cudaError_t launch_pack_rows(const int8_t *t, uint8_t *packed, int64_t N, int64_t K,
                             unsigned long long *invalid, int sm_count, cudaStream_t st);

// ------------------------------------------------------------ zero-block map
// bit kb%32 of word [rb][kb/32]: rows [128 rb, +128) x k [64 kb, +64) hold a non-zero weight
constexpr int kMaskRows = 128, kMaskK = 64;
inline int mask_words(int64_t K) { return (int)((((K + 63) / 64) + 31) / 32); }
cudaError_t launch_block_mask(const uint8_t *packed, int64_t N, int64_t K, uint32_t *mask,
                              unsigned long long *zero_count, cudaStream_t st);

// ------------------------------------------------------------ skinny path
constexpr int kSkinnyWarps = 8;            // warps per CTA
constexpr int kSkinnyMaxCluster = 8;       // portable cluster size
constexpr int64_t kSkinnyMaxSmem = 200 * 1024;
constexpr int64_t kSkinnyTargetSmem = 100 * 1024;  // two CTAs per SM (overlap of layers)

// SkinnyArgs::flags
constexpr int kSkinnyStaticWeights = 1;  // packed/scale may be read before griddepcontrol.wait
constexpr int kSkinnyTriggerLate = 2;    // launch dependents after the main loop, not at entry
constexpr int kSkinnyTriggerNever = 8;   // no explicit trigger (dependents start at exit)

struct SkinnyArgs {
    const uint16_t *x;       // [M,K] fp16 or bf16 bits
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/G]
    void *out;               // [M,N]
    int M, N, K;
    int gshift;              // log2 of the group size G (7 or 8) in group mode
    int kc;                  // k per CTA (multiple of 128), set from the plan
    int row_stride;          // shared-memory bytes per staged packed row
    int x_off;               // byte offsets in shared memory: staged x fragments,
    int red_off;             //   per-warp partial tiles,
    int recv_off;            //   split-K receive buffer
    int flags;               // kSkinny* bits
    int xts;                 // token stride of the staged x fragments (1, 2, 4 or 8)
    int *status;             // device status word (bounded-wait failures)
};

struct SkinnyPlan {
    int nt8;           // 8-token MMA tiles
    int rows_per_cta;  // 16, 32, 64 or 128
    int sk;            // K split = cluster size
    int kc;            // k per CTA
    int row_stride;
    int x_off;
    int xts;
    size_t smem;
    int red_off;
    int recv_off;
    bool ok;
};

SkinnyPlan plan_skinny(int64_t M, int64_t N, int64_t K, int sm_count, int force_sk = 0);
cudaError_t launch_skinny(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                          const SkinnyPlan &p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------ skinny path, tensor cores
struct SkinnyTcArgs {
    const uint16_t *x;       // [M,K] fp16 or bf16 bits
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/G]
    void *out;               // [M,N]
    int M, N, K;
    int gshift;              // log2 of the group size G (7 or 8) in group mode
    int nh;                  // SiLU-gated call: gate rows [0, nh), up rows [nh, 2 nh), out [M, nh]
    int kc;                  // k per CTA (multiple of 128), set from the plan
    int flags;               // kSkinny* bits
    int *status;             // device status word (bounded-wait failures)
    const uint32_t *mask;    // zero-block map (channel scales only; nullptr: every block is read)
    int mask_words;          // map words per 128-row block
};

struct SkinnyTcPlan {
    int nt;         // MMA N (tokens padded to 16 or 32)
    int row_tiles;  // 128-row blocks
    int sk;         // K split = cluster size (<= 8)
    int kc;         // k per CTA
    bool ok;
};

SkinnyTcPlan plan_skinny_tc(int64_t M, int64_t N, int64_t K, int sm_count, int force_sk = 0,
                            int ctas_per_sm = 2);
cudaError_t launch_skinny_tc(const SkinnyTcArgs &a, bool bf, bool group, int out_dtype,
                             const SkinnyTcPlan &p, cudaStream_t st, bool pdl);
// SiLU-gated gate/up product: a.N = 2 * a.nh stacked rows, out [M, nh]; plan with
// plan_skinny_tc(M, 2 * nh, K, ...) (64 row pairs per CTA = 128 rows)
cudaError_t launch_skinny_silu(const SkinnyTcArgs &a, bool bf, bool group, int out_dtype,
                               const SkinnyTcPlan &p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------ decode path (gemv.cuh)
// GemvArgs::flags
constexpr int kGemvStaticWeights = 1;  // packed / scale may be read before griddepcontrol.wait
constexpr int kGemvTestStall = 2;      // testing aid: consumers first wait on a barrier nothing arrives on

struct GemvArgs {
    const uint16_t *x;       // [M,K] fp16 or bf16 bits
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/G]
    void *out;               // [M,N] (gated: [M,nh])
    int M, N, K;             // N = every stacked row (gated: 2 * nh)
    int gshift;              // log2 of the group size G (6, 7 or 8) in group mode
    int nh;                  // gated call: gate rows [0, nh), up rows [nh, 2 nh)
    int rg;                  // row groups (16 rows) per CTA, from the plan
    int kc;                  // k per CTA (multiple of 256), from the plan
    int ws;                  // weight stages in the ring, from the plan
    int flags;               // kGemv* bits
    int odt;                 // output dtype: 0 fp16, 1 bf16, 2 fp32
    int *status;             // device status word (bounded-wait failures)
    long long wait_limit;    // give-up time of the main-loop waits, SM cycles
    const uint32_t *mask;    // zero-block map of packed (nullptr: every block is read)
    int mask_words;          // map words per 128-row block
};

struct GemvPlan {
    int nt8;    // 8-token MMA tiles (1 or 2)
    int rg;     // row groups per CTA
    int tiles;  // row blocks (grid x)
    int sk;     // K split = cluster size (grid y)
    int kc;     // k per CTA
    int ws;     // ring stages
    bool ok;
};

constexpr int kGemvMaxM = 16;
// rows = stacked weight rows (gated: 2 * nh); gated plans pair rows within a CTA
GemvPlan plan_gemv(int64_t M, int64_t rows, int64_t K, int sm_count, bool gated, bool group,
                   int force_sk = 0);
// a.odt selects the output dtype
cudaError_t launch_gemv(const GemvArgs &a, bool bf, bool group, const GemvPlan &p, cudaStream_t st,
                        bool pdl);
cudaError_t launch_gemv_silu(const GemvArgs &a, bool bf, bool group, const GemvPlan &p,
                             cudaStream_t st, bool pdl);

// ------------------------------------------------------------ tile path
struct TileArgs {
    const uint16_t *x;       // [M,K]
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/G]
    void *out;               // [M,N]
    int M, N, K;
    int gshift;              // log2 of the group size G (6, 7 or 8) in group mode
    int nh;                  // SiLU-gated call: gate rows [0, nh), up rows [nh, 2 nh), out [M, nh]
    int *status;             // device status word (bounded-wait failures)
    const uint32_t *mask;    // zero-block map of packed (nullptr: every block is read)
    int mask_words;          // map words per 128-row block
    int sk;                  // K split = cluster size along grid z (set by the launcher)
    int cpc;                 // 64-k chunks per CTA of the split (set by the launcher)
    int persist;             // -1: the launcher decides; 0: one tile per CTA; 1: persistent CTAs,
                             // 192-token tiles; 2: persistent, 256-token tiles (per-channel scales)
};

bool tile_supported(int64_t M, int64_t N, int64_t K);  // K % 64 == 0
cudaError_t launch_tile(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                        cudaStream_t st, bool pdl);
// SiLU-gated gate/up product on the tile kernel: a.N = 2 * a.nh stacked rows, out [M, nh]
cudaError_t launch_tile_silu(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                             cudaStream_t st, bool pdl);

// ------------------------------------------------------------ generic path (K % 64 != 0)
struct GenArgs {
    const uint16_t *x;       // [M,K] fp16 or bf16 bits
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/G]
    void *out;               // [M,N] (gated: [M,nh])
    int M, N, K;             // packed rows of ceil(K/4) bytes; N = every stacked row (gated: 2 * nh)
    int gshift;              // log2 of the group size G (5, 6, 7 or 8) in group mode
    int nh;                  // gated call: gate rows [0, nh), up rows [nh, 2 nh)
    int odt;                 // output dtype: 0 fp16, 1 bf16, 2 fp32
};
cudaError_t launch_generic(const GenArgs &a, bool bf, bool group, bool silu, cudaStream_t st,
                           bool pdl);

}  // namespace tl
