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

// ------------------------------------------------------------ skinny path
constexpr int kSkinnyThreads = 128;        // 4 warps, 16*MT rows each
constexpr int kSkinnyMaxCluster = 8;       // portable cluster size
constexpr int64_t kSkinnyMaxSmem = 200 * 1024;

struct SkinnyArgs {
    const uint16_t *x;       // [M,K] fp16 or bf16 bits
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/128]
    void *out;               // [M,N]
    int M, N, K;
    int kc;                  // k per CTA (multiple of 128), set from the plan
};

struct SkinnyPlan {
    int nt8;           // 8-token MMA tiles
    int mt;            // 16-row MMA tiles per warp
    int rows_per_cta;
    int sk;            // K split = cluster size
    int kc;            // k per CTA
    size_t smem;
    bool ok;
};

SkinnyPlan plan_skinny(int64_t M, int64_t N, int64_t K, int sm_count);
cudaError_t launch_skinny(const SkinnyArgs &a, bool bf, bool group, int out_dtype,
                          const SkinnyPlan &p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------ tile path
struct TileArgs {
    const uint16_t *x;       // [M,K]
    const uint8_t *packed;   // [N,K/4]
    const uint16_t *scale;   // fp16 [N] or [N,K/128]
    void *out;               // [M,N]
    int M, N, K;
    int *status;             // device status word (bounded-wait failures)
};

bool tile_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_tile(const TileArgs &a, bool bf, bool group, int out_dtype, int sm_count,
                        cudaStream_t st, bool pdl);

}  // namespace tl
