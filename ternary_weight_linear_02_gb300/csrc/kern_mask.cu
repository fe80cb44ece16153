// kern_mask.cu -- the zero-block map of a packed weight matrix, for skipping
// all-zero blocks in the linear kernels ("三元量化模型接入vLLM：从逆向加载到
// Kernel优化的完整实战", trdm.cn/news/729035, §6: ternary weights often come
// with sparse structure, and a mask of zero blocks lets the kernel skip them).
//
// Block (rb, kb) = rows [128 rb, 128 rb + 128) x weights k in [64 kb, 64 kb + 64)
// (16 packed bytes per row), clipped to the matrix.  Its bit is set when any of
// its weights decodes to a non-zero value: with code bits (b1 b0) a weight is
// non-zero exactly when b0 != b1, so a byte holds a non-zero weight when
// (byte ^ (byte >> 1)) & 0x55 != 0.
//
// Rows are ceil(K/4) bytes; when K % 4 != 0 the last byte's fields past K are
// padding (the Qwen2.5-7B write-up §2.3) and are masked off before the test.
//
// One thread per block: a warp covers 32 consecutive k-blocks of one row block
// (512 contiguous bytes of each row, so its loads are coalesced) and writes
// one 32-bit word of the map with a ballot.  HBM-bound: the packed matrix is
// read once.
#include "common.cuh"
#include "kernels.h"

namespace tl {

__global__ void __launch_bounds__(256) block_mask_kernel(const uint8_t *packed, int64_t N, int64_t K,
                                                         int words, uint32_t *mask,
                                                         unsigned long long *zero_count) {
    const int lane = threadIdx.x & 31;
    const int64_t rb = blockIdx.x;
    const int w = blockIdx.y * 8 + (threadIdx.x >> 5);  // map word of this warp
    if (w >= words) return;
    const int64_t Kq = (K + 3) >> 2;                    // bytes per packed row
    // weight fields of the row's last byte (padding fields cleared)
    const uint32_t last = (K & 3) ? (1u << (2 * (K & 3))) - 1u : 0xFFu;
    const int64_t KB = (K + 63) >> 6;
    const int64_t kb = (int64_t)w * 32 + lane;
    const bool valid = kb < KB;
    uint32_t nz = 0;
    if (valid) {
        const int64_t b0 = kb * 16, b1 = b0 + 16 < Kq ? b0 + 16 : Kq;
        const int64_t r0 = rb * 128, r1 = r0 + 128 < N ? r0 + 128 : N;
        if ((K & 63) == 0) {  // whole 16-byte segments, no padding
            for (int64_t n = r0; n < r1; ++n) {
                const uint4 v = ldg_nc_v4(packed + n * Kq + b0);
                nz |= ((v.x ^ (v.x >> 1)) | (v.y ^ (v.y >> 1)) | (v.z ^ (v.z >> 1)) |
                       (v.w ^ (v.w >> 1))) & 0x55555555u;
            }
        } else {
            for (int64_t n = r0; n < r1; ++n)
                for (int64_t b = b0; b < b1; ++b) {
                    const uint32_t v = packed[n * Kq + b] & (b == Kq - 1 ? last : 0xFFu);
                    nz |= (v ^ (v >> 1)) & 0x55u;
                }
        }
    }
    const uint32_t live = __ballot_sync(0xffffffffu, valid && nz != 0);
    const uint32_t inside = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) {
        mask[rb * words + w] = live;
        if (zero_count) atomicAdd(zero_count, (unsigned long long)__popc(inside & ~live));
    }
}

cudaError_t launch_block_mask(const uint8_t *packed, int64_t N, int64_t K, uint32_t *mask,
                              unsigned long long *zero_count, cudaStream_t st) {
    const int64_t RB = (N + 127) / 128;
    const int words = (int)((((K + 63) / 64) + 31) / 32);
    if (RB == 0 || words == 0) return cudaSuccess;
    dim3 grid((unsigned)RB, (unsigned)((words + 7) / 8), 1);
    block_mask_kernel<<<grid, 256, 0, st>>>(packed, N, K, words, mask, zero_count);
    return cudaGetLastError();
}

}  // namespace tl
