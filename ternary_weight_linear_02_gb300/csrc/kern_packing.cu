// kern_packing.cu -- ternary_pack / ternary_unpack kernels.
//
// Code table and byte layout: "三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战"
// (trdm.cn/news/729035) §3.1; the Qwen2.5-7B ternary-in-vLLM write-up
// (m.nxbn.cn/news/169761) §2.2 (reserved code counted as a format check).
//
// K % 4 == 0: both kernels are pure streaming: packed byte i holds the four
// weights 4i..4i+3 of the flattened [N,K] matrix (rows are dense, so the row
// split does not matter).  One thread handles 16 packed bytes (one 16-byte
// load) and the 64 int8 weights they expand to; a scalar loop covers the
// ragged tail.  The grid is a multiple of the SM count, grid-striding over the
// array.
//
// K % 4 != 0: a row takes ceil(K/4) bytes and the last byte's fields past K are
// padding (the Qwen2.5-7B write-up §2.3: an export pads rows to whole bytes and
// the padding is cut off after unpacking).  The *_rows kernels take one packed
// byte per thread; pack writes padding fields as 00, unpack neither writes nor
// counts them.
#include "common.cuh"

namespace tl {

// byte b (0..255, in the low 8 bits of `b`) -> four int8 weights in one word,
// weight j in byte j.  value = b0 - b1 for every code (11 -> 1-1 = 0).
__device__ __forceinline__ uint32_t unpack_byte(uint32_t b) {
    // move field j to bits [8j+1 : 8j]
    uint32_t s = (b & 0x3u) | ((b & 0xCu) << 6) | ((b & 0x30u) << 12) | ((b & 0xC0u) << 18);
    uint32_t lo = s & 0x01010101u;          // b0 of each field
    uint32_t hi = (s >> 1) & 0x01010101u;   // b1 of each field
    return __vsub4(lo, hi);                 // per-byte b0 - b1 (wraps to 0xFF for -1)
}

__device__ __forceinline__ uint32_t reserved_in_byte(uint32_t b) {
    uint32_t both = b & (b >> 1) & 0x55u;   // fields whose two bits are both set
    return __popc(both);
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t *__restrict__ packed,
                                                     int8_t *__restrict__ t, int64_t nbytes,
                                                     unsigned long long *reserved) {
    const int64_t nvec = nbytes / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t cnt = 0;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        uint4 in = *reinterpret_cast<const uint4 *>(packed + v * 16);
        uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint4 *dst = reinterpret_cast<uint4 *>(t + v * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = unpack_byte(w[q] & 0xFFu);
            o.y = unpack_byte((w[q] >> 8) & 0xFFu);
            o.z = unpack_byte((w[q] >> 16) & 0xFFu);
            o.w = unpack_byte(w[q] >> 24);
            if (reserved) {
                cnt += reserved_in_byte(w[q] & 0xFFu) + reserved_in_byte((w[q] >> 8) & 0xFFu) +
                       reserved_in_byte((w[q] >> 16) & 0xFFu) + reserved_in_byte(w[q] >> 24);
            }
            dst[q] = o;
        }
    }
    // ragged tail: bytes [16*nvec, nbytes)
    for (int64_t i = nvec * 16 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes;
         i += stride) {
        uint32_t b = packed[i];
        uint32_t o = unpack_byte(b);
        t[4 * i + 0] = (int8_t)(o & 0xFF);
        t[4 * i + 1] = (int8_t)((o >> 8) & 0xFF);
        t[4 * i + 2] = (int8_t)((o >> 16) & 0xFF);
        t[4 * i + 3] = (int8_t)(o >> 24);
        if (reserved) cnt += reserved_in_byte(b);
    }
    if (reserved) {
        for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(reserved, (unsigned long long)cnt);
    }
}

// four int8 weights (one per byte of w) -> one packed byte; counts entries
// outside {-1,0,+1}, which are written as 00.
__device__ __forceinline__ uint32_t pack_word(uint32_t w, uint32_t &invalid) {
    uint32_t pos = __vcmpeq4(w, 0x01010101u);   // 0xFF where +1
    uint32_t neg = __vcmpeq4(w, 0xFFFFFFFFu);   // 0xFF where -1
    uint32_t zer = __vcmpeq4(w, 0u);
    invalid += 4u - (uint32_t)__popc((pos | neg | zer) & 0x01010101u);
    uint32_t c = (pos & 0x01010101u) | (neg & 0x02020202u);  // code j in byte j
    return (c & 0x3u) | ((c >> 6) & 0xCu) | ((c >> 12) & 0x30u) | ((c >> 18) & 0xC0u);
}

__global__ void __launch_bounds__(256) pack_kernel(const int8_t *__restrict__ t,
                                                   uint8_t *__restrict__ packed, int64_t nbytes,
                                                   unsigned long long *invalid_out) {
    const int64_t nvec = nbytes / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t bad = 0;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        const uint4 *src = reinterpret_cast<const uint4 *>(t + v * 64);
        uint32_t ob[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 in = src[q];
            ob[q] = pack_word(in.x, bad) | (pack_word(in.y, bad) << 8) |
                    (pack_word(in.z, bad) << 16) | (pack_word(in.w, bad) << 24);
        }
        *reinterpret_cast<uint4 *>(packed + v * 16) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
    for (int64_t i = nvec * 16 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes;
         i += stride) {
        uint32_t w = (uint32_t)(uint8_t)t[4 * i] | ((uint32_t)(uint8_t)t[4 * i + 1] << 8) |
                     ((uint32_t)(uint8_t)t[4 * i + 2] << 16) |
                     ((uint32_t)(uint8_t)t[4 * i + 3] << 24);
        packed[i] = (uint8_t)pack_word(w, bad);
    }
    if (invalid_out) {
        for (int off = 16; off; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(invalid_out, (unsigned long long)bad);
    }
}

__global__ void __launch_bounds__(256) unpack_rows_kernel(const uint8_t *__restrict__ packed,
                                                          int8_t *__restrict__ t, int64_t N,
                                                          int64_t K, unsigned long long *reserved) {
    const int64_t Kq = (K + 3) >> 2, nbytes = N * Kq;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t cnt = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes; i += stride) {
        const int64_t n = i / Kq, b = i - n * Kq;
        const int nf = (int)min((int64_t)4, K - 4 * b);  // fields of this byte that are weights
        uint32_t byte = packed[i];
        if (nf < 4) byte &= (1u << (2 * nf)) - 1u;       // drop the padding fields
        const uint32_t o = unpack_byte(byte);
        int8_t *dst = t + n * K + 4 * b;
        for (int j = 0; j < nf; ++j) dst[j] = (int8_t)((o >> (8 * j)) & 0xFFu);
        if (reserved) cnt += reserved_in_byte(byte);
    }
    if (reserved) {
        for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(reserved, (unsigned long long)cnt);
    }
}

__global__ void __launch_bounds__(256) pack_rows_kernel(const int8_t *__restrict__ t,
                                                        uint8_t *__restrict__ packed, int64_t N,
                                                        int64_t K, unsigned long long *invalid_out) {
    const int64_t Kq = (K + 3) >> 2, nbytes = N * Kq;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t bad = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes; i += stride) {
        const int64_t n = i / Kq, b = i - n * Kq;
        const int nf = (int)min((int64_t)4, K - 4 * b);
        const int8_t *src = t + n * K + 4 * b;
        uint32_t w = 0;  // padding lanes stay 0: written 00, never counted invalid
        for (int j = 0; j < nf; ++j) w |= (uint32_t)(uint8_t)src[j] << (8 * j);
        packed[i] = (uint8_t)pack_word(w, bad);
    }
    if (invalid_out) {
        for (int off = 16; off; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
        if ((threadIdx.x & 31) == 0 && bad) atomicAdd(invalid_out, (unsigned long long)bad);
    }
}

static int grid_for(int64_t work_items, int sm_count) {
    int64_t blocks = (work_items + 255) / 256;
    int64_t cap = (int64_t)sm_count * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

cudaError_t launch_unpack(const uint8_t *packed, int8_t *t, int64_t nbytes,
                          unsigned long long *reserved, int sm_count, cudaStream_t st) {
    int64_t items = nbytes / 16 > 0 ? nbytes / 16 : nbytes;
    unpack_kernel<<<grid_for(items, sm_count), 256, 0, st>>>(packed, t, nbytes, reserved);
    return cudaGetLastError();
}

cudaError_t launch_pack(const int8_t *t, uint8_t *packed, int64_t nbytes,
                        unsigned long long *invalid, int sm_count, cudaStream_t st) {
    int64_t items = nbytes / 16 > 0 ? nbytes / 16 : nbytes;
    pack_kernel<<<grid_for(items, sm_count), 256, 0, st>>>(t, packed, nbytes, invalid);
    return cudaGetLastError();
}

cudaError_t launch_unpack_rows(const uint8_t *packed, int8_t *t, int64_t N, int64_t K,
                               unsigned long long *reserved, int sm_count, cudaStream_t st) {
    unpack_rows_kernel<<<grid_for(N * ((K + 3) / 4), sm_count), 256, 0, st>>>(packed, t, N, K,
                                                                             reserved);
    return cudaGetLastError();
}

cudaError_t launch_pack_rows(const int8_t *t, uint8_t *packed, int64_t N, int64_t K,
                             unsigned long long *invalid, int sm_count, cudaStream_t st) {
    pack_rows_kernel<<<grid_for(N * ((K + 3) / 4), sm_count), 256, 0, st>>>(t, packed, N, K,
                                                                           invalid);
    return cudaGetLastError();
}

}  // namespace tl
