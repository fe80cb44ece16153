// api.cu -- the C ABI of libternary_gb300.so (declared in include/ternary_linear.h).
//
// Host-side duties only: argument validation (synchronous, before anything is
// enqueued), per-device facts (SM count, architecture), the per-device status
// word used by kernels with bounded waits, and the choice between the skinny
// path (decode-shaped M) and the tcgen05 tile path.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "ternary_linear.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
    bool init = false;
    bool sm103 = false;
    int sm_count = 0;
    int *status = nullptr;  // 1 int, cudaMalloc'd on the first ternary_linear call
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
std::atomic<int> g_inject_launch_failures{0};
// testing aids for the decode kernel's bounded waits (ternary_test_set_wait_limit)
std::atomic<long long> g_wait_limit{0};  // 0 = the default (~0.5 s)
std::atomic<int> g_stall{0};
// testing aid: the tile kernel's form (ternary_test_set_tile_mode): 0 = chosen
// per call, 1 = one tile per CTA, 2 = persistent CTAs (192-token tiles), 3 = persistent
// CTAs with 256-token tiles where the scales are per channel
std::atomic<int> g_tile_mode{0};

int env_int(const char *name, int dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

int skinny_max_m() {
    static const int v = [] {
        int m = env_int("TERNARY_SKINNY_MAX_M", 32);
        if (m < 0) m = 0;
        if (m > 32) m = 32;
        return m;
    }();
    return v;
}

// Launch tuning knobs (environment, read once):
//   TERNARY_PDL=0          launch without programmatic dependent launch
//   TERNARY_PDL_TRIGGER=1  release dependents after the main loop instead of at entry
//                      =2  no explicit release (dependents start when the grid exits)
//   TERNARY_SKINNY_SK=n    force the skinny path's K split (cluster size), 0 = automatic
//   TERNARY_SKINNY_CTAS_PER_SM=n  CTAs per SM the tensor-core skinny path aims for (default 2)
bool pdl_enabled() {
    static const bool v = env_int("TERNARY_PDL", 1) != 0;
    return v;
}

int skinny_launch_flags(uint32_t api_flags) {
    static const int trig = env_int("TERNARY_PDL_TRIGGER", 0);
    static const int base = (trig == 1 ? tl::kSkinnyTriggerLate : 0) |
                            (trig == 2 ? tl::kSkinnyTriggerNever : 0);
    return base | ((api_flags & TL_FLAG_STATIC_WEIGHTS) ? tl::kSkinnyStaticWeights : 0);
}

// Skinny-path kernel choice (prefer_skinny_tc below).  The decode kernel of
// gemv.cuh (register-fed warp MMAs, TMA-staged weights, x fragments held in
// registers per 64-k column) serves M <= 8 except plain layers of 2049..4608
// rows, 64-wide groups and zero-block maps at M <= 16; the tcgen05 kernel
// (decoded weights in TMEM, 128-row tiles) serves the rest up to M = 32.
//   TERNARY_SKINNY_IMPL=tc | mma   force the tcgen05 kernel, or the older warp-MMA
//                                  kernel of kern_skinny.cu, for every M <= 32
enum { kImplAuto = 0, kImplMma = 1, kImplTc = 2 };
int skinny_impl() {
    static const int mode = [] {
        const char *e = std::getenv("TERNARY_SKINNY_IMPL");
        if (e && e[0] == 'm') return (int)kImplMma;
        if (e && e[0] == 't') return (int)kImplTc;
        return (int)kImplAuto;
    }();
    return mode;
}

int gemv_flags(uint32_t api_flags) {
    return ((api_flags & TL_FLAG_STATIC_WEIGHTS) ? tl::kGemvStaticWeights : 0) |
           (g_stall.load() ? tl::kGemvTestStall : 0);
}

long long wait_limit() {
    const long long v = g_wait_limit.load();
    return v > 0 ? v : (1ll << 30);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device's facts; optionally make sure the status word exists.
tl_status current_device(DevInfo **out, bool need_status) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TL_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return TL_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TL_ERR_CUDA;
        }
        d.sm103 = (major == 10 && minor == 3);
        d.sm_count = sms;
        d.init = true;
    }
    if (!d.sm103) return TL_ERR_UNSUPPORTED;
    if (need_status && d.status == nullptr) {
        int *p = nullptr;
        if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return TL_ERR_CUDA;
        }
        if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p);
            return TL_ERR_CUDA;
        }
        d.status = p;
    }
    *out = &d;
    return TL_OK;
}

// Host-side fault injection for tests: the next n launch attempts fail with
// TL_ERR_CUDA before touching the GPU.
bool take_injected_failure() {
    int n = g_inject_launch_failures.load();
    while (n > 0) {
        if (g_inject_launch_failures.compare_exchange_weak(n, n - 1)) return true;
    }
    return false;
}

tl_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TL_OK;
    cudaGetLastError();  // clear the sticky-free error state
    return TL_ERR_CUDA;
}

size_t dtype_size(int32_t d) { return d == TL_F32 ? 4 : 2; }

// Validation shared by ternary_linear / ternary_linear_path.  Returns TL_OK
// and sets *noop when nothing needs to be enqueued.
tl_status check_linear(const void *x, int32_t x_dtype, const uint8_t *packed, const void *scale,
                       int32_t group_size, void *out, int32_t out_dtype, int64_t M, int64_t N,
                       int64_t K, bool *noop) {
    *noop = false;
    if (x_dtype != TL_F16 && x_dtype != TL_BF16) return TL_ERR_DTYPE;
    if (out_dtype != TL_F16 && out_dtype != TL_BF16 && out_dtype != TL_F32) return TL_ERR_DTYPE;
    if (group_size != 0 && group_size != 32 && group_size != 64 && group_size != 128 &&
        group_size != 256)
        return TL_ERR_DTYPE;
    if (M < 0 || N < 0 || K < 0) return TL_ERR_SHAPE;
    if (group_size > 0 && K % group_size != 0) return TL_ERR_SHAPE;
    const int64_t lim = (int64_t)1 << 30;
    if (M >= lim || N >= lim || K >= lim) return TL_ERR_SHAPE;
    if (M == 0 || N == 0) {
        *noop = true;
        return TL_OK;
    }
    if (out == nullptr) return TL_ERR_NULL;
    if (K > 0 && (x == nullptr || packed == nullptr)) return TL_ERR_NULL;
    if (scale == nullptr && (group_size == 0 || K > 0)) return TL_ERR_NULL;
    if (!aligned16(out) || (x && !aligned16(x)) || (packed && !aligned16(packed)) ||
        (scale && !aligned16(scale)))
        return TL_ERR_ALIGN;
    return TL_OK;
}

// Decode shapes that the tcgen05 skinny kernel serves faster than the register-fed
// decode kernel (timed per layer on the 7B, 27B and 7B-stack shapes): two token
// tiles of the decode kernel (M > 8) double its MMAs, where the tcgen05 kernel's
// N = 16 MMA costs the same; at M <= 8, plain layers of 2049..4608 rows.
bool prefer_skinny_tc(int64_t M, int64_t rows, bool gated) {
    if (M > 8) return true;
    return !gated && rows > 2048 && rows <= 4608;
}

int gshift_of(int32_t group_size) {
    return group_size == 32 ? 5 : group_size == 64 ? 6 : group_size == 256 ? 8 : 7;
}

// The CUDA-core kernel for shapes the TMA-fed kernels cannot take (K % 64 != 0:
// packed rows are not 16-byte pitched).  It does not read a zero-block map.
tl_status run_generic(const void *x, bool bf, const uint8_t *packed, const void *scale,
                      int32_t group_size, void *out, int32_t out_dtype, int64_t M, int64_t N,
                      int64_t K, int64_t nh, cudaStream_t st) {
    tl::GenArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.packed = packed;
    a.scale = static_cast<const uint16_t *>(scale);
    a.out = out;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.gshift = gshift_of(group_size);
    a.nh = (int)nh;
    a.odt = out_dtype;
    return from_cuda(tl::launch_generic(a, bf, group_size != 0, nh > 0, st, pdl_enabled()));
}

tl_status run_linear(const void *x, int32_t x_dtype, const uint8_t *packed, const void *scale,
                     int32_t group_size, void *out, int32_t out_dtype, int64_t M, int64_t N,
                     int64_t K, int32_t path, uint32_t flags, void *stream,
                     const uint32_t *mask = nullptr) {
    bool noop = false;
    tl_status s = check_linear(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K,
                               &noop);
    if (s != TL_OK || noop) return s;
    if (path != TL_PATH_AUTO && path != TL_PATH_SKINNY && path != TL_PATH_TILE &&
        path != TL_PATH_GENERIC)
        return TL_ERR_DTYPE;
    if (flags & ~(uint32_t)TL_FLAG_STATIC_WEIGHTS) return TL_ERR_DTYPE;
    if (take_injected_failure()) return TL_ERR_CUDA;
    DevInfo *d = nullptr;
    s = current_device(&d, true);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(out, 0, (size_t)(M * N) * dtype_size(out_dtype), st));

    const bool bf = x_dtype == TL_BF16;
    if (path == TL_PATH_GENERIC || (path == TL_PATH_AUTO && K % 64 != 0))
        return run_generic(x, bf, packed, scale, group_size, out, out_dtype, M, N, K, 0, st);
    if (K % 64 != 0) return TL_ERR_UNSUPPORTED;
    const bool group = group_size != 0;
    // groups narrower than 128: no tcgen05 skinny kernel; 32-wide: tile kernel only
    const bool narrow = group_size == 64 || group_size == 32;
    const bool g32 = group_size == 32;
    const int gshift = gshift_of(group_size);
    static const int force_sk = env_int("TERNARY_SKINNY_SK", 0);
    const int impl = skinny_impl();
    const bool tile_ok = tl::tile_supported(M, N, K);
    // skinny candidates: the decode kernel (M <= 16, any group size), then the
    // tcgen05 skinny kernel (M <= 32, not 64-wide groups)
    tl::GemvPlan gp{};
    // the tcgen05 skinny kernel takes groups 0 / 128 / 256, and a zero-block map
    // with per-channel scales
    const bool tc_can = !narrow && (mask == nullptr || !group);
    if (impl == kImplAuto && M <= tl::kGemvMaxM && !g32 && !(tc_can && prefer_skinny_tc(M, N, false)))
        gp = tl::plan_gemv(M, N, K, d->sm_count, false, group, force_sk);
    tl::SkinnyTcPlan tp{};
    tl::SkinnyPlan mp{};
    // the zero-block map is read by the decode, tile and (channel scales) tcgen05 skinny kernels
    if (!gp.ok && tc_can && impl != kImplMma) {
        static const int per_sm = env_int("TERNARY_SKINNY_CTAS_PER_SM", 2);
        tp = tl::plan_skinny_tc(M, N, K, d->sm_count, force_sk, per_sm);
    }
    if (!narrow && impl == kImplMma && mask == nullptr) mp = tl::plan_skinny(M, N, K, d->sm_count, force_sk);
    const bool skinny_ok = gp.ok || tp.ok || mp.ok;
    int use = path;
    if (use == TL_PATH_AUTO) {
        use = (M <= skinny_max_m() && skinny_ok) ? TL_PATH_SKINNY : TL_PATH_TILE;
        if (use == TL_PATH_TILE && !tile_ok && skinny_ok) use = TL_PATH_SKINNY;
    }
    if (use == TL_PATH_SKINNY) {
        if (!skinny_ok) return TL_ERR_UNSUPPORTED;
        if (gp.ok) {
            tl::GemvArgs a{};
            a.x = static_cast<const uint16_t *>(x);
            a.packed = packed;
            a.scale = static_cast<const uint16_t *>(scale);
            a.out = out;
            a.M = (int)M;
            a.N = (int)N;
            a.K = (int)K;
            a.gshift = gshift;
            a.nh = 0;
            a.flags = gemv_flags(flags);
            a.odt = out_dtype;
            a.status = d->status;
            a.wait_limit = wait_limit();
            a.mask = mask;
            a.mask_words = tl::mask_words(K);
            return from_cuda(tl::launch_gemv(a, bf, group, gp, st, pdl_enabled()));
        }
        if (tp.ok) {
            tl::SkinnyTcArgs a{};
            a.x = static_cast<const uint16_t *>(x);
            a.packed = packed;
            a.scale = static_cast<const uint16_t *>(scale);
            a.out = out;
            a.M = (int)M;
            a.N = (int)N;
            a.K = (int)K;
            a.gshift = gshift;
            a.flags = skinny_launch_flags(flags);
            a.status = d->status;
            a.mask = mask;
            a.mask_words = tl::mask_words(K);
            return from_cuda(tl::launch_skinny_tc(a, bf, group, out_dtype, tp, st, pdl_enabled()));
        }
        tl::SkinnyArgs a{};
        a.x = static_cast<const uint16_t *>(x);
        a.packed = packed;
        a.scale = static_cast<const uint16_t *>(scale);
        a.out = out;
        a.M = (int)M;
        a.N = (int)N;
        a.K = (int)K;
        a.gshift = gshift;
        a.flags = skinny_launch_flags(flags);
        a.status = d->status;
        return from_cuda(tl::launch_skinny(a, bf, group, out_dtype, mp, st, pdl_enabled()));
    }
    if (!tile_ok) return TL_ERR_UNSUPPORTED;
    tl::TileArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.packed = packed;
    a.scale = static_cast<const uint16_t *>(scale);
    a.out = out;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.gshift = gshift;
    a.status = d->status;
    a.mask = mask;
    a.mask_words = tl::mask_words(K);
    a.persist = g_tile_mode.load() - 1;
    return from_cuda(tl::launch_tile(a, bf, group, out_dtype, d->sm_count, st, pdl_enabled()));
}

// Fused gate/up with the SiLU-gated product: packed / scale hold 2N stacked rows
// (gate, then up), out is [M, N].  Decode shapes run on the tcgen05 decode
// kernel, larger M (and 64-wide groups) on the tile kernel.
tl_status run_silu_mul(const void *x, int32_t x_dtype, const uint8_t *packed, const void *scale,
                       int32_t group_size, void *out, int32_t out_dtype, int64_t M, int64_t N,
                       int64_t K, uint32_t flags, void *stream, const uint32_t *mask = nullptr) {
    if (N < 0 || N >= ((int64_t)1 << 29)) return TL_ERR_SHAPE;
    bool noop = false;
    tl_status s = check_linear(x, x_dtype, packed, scale, group_size, out, out_dtype, M, 2 * N, K,
                               &noop);
    if (s != TL_OK || noop) return s;
    if (flags & ~(uint32_t)TL_FLAG_STATIC_WEIGHTS) return TL_ERR_DTYPE;
    if (take_injected_failure()) return TL_ERR_CUDA;
    DevInfo *d = nullptr;
    s = current_device(&d, true);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // K == 0: g = u = 0 and silu(0) * 0 = 0
    if (K == 0) return from_cuda(cudaMemsetAsync(out, 0, (size_t)(M * N) * dtype_size(out_dtype), st));
    const bool bf = x_dtype == TL_BF16;
    if (K % 64 != 0)
        return run_generic(x, bf, packed, scale, group_size, out, out_dtype, M, 2 * N, K, N, st);
    const bool group = group_size != 0;
    const int gshift = gshift_of(group_size);
    static const int force_sk = env_int("TERNARY_SKINNY_SK", 0);
    const bool tc_can = group_size != 64 && group_size != 32 && (mask == nullptr || group_size == 0);
    if (M <= skinny_max_m() && M <= tl::kGemvMaxM && skinny_impl() == kImplAuto &&
        group_size != 32 && !(tc_can && prefer_skinny_tc(M, 2 * N, true))) {
        tl::GemvPlan gp = tl::plan_gemv(M, 2 * N, K, d->sm_count, true, group_size != 0, force_sk);
        if (gp.ok) {
            tl::GemvArgs a{};
            a.x = static_cast<const uint16_t *>(x);
            a.packed = packed;
            a.scale = static_cast<const uint16_t *>(scale);
            a.out = out;
            a.M = (int)M;
            a.N = (int)(2 * N);
            a.K = (int)K;
            a.gshift = gshift;
            a.nh = (int)N;
            a.flags = gemv_flags(flags);
            a.odt = out_dtype;
            a.status = d->status;
            a.wait_limit = wait_limit();
            a.mask = mask;
            a.mask_words = tl::mask_words(K);
            return from_cuda(tl::launch_gemv_silu(a, bf, group, gp, st, pdl_enabled()));
        }
    }
    if (M <= skinny_max_m() && tc_can) {
        static const int per_sm = env_int("TERNARY_SKINNY_CTAS_PER_SM", 2);
        tl::SkinnyTcPlan tp = tl::plan_skinny_tc(M, 2 * N, K, d->sm_count, force_sk, per_sm);
        if (tp.ok) {
            tl::SkinnyTcArgs a{};
            a.x = static_cast<const uint16_t *>(x);
            a.packed = packed;
            a.scale = static_cast<const uint16_t *>(scale);
            a.out = out;
            a.M = (int)M;
            a.N = (int)(2 * N);
            a.K = (int)K;
            a.nh = (int)N;
            a.gshift = gshift;
            a.flags = skinny_launch_flags(flags);
            a.status = d->status;
            a.mask = mask;
            a.mask_words = tl::mask_words(K);
            return from_cuda(tl::launch_skinny_silu(a, bf, group, out_dtype, tp, st, pdl_enabled()));
        }
    }
    if (!tl::tile_supported(M, 2 * N, K)) return TL_ERR_UNSUPPORTED;
    tl::TileArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.packed = packed;
    a.scale = static_cast<const uint16_t *>(scale);
    a.out = out;
    a.M = (int)M;
    a.N = (int)(2 * N);
    a.K = (int)K;
    a.nh = (int)N;
    a.gshift = gshift;
    a.status = d->status;
    a.mask = mask;
    a.mask_words = tl::mask_words(K);
    a.persist = g_tile_mode.load() - 1;
    return from_cuda(tl::launch_tile_silu(a, bf, group, out_dtype, d->sm_count, st, pdl_enabled()));
}

tl_status check_packing(const void *t, const void *packed, int64_t N, int64_t K,
                        const int64_t *count) {
    if (N < 0 || K < 0) return TL_ERR_SHAPE;
    // N * K must stay representable (and addressable): cap the element count at 2^48
    if (N >= ((int64_t)1 << 40) || K >= ((int64_t)1 << 40)) return TL_ERR_SHAPE;
    if (K > 0 && N > (((int64_t)1 << 48) / K)) return TL_ERR_SHAPE;
    if (N * K > 0 && (t == nullptr || packed == nullptr)) return TL_ERR_NULL;
    if ((t && !aligned16(t)) || (packed && !aligned16(packed))) return TL_ERR_ALIGN;
    if (count && (reinterpret_cast<uintptr_t>(count) & 7u)) return TL_ERR_ALIGN;
    return TL_OK;
}

}  // namespace

extern "C" {

tl_status ternary_pack(const int8_t *t, uint8_t *packed, int64_t N, int64_t K,
                       int64_t *invalid_count, void *stream) {
    tl_status s = check_packing(t, packed, N, K, invalid_count);
    if (s != TL_OK) return s;
    if (take_injected_failure()) return TL_ERR_CUDA;
    DevInfo *d = nullptr;
    s = current_device(&d, false);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (invalid_count) {
        s = from_cuda(cudaMemsetAsync(invalid_count, 0, sizeof(int64_t), st));
        if (s != TL_OK) return s;
    }
    if (N * K == 0) return TL_OK;
    auto *cnt = reinterpret_cast<unsigned long long *>(invalid_count);
    if (K % 4 != 0) return from_cuda(tl::launch_pack_rows(t, packed, N, K, cnt, d->sm_count, st));
    return from_cuda(tl::launch_pack(t, packed, N * (K / 4), cnt, d->sm_count, st));
}

tl_status ternary_unpack(const uint8_t *packed, int8_t *t, int64_t N, int64_t K,
                         int64_t *reserved_count, void *stream) {
    tl_status s = check_packing(t, packed, N, K, reserved_count);
    if (s != TL_OK) return s;
    if (take_injected_failure()) return TL_ERR_CUDA;
    DevInfo *d = nullptr;
    s = current_device(&d, false);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (reserved_count) {
        s = from_cuda(cudaMemsetAsync(reserved_count, 0, sizeof(int64_t), st));
        if (s != TL_OK) return s;
    }
    if (N * K == 0) return TL_OK;
    auto *cnt = reinterpret_cast<unsigned long long *>(reserved_count);
    if (K % 4 != 0)
        return from_cuda(tl::launch_unpack_rows(packed, t, N, K, cnt, d->sm_count, st));
    return from_cuda(tl::launch_unpack(packed, t, N * (K / 4), cnt, d->sm_count, st));
}

tl_status ternary_linear(const void *x, int32_t x_dtype, const uint8_t *packed, const void *scale,
                         int32_t group_size, void *out, int32_t out_dtype, int64_t M, int64_t N,
                         int64_t K, void *stream) {
    return run_linear(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K,
                      TL_PATH_AUTO, 0u, stream);
}

tl_status ternary_linear_ex(const void *x, int32_t x_dtype, const uint8_t *packed,
                            const void *scale, int32_t group_size, void *out, int32_t out_dtype,
                            int64_t M, int64_t N, int64_t K, int32_t path, uint32_t flags,
                            void *stream) {
    return run_linear(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K, path,
                      flags, stream);
}

tl_status ternary_linear_silu_mul(const void *x, int32_t x_dtype, const uint8_t *packed,
                                  const void *scale, int32_t group_size, void *out,
                                  int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                                  uint32_t flags, void *stream) {
    return run_silu_mul(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K, flags,
                        stream);
}

int64_t ternary_block_mask_words(int64_t N, int64_t K) {
    if (N < 0 || K < 0) return -1;
    return ((N + 127) / 128) * (int64_t)tl::mask_words(K);
}

tl_status ternary_block_mask(const uint8_t *packed, int64_t N, int64_t K, uint32_t *mask,
                             int64_t *zero_blocks, void *stream) {
    if (N < 0 || K < 0) return TL_ERR_SHAPE;
    if (N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) return TL_ERR_SHAPE;
    if (N * K > 0 && (packed == nullptr || mask == nullptr)) return TL_ERR_NULL;
    if ((mask && (reinterpret_cast<uintptr_t>(mask) & 3u)) ||
        (zero_blocks && (reinterpret_cast<uintptr_t>(zero_blocks) & 7u)))
        return TL_ERR_ALIGN;
    if (take_injected_failure()) return TL_ERR_CUDA;
    DevInfo *d = nullptr;
    tl_status s = current_device(&d, false);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (zero_blocks) {
        s = from_cuda(cudaMemsetAsync(zero_blocks, 0, sizeof(int64_t), st));
        if (s != TL_OK) return s;
    }
    if (N * K == 0) return TL_OK;
    return from_cuda(tl::launch_block_mask(packed, N, K, mask,
                                           reinterpret_cast<unsigned long long *>(zero_blocks), st));
}

tl_status ternary_linear_masked(const void *x, int32_t x_dtype, const uint8_t *packed,
                                const void *scale, int32_t group_size, const uint32_t *mask,
                                void *out, int32_t out_dtype, int64_t M, int64_t N, int64_t K,
                                uint32_t flags, void *stream) {
    if (mask == nullptr && M > 0 && N > 0 && K > 0) return TL_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(mask) & 3u) return TL_ERR_ALIGN;
    return run_linear(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K,
                      TL_PATH_AUTO, flags, stream, mask);
}

tl_status ternary_linear_silu_mul_masked(const void *x, int32_t x_dtype, const uint8_t *packed,
                                         const void *scale, int32_t group_size,
                                         const uint32_t *mask, void *out, int32_t out_dtype,
                                         int64_t M, int64_t N, int64_t K, uint32_t flags,
                                         void *stream) {
    if (mask == nullptr && M > 0 && N > 0 && K > 0) return TL_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(mask) & 3u) return TL_ERR_ALIGN;
    return run_silu_mul(x, x_dtype, packed, scale, group_size, out, out_dtype, M, N, K, flags,
                        stream, mask);
}

int32_t ternary_skinny_max_m(void) { return skinny_max_m(); }

tl_status ternary_device_status(int32_t *code, int32_t clear) {
    if (code == nullptr) return TL_ERR_NULL;
    *code = TL_OK;
    DevInfo *d = nullptr;
    tl_status s = current_device(&d, false);
    if (s != TL_OK) return s;
    if (d->status == nullptr) return TL_OK;
    int v = 0;
    s = from_cuda(cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (s != TL_OK) return s;
    if (v != 0) *code = TL_ERR_TIMEOUT;
    if (clear && v != 0) s = from_cuda(cudaMemset(d->status, 0, sizeof(int)));
    return s;
}

const char *ternary_status_string(int32_t status) {
    switch (status) {
    case TL_OK: return "TL_OK";
    case TL_ERR_NULL: return "TL_ERR_NULL: a required pointer is NULL";
    case TL_ERR_SHAPE: return "TL_ERR_SHAPE: invalid or unsupported sizes";
    case TL_ERR_DTYPE: return "TL_ERR_DTYPE: unknown dtype, group size (0, 32, 64, 128, 256) or path code";
    case TL_ERR_ALIGN: return "TL_ERR_ALIGN: pointer not 16-byte aligned";
    case TL_ERR_VALUE: return "TL_ERR_VALUE: invalid or reserved values present";
    case TL_ERR_CUDA: return "TL_ERR_CUDA: a CUDA call or kernel launch failed";
    case TL_ERR_TIMEOUT: return "TL_ERR_TIMEOUT: a bounded device-side wait gave up";
    case TL_ERR_UNSUPPORTED: return "TL_ERR_UNSUPPORTED: no sm_103 device, or the forced path "
                                    "cannot serve these arguments";
    default: return "unknown tl_status";
    }
}

int32_t ternary_version(void) { return 100; }

void ternary_test_inject_launch_failures(int32_t n) {
    g_inject_launch_failures.store(n < 0 ? 0 : n);
}

void ternary_test_set_wait_limit(int64_t cycles, int32_t stall) {
    g_wait_limit.store(cycles > 0 ? cycles : 0);
    g_stall.store(stall ? 1 : 0);
}

void ternary_test_set_tile_mode(int32_t mode) { g_tile_mode.store(mode >= 1 && mode <= 3 ? mode : 0); }

tl_status ternary_device_status_async(int32_t *dst, int32_t clear, void *stream) {
    if (dst == nullptr) return TL_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(dst) & 3u) != 0) return TL_ERR_ALIGN;
    DevInfo *d = nullptr;
    tl_status s = current_device(&d, true);
    if (s != TL_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    s = from_cuda(cudaMemcpyAsync(dst, d->status, sizeof(int), cudaMemcpyDefault, st));
    if (s == TL_OK && clear) s = from_cuda(cudaMemsetAsync(d->status, 0, sizeof(int), st));
    return s;
}

}  // extern "C"
