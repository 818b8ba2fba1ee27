// abi.cu -- the extern "C" boundary of librz: argument checks, error reporting,
// device queries and the device error word.  Every check runs on the host before
// any launch; a failed check launches nothing.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/rz.h"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {

bool g_use_pdl = true;
uint32_t g_stall_next_gemv = 0;

namespace {

thread_local std::string t_last_error;

// First-error-wins device error word; one instance per device that loads the library.
__device__ unsigned g_dev_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
unsigned *g_err_ptr[kMaxDevices];

rz_status fail(rz_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

rz_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(RZ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device must be sm_103 (GB300); everything else is refused before any launch.
rz_status check_device()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(RZ_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_info_ok[dev]) {
        DevInfo d{};
        d.device = dev;
        cudaDeviceProp p;
        e = cudaGetDeviceProperties(&p, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        d.sm_count = p.multiProcessorCount;
        d.cc_major = p.major;
        d.cc_minor = p.minor;
        d.smem_optin = p.sharedMemPerBlockOptin;
        if (!(d.cc_major == 10 && d.cc_minor == 3))
            return fail(RZ_ERR_UNSUPPORTED, "librz is built for sm_103a; device %d is sm_%d%d", dev,
                        d.cc_major, d.cc_minor);
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_dev_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        g_err_ptr[dev] = static_cast<unsigned *>(ptr);
        g_info[dev] = d;
        g_info_ok[dev] = true;
    }
    return RZ_OK;
}

#define RZ_TRY(expr)                         \
    do {                                     \
        rz_status _st = (expr);              \
        if (_st != RZ_OK) return _st;        \
    } while (0)

#define RZ_CUDA(expr, what)                              \
    do {                                                 \
        cudaError_t _e = (expr);                         \
        if (_e != cudaSuccess) return cuda_fail(_e, what); \
    } while (0)

}  // namespace

// Shared with entry points defined in other files: set this thread's last-error
// message, and run the device check (and the per-device set-up) of this file.
rz_status record_error(rz_status st, const char *msg)
{
    t_last_error = msg;
    return st;
}

rz_status ensure_device() { return check_device(); }

const DevInfo &dev_info()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return g_info[dev];
}

unsigned *dev_error_word()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return g_err_ptr[dev];
}

}  // namespace rz

using namespace rz;

extern "C" {

const char *rz_last_error(void) { return t_last_error.c_str(); }

const char *rz_version(void) { return "librz 0.1 (sm_103a)"; }

rz_status rz_q8_1_quantize(const float *x, void *q8, int64_t m, int64_t n, rz_stream stream)
{
    t_last_error.clear();
    if (!x || !q8) return fail(RZ_ERR_INVALID_ARG, "rz_q8_1_quantize: null pointer");
    if (m < 1 || n < 1) return fail(RZ_ERR_INVALID_ARG, "rz_q8_1_quantize: m=%lld n=%lld", (long long)m, (long long)n);
    if (n % 32) return fail(RZ_ERR_SHAPE, "rz_q8_1_quantize: n=%lld is not a multiple of 32", (long long)n);
    if (!aligned16(x) || !aligned16(q8)) return fail(RZ_ERR_ALIGN, "rz_q8_1_quantize: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    RZ_CUDA(launch_q8_1_quantize(x, q8, m, n, static_cast<cudaStream_t>(stream)), "rz_q8_1_quantize launch");
    return RZ_OK;
}

rz_status rz_q4k_q8_gemv(const void *w, const void *q8, float *y, int64_t m, int64_t out_dim,
                         int64_t in_dim, rz_stream stream)
{
    t_last_error.clear();
    if (!w || !q8 || !y) return fail(RZ_ERR_INVALID_ARG, "rz_q4k_q8_gemv: null pointer");
    if (m < 1 || out_dim < 1 || in_dim < 1)
        return fail(RZ_ERR_INVALID_ARG, "rz_q4k_q8_gemv: m=%lld out_dim=%lld in_dim=%lld", (long long)m,
                    (long long)out_dim, (long long)in_dim);
    if (m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "rz_q4k_q8_gemv: m=%lld > %d", (long long)m, RZ_MAX_BATCH);
    if (in_dim % 256) return fail(RZ_ERR_SHAPE, "rz_q4k_q8_gemv: in_dim=%lld is not a multiple of 256", (long long)in_dim);
    if (in_dim / 256 > (1 << 20)) return fail(RZ_ERR_SHAPE, "rz_q4k_q8_gemv: in_dim too large");
    if (!aligned16(w) || !aligned16(q8) || !aligned16(y))
        return fail(RZ_ERR_ALIGN, "rz_q4k_q8_gemv: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    if (!q4k_gemv_supported(m, in_dim, EPI_STORE))
        return fail(RZ_ERR_UNSUPPORTED, "rz_q4k_q8_gemv: in_dim=%lld exceeds the shared-memory stage ring", (long long)in_dim);
    Q4kSegment seg{w, y, nullptr, out_dim};
    RZ_CUDA(launch_q4k_gemv(&seg, 1, EPI_STORE, q8, m, in_dim, static_cast<cudaStream_t>(stream)),
            "rz_q4k_q8_gemv launch");
    return RZ_OK;
}

rz_status rz_q4k_q8_subblock_dots(const void *w, const void *q8, int32_t *I, int64_t out_dim,
                                  int64_t in_dim, rz_stream stream)
{
    t_last_error.clear();
    if (!w || !q8 || !I) return fail(RZ_ERR_INVALID_ARG, "rz_q4k_q8_subblock_dots: null pointer");
    if (out_dim < 1 || in_dim < 1) return fail(RZ_ERR_INVALID_ARG, "rz_q4k_q8_subblock_dots: bad sizes");
    if (in_dim % 256) return fail(RZ_ERR_SHAPE, "rz_q4k_q8_subblock_dots: in_dim %% 256 != 0");
    if (!aligned16(w) || !aligned16(q8) || !aligned16(I))
        return fail(RZ_ERR_ALIGN, "rz_q4k_q8_subblock_dots: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    RZ_CUDA(launch_q4k_subblock_dots(w, q8, I, out_dim, in_dim, static_cast<cudaStream_t>(stream)),
            "rz_q4k_q8_subblock_dots launch");
    return RZ_OK;
}

rz_status rz_q4k_q8_gemv_ex(const void *w, const void *q8, const float *bias, const float *residual, float *y,
                            int64_t ld, int64_t m, int64_t out_dim, int64_t in_dim, rz_stream stream)
{
    const char *fn = "rz_q4k_q8_gemv_ex";
    t_last_error.clear();
    if (!w || !q8 || !y) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (bias && residual) return fail(RZ_ERR_UNSUPPORTED, "%s: a bias and a residual in one call", fn);
    if (m < 1 || out_dim < 1 || in_dim < 1)
        return fail(RZ_ERR_INVALID_ARG, "%s: m=%lld out_dim=%lld in_dim=%lld", fn, (long long)m, (long long)out_dim,
                    (long long)in_dim);
    if (ld == 0) ld = out_dim;
    if (ld < out_dim) return fail(RZ_ERR_SHAPE, "%s: ld=%lld < out_dim", fn, (long long)ld);
    if (m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld > %d", fn, (long long)m, RZ_MAX_BATCH);
    if (in_dim % 256) return fail(RZ_ERR_SHAPE, "%s: in_dim=%lld is not a multiple of 256", fn, (long long)in_dim);
    if (in_dim / 256 > (1 << 20)) return fail(RZ_ERR_SHAPE, "%s: in_dim too large", fn);
    if (!aligned16(w) || !aligned16(q8) || !aligned16(y) || (residual && !aligned16(residual)))
        return fail(RZ_ERR_ALIGN, "%s: buffers must be 16-byte aligned", fn);
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return fail(RZ_ERR_ALIGN, "%s: bias must be 4-byte aligned", fn);
    RZ_TRY(check_device());
    const int epi = residual ? EPI_RESID : EPI_STORE;
    if (!q4k_gemv_supported(m, in_dim, epi))
        return fail(RZ_ERR_UNSUPPORTED, "%s: in_dim=%lld exceeds the shared-memory stage ring", fn, (long long)in_dim);
    Q4kSegment seg{w, y, residual, out_dim, ld, ld, bias};
    RZ_CUDA(launch_q4k_gemv(&seg, 1, epi, q8, m, in_dim, static_cast<cudaStream_t>(stream)), "rz_q4k_q8_gemv_ex launch");
    return RZ_OK;
}

size_t rz_q4k_q8_gemm_workspace_bytes(int64_t m, int64_t in_dim)
{
    if (m < 1 || in_dim < 256 || in_dim % 256) return 0;
    return (size_t)q4k_gemm_tc_workspace_bytes(m, in_dim);
}

rz_status rz_q4k_q8_gemm(const void *w, const void *q8, float *y, int64_t ldy, int64_t m, int64_t out_dim,
                         int64_t in_dim, void *workspace, size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_q4k_q8_gemm";
    t_last_error.clear();
    if (!w || !q8 || !y || !workspace) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (m < 1 || out_dim < 1 || in_dim < 1)
        return fail(RZ_ERR_INVALID_ARG, "%s: m=%lld out_dim=%lld in_dim=%lld", fn, (long long)m, (long long)out_dim,
                    (long long)in_dim);
    if (in_dim % 256) return fail(RZ_ERR_SHAPE, "%s: in_dim=%lld is not a multiple of 256", fn, (long long)in_dim);
    if (ldy == 0) ldy = out_dim;
    if (ldy < out_dim) return fail(RZ_ERR_SHAPE, "%s: ldy=%lld < out_dim", fn, (long long)ldy);
    // grid limits: 128-token tiles in the second grid dimension; int32 indexing
    if (m > 65535LL * 128 || out_dim > (1LL << 30) || in_dim > (1LL << 24) || m * in_dim > (1LL << 40))
        return fail(RZ_ERR_SHAPE, "%s: m=%lld out_dim=%lld in_dim=%lld beyond the supported range", fn, (long long)m,
                    (long long)out_dim, (long long)in_dim);
    if (!aligned16(w) || !aligned16(q8) || !aligned16(workspace))
        return fail(RZ_ERR_ALIGN, "%s: w, q8 and the workspace must be 16-byte aligned", fn);
    if (reinterpret_cast<uintptr_t>(y) & 3u) return fail(RZ_ERR_ALIGN, "%s: y must be 4-byte aligned", fn);
    const size_t need = (size_t)q4k_gemm_tc_workspace_bytes(m, in_dim);
    if (ws_bytes < need) return fail(RZ_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
    RZ_TRY(check_device());
    RZ_CUDA(launch_q4k_gemm_tc(w, q8, y, ldy, m, out_dim, in_dim, workspace, static_cast<cudaStream_t>(stream)),
            "rz_q4k_q8_gemm launch");
    return RZ_OK;
}

rz_status rz_rmsnorm_q4k_gemv(const float *x, int64_t ldx, const float *gamma, int64_t n, float eps, int32_t n_mats,
                              const void *const *w, const int64_t *rows, const float *const *bias, float *y,
                              int64_t ldy, int64_t m, int64_t in_dim, rz_stream stream)
{
    const char *fn = "rz_rmsnorm_q4k_gemv";
    t_last_error.clear();
    if (!x || !gamma || !w || !rows || !y) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (n_mats < 1 || n_mats > 3) return fail(RZ_ERR_INVALID_ARG, "%s: n_mats=%d not in [1, 3]", fn, n_mats);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld", fn, (long long)m);
    if (in_dim < 256 || in_dim % 256) return fail(RZ_ERR_SHAPE, "%s: in_dim=%lld is not a multiple of 256", fn,
                                                  (long long)in_dim);
    if (n < 1 || n > in_dim) return fail(RZ_ERR_SHAPE, "%s: n=%lld not in [1, in_dim]", fn, (long long)n);
    if (ldx < in_dim) return fail(RZ_ERR_SHAPE, "%s: ldx < in_dim", fn);
    if (!(eps >= 0.0f)) return fail(RZ_ERR_INVALID_ARG, "%s: eps", fn);
    int64_t total = 0;
    Q4kSegment seg[3];
    for (int k = 0; k < n_mats; ++k) {
        if (!w[k] || rows[k] < 1) return fail(RZ_ERR_INVALID_ARG, "%s: matrix %d", fn, k);
        if (!aligned16(w[k])) return fail(RZ_ERR_ALIGN, "%s: weights must be 16-byte aligned", fn);
        const float *b = bias ? bias[k] : nullptr;
        if (b && (reinterpret_cast<uintptr_t>(b) & 3u)) return fail(RZ_ERR_ALIGN, "%s: bias alignment", fn);
        seg[k] = Q4kSegment{w[k], y + total, nullptr, rows[k], ldy, 0, b};
        total += rows[k];
    }
    if (ldy < total) return fail(RZ_ERR_SHAPE, "%s: ldy=%lld < the %lld rows of the matrices", fn, (long long)ldy,
                                 (long long)total);
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y) || (ldx % 4) || (ldy % 4))
        return fail(RZ_ERR_ALIGN, "%s: x, gamma, y must be 16-byte aligned (ldx, ldy multiples of 4)", fn);
    RZ_TRY(check_device());
    if (!q4k_gemv_supported(m, in_dim, EPI_STORE) || !q4k_gemv_f32_input_ok(m, in_dim))
        return fail(RZ_ERR_UNSUPPORTED, "%s: in_dim=%lld with m=%lld does not fit the fused prologue", fn,
                    (long long)in_dim, (long long)m);
    RZ_CUDA(launch_q4k_gemv_f32(seg, n_mats, EPI_STORE, F32Input{x, ldx, gamma, n, eps}, m, in_dim,
                                static_cast<cudaStream_t>(stream)),
            "rz_rmsnorm_q4k_gemv launch");
    return RZ_OK;
}

rz_status rz_q4k_q8_gemv_multi(const void *q8, int32_t n_mats, const void *const *w, const int64_t *rows,
                               const float *const *bias, float *y, int64_t ldy, int64_t m, int64_t in_dim,
                               rz_stream stream)
{
    const char *fn = "rz_q4k_q8_gemv_multi";
    t_last_error.clear();
    if (!q8 || !w || !rows || !y) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (n_mats < 1 || n_mats > 3) return fail(RZ_ERR_INVALID_ARG, "%s: n_mats=%d not in [1, 3]", fn, n_mats);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld", fn, (long long)m);
    if (in_dim < 256 || in_dim % 256) return fail(RZ_ERR_SHAPE, "%s: in_dim=%lld is not a multiple of 256", fn,
                                                  (long long)in_dim);
    int64_t total = 0;
    Q4kSegment seg[3];
    for (int k = 0; k < n_mats; ++k) {
        if (!w[k] || rows[k] < 1) return fail(RZ_ERR_INVALID_ARG, "%s: matrix %d", fn, k);
        if (!aligned16(w[k])) return fail(RZ_ERR_ALIGN, "%s: weights must be 16-byte aligned", fn);
        const float *b = bias ? bias[k] : nullptr;
        if (b && (reinterpret_cast<uintptr_t>(b) & 3u)) return fail(RZ_ERR_ALIGN, "%s: bias alignment", fn);
        seg[k] = Q4kSegment{w[k], y + total, nullptr, rows[k], ldy, 0, b};
        total += rows[k];
    }
    if (ldy < total) return fail(RZ_ERR_SHAPE, "%s: ldy=%lld < the %lld rows of the matrices", fn, (long long)ldy,
                                 (long long)total);
    if (!aligned16(q8) || (reinterpret_cast<uintptr_t>(y) & 3u))
        return fail(RZ_ERR_ALIGN, "%s: q8 must be 16-byte aligned, y 4-byte aligned", fn);
    RZ_TRY(check_device());
    if (!q4k_gemv_supported(m, in_dim, EPI_STORE))
        return fail(RZ_ERR_UNSUPPORTED, "%s: in_dim=%lld with m=%lld does not fit the stage ring", fn,
                    (long long)in_dim, (long long)m);
    RZ_CUDA(launch_q4k_gemv(seg, n_mats, EPI_STORE, q8, m, in_dim, static_cast<cudaStream_t>(stream)),
            "rz_q4k_q8_gemv_multi launch");
    return RZ_OK;
}

rz_status rz_q4k_f32_gemv(const void *w, const float *x, const float *bias, float *y, int64_t m, int64_t out_dim,
                          int64_t in_dim, rz_stream stream)
{
    const char *fn = "rz_q4k_f32_gemv";
    t_last_error.clear();
    if (!w || !x || !y) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (m < 1 || out_dim < 1 || in_dim < 1) return fail(RZ_ERR_INVALID_ARG, "%s: bad sizes", fn);
    if (m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld > %d", fn, (long long)m, RZ_MAX_BATCH);
    if (in_dim % 256) return fail(RZ_ERR_SHAPE, "%s: in_dim=%lld is not a multiple of 256", fn, (long long)in_dim);
    if (!aligned16(w) || !aligned16(x) || (reinterpret_cast<uintptr_t>(y) & 3u) ||
        (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
        return fail(RZ_ERR_ALIGN, "%s: w and x must be 16-byte aligned, y and bias 4-byte aligned", fn);
    RZ_TRY(check_device());
    if (q4k_f32_gemv_group(in_dim) < 1)
        return fail(RZ_ERR_UNSUPPORTED, "%s: in_dim=%lld does not fit in shared memory", fn, (long long)in_dim);
    RZ_CUDA(launch_q4k_f32_gemv(w, x, in_dim, y, out_dim, bias, m, out_dim, in_dim, static_cast<cudaStream_t>(stream)),
            "rz_q4k_f32_gemv launch");
    return RZ_OK;
}

rz_status rz_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                       int64_t in_dim, rz_stream stream)
{
    t_last_error.clear();
    if (!w || !x || !y) return fail(RZ_ERR_INVALID_ARG, "rz_q4_0_gemv: null pointer");
    if (m < 1 || out_dim < 1 || in_dim < 1) return fail(RZ_ERR_INVALID_ARG, "rz_q4_0_gemv: bad sizes");
    if (m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "rz_q4_0_gemv: m=%lld > %d", (long long)m, RZ_MAX_BATCH);
    if (in_dim % 32) return fail(RZ_ERR_SHAPE, "rz_q4_0_gemv: in_dim=%lld is not a multiple of 32", (long long)in_dim);
    if (!aligned16(w) || !aligned16(x) || !aligned16(y))
        return fail(RZ_ERR_ALIGN, "rz_q4_0_gemv: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    RZ_CUDA(launch_q4_0_gemv(w, x, y, m, out_dim, in_dim, static_cast<cudaStream_t>(stream)),
            "rz_q4_0_gemv launch");
    return RZ_OK;
}

rz_status rz_q4_0_gemv_bias(const void *w, const float *x, const float *bias, float *y, int64_t m, int64_t out_dim,
                            int64_t in_dim, rz_stream stream)
{
    t_last_error.clear();
    if (!w || !x || !y || !bias) return fail(RZ_ERR_INVALID_ARG, "rz_q4_0_gemv_bias: null pointer");
    if (m < 1 || out_dim < 1 || in_dim < 1) return fail(RZ_ERR_INVALID_ARG, "rz_q4_0_gemv_bias: bad sizes");
    if (m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "rz_q4_0_gemv_bias: m=%lld > %d", (long long)m, RZ_MAX_BATCH);
    if (in_dim % 32) return fail(RZ_ERR_SHAPE, "rz_q4_0_gemv_bias: in_dim %% 32 != 0");
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(bias) & 3u))
        return fail(RZ_ERR_ALIGN, "rz_q4_0_gemv_bias: alignment");
    RZ_TRY(check_device());
    RZ_CUDA(launch_q4_0_gemv(w, x, y, m, out_dim, in_dim, static_cast<cudaStream_t>(stream), bias),
            "rz_q4_0_gemv_bias launch");
    return RZ_OK;
}

rz_status rz_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m, int64_t n,
                     int64_t n_pad, float eps, rz_stream stream)
{
    t_last_error.clear();
    if (!x || !gamma || (!y && !q8)) return fail(RZ_ERR_INVALID_ARG, "rz_rmsnorm: null pointer");
    if (m < 1 || n < 1 || n_pad < n) return fail(RZ_ERR_INVALID_ARG, "rz_rmsnorm: bad sizes");
    if (m > (1 << 30)) return fail(RZ_ERR_SHAPE, "rz_rmsnorm: m too large");
    if (n_pad > 16384) return fail(RZ_ERR_UNSUPPORTED, "rz_rmsnorm: rows longer than 16384 values");
    if (q8 && (n_pad % 32)) return fail(RZ_ERR_SHAPE, "rz_rmsnorm: n_pad %% 32 != 0 with a Q8_1 output");
    if (!(eps >= 0.0f)) return fail(RZ_ERR_INVALID_ARG, "rz_rmsnorm: eps must be >= 0");
    if (!aligned16(x) || !aligned16(gamma) || (y && !aligned16(y)) || (q8 && !aligned16(q8)))
        return fail(RZ_ERR_ALIGN, "rz_rmsnorm: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    RZ_CUDA(launch_rmsnorm(x, gamma, y, q8, m, n, n_pad, eps, static_cast<cudaStream_t>(stream)),
            "rz_rmsnorm launch");
    return RZ_OK;
}

rz_status rz_residual_add(const float *a, const float *b, float *out, int64_t n, rz_stream stream)
{
    t_last_error.clear();
    if (!a || !b || !out) return fail(RZ_ERR_INVALID_ARG, "rz_residual_add: null pointer");
    if (n < 1) return fail(RZ_ERR_INVALID_ARG, "rz_residual_add: n=%lld", (long long)n);
    if (!aligned16(a) || !aligned16(b) || !aligned16(out))
        return fail(RZ_ERR_ALIGN, "rz_residual_add: buffers must be 16-byte aligned");
    RZ_TRY(check_device());
    RZ_CUDA(launch_residual_add(a, b, out, n, static_cast<cudaStream_t>(stream)), "rz_residual_add launch");
    return RZ_OK;
}

rz_status rz_check_device_error(rz_stream stream, uint32_t *code_out)
{
    t_last_error.clear();
    RZ_TRY(check_device());
    unsigned code = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RZ_CUDA(cudaMemcpyFromSymbolAsync(&code, g_dev_error, sizeof code, 0, cudaMemcpyDeviceToHost, s),
            "read device error word");
    RZ_CUDA(cudaStreamSynchronize(s), "synchronize");
    if (code_out) *code_out = code;
    if (code == 0) return RZ_OK;
    const unsigned zero = 0;
    RZ_CUDA(cudaMemcpyToSymbolAsync(g_dev_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s),
            "clear device error word");
    RZ_CUDA(cudaStreamSynchronize(s), "synchronize");
    if ((code & 0xf00u) == 0x100u || (code & 0xf00u) == 0x300u)
        return fail(RZ_ERR_TIMEOUT, "device error 0x%x: a bounded wait ran out", code);
    return fail(RZ_ERR_DEVICE, "device error 0x%x: a device-side range check failed", code);
}

rz_status rz_set_pdl(int enable)
{
    t_last_error.clear();
    g_use_pdl = enable != 0;
    return RZ_OK;
}

rz_status rz_debug_stall_next_gemv(uint32_t wait_limit)
{
    t_last_error.clear();
    if (wait_limit < 1024 || wait_limit > (1u << 22))
        return fail(RZ_ERR_INVALID_ARG, "rz_debug_stall_next_gemv: wait_limit=%u outside [1024, 2^22]", wait_limit);
    g_stall_next_gemv = wait_limit;
    return RZ_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- layer-level helpers
namespace {

rz_status check_layer(const rz_layer_weights *w, const char *fn, int64_t m, LayerDesc *out)
{
    if (!w) return fail(RZ_ERR_INVALID_ARG, "%s: null layer descriptor", fn);
    const bool fused = !w->wk && !w->wv;
    const void *ptrs[] = {w->wq, fused ? w->wq : w->wk, fused ? w->wq : w->wv, w->wo, w->wgate, w->wup, w->wdown,
                          w->attn_gamma, w->ffn_gamma};
    for (const void *p : ptrs) {
        if (!p) return fail(RZ_ERR_INVALID_ARG, "%s: null weight pointer (wk and wv are both NULL or both set)", fn);
        if (!aligned16(p)) return fail(RZ_ERR_ALIGN, "%s: weights must be 16-byte aligned", fn);
    }
    if (fused && (w->bk || w->bv))
        return fail(RZ_ERR_INVALID_ARG, "%s: a fused Q|K|V matrix takes its bias in bq alone", fn);
    const float *biases[] = {w->bq, w->bk, w->bv};
    for (const float *b : biases)
        if (b && (reinterpret_cast<uintptr_t>(b) & 3u)) return fail(RZ_ERR_ALIGN, "%s: biases must be 4-byte aligned", fn);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld not in [1, %d]", fn, (long long)m, RZ_MAX_BATCH);
    if (w->hidden < 1 || w->hidden_pad < w->hidden || w->hidden_pad % 256)
        return fail(RZ_ERR_SHAPE, "%s: hidden=%d hidden_pad=%d (hidden_pad must be a multiple of 256 >= hidden)", fn,
                    w->hidden, w->hidden_pad);
    if (w->n_heads < 1 || w->n_kv_heads < 1 || w->n_heads % w->n_kv_heads)
        return fail(RZ_ERR_SHAPE, "%s: n_heads=%d n_kv_heads=%d", fn, w->n_heads, w->n_kv_heads);
    if (w->n_heads / w->n_kv_heads > 16) return fail(RZ_ERR_UNSUPPORTED, "%s: more than 16 query heads per kv head", fn);
    if (w->head_dim < 32 || w->head_dim > 256 || w->head_dim % 32)
        return fail(RZ_ERR_SHAPE, "%s: head_dim=%d (multiple of 32 in [32, 256])", fn, w->head_dim);
    // the limits from here on depend on the device's shared memory
    RZ_TRY(check_device());
    if (attention_smem_bytes(w->n_heads / w->n_kv_heads, w->head_dim, 0) > dev_info().smem_optin)
        return fail(RZ_ERR_UNSUPPORTED, "%s: head_dim=%d with %d query heads per kv head needs more shared memory "
                    "than a CTA has", fn, w->head_dim, w->n_heads / w->n_kv_heads);
    if (w->inter < 256 || w->inter % 256) return fail(RZ_ERR_SHAPE, "%s: inter=%d is not a multiple of 256", fn, w->inter);
    if (!(w->eps >= 0.0f) || !(w->rope_theta > 0.0f)) return fail(RZ_ERR_INVALID_ARG, "%s: eps/rope_theta", fn);
    if (w->rope_mode != 0 && w->rope_mode != 1) return fail(RZ_ERR_INVALID_ARG, "%s: rope_mode=%d", fn, w->rope_mode);
    const int q_dim = w->n_heads * w->head_dim;
    const int q_pad = (q_dim + 255) / 256 * 256;
    if (!q4k_gemv_supported(m, w->hidden_pad, EPI_SWIGLU) || !q4k_gemv_supported(m, q_pad, EPI_STORE) ||
        !q4k_gemv_supported(m, w->inter, EPI_STORE))
        return fail(RZ_ERR_UNSUPPORTED, "%s: a GEMV row is too wide for the shared-memory stage ring", fn);
    LayerDesc d{w->wq, w->wk, w->wv, w->wo, w->wgate, w->wup, w->wdown, w->attn_gamma, w->ffn_gamma,
                w->hidden, w->hidden_pad, w->n_heads, w->n_kv_heads, w->head_dim, w->inter,
                w->eps, w->rope_theta, w->rope_mode, w->bq, w->bk, w->bv};
    *out = d;
    return RZ_OK;
}

rz_status check_kv(const rz_kv_cache *kv, const char *fn, int64_t m, int kv_dim, KvDesc *out)
{
    if (!kv || !kv->k || !kv->v) return fail(RZ_ERR_INVALID_ARG, "%s: null KV cache", fn);
    if (!aligned16(kv->k) || !aligned16(kv->v)) return fail(RZ_ERR_ALIGN, "%s: KV cache must be 16-byte aligned", fn);
    if (kv->max_seq < 1) return fail(RZ_ERR_INVALID_ARG, "%s: max_seq=%d", fn, kv->max_seq);
    if (kv->max_seq > 4096) return fail(RZ_ERR_UNSUPPORTED, "%s: max_seq=%d > 4096", fn, kv->max_seq);
    if (m > 1 && kv->seq_stride < (int64_t)kv->max_seq * kv_dim)
        return fail(RZ_ERR_SHAPE, "%s: seq_stride=%lld < max_seq*kv_dim", fn, (long long)kv->seq_stride);
    if (m > 1 && kv->seq_stride % 4)
        return fail(RZ_ERR_ALIGN, "%s: seq_stride=%lld is not a multiple of 4 (16-byte sequence starts)", fn,
                    (long long)kv->seq_stride);
    *out = KvDesc{kv->k, kv->v, m > 1 ? kv->seq_stride : 0, kv->max_seq};
    return RZ_OK;
}

rz_status check_position(const int32_t *positions, int32_t position, int max_seq, const char *fn)
{
    if (positions) {
        if (!aligned16(positions) && (reinterpret_cast<uintptr_t>(positions) & 3u))
            return fail(RZ_ERR_ALIGN, "%s: positions must be 4-byte aligned", fn);
        return RZ_OK;
    }
    if (position < 0 || position >= max_seq)
        return fail(RZ_ERR_INVALID_ARG, "%s: position=%d outside [0, %d)", fn, position, max_seq);
    return RZ_OK;
}

rz_status check_ws(const void *ws, size_t have, size_t need, const char *fn)
{
    if (!ws) return fail(RZ_ERR_INVALID_ARG, "%s: null workspace", fn);
    if (!aligned16(ws)) return fail(RZ_ERR_ALIGN, "%s: workspace must be 16-byte aligned", fn);
    if (have < need) return fail(RZ_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, have, need);
    return RZ_OK;
}

}  // namespace

extern "C" {

size_t rz_swiglu_ffn_workspace_bytes(int64_t m, int64_t hidden_pad, int64_t inter)
{
    if (m < 1 || hidden_pad < 1 || inter < 1) return 0;
    return ffn_workspace_bytes(m, hidden_pad, inter);
}

rz_status rz_swiglu_ffn(const float *x, const float *gamma, const void *w_gate, const void *w_up,
                        const void *w_down, float *out, int64_t m, int64_t hidden, int64_t hidden_pad,
                        int64_t inter, float eps, void *workspace, size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_swiglu_ffn";
    t_last_error.clear();
    if (!x || !gamma || !w_gate || !w_up || !w_down || !out) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    const void *ptrs[] = {x, gamma, w_gate, w_up, w_down, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(RZ_ERR_ALIGN, "%s: buffers must be 16-byte aligned", fn);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld", fn, (long long)m);
    if (hidden < 1 || hidden_pad < hidden || hidden_pad % 256 || inter < 256 || inter % 256)
        return fail(RZ_ERR_SHAPE, "%s: hidden=%lld hidden_pad=%lld inter=%lld", fn, (long long)hidden,
                    (long long)hidden_pad, (long long)inter);
    if (!(eps >= 0.0f)) return fail(RZ_ERR_INVALID_ARG, "%s: eps", fn);
    RZ_TRY(check_ws(workspace, ws_bytes, ffn_workspace_bytes(m, hidden_pad, inter), fn));
    RZ_TRY(check_device());
    if (!q4k_gemv_supported(m, hidden_pad, EPI_SWIGLU) || !q4k_gemv_supported(m, inter, EPI_STORE))
        return fail(RZ_ERR_UNSUPPORTED, "%s: a GEMV row is too wide for the shared-memory stage ring", fn);
    RZ_CUDA(launch_swiglu_ffn(x, gamma, w_gate, w_up, w_down, out, m, hidden, hidden_pad, inter, eps, workspace,
                              static_cast<cudaStream_t>(stream)),
            "rz_swiglu_ffn launch");
    return RZ_OK;
}

size_t rz_attention_workspace_bytes(int64_t m, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                    int32_t max_seq)
{
    if (m < 1 || n_heads < 1 || n_kv_heads < 1 || head_dim < 1 || max_seq < 1) return 0;
    if (check_device() != RZ_OK) return 0;
    auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
    return a256(attention_part_bytes(m, n_kv_heads, n_heads / n_kv_heads, head_dim, max_seq)) +
           a256((size_t)m * n_kv_heads * 4);
}

rz_status rz_attention_decode(const float *q, const float *k, const float *v, int64_t ld_qkv,
                              const rz_kv_cache *kv, const int32_t *positions, int32_t position, int64_t m,
                              int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float rope_theta,
                              int32_t rope_mode, float *att, void *att_q8, void *workspace, size_t ws_bytes,
                              rz_stream stream)
{
    const char *fn = "rz_attention_decode";
    t_last_error.clear();
    if (!q || !k || !v || (!att && !att_q8)) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld", fn, (long long)m);
    if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || n_heads / n_kv_heads > 16)
        return fail(RZ_ERR_SHAPE, "%s: n_heads=%d n_kv_heads=%d", fn, n_heads, n_kv_heads);
    if (head_dim < 32 || head_dim > 256 || head_dim % 32) return fail(RZ_ERR_SHAPE, "%s: head_dim=%d", fn, head_dim);
    if (rope_mode != 0 && rope_mode != 1) return fail(RZ_ERR_INVALID_ARG, "%s: rope_mode", fn);
    if (!(rope_theta > 0.0f)) return fail(RZ_ERR_INVALID_ARG, "%s: rope_theta", fn);
    const int64_t q_dim = (int64_t)n_heads * head_dim, kv_dim = (int64_t)n_kv_heads * head_dim;
    if (m > 1 && ld_qkv < q_dim) return fail(RZ_ERR_SHAPE, "%s: ld_qkv", fn);
    if ((att && !aligned16(att)) || (att_q8 && !aligned16(att_q8)))
        return fail(RZ_ERR_ALIGN, "%s: outputs must be 16-byte aligned", fn);
    KvDesc kd;
    RZ_TRY(check_kv(kv, fn, m, (int)kv_dim, &kd));
    RZ_TRY(check_position(positions, position, kv->max_seq, fn));
    const size_t need = rz_attention_workspace_bytes(m, n_heads, n_kv_heads, head_dim, kv->max_seq);
    RZ_TRY(check_device());
    if (attention_smem_bytes(n_heads / n_kv_heads, head_dim, 0) > dev_info().smem_optin)
        return fail(RZ_ERR_UNSUPPORTED, "%s: head_dim=%d with %d query heads per kv head needs more shared memory "
                    "than a CTA has", fn, head_dim, n_heads / n_kv_heads);
    RZ_TRY(check_ws(workspace, ws_bytes, need, fn));
    LayerDesc L{};
    L.n_heads = n_heads;
    L.n_kv_heads = n_kv_heads;
    L.head_dim = head_dim;
    L.rope_theta = rope_theta;
    L.rope_mode = rope_mode;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
    float *part = reinterpret_cast<float *>(ws);
    ws += a256(attention_part_bytes(m, n_kv_heads, n_heads / n_kv_heads, head_dim, kv->max_seq));
    int *counters = reinterpret_cast<int *>(ws);
    AttnArgs a = make_attn_args(L, m, kd, positions, position, part, counters, q, k, v, ld_qkv, att,
                                att_q8);
    RZ_CUDA(launch_attention(a, static_cast<cudaStream_t>(stream)), "rz_attention_decode launch");
    return RZ_OK;
}

size_t rz_decode_layer_workspace_bytes(const rz_layer_weights *w, int64_t m, int32_t max_seq)
{
    LayerDesc L;
    if (max_seq < 1 || check_layer(w, "rz_decode_layer_workspace_bytes", m, &L) != RZ_OK) return 0;
    if (check_device() != RZ_OK) return 0;
    return layer_workspace_bytes(L, m, max_seq);
}

rz_status rz_decode_layer(const float *input, const rz_layer_weights *w, const rz_kv_cache *kv,
                          const int32_t *positions, int32_t position, int64_t m, float *output, void *workspace,
                          size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_decode_layer";
    t_last_error.clear();
    if (!input || !output) return fail(RZ_ERR_INVALID_ARG, "%s: null input/output", fn);
    if (!aligned16(input) || !aligned16(output)) return fail(RZ_ERR_ALIGN, "%s: input/output alignment", fn);
    LayerDesc L;
    RZ_TRY(check_layer(w, fn, m, &L));
    KvDesc kd;
    RZ_TRY(check_kv(kv, fn, m, L.n_kv_heads * L.head_dim, &kd));
    RZ_TRY(check_position(positions, position, kv->max_seq, fn));
    RZ_TRY(check_device());
    RZ_TRY(check_ws(workspace, ws_bytes, layer_workspace_bytes(L, m, kd.max_seq), fn));
    RZ_CUDA(launch_decode_layer(input, L, kd, positions, position, m, output, workspace,
                                static_cast<cudaStream_t>(stream)),
            "rz_decode_layer launch");
    return RZ_OK;
}

size_t rz_decode_stack_workspace_bytes(const rz_layer_weights *layers, int32_t n_layers, int64_t m, int32_t max_seq)
{
    LayerDesc L;
    if (!layers || n_layers < 1 || max_seq < 1) return 0;
    if (check_layer(&layers[0], "rz_decode_stack_workspace_bytes", m, &L) != RZ_OK) return 0;
    if (check_device() != RZ_OK) return 0;
    return stack_workspace_bytes(L, m, max_seq);
}

// Checks shared by rz_decode_stack and rz_decode_layers.
static rz_status check_stack(const char *fn, const float *input, const rz_layer_weights *layers,
                             const rz_kv_cache *kvs, int32_t n_layers, const int32_t *positions, int32_t position,
                             int64_t m, std::vector<LayerDesc> &Ls, std::vector<KvDesc> &Ks)
{
    if (!input || !layers || !kvs) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (n_layers < 1 || n_layers > 4096) return fail(RZ_ERR_INVALID_ARG, "%s: n_layers=%d", fn, n_layers);
    if (!aligned16(input)) return fail(RZ_ERR_ALIGN, "%s: buffers must be 16-byte aligned", fn);
    Ls.resize((size_t)n_layers);
    Ks.resize((size_t)n_layers);
    for (int l = 0; l < n_layers; ++l) {
        RZ_TRY(check_layer(&layers[l], fn, m, &Ls[l]));
        RZ_TRY(check_kv(&kvs[l], fn, m, Ls[l].n_kv_heads * Ls[l].head_dim, &Ks[l]));
        if (Ls[l].hidden != Ls[0].hidden || Ls[l].hidden_pad != Ls[0].hidden_pad || Ls[l].eps != Ls[0].eps ||
            Ks[l].max_seq != Ks[0].max_seq || Ls[l].n_heads != Ls[0].n_heads ||
            Ls[l].n_kv_heads != Ls[0].n_kv_heads || Ls[l].head_dim != Ls[0].head_dim || Ls[l].inter != Ls[0].inter)
            return fail(RZ_ERR_SHAPE, "%s: layer %d differs in shape from layer 0", fn, l);
    }
    RZ_TRY(check_position(positions, position, Ks[0].max_seq, fn));
    return check_device();
}

rz_status rz_decode_stack(const float *input, const rz_layer_weights *layers, const rz_kv_cache *kvs,
                          int32_t n_layers, const int32_t *positions, int32_t position, int64_t m,
                          const float *out_gamma, const void *lm_head, const float *lm_bias, int64_t vocab,
                          float *hidden_out, float *logits, void *workspace, size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_decode_stack";
    t_last_error.clear();
    if (!out_gamma || !lm_head || !logits) return fail(RZ_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (vocab < 1) return fail(RZ_ERR_INVALID_ARG, "%s: vocab", fn);
    const void *ptrs[] = {out_gamma, lm_head, logits};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(RZ_ERR_ALIGN, "%s: buffers must be 16-byte aligned", fn);
    if (hidden_out && !aligned16(hidden_out)) return fail(RZ_ERR_ALIGN, "%s: hidden_out alignment", fn);
    if (lm_bias && (reinterpret_cast<uintptr_t>(lm_bias) & 3u)) return fail(RZ_ERR_ALIGN, "%s: lm_bias alignment", fn);
    std::vector<LayerDesc> Ls;
    std::vector<KvDesc> Ks;
    RZ_TRY(check_stack(fn, input, layers, kvs, n_layers, positions, position, m, Ls, Ks));
    if (Ls[0].hidden % 32) return fail(RZ_ERR_SHAPE, "%s: hidden %% 32 != 0 (Q4_0 LM head blocks)", fn);
    RZ_TRY(check_ws(workspace, ws_bytes, stack_workspace_bytes(Ls[0], m, Ks[0].max_seq), fn));
    RZ_CUDA(launch_decode_stack(input, Ls.data(), n_layers, Ks.data(), positions, position, m, out_gamma, lm_head,
                                lm_bias, vocab, hidden_out, logits, workspace, static_cast<cudaStream_t>(stream)),
            "rz_decode_stack launch");
    return RZ_OK;
}

rz_status rz_decode_layers(const float *input, const rz_layer_weights *layers, const rz_kv_cache *kvs,
                           int32_t n_layers, const int32_t *positions, int32_t position, int64_t m, float *output,
                           void *workspace, size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_decode_layers";
    t_last_error.clear();
    if (!output) return fail(RZ_ERR_INVALID_ARG, "%s: null output", fn);
    if (!aligned16(output)) return fail(RZ_ERR_ALIGN, "%s: output alignment", fn);
    std::vector<LayerDesc> Ls;
    std::vector<KvDesc> Ks;
    RZ_TRY(check_stack(fn, input, layers, kvs, n_layers, positions, position, m, Ls, Ks));
    RZ_TRY(check_ws(workspace, ws_bytes, stack_workspace_bytes(Ls[0], m, Ks[0].max_seq), fn));
    RZ_CUDA(launch_decode_stack(input, Ls.data(), n_layers, Ks.data(), positions, position, m, nullptr, nullptr,
                                nullptr, 0, output, nullptr, workspace, static_cast<cudaStream_t>(stream)),
            "rz_decode_layers launch");
    return RZ_OK;
}

static rz_status check_layer_q4_0(const rz_layer_weights_q4_0 *w, const char *fn, int64_t m, LayerQ40Desc *out)
{
    if (!w) return fail(RZ_ERR_INVALID_ARG, "%s: null layer descriptor", fn);
    const void *ptrs[] = {w->wqkv, w->wo, w->wup, w->wdown, w->attn_gamma, w->ffn_gamma};
    for (const void *p : ptrs) {
        if (!p) return fail(RZ_ERR_INVALID_ARG, "%s: null weight pointer", fn);
        if (!aligned16(p)) return fail(RZ_ERR_ALIGN, "%s: weights must be 16-byte aligned", fn);
    }
    if (w->wgate && !aligned16(w->wgate)) return fail(RZ_ERR_ALIGN, "%s: weights must be 16-byte aligned", fn);
    if (m < 1 || m > RZ_MAX_BATCH) return fail(RZ_ERR_SHAPE, "%s: m=%lld not in [1, %d]", fn, (long long)m, RZ_MAX_BATCH);
    if (w->hidden < 32 || w->hidden % 32 || w->hidden > 16384)
        return fail(RZ_ERR_SHAPE, "%s: hidden=%d (a multiple of 32, at most 16384)", fn, w->hidden);
    if (w->inter < 32 || w->inter % 32) return fail(RZ_ERR_SHAPE, "%s: inter=%d is not a multiple of 32", fn, w->inter);
    if (w->n_heads < 1 || w->n_kv_heads < 1 || w->n_heads % w->n_kv_heads || w->n_heads / w->n_kv_heads > 16)
        return fail(RZ_ERR_SHAPE, "%s: n_heads=%d n_kv_heads=%d", fn, w->n_heads, w->n_kv_heads);
    if (w->head_dim < 32 || w->head_dim > 256 || w->head_dim % 32)
        return fail(RZ_ERR_SHAPE, "%s: head_dim=%d (multiple of 32 in [32, 256])", fn, w->head_dim);
    // the limits from here on depend on the device's shared memory
    RZ_TRY(check_device());
    if (attention_smem_bytes(w->n_heads / w->n_kv_heads, w->head_dim, 0) > dev_info().smem_optin)
        return fail(RZ_ERR_UNSUPPORTED, "%s: the attention of this head shape does not fit a CTA", fn);
    if (!(w->eps >= 0.0f) || !(w->rope_theta > 0.0f)) return fail(RZ_ERR_INVALID_ARG, "%s: eps/rope_theta", fn);
    if (w->rope_mode != 0 && w->rope_mode != 1) return fail(RZ_ERR_INVALID_ARG, "%s: rope_mode=%d", fn, w->rope_mode);
    *out = LayerQ40Desc{w->wqkv, w->wo, w->wgate, w->wup, w->wdown, w->attn_gamma, w->ffn_gamma, w->hidden,
                        w->n_heads, w->n_kv_heads, w->head_dim, w->inter, w->eps, w->rope_theta, w->rope_mode};
    return RZ_OK;
}

size_t rz_decode_layer_q4_0_workspace_bytes(const rz_layer_weights_q4_0 *w, int64_t m, int32_t max_seq)
{
    LayerQ40Desc L;
    if (max_seq < 1 || check_layer_q4_0(w, "rz_decode_layer_q4_0_workspace_bytes", m, &L) != RZ_OK) return 0;
    return layer_q4_0_workspace_bytes(L, m, max_seq);
}

rz_status rz_decode_layer_q4_0(const float *input, const rz_layer_weights_q4_0 *w, const rz_kv_cache *kv,
                               const int32_t *positions, int32_t position, int64_t m, float *output, void *workspace,
                               size_t ws_bytes, rz_stream stream)
{
    const char *fn = "rz_decode_layer_q4_0";
    t_last_error.clear();
    if (!input || !output) return fail(RZ_ERR_INVALID_ARG, "%s: null input/output", fn);
    if (!aligned16(input) || !aligned16(output)) return fail(RZ_ERR_ALIGN, "%s: input/output alignment", fn);
    LayerQ40Desc L;
    RZ_TRY(check_layer_q4_0(w, fn, m, &L));
    KvDesc kd;
    RZ_TRY(check_kv(kv, fn, m, L.n_kv_heads * L.head_dim, &kd));
    RZ_TRY(check_position(positions, position, kv->max_seq, fn));
    RZ_TRY(check_ws(workspace, ws_bytes, layer_q4_0_workspace_bytes(L, m, kd.max_seq), fn));
    RZ_CUDA(launch_decode_layer_q4_0(input, L, kd, positions, position, m, output, workspace,
                                     static_cast<cudaStream_t>(stream)),
            "rz_decode_layer_q4_0 launch");
    return RZ_OK;
}

int32_t rz_decode_stack_launches(const rz_layer_weights *layers, int32_t n_layers, int64_t m, int32_t max_seq,
                                 int32_t with_head, int64_t vocab)
{
    if (!layers || n_layers < 1 || n_layers > 4096 || max_seq < 1 || (with_head && vocab < 1)) return 0;
    std::vector<LayerDesc> Ls((size_t)n_layers);
    for (int l = 0; l < n_layers; ++l)
        if (check_layer(&layers[l], "rz_decode_stack_launches", m, &Ls[l]) != RZ_OK) return 0;
    if (check_device() != RZ_OK) return 0;
    return stack_kernel_launches(Ls.data(), n_layers, m, max_seq, with_head != 0, vocab);
}

}  // extern "C"
