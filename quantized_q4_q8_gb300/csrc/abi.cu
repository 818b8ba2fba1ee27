// abi.cu -- the extern "C" boundary of librz: argument checks, error reporting,
// device queries and the device error word.  Every check runs on the host before
// any launch; a failed check launches nothing.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/rz.h"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {

bool g_use_pdl = true;

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

rz_status rz_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m, int64_t n,
                     int64_t n_pad, float eps, rz_stream stream)
{
    t_last_error.clear();
    if (!x || !gamma || (!y && !q8)) return fail(RZ_ERR_INVALID_ARG, "rz_rmsnorm: null pointer");
    if (m < 1 || n < 1 || n_pad < n) return fail(RZ_ERR_INVALID_ARG, "rz_rmsnorm: bad sizes");
    if (m > (1 << 30)) return fail(RZ_ERR_SHAPE, "rz_rmsnorm: m too large");
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
    if ((code & 0xf00u) == 0x100u)
        return fail(RZ_ERR_TIMEOUT, "device error 0x%x: a bounded wait ran out", code);
    return fail(RZ_ERR_DEVICE, "device error 0x%x: a device-side range check failed", code);
}

rz_status rz_set_pdl(int enable)
{
    t_last_error.clear();
    g_use_pdl = enable != 0;
    return RZ_OK;
}

}  // extern "C"
