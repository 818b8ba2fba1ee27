// noalloc.cu -- rz_swiglu_ffn_static: the SwiGLU FFN with its intermediates in a
// fixed device array owned by the library instead of a caller workspace.
//
// Some callers cannot hand the library any device memory: code that runs where
// allocation is not allowed (a latency-critical serving loop that must never
// enter the CUDA allocator, a plugin that lives inside another runtime which owns
// every device buffer, or a host thread that only holds borrowed pointers to the
// inputs and outputs).  For them this entry point keeps its scratch in a
// file-scope __device__ array of kStaticScratchBytes.  Every GPU that loads the
// library holds one copy of that array until the process exits.
//
// In host code the array's name is only a host-side stand-in, not a device
// address, so the device address is looked up once per device with
// cudaGetSymbolAddress (on that device's first call, with that device current)
// and passed to the kernels.  That first call therefore makes a runtime query and
// should come before any stream capture.  All calls share the one array: calls
// that overlap on the GPU (two streams, or two threads) race on it and must be
// ordered by the caller.  Nothing in the FFN scratch needs to start at zero; the
// array keeps whatever the last call left in it.
#include <mutex>
#include <string>

#include "../../include/rz.h"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
rz_status record_error(rz_status st, const char *msg);
rz_status ensure_device();
}  // namespace rz

namespace {
// RZ_ERR_CUDA with the CUDA error's name and text, like the other entry points
rz_status cuda_error(const char *what, cudaError_t e)
{
    std::string msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return rz::record_error(RZ_ERR_CUDA, msg.c_str());
}
}  // namespace

namespace {

constexpr size_t kStaticScratchBytes = 512 * 1024;

static __device__ __align__(256) uint8_t g_ffn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_dev[64];  // device address of g_ffn_scratch, per device

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" rz_status rz_swiglu_ffn_static(const float *x, const float *gamma, const void *w_gate,
                                          const void *w_up, const void *w_down, float *out, int64_t m,
                                          int64_t hidden, int64_t hidden_pad, int64_t inter, float eps,
                                          rz_stream stream)
{
    using namespace rz;
    record_error(RZ_OK, "");
    if (!x || !gamma || !w_gate || !w_up || !w_down || !out)
        return record_error(RZ_ERR_INVALID_ARG, "rz_swiglu_ffn_static: null pointer");
    const void *ptrs[] = {x, gamma, w_gate, w_up, w_down, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return record_error(RZ_ERR_ALIGN, "rz_swiglu_ffn_static: buffers must be 16-byte aligned");
    if (m < 1 || m > RZ_MAX_BATCH || hidden < 1 || hidden_pad < hidden || hidden_pad % 256 || inter < 256 ||
        inter % 256)
        return record_error(RZ_ERR_SHAPE, "rz_swiglu_ffn_static: bad m / hidden / hidden_pad / inter");
    if (!(eps >= 0.0f)) return record_error(RZ_ERR_INVALID_ARG, "rz_swiglu_ffn_static: eps");
    const size_t need = ffn_workspace_bytes(m, hidden_pad, inter);
    if (need > kStaticScratchBytes)
        return record_error(RZ_ERR_UNSUPPORTED,
                            "rz_swiglu_ffn_static: this shape needs more scratch than the 512 KiB static "
                            "buffer; use rz_swiglu_ffn with a workspace");
    rz_status st = ensure_device();
    if (st != RZ_OK) return st;
    if (!q4k_gemv_supported(m, hidden_pad, EPI_SWIGLU) || !q4k_gemv_supported(m, inter, EPI_STORE))
        return record_error(RZ_ERR_UNSUPPORTED, "rz_swiglu_ffn_static: a GEMV row is too wide");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error("rz_swiglu_ffn_static: cudaGetDevice", e);
    if (dev < 0 || dev >= 64) return record_error(RZ_ERR_UNSUPPORTED, "rz_swiglu_ffn_static: device index");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_dev[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_ffn_scratch);
            if (e != cudaSuccess)
                return cuda_error("rz_swiglu_ffn_static: cudaGetSymbolAddress of the static scratch", e);
            g_scratch_dev[dev] = p;
        }
        scratch = g_scratch_dev[dev];
    }
    e = launch_swiglu_ffn(x, gamma, w_gate, w_up, w_down, out, m, hidden, hidden_pad, inter, eps, scratch,
                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error("rz_swiglu_ffn_static: launch", e);
    return RZ_OK;
}
