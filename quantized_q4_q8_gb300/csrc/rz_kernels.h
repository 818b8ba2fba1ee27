// rz_kernels.h -- host-side launchers shared between the librz translation units.
// Arguments are already validated by the C-ABI layer (abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rz {

// Device properties of the current device (cached per device).
struct DevInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
};
const DevInfo &dev_info();

// Device error word of the current device (a file-scope __device__ variable).
unsigned *dev_error_word();

// Launch with the programmatic-stream-serialization attribute (PDL) so that the
// kernel's weight prefetch overlaps the tail of the previous kernel in the stream.
extern bool g_use_pdl;

// ---------------------------------------------------------------- Q8_1
cudaError_t launch_q8_1_quantize(const float *x, void *q8, int64_t m, int64_t n, cudaStream_t s);

// ---------------------------------------------------------------- norms / elementwise
cudaError_t launch_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m,
                           int64_t n, int64_t n_pad, float eps, cudaStream_t s);
cudaError_t launch_residual_add(const float *a, const float *b, float *out, int64_t n,
                                cudaStream_t s);

// ---------------------------------------------------------------- Q4_K x Q8_1 GEMV
enum Q4kEpilogue { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2 };

struct Q4kSegment {
    const void *w;     // Q4_K [rows][in_dim]
    float *y;          // [m][rows]
    const float *res;  // [m][rows] (EPI_RESID) or nullptr
    int64_t rows;
};

// Up to three weight matrices with the same in_dim read against one Q8_1
// activation (the fused Q|K|V launch).  For EPI_SWIGLU seg[0] is the gate
// matrix, seg[1] the up matrix, and seg[0].y receives silu(gate) * up.
cudaError_t launch_q4k_gemv(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                            int64_t m, int64_t in_dim, cudaStream_t s);

cudaError_t launch_q4k_subblock_dots(const void *w, const void *q8, int32_t *I, int64_t out_dim,
                                     int64_t in_dim, cudaStream_t s);

// ---------------------------------------------------------------- Q4_0 GEMV
cudaError_t launch_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                             int64_t in_dim, cudaStream_t s);

}  // namespace rz
