// elementwise.cu -- Q8_1 quantisation, RMSNorm (with fused Q8_1), residual add and
// the FFN activations of the Q4_0 layer.
//
// Q8_1 (q8_quantize_async in realizar 0.8.5 src/cuda/executor/cached.rs,
// transformer_layer_gpu_true_dp4a steps 2 and 5): per block of 32 values,
// d = max|x| / 127, q = round-half-away(x / d) in [-127, 127], s = d * sum(q);
// f32 IEEE division and rounding so the codes are bit-exact with the format.
// One warp per block: the max and the integer sum are warp reductions (order
// independent), so the result does not depend on the launch shape.
//
// RMSNorm (rms_norm_inplace in realizar 0.8.4 src/gpu/adapters/using.rs):
// rms = sqrt(sum x^2 / n + eps), y = x * (1 / rms) * gamma over the logical n,
// zeros in the padding up to n_pad (pad_and_upload_input in
// realizar 0.8.5 src/cuda/executor/layers/forward_utils.rs).  One CTA per row;
// the sum of squares is reduced in a fixed order (deterministic).  When a Q8_1
// output is requested the same kernel quantises the f32 y it just produced.
#include <algorithm>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

__device__ __forceinline__ void q8_block_store(float v, int lane, int8_t *q, float *d_out,
                                               float *s_out)
{
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    const int qi = q8_code(v, q8_scale(d));
    const int sum = warp_sum_int(qi);
    q[lane] = (int8_t)qi;
    if (lane == 0) {
        *d_out = d;
        *s_out = __fmul_rn(d, (float)sum);
    }
}

__global__ void q8_1_quantize_kernel(const float *__restrict__ x, int8_t *__restrict__ q,
                                     float *__restrict__ qd, float *__restrict__ qs,
                                     int64_t nblocks)
{
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (blk >= nblocks) return;
    // blocks of consecutive rows are consecutive: block blk covers x[32 blk, 32 blk + 32)
    const float v = x[blk * 32 + lane];
    q8_block_store(v, lane, q + blk * 32, qd + blk, qs + blk);
}

constexpr int kNormThreads = 32 * kRowWarps;  // 512: the register-row layout

// Rows up to kRowWarps * kRowBlocksPerWarp * 32 values, reduced in the same
// fixed order as the GEMV prologue, so the fused and the separate paths give
// identical bits.  `parts` CTAs share a row: each reduces the whole row (the
// same order, so the same scale) and writes its share of the blocks -- block
// warp + 16 k goes to part k % parts -- so that a warp's quantisations, a chain
// of shuffles each, are few (one CTA per row took about 8 us for four rows of
// 4096 values, most of it eight blocks in turn per warp).
__global__ void __launch_bounds__(kNormThreads, 1) rmsnorm_kernel(
    const float *__restrict__ x, const float *__restrict__ gamma, float *__restrict__ y,
    int8_t *__restrict__ q, float *__restrict__ qd, float *__restrict__ qs, int64_t n,
    int64_t n_pad, float eps, int parts)
{
    __shared__ float red[kRowWarps + 1];
    const int64_t row = blockIdx.x / parts;
    const int part = (int)(blockIdx.x % parts);
    const float *xr = x + row * n_pad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    pdl_wait();
    const int64_t nb = (n_pad + 31) / 32;
    const float scale = rms_scale(row_sumsq(xr, nb, n, warp, lane, red, [] { __syncthreads(); }), n, eps);
    for (int k0 = part; k0 < kRowBlocksPerWarp; k0 += 8 * parts) {
        if (warp + (int64_t)kRowWarps * k0 >= nb) break;
        float rv[8], rg[8];  // values and gammas of 8 blocks, loaded before any use
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t b = warp + (int64_t)kRowWarps * (k0 + u * parts);
            const int64_t i = b * 32 + lane;
            const bool in = b < nb && i < n;
            rv[u] = in ? __ldg(xr + i) : 0.0f;
            rg[u] = (in && gamma) ? __ldg(gamma + i) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t b = warp + (int64_t)kRowWarps * (k0 + u * parts);
            if (b >= nb) break;
            const int64_t i = b * 32 + lane;
            const float v = (i < n) ? __fmul_rn(__fmul_rn(rv[u], scale), rg[u]) : 0.0f;
            if (y && i < n_pad) y[row * n_pad + i] = v;
            if (q) q8_block_store(v, lane, q + row * n_pad + b * 32, qd + row * (n_pad / 32) + b,
                                  qs + row * (n_pad / 32) + b);
        }
    }
}

__global__ void residual_add_kernel(const float *a, const float *b, float *out, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = n / 4;
    if (i < n4) {
        const float4 va = reinterpret_cast<const float4 *>(a)[i];
        const float4 vb = reinterpret_cast<const float4 *>(b)[i];
        float4 r;
        r.x = __fadd_rn(va.x, vb.x);
        r.y = __fadd_rn(va.y, vb.y);
        r.z = __fadd_rn(va.z, vb.z);
        r.w = __fadd_rn(va.w, vb.w);
        reinterpret_cast<float4 *>(out)[i] = r;
    }
    if (i < n - n4 * 4) out[n4 * 4 + i] = __fadd_rn(a[n4 * 4 + i], b[n4 * 4 + i]);
}

// FFN activation of the Q4_0 layer (GpuModelQ4::forward_layer): h = silu(g) * u
// (ffn_swiglu_gpu's fused SwiGLU) when g is given, else h = GELU(u) in its tanh
// form (ffn_standard_gpu's gelu_gpu).
__global__ void ffn_act_kernel(const float *g, const float *u, float *h, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float x = u[i];
    if (g) {
        const float gv = g[i];
        h[i] = gv / (1.0f + expf(-gv)) * x;
    } else {
        const float c = 0.7978845608028654f;  // sqrt(2 / pi)
        h[i] = 0.5f * x * (1.0f + tanhf(c * (x + 0.044715f * x * x * x)));
    }
}

}  // namespace

cudaError_t launch_ffn_act(const float *g, const float *u, float *h, int64_t n, cudaStream_t s)
{
    const int threads = 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n + threads - 1) / threads));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ffn_act_kernel, g, u, h, n);
}

cudaError_t launch_q8_1_quantize(const float *x, void *q8, int64_t m, int64_t n, cudaStream_t s)
{
    int8_t *q = static_cast<int8_t *>(q8);
    float *qd = reinterpret_cast<float *>(q + m * n);
    float *qs = qd + m * (n / 32);
    const int64_t nblocks = m * (n / 32);
    const int warps = 8;
    const int64_t grid = (nblocks + warps - 1) / warps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(warps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q8_1_quantize_kernel, x, q, qd, qs, nblocks);
}

cudaError_t launch_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m,
                           int64_t n, int64_t n_pad, float eps, cudaStream_t s)
{
    int8_t *q = static_cast<int8_t *>(q8);
    float *qd = q ? reinterpret_cast<float *>(q + m * n_pad) : nullptr;
    float *qs = q ? qd + m * (n_pad / 32) : nullptr;
    // CTAs per row: about one block per warp (16 blocks a CTA), bounded by the SMs
    const int64_t nb = (n_pad + 31) / 32;
    int parts = (int)std::max<int64_t>(1, std::min<int64_t>((nb + kRowWarps - 1) / kRowWarps, 8));
    while (parts > 1 && m * parts > dev_info().sm_count) --parts;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(m * parts));
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, gamma, y, q, qd, qs, n, n_pad, eps, parts);
}

cudaError_t launch_residual_add(const float *a, const float *b, float *out, int64_t n,
                                cudaStream_t s)
{
    const int threads = 256;
    int64_t work = n / 4;
    if (work < n % 4) work = n % 4;
    const int64_t grid = (work + threads - 1) / threads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, residual_add_kernel, a, b, out, n);
}

}  // namespace rz
