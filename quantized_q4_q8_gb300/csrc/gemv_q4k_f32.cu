// gemv_q4k_f32.cu -- Q4_K weights times f32 activations, without Q8_1
// quantisation of the activations (q4k_gemv_cached_async of realizar 0.8.5
// src/cuda/executor/cached.rs, transformer_layer_gpu_cached: the accuracy
// reference variant of the dp4a path).
//
// For every row r and token t
//   y[t][r] = sum_b [ d_b * sum_j sc_bj * (sum_k q_bjk x_tbjk) - dmin_b * sum_j m_bj * X_tbj ],
// X_tbj the sum of the 32 activations of sub-block j, which is the dot of the
// dequantised row d * sc_j * q - dmin * m_j with x, rearranged so that the
// per-element work is one multiply-add of the 4-bit code (as an exact float)
// with the activation.
//
// Layout.  The activations of up to four tokens and their 32-value block sums
// are staged in shared memory once per CTA.  A warp takes one row at a time;
// lane group g = lane / 4 takes super-blocks g, g + 8, ... of it (the loads of two
// of them issued together), lane c = lane % 4 one 32-byte chunk (sub-blocks 2c and
// 2c + 1: the low and the high nibbles).  A code becomes an exact float through
// its bit pattern (2^23 + q, minus 2^23).  The f32 partial sums of the lanes are
// added by a fixed-order butterfly (deterministic).  The f32 products make this
// path issue-bound, not HBM-bound, at one token (about four instructions per
// weight against the dp4a path's one per four).
#include <algorithm>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFMaxTokens = 4;

__device__ __forceinline__ float nib_f(uint32_t w, int shift)
{
    // 2^23 + q as a float bit pattern, minus 2^23: q exactly
    return __int_as_float((int)(0x4B000000u | ((w >> shift) & 0xFu))) - 8388608.0f;
}

template <int MT>
__global__ void __launch_bounds__(kFThreads) q4k_f32_gemv_kernel(const uint8_t *__restrict__ w,
                                                                 const float *__restrict__ x, int64_t ldx,
                                                                 float *__restrict__ y, int64_t ldy,
                                                                 const float *__restrict__ bias, int m,
                                                                 int64_t out_dim, int in_dim)
{
    extern __shared__ __align__(16) float fsm[];
    float *xs = fsm;                          // [m][in_dim]
    float *bs = fsm + (int64_t)m * in_dim;    // [m][in_dim / 32] block sums
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = in_dim / 32, nsb = in_dim / 256;
    pdl_wait();  // the activations may come from the previous kernel
    for (int t = 0; t < m; ++t) {
        const float4 *src = reinterpret_cast<const float4 *>(x + t * ldx);
        float4 *dst = reinterpret_cast<float4 *>(xs + (int64_t)t * in_dim);
        for (int i = tid; i < in_dim / 4; i += kFThreads) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    // block sums, warp per block, fixed order (butterfly)
    for (int b = warp; b < m * nb; b += kFWarps) {
        const float v = xs[(int64_t)b * 32 + lane];
        const float s = warp_sum(v);
        if (lane == 0) bs[b] = s;
    }
    __syncthreads();
    pdl_launch_dependents();

    const int g = lane >> 2, c = lane & 3;
    const int64_t row_bytes = (int64_t)nsb * 144;
    for (int64_t row = (int64_t)blockIdx.x * kFWarps + warp; row < out_dim; row += (int64_t)gridDim.x * kFWarps) {
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
        const uint8_t *rw = w + row * row_bytes;
        for (int sb0 = g; sb0 < nsb; sb0 += 16) {
            // two super-blocks per step, their loads in flight together
            int4 hdr[2], qa[2], qb[2];
            bool on[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int sb = sb0 + 8 * u;
                on[u] = sb < nsb;
                const uint8_t *blk = rw + (int64_t)(on[u] ? sb : sb0) * 144;
                hdr[u] = __ldg(reinterpret_cast<const int4 *>(blk));
                qa[u] = __ldg(reinterpret_cast<const int4 *>(blk + 16 + 32 * c));
                qb[u] = __ldg(reinterpret_cast<const int4 *>(blk + 32 + 32 * c));
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (!on[u]) continue;
                const int sb = sb0 + 8 * u;
                const float d = h2f((uint16_t)((uint32_t)hdr[u].x & 0xffffu));
                const float dmin = h2f((uint16_t)((uint32_t)hdr[u].x >> 16));
                // 6-bit scales and mins of sub-blocks 2c, 2c + 1 (bytes 4-15 of the header:
                // s0-3 in .y, s4-7 in .z, s8-11 in .w)
                const uint32_t A = (uint32_t)hdr[u].y, B = (uint32_t)hdr[u].z, C = (uint32_t)hdr[u].w;
                int sc[2], mn[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = 2 * c + h, k = j & 3;
                    const int a = (int)((A >> (8 * k)) & 0xFFu), b = (int)((B >> (8 * k)) & 0xFFu);
                    const int cc = (int)((C >> (8 * k)) & 0xFFu);
                    if (j < 4) {
                        sc[h] = a & 63;
                        mn[h] = b & 63;
                    } else {
                        sc[h] = (cc & 15) | ((a >> 6) << 4);
                        mn[h] = (cc >> 4) | ((b >> 6) << 4);
                    }
                }
                const uint32_t q[8] = {(uint32_t)qa[u].x, (uint32_t)qa[u].y, (uint32_t)qa[u].z, (uint32_t)qa[u].w,
                                       (uint32_t)qb[u].x, (uint32_t)qb[u].y, (uint32_t)qb[u].z, (uint32_t)qb[u].w};
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t < m) {
                        const float *xb = xs + (int64_t)t * in_dim + sb * 256 + 64 * c;
                        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 xl = *reinterpret_cast<const float4 *>(xb + 4 * k);
                            const float4 xh = *reinterpret_cast<const float4 *>(xb + 32 + 4 * k);
                            s0 = fmaf(nib_f(q[k], 0), xl.x, s0);
                            s0 = fmaf(nib_f(q[k], 8), xl.y, s0);
                            s0 = fmaf(nib_f(q[k], 16), xl.z, s0);
                            s0 = fmaf(nib_f(q[k], 24), xl.w, s0);
                            s1 = fmaf(nib_f(q[k], 4), xh.x, s1);
                            s1 = fmaf(nib_f(q[k], 12), xh.y, s1);
                            s1 = fmaf(nib_f(q[k], 20), xh.z, s1);
                            s1 = fmaf(nib_f(q[k], 28), xh.w, s1);
                        }
                        const float *bt = bs + (int64_t)t * nb + sb * 8 + 2 * c;
                        acc[t] = fmaf(d, (float)sc[0] * s0 + (float)sc[1] * s1, acc[t]) -
                                 dmin * ((float)mn[0] * bt[0] + (float)mn[1] * bt[1]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const float v = warp_sum(acc[t]);
            if (lane == t && t < m) y[t * ldy + row] = bias ? v + bias[row] : v;
        }
    }
}

size_t f32_smem(int m, int in_dim) { return (size_t)m * in_dim * 4 + (size_t)m * (in_dim / 32) * 4; }

template <int MT>
cudaError_t f32_launch(const void *w, const float *x, int64_t ldx, float *y, int64_t ldy, const float *bias, int m,
                       int64_t out_dim, int in_dim, cudaStream_t s)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_f32_gemv_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const size_t smem = f32_smem(m, in_dim);
    const int64_t rows_per_cta = kFWarps;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((out_dim + rows_per_cta - 1) / rows_per_cta,
                                                                 (int64_t)dev_info().sm_count * 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4k_f32_gemv_kernel<MT>, static_cast<const uint8_t *>(w), x, ldx, y, ldy, bias,
                              m, out_dim, in_dim);
}

}  // namespace

// Tokens one launch takes for this in_dim (the activations must fit in shared
// memory); 0 if not even one does.
int q4k_f32_gemv_group(int64_t in_dim)
{
    int mt = kFMaxTokens;
    while (mt > 0 && f32_smem(mt, (int)in_dim) > dev_info().smem_optin) --mt;
    return mt;
}

cudaError_t launch_q4k_f32_gemv(const void *w, const float *x, int64_t ldx, float *y, int64_t ldy, const float *bias,
                                int64_t m, int64_t out_dim, int64_t in_dim, cudaStream_t s)
{
    const int mg = q4k_f32_gemv_group(in_dim);
    if (mg < 1) return cudaErrorInvalidConfiguration;
    for (int64_t t0 = 0; t0 < m; t0 += mg) {
        const int n = (int)std::min<int64_t>(mg, m - t0);
        cudaError_t e;
        if (n == 1)
            e = f32_launch<1>(w, x + t0 * ldx, ldx, y + t0 * ldy, ldy, bias, n, out_dim, (int)in_dim, s);
        else if (n == 2)
            e = f32_launch<2>(w, x + t0 * ldx, ldx, y + t0 * ldy, ldy, bias, n, out_dim, (int)in_dim, s);
        else
            e = f32_launch<4>(w, x + t0 * ldx, ldx, y + t0 * ldy, ldy, bias, n, out_dim, (int)in_dim, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rz
