// gemv_q4_0.cu -- Q4_0 weight x f32 activation GEMV (the LM head).
//
// Operation (q4_0_gemv_into in GpuModelQ4::forward, realizar 0.8.4
// src/gpu/adapters/using.rs): y[t][r] = sum_b d_rb * sum_i (q_rbi - 8) * x[t][32 b + i]
// with f32 activations (the normed hidden state is passed as f32).
//
// Layout on the GPU.  A row is in_dim / 32 blocks of 18 bytes, so rows and blocks
// are only 2-byte aligned.  Lanes own blocks (lane L of column warp cw owns block
// 32 cw + L) and walk down the rows of the CTA, so each lane keeps its 32
// activations in registers (m == 1) and reuses them for every row; each warp
// load instruction reads 32 consecutive blocks (576 contiguous bytes).  Nibbles
// become exact floats (q - 8) with the exponent trick 0x4B000000 | q minus
// (2^23 + 8), so the inner loop is one integer op, one add and one FMA per
// weight.  Partial sums of the column warps of a row are combined in a fixed
// order in shared memory (deterministic).
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowUnroll = 4;

struct Args {
    const uint8_t *w;
    const float *x;
    float *y;
    int64_t out_dim, in_dim;
    int nb;        // blocks per row
    int cw;        // column chunks of 32 blocks
    int wg;        // warps per row group
    int rp;        // row groups per CTA
    int m;
    int64_t ldx;   // elements between tokens' activation rows
    int64_t rows_per_cta_max;
    const float *bias;  // [out_dim] added to every token's row, or nullptr (the LM-head bias)
};

__device__ __forceinline__ float nib_minus8(uint32_t word, int shift)
{
    return __int_as_float((int)(0x4B000000u | ((word >> shift) & 15u))) - 8388616.0f;
}

// partial dot of one block (18 bytes at p) with 32 activations xv
__device__ __forceinline__ float block_dot(const uint8_t *p, const float (&xv)[32])
{
    const uint16_t *p16 = reinterpret_cast<const uint16_t *>(p);
    const float d = h2f(__ldg(p16));
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t w = (uint32_t)__ldg(p16 + 1 + 2 * k) | ((uint32_t)__ldg(p16 + 2 + 2 * k) << 16);
        // bytes 4k..4k+3: low nibbles are elements 4k..4k+3, high nibbles 16+4k..
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            acc = fmaf(nib_minus8(w, 8 * b), xv[4 * k + b], acc);
            acc = fmaf(nib_minus8(w, 8 * b + 4), xv[16 + 4 * k + b], acc);
        }
    }
    return d * acc;
}

__device__ __forceinline__ void load_x(const float *xp_f, float (&xv)[32])
{
    const float4 *xp = reinterpret_cast<const float4 *>(xp_f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(xp + i);
        xv[4 * i] = v.x;
        xv[4 * i + 1] = v.y;
        xv[4 * i + 2] = v.z;
        xv[4 * i + 3] = v.w;
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads) q4_0_gemv_kernel(const Args a)
{
    extern __shared__ float part[];  // [rows of this CTA][MT][wg]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t r0 = a.out_dim * blockIdx.x / G, r1 = a.out_dim * (blockIdx.x + 1) / G;
    const int rg = warp / a.wg, wc = warp % a.wg;
    const int64_t row_bytes = (int64_t)a.nb * 18;
    const bool direct = (a.wg == 1 && a.cw == 1);
    pdl_launch_dependents();
    pdl_wait();

    if (rg < a.rp) {
        for (int cw = wc; cw < a.cw; cw += a.wg) {
            const int b = cw * 32 + lane;
            const bool active = b < a.nb;
            float xv[32];
            if (MT == 1) {
                if (active) load_x(a.x + (int64_t)b * 32, xv);
            }
            for (int64_t r = r0 + rg; r < r1; r += (int64_t)a.rp * kRowUnroll) {
                float res[kRowUnroll][MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (MT > 1 && t < a.m && active) load_x(a.x + t * a.ldx + (int64_t)b * 32, xv);
#pragma unroll
                    for (int u = 0; u < kRowUnroll; ++u) {
                        const int64_t rr = r + (int64_t)u * a.rp;
                        float v = 0.0f;
                        if (t < a.m && active && rr < r1)
                            v = block_dot(a.w + rr * row_bytes + (int64_t)b * 18, xv);
                        res[u][t] = warp_sum(v);
                    }
                }
                if (lane == 0) {
#pragma unroll
                    for (int u = 0; u < kRowUnroll; ++u) {
                        const int64_t rr = r + (int64_t)u * a.rp;
                        if (rr >= r1) continue;
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
                            if (t >= a.m) continue;
                            if (direct) {
                                a.y[t * a.out_dim + rr] = a.bias ? res[u][t] + a.bias[rr] : res[u][t];
                            } else {
                                float *slot = &part[((rr - r0) * MT + t) * a.wg + wc];
                                *slot = (cw == wc) ? res[u][t] : *slot + res[u][t];
                            }
                        }
                    }
                }
            }
        }
    }
    if (direct) return;
    __syncthreads();
    // combine the column warps of each row in a fixed order
    for (int64_t i = threadIdx.x; i < (r1 - r0) * MT; i += kThreads) {
        const int64_t rl = i / MT;
        const int t = (int)(i % MT);
        if (t >= a.m) continue;
        float sum = 0.0f;
        for (int k = 0; k < a.wg; ++k) sum += part[(rl * MT + t) * a.wg + k];
        a.y[t * a.out_dim + r0 + rl] = a.bias ? sum + a.bias[r0 + rl] : sum;
    }
}

template <int MT>
cudaError_t launch_t(const Args &a, int grid, size_t smem, cudaStream_t s)
{
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(q4_0_gemv_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4_0_gemv_kernel<MT>, a);
}

}  // namespace

cudaError_t launch_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                             int64_t in_dim, cudaStream_t s, const float *bias)
{
    return launch_q4_0_gemv_ld(w, x, in_dim, y, m, out_dim, in_dim, s, bias);
}

cudaError_t launch_q4_0_gemv_ld(const void *w, const float *x, int64_t ldx, float *y, int64_t m,
                                int64_t out_dim, int64_t in_dim, cudaStream_t s, const float *bias)
{
    Args a = {};
    a.bias = bias;
    a.ldx = ldx;
    a.w = static_cast<const uint8_t *>(w);
    a.x = x;
    a.y = y;
    a.out_dim = out_dim;
    a.in_dim = in_dim;
    a.nb = (int)(in_dim / 32);
    a.cw = (a.nb + 31) / 32;
    a.wg = a.cw < kWarps ? a.cw : kWarps;
    a.rp = kWarps / a.wg;
    a.m = (int)m;
    const int sms = dev_info().sm_count;
    // enough CTAs to fill the GPU several times over, rows per CTA bounded so the
    // partial-sum table stays small
    int64_t grid = 4 * (int64_t)sms;
    const int mt = m <= 1 ? 1 : (m <= 4 ? 4 : 16);
    int64_t rows = (out_dim + grid - 1) / grid;
    const int64_t max_rows = (48 * 1024) / (4 * mt * a.wg);
    if (rows > max_rows) {
        grid = (out_dim + max_rows - 1) / max_rows;
        rows = (out_dim + grid - 1) / grid;
    }
    if (grid > out_dim) grid = out_dim;
    rows = (out_dim + grid - 1) / grid;
    a.rows_per_cta_max = rows;
    const size_t smem = (a.wg == 1 && a.cw == 1) ? 0 : (size_t)rows * mt * a.wg * sizeof(float);
    if (mt == 1) return launch_t<1>(a, (int)grid, smem, s);
    if (mt == 4) return launch_t<4>(a, (int)grid, smem, s);
    return launch_t<16>(a, (int)grid, smem, s);
}

}  // namespace rz
