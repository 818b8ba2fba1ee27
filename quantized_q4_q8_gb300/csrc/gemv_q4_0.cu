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
#include <algorithm>

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

// ---------------------------------------------------------------------------
// One token (the LM head of a decode step): the weights stream through a ring of
// shared-memory stages filled by bulk copies, as the Q4_K GEMV does.  A CTA per
// SM owns a contiguous range of rows (a whole number of copy units: rows whose
// bytes are a multiple of 16); a producer warp keeps the ring full, 16 consumer
// warps are (nb / 32) column warps x row groups: lane L of column warp c owns
// block 32 c + L of every row and keeps its 32 activations in registers,
// pre-scaled by 2^-s for the bit position s its nibble has inside a 16-bit half
// of the packed word.  A nibble then becomes an exact float with one LOP3
// (0x4B000000 | (half & (0xF << s)) = 2^23 + q 2^s) and one subtraction of 2^23,
// and the dot runs on fma.rn.f32x2 pairs:
//   sum_i (q_i - 8) x_i = sum_i (q_i 2^s_i)(x_i 2^-s_i) - 8 sum_i x_i.
// Per-row partial sums of the column warps are added in a fixed order at the end.
constexpr int kRW = 16;                  // consumer warps
constexpr int kRThreads = (kRW + 1) * 32;
constexpr int kRingBytes = 196 * 1024;
// 64 KB stages: every mbarrier wait costs a warp a few hundred cycles here, so fewer,
// larger stages keep more of the consumers' time on the dot products.
constexpr int kStageBytes = 64 * 1024;

struct RArgs {
    const uint8_t *w;
    const float *x;
    float *y;
    const float *bias;
    int64_t out_dim, row_bytes;
    int nb;          // blocks per row
    int cw, rg;      // column warps per row, row groups (cw * rg == kRW)
    int unit;        // rows per copy unit
    int64_t units;   // copy units of the matrix
    int stage_rows;  // rows per ring stage (a multiple of unit)
    int NS;          // stages in the ring
    int64_t rows_max;  // rows of the largest CTA range
    unsigned *err;
};

__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ uint32_t lds_b32(uint32_t addr)
{
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// 2^23 + v as a float (v < 2^23 in the mantissa bits)
__device__ __forceinline__ float magic(uint32_t v) { return __uint_as_float(v | 0x4B000000u); }

// bit position of element i's nibble inside its 16-bit half: byte k = i % 16,
// nibble i / 16 (high), byte k % 2 inside the half
__host__ __device__ constexpr int nib_shift(int i) { return 8 * ((i % 16) % 2) + 4 * (i / 16); }

// sum_i q_i 2^s_i xs_i of one block whose 16 code bytes are q[0..3]
__device__ __forceinline__ float block_dot_scaled(const uint32_t (&q)[4], const float (&xs)[32])
{
    const float2 off = make_float2(-8388608.0f, -8388608.0f);
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;  // two chains
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint32_t v = hh ? (q[wd] >> 16) : q[wd];
            const int k0 = 4 * wd + 2 * hh;  // bytes k0 (bits 0-7) and k0 + 1 (bits 8-15)
            // elements: k0 (s 0), k0 + 16 (s 4), k0 + 1 (s 8), k0 + 17 (s 12)
            const float2 fa = f2_add(make_float2(magic(v & 0xFu), magic(v & 0xF0u)), off);
            const float2 fb = f2_add(make_float2(magic(v & 0xF00u), magic(v & 0xF000u)), off);
            acc0 = f2_fma(fa, make_float2(xs[k0], xs[k0 + 16]), acc0);
            acc1 = f2_fma(fb, make_float2(xs[k0 + 1], xs[k0 + 17]), acc1);
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

__global__ void __launch_bounds__(kRThreads, 1) q4_0_gemv_ring_kernel(const RArgs a)
{
    extern __shared__ __align__(128) uint8_t rsm[];
    const int64_t stage_bytes = (int64_t)a.stage_rows * a.row_bytes;
    uint8_t *ring = rsm;
    float *part = reinterpret_cast<float *>(rsm + (int64_t)a.NS * stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(part + a.rows_max * a.cw) + 7) & ~uintptr_t(7));
    uint64_t *empty = full + a.NS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t r0 = (a.units * blockIdx.x / G) * a.unit;
    const int64_t r1 = min((a.units * (blockIdx.x + 1) / G) * a.unit, a.out_dim);
    const int64_t nrows = r1 > r0 ? r1 - r0 : 0;
    const int64_t nstages = (nrows + a.stage_rows - 1) / a.stage_rows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kRW) {
        // ---- producer: the weights do not depend on the previous kernel
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            RingPos rp{0, 0u};
            for (int64_t k = 0; k < nstages; ++k, ring_next(rp, a.NS)) {
                if (k >= a.NS && !mbar_wait(&empty[rp.s], rp.par ^ 1u)) {
                    set_error(a.err, DEV_TIMEOUT_Q40);
                    // copies issued before must land before the CTA exits
                    for (int64_t q = (k > a.NS ? k - a.NS : 0); q < k; ++q)
                        if (!mbar_wait(&full[q % a.NS], (unsigned)((q / a.NS) & 1))) set_error(a.err, DEV_TIMEOUT_DRAIN);
                    break;
                }
                const int64_t u0 = r0 + k * a.stage_rows;
                const int64_t n = min((int64_t)a.stage_rows, r1 - u0);
                const unsigned bytes = (unsigned)(n * a.row_bytes);
                mbar_arrive_expect_tx(&full[rp.s], bytes);
                bulk_g2s_hint(ring + (int64_t)rp.s * stage_bytes, a.w + u0 * a.row_bytes, bytes, &full[rp.s], pol);
            }
        }
        return;
    }

    // ---- consumers
    pdl_wait();  // the activations come from the previous kernel
    const int cwi = warp % a.cw, rgi = warp / a.cw;
    const int b = 32 * cwi + lane;  // this lane's block
    const bool active = b < a.nb;
    float xs[32];
    float sx = 0.0f;
    {
        const float4 *xp = reinterpret_cast<const float4 *>(a.x + (int64_t)(active ? b : 0) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = active ? __ldg(xp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            xs[4 * i] = v.x;
            xs[4 * i + 1] = v.y;
            xs[4 * i + 2] = v.z;
            xs[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            sx += xs[i];
            xs[i] = ldexpf(xs[i], -nib_shift(i));  // exact: a power-of-two scale
        }
    }
    const uint32_t ring_s = smem_u32(ring);
    RingPos rp{0, 0u};
    bool ok = true;
    for (int64_t k = 0; k < nstages; ++k, ring_next(rp, a.NS)) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full[rp.s], rp.par));
        if (!ok) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_Q40);
            break;
        }
        const int64_t u0 = r0 + k * a.stage_rows;
        const int n = (int)min((int64_t)a.stage_rows, r1 - u0);
        const uint32_t slot = ring_s + (uint32_t)((int64_t)rp.s * stage_bytes);
        // two rows in flight per warp: independent loads, dots and reductions
        for (int rr = rgi; rr < n; rr += 2 * a.rg) {
            float v[2] = {0.0f, 0.0f};
            const bool has1 = rr + a.rg < n;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (active && (u == 0 || has1)) {
                    // the 18 bytes of the block: five aligned words, realigned by funnel shifts
                    const uint32_t addr = slot + (uint32_t)((int64_t)(rr + u * a.rg) * a.row_bytes) + 18u * (uint32_t)b;
                    const uint32_t base = addr & ~3u, off = addr & 3u;  // off is 0 or 2
                    uint32_t w5[5];
#pragma unroll
                    for (int i = 0; i < 5; ++i) w5[i] = lds_b32(base + 4u * i);
                    const uint32_t sh = 16u - 8u * off;  // 16 (off 0) or 0 (off 2)
                    uint32_t q[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t lo = off ? w5[i + 1] : w5[i];
                        const uint32_t hi = off ? (i + 2 < 5 ? w5[i + 2] : 0u) : w5[i + 1];
                        q[i] = __funnelshift_r(lo, hi, sh);
                    }
                    const float d = h2f((uint16_t)(off ? (w5[0] >> 16) : (w5[0] & 0xffffu)));
                    v[u] = d * (block_dot_scaled(q, xs) - 8.0f * sx);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
                v[1] += __shfl_xor_sync(0xffffffffu, v[1], o);
            }
            if (lane == 0) {
                part[(u0 - r0 + rr) * a.cw + cwi] = v[0];
                if (has1) part[(u0 - r0 + rr + a.rg) * a.cw + cwi] = v[1];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[rp.s]);
    }
    // the column warps' partial sums of every row, in a fixed order
    asm volatile("bar.sync 1, %0;" ::"r"(kRW * 32) : "memory");
    if (!ok) return;
    for (int64_t i = threadIdx.x; i < nrows; i += kRW * 32) {
        float sum = 0.0f;
        for (int c = 0; c < a.cw; ++c) sum += part[i * a.cw + c];
        a.y[r0 + i] = a.bias ? sum + a.bias[r0 + i] : sum;
    }
}

// The ring kernel's geometry for these shapes; false when they do not suit it.
bool ring_plan(int64_t out_dim, int64_t in_dim, RArgs &a, int64_t &grid, size_t &smem)
{
    a = RArgs{};
    a.nb = (int)(in_dim / 32);
    a.cw = (a.nb + 31) / 32;
    if (a.cw > kRW || kRW % a.cw) return false;
    a.rg = kRW / a.cw;
    a.row_bytes = (int64_t)a.nb * 18;
    int g = 16;
    while (a.row_bytes % g) g >>= 1;
    a.unit = 16 / g;  // rows whose bytes are a multiple of 16
    if ((out_dim * a.row_bytes) % 16) return false;
    a.units = (out_dim + a.unit - 1) / a.unit;
    const int64_t per_stage = std::max<int64_t>(1, kStageBytes / (a.row_bytes * a.unit));
    a.stage_rows = (int)(per_stage * a.unit);
    const int64_t stage_bytes = (int64_t)a.stage_rows * a.row_bytes;
    a.NS = (int)std::min<int64_t>(32, kRingBytes / stage_bytes);
    if (a.NS < 2) return false;
    grid = std::min<int64_t>(dev_info().sm_count, a.units);
    a.rows_max = ((a.units + grid - 1) / grid) * a.unit;
    smem = (size_t)(a.NS * stage_bytes) + (size_t)a.rows_max * a.cw * 4 + 8 + 16 * (size_t)a.NS;
    return smem <= dev_info().smem_optin;
}

// One token through the ring kernel, when the shapes allow it (else *used = false).
cudaError_t launch_ring(const void *w, const float *x, float *y, int64_t out_dim, int64_t in_dim, const float *bias,
                        cudaStream_t s, bool *used)
{
    *used = false;
    RArgs a;
    int64_t grid;
    size_t smem;
    if (!ring_plan(out_dim, in_dim, a, grid, smem)) return cudaSuccess;
    a.w = static_cast<const uint8_t *>(w);
    a.x = x;
    a.y = y;
    a.bias = bias;
    a.out_dim = out_dim;
    a.err = dev_error_word();
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4_0_gemv_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    *used = true;
    return cudaLaunchKernelEx(&cfg, q4_0_gemv_ring_kernel, a);
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

int q4_0_gemv_launches(int64_t m, int64_t out_dim, int64_t in_dim)
{
    RArgs a;
    int64_t grid;
    size_t smem;
    if (q4_0_head_mma_ok(m, out_dim, in_dim, nullptr, in_dim)) return q4_0_head_mma_launches(m);
    return ring_plan(out_dim, in_dim, a, grid, smem) ? (int)m : 1;
}

cudaError_t launch_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                             int64_t in_dim, cudaStream_t s, const float *bias)
{
    return launch_q4_0_gemv_ld(w, x, in_dim, y, m, out_dim, in_dim, s, bias);
}

cudaError_t launch_q4_0_gemv_ld(const void *w, const float *x, int64_t ldx, float *y, int64_t m,
                                int64_t out_dim, int64_t in_dim, cudaStream_t s, const float *bias)
{
    // the tensor-core kernel (rows of a whole number of 144-byte slices): it reads
    // the weights once per eight tokens, and even for one token it is faster
    // than the ring kernel below (32000 x 4096: 22.8 against 30.1 us)
    if (q4_0_head_mma_ok(m, out_dim, in_dim, x, ldx))
        return launch_q4_0_head_mma(w, x, ldx, y, m, out_dim, in_dim, bias, s);
    {
        // the ring kernel, once per token: each launch streams the weights at the
        // bandwidth the one-token kernel reaches, where the multi-token kernel
        // below re-reads every block per token from the cache hierarchy
        bool used = false;
        cudaError_t e = launch_ring(w, x, y, out_dim, in_dim, bias, s, &used);
        for (int64_t t = 1; used && e == cudaSuccess && t < m; ++t)
            e = launch_ring(w, x + t * ldx, y + t * out_dim, out_dim, in_dim, bias, s, &used);
        if (used || e != cudaSuccess) return e;
    }
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
