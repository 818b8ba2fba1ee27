// gemv_q4_0_mma.cu -- the Q4_0 weight x f32 activation GEMV (the LM head) for
// one to eight tokens per launch on the tensor cores.
//
// Operation: that of gemv_q4_0.cu (q4_0_gemv_into in GpuModelQ4::forward,
// realizar 0.8.4 src/gpu/adapters/using.rs): for every row r and token t
//   y[t][r] = bias[r] + sum_b d_rb * sum_{k < 32} (q_rbk - 8) x[t][32 b + k].
//
// Per block of 32 values the dot of the codes with the activations comes out of
// mma.sync.m16n8k16 with f16 operands and f32 accumulation:
//   A (16 rows x 16 k)  = q - 8, exact in f16 (from the 1024 + q bit pattern);
//   B (16 k x 8 tokens) = x in two f16 pieces, hi = f16(x) and lo = f16(x - hi)
//                         (x - hi is exact in f32), so that hi + lo is x to about
//                         2^-22 relative (|x| below the f16 range, 65504);
//   D                   = the block's dot: the low nibbles (values 0..15) and
//                         the high nibbles (16..31), each against both pieces,
//                         four MMAs into one f32 accumulator;
// then acc += d_rb * D in f32.  The one-token kernel computes the same sums in
// f32 FMAs; the two orders differ by f32 rounding only.
//
// Structure (that of gemv_q4k_mma.cu): one CTA per SM owns rpc rows, cut into
// 16-row tiles; a producer warp streams stages through a ring with the tensor
// memory access engine, a stage being one 2-D box -- the rpc rows over a slice
// of eight blocks, 144 bytes, landing with a row pitch of 144 (16 mod 128:
// conflict-free 16-bit code loads).  Consumer warp w takes tile w over every
// slice, so each warp holds the sums of its 16 rows x 8 tokens in registers for
// the whole row and stores them itself.  The activations are staged once per
// CTA: per four values the hi pieces, then the lo pieces (16 bytes), so that a
// lane's two B fragments of a block half are one 16-byte load; token pitch 64
// mod 128.  A block's code bytes start 2 mod 4 in every other block, so a lane
// reads its four code bytes of a row as two 16-bit loads.  Rows whose length is
// not a multiple of 16 bytes (in_dim not a multiple of 256) cannot be described
// to the copy engine: those heads run the one-token kernel once per token.
// Every wait is bounded.
#include <cuda_fp16.h>

#include <algorithm>

#include "mma_f16.cuh"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kHW = 15;                    // consumer warps (16 warps: 128 registers a thread)
constexpr int kHThreads = (kHW + 1) * 32;  // + 1 producer warp
constexpr int kHSmem = 224 * 1024;         // shared-memory budget of a CTA
constexpr int kHSlice = 144;               // eight blocks of 18 bytes
constexpr int kHMaxTokens = 8;             // one n-tile of the MMA

struct HArgs {
    CUtensorMap map;    // the weights as [out_dim][row_bytes / 4] u32, box (36, rpc)
    const float *x;     // [m][ldx]
    int64_t ldx;
    float *y;           // [m][out_dim]
    const float *bias;  // [out_dim] or nullptr
    int64_t out_dim;
    int in_dim, nsl;    // nsl = in_dim / 256 slices
    int m;              // tokens of this launch, 1..8
    int rpc;            // rows per CTA (<= 16 kHW)
    int NS;             // ring stages
    int stage_bytes;    // ceil(rpc / 16) tiles of 16 rows x 144 bytes
    unsigned *err;
};

__host__ __device__ inline int64_t head_x_pitch(int in_dim) { return 4 * (int64_t)in_dim + 64; }
__host__ __device__ inline int64_t head_x_bytes(int m, int in_dim) { return (int64_t)m * head_x_pitch(in_dim); }

__device__ __forceinline__ uint32_t lds_u16(uint32_t a)
{
    uint16_t v;
    asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Two code bytes (b0 in bits 0-7, b1 in 8-15) as the f16 pairs (lo(b0) - 8,
// lo(b1) - 8) and (hi(b0) - 8, hi(b1) - 8): 1024 + q from the bit pattern minus
// 1032; 1024 + 16 q times 1/16 minus 72.  Exact.
__device__ __forceinline__ void nib_pairs(uint32_t h, uint32_t &lo, uint32_t &hi)
{
    uint32_t v;
    asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(v) : "r"(h));  // bytes: b0, 0, b1, 0
    lo = hsub2u(lop_and_or(v, 0x000F000Fu, 0x64006400u), 0x64086408u /* 1032 */);
    hi = hfma2u(lop_and_or(v, 0x00F000F0u, 0x64006400u), 0x2C002C00u /* 1/16 */, 0xD480D480u /* -72 */);
}

__global__ void __launch_bounds__(kHThreads, 1) q4_0_head_mma_kernel(const __grid_constant__ HArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *xs = ring + (int64_t)a.NS * a.stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(xs + head_x_bytes(a.m, a.in_dim));
    uint64_t *empty = full + a.NS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)blockIdx.x * a.rpc;
    const int rows = (int)min((int64_t)a.rpc, a.out_dim - r0);
    const int ntiles = (a.rpc + 15) / 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kHW);  // one arrival per consumer warp
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kHW) {
        // ------------------------------------------------ producer: the weights do
        // not depend on the previous kernel
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            tma_prefetch_desc(&a.map);
            const unsigned box_bytes = (unsigned)a.rpc * (unsigned)kHSlice;
            int64_t q = 0;
            bool ok = true;
            RingPos rp{0, 0u};
            for (; q < a.nsl; ++q, ring_next(rp, a.NS)) {
                if (q >= a.NS && !mbar_wait(&empty[rp.s], rp.par ^ 1u)) {
                    set_error(a.err, DEV_TIMEOUT_Q40);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[rp.s], box_bytes);
                tma_load_2d(ring + (int64_t)rp.s * a.stage_bytes, &a.map, (int)q * (kHSlice / 4), (int)r0,
                            &full[rp.s], pol);
            }
            if (!ok) {
                // copies issued but possibly not complete must land before exit
                for (int64_t p = (q > a.NS ? q - a.NS : 0); p < q; ++p)
                    if (!mbar_wait(&full[p % a.NS], (unsigned)((p / a.NS) & 1))) set_error(a.err, DEV_TIMEOUT_DRAIN);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();  // the activations come from the previous kernel
    const int tid = threadIdx.x;
    {
        // x -> (hi, lo) f16 pieces: per four values, hi[4] then lo[4].  Each thread
        // issues kQ loads before it converts any (one round trip to L2 per kQ
        // values rather than one each: 8 tokens x 4096 values is 17 per thread).
        constexpr int kQ = 12;
        const int64_t pitch = head_x_pitch(a.in_dim);
        const int n4 = a.in_dim / 4, nq = a.m * n4;
        for (int q0 = 0; q0 < nq; q0 += kQ * kHW * 32) {
            float4 v[kQ];
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kHW * 32 + tid;
                if (q < nq) {
                    const int t = q / n4;
                    v[u] = __ldg(reinterpret_cast<const float4 *>(a.x + t * a.ldx) + (q - t * n4));
                }
            }
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kHW * 32 + tid;
                if (q < nq) {
                    const int t = q / n4;
                    const __half2 h01 = __floats2half2_rn(v[u].x, v[u].y), h23 = __floats2half2_rn(v[u].z, v[u].w);
                    const __half2 l01 = __floats2half2_rn(v[u].x - __low2float(h01), v[u].y - __high2float(h01));
                    const __half2 l23 = __floats2half2_rn(v[u].z - __low2float(h23), v[u].w - __high2float(h23));
                    uint4 o;
                    o.x = *reinterpret_cast<const uint32_t *>(&h01);
                    o.y = *reinterpret_cast<const uint32_t *>(&h23);
                    o.z = *reinterpret_cast<const uint32_t *>(&l01);
                    o.w = *reinterpret_cast<const uint32_t *>(&l23);
                    *reinterpret_cast<uint4 *>(xs + t * pitch + (int64_t)(q - t * n4) * 16) = o;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kHW * 32) : "memory");
    }

    const int g = lane >> 2, i = lane & 3;
    const uint32_t ring_s = smem_u32(ring);
    // this lane's 16 bytes of block 0 (token g, clamped into the staged tokens)
    const uint32_t xrow = smem_u32(xs) + (uint32_t)(min(g, a.m - 1) * head_x_pitch(a.in_dim)) + 16u * i;
    const bool active = warp < ntiles;
    const int tile = warp;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool failed = false;
    RingPos rp{0, 0u};
    for (int sl = 0; sl < a.nsl; ++sl, ring_next(rp, a.NS)) {
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(&full[rp.s], rp.par))) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_Q40);
            failed = true;
        }
        if (!failed && active) {
            const uint32_t base = smem_after(ring_s);  // ordered after the wait
            const uint32_t rowA = base + (uint32_t)(rp.s * a.stage_bytes + (tile * 16 + g) * kHSlice);
            const uint32_t rowB = rowA + 8u * kHSlice;
            const uint32_t xb = xrow + (base - ring_s) + (uint32_t)sl * 1024u;  // 256 values x 4 bytes
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                const uint32_t ba = rowA + 18u * bb, bbB = rowB + 18u * bb;
                uint32_t lo[4], hi[4];  // A fragments: values 4i..4i+3 of the block (low / high nibbles)
                nib_pairs(lds_u16(ba + 2 + 4 * i), lo[0], hi[0]);       // row g, values 4i, 4i+1
                nib_pairs(lds_u16(bbB + 2 + 4 * i), lo[1], hi[1]);      // row g + 8
                nib_pairs(lds_u16(ba + 2 + 4 * i + 2), lo[2], hi[2]);   // row g, values 4i+2, 4i+3
                nib_pairs(lds_u16(bbB + 2 + 4 * i + 2), lo[3], hi[3]);  // row g + 8
                const float dA = h2f((uint16_t)lds_u16(ba)), dB = h2f((uint16_t)lds_u16(bbB));
                const uint4 X0 = lds_u4(xb + 128u * bb), X1 = lds_u4(xb + 128u * bb + 64u);
                float d[4];
                mma16816(d, lo, X0.x, X0.y, zero);  // values 0..15: hi piece
                mma16816(d, lo, X0.z, X0.w, d);     // lo piece
                mma16816(d, hi, X1.x, X1.y, d);     // values 16..31
                mma16816(d, hi, X1.z, X1.w, d);
                acc[0] = fmaf(dA, d[0], acc[0]);
                acc[1] = fmaf(dA, d[1], acc[1]);
                acc[2] = fmaf(dB, d[2], acc[2]);
                acc[3] = fmaf(dB, d[3], acc[3]);
            }
        }
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(&empty[rp.s]);
    }
    if (!active || failed) return;
    // accumulators: rows g, g + 8 of the tile x tokens 2i, 2i + 1
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int rr = tile * 16 + g + ((e >> 1) << 3), t = 2 * i + (e & 1);
        if (rr < rows && t < a.m) {
            const int64_t r = r0 + rr;
            a.y[t * a.out_dim + r] = acc[e] + (a.bias ? a.bias[r] : 0.0f);
        }
    }
}

// Rows per CTA, ring stages, shared memory of a launch of mt tokens (false when
// two stages do not fit beside the activations).
bool head_plan(int64_t out_dim, int64_t in_dim, int mt, int &rpc, int64_t &grid, int &ns, int &stage_bytes,
               size_t &smem)
{
    const int sms = dev_info().sm_count;
    int64_t r = (out_dim + sms - 1) / sms;
    if (r > 16 * kHW) r = 16 * kHW;
    rpc = (int)r;
    grid = (out_dim + rpc - 1) / rpc;
    stage_bytes = (rpc + 15) / 16 * 16 * kHSlice;
    const int64_t xb = head_x_bytes(mt, (int)in_dim);
    const int64_t budget = (int64_t)std::min<int64_t>(kHSmem, dev_info().smem_optin) - xb - 1024;
    ns = (int)std::min<int64_t>(8, budget / (stage_bytes + 16));
    if (ns < 2) return false;
    smem = (size_t)((int64_t)ns * stage_bytes + xb + 16 * ns);
    return true;
}

cudaError_t launch_head_group(const void *w, const float *x, int64_t ldx, float *y, int mt, int64_t out_dim,
                              int64_t in_dim, const float *bias, cudaStream_t s)
{
    HArgs a = {};
    int64_t grid;
    size_t smem;
    if (!head_plan(out_dim, in_dim, mt, a.rpc, grid, a.NS, a.stage_bytes, smem)) return cudaErrorInvalidConfiguration;
    const int64_t row_bytes = in_dim / 32 * 18;
    const cudaError_t e = encode_tensor_map_2d(&a.map, w, 4, (uint64_t)row_bytes / 4, (uint64_t)out_dim,
                                               (uint64_t)row_bytes, (uint32_t)(kHSlice / 4), (uint32_t)a.rpc);
    if (e != cudaSuccess) return e;
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.bias = bias;
    a.out_dim = out_dim;
    a.in_dim = (int)in_dim;
    a.nsl = (int)(in_dim / 256);
    a.m = mt;
    a.err = dev_error_word();
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if (dev < 64 && !attr_done[dev]) {
        const cudaError_t ea = cudaFuncSetAttribute(q4_0_head_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    (int)dev_info().smem_optin);
        if (ea != cudaSuccess) return ea;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kHThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4_0_head_mma_kernel, a);
}

}  // namespace

bool q4_0_head_mma_ok(int64_t m, int64_t out_dim, int64_t in_dim, const float *x, int64_t ldx)
{
    if (m < 1 || out_dim < 1 || in_dim < 256 || in_dim % 256 || ldx % 4 ||
        (reinterpret_cast<uintptr_t>(x) & 15))
        return false;
    int rpc, ns, sb;
    int64_t grid;
    size_t smem;
    return head_plan(out_dim, in_dim, kHMaxTokens, rpc, grid, ns, sb, smem);
}

int q4_0_head_mma_launches(int64_t m) { return (int)((m + kHMaxTokens - 1) / kHMaxTokens); }

cudaError_t launch_q4_0_head_mma(const void *w, const float *x, int64_t ldx, float *y, int64_t m, int64_t out_dim,
                                 int64_t in_dim, const float *bias, cudaStream_t s)
{
    // equal token groups of at most eight (one n-tile each)
    const int64_t ng = q4_0_head_mma_launches(m);
    const int64_t mc = (m + ng - 1) / ng;
    for (int64_t t0 = 0; t0 < m; t0 += mc) {
        const int mt = (int)std::min<int64_t>(mc, m - t0);
        const cudaError_t e = launch_head_group(w, x + t0 * ldx, ldx, y + t0 * out_dim, mt, out_dim, in_dim, bias, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rz
