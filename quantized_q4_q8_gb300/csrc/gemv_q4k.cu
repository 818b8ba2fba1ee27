// gemv_q4k.cu -- Q4_K weight x Q8_1 activation GEMV for decode (m <= 16 tokens).
//
// Operation (q4k_q8_gemv_async of realizar 0.8.5 src/cuda/executor/cached.rs,
// transformer_layer_gpu_true_dp4a): for every output row r and token t
//   y[t][r] = sum_b d_b * sum_j sc_bj * d8_tbj * I_tbj - dmin_b * sum_j m_bj * s_tbj,
// I_tbj the exact int32 dot of the 32 4-bit codes of sub-block j with the 32
// int8 codes of the matching Q8_1 block.
//
// GB300 design.  The kernel is bound by streaming the 144-byte super-blocks
// from HBM.  Each warp owns a contiguous range of output rows and runs its own
// ring of shared-memory slots fed by the 1-D bulk copy engine (cp.async.bulk,
// completion on an mbarrier): lane 0 keeps kSlots pieces of 8 super-blocks
// (1152 bytes) in flight while the warp computes on the oldest one, so the
// bytes in flight live in shared memory instead of registers.  Inside a piece
// each group of 4 lanes takes one super-block and each lane one 32-byte chunk of
// its quants (two sub-blocks: low and high nibbles), so the 32-element integer
// dots are complete within a lane (dp4a on unsigned nibbles x signed int8) and
// only the f32 combination crosses lanes, once per row, in a fixed order (the
// result is deterministic).  Rows shorter than 8 super-blocks are packed
// several to a piece.  Weights are read once for all m tokens.  Every wait on a
// bulk copy is bounded; on expiry the warp records an error and drains.
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 6;
constexpr int kPieceSB = 8;
constexpr int kSB = 144;
constexpr int kPieceBytes = kPieceSB * kSB;
constexpr int kWarpSmem = kSlots * kPieceBytes;
constexpr int kSmemBytes = kWarps * kWarpSmem + kWarps * kSlots * 8;

struct Args {
    const uint8_t *w[3];
    float *y[3];
    const float *res[3];
    int64_t seg_begin[4];  // first unit of segment k; seg_begin[nseg] == units
    int nseg;
    int64_t units;
    int nsb;               // super-blocks per row
    int64_t row_bytes;
    int m;
    const int8_t *xq;      // [m][in_dim]
    const float *xd;       // [m][in_dim/32]
    const float *xs;       // [m][in_dim/32]
    int64_t in_dim;
    unsigned *err;
};

struct Piece {
    int64_t unit;  // first unit of the piece
    int rows;      // whole rows in the piece (packed mode), else 1
    int half;      // 0: gate / plain row, 1: up row (SwiGLU)
    int sb0;       // first super-block of the row in this piece
    int cnt;       // super-blocks per row in this piece
    bool row_end;  // the piece ends its row
};

__device__ __forceinline__ Piece piece_of(int64_t p, int64_t u0, int64_t u1, int rpp, int ppr,
                                          int R, int nsb)
{
    Piece pc;
    if (rpp > 1) {
        pc.unit = u0 + p * rpp;
        pc.rows = (int)min((int64_t)rpp, u1 - pc.unit);
        pc.half = 0;
        pc.sb0 = 0;
        pc.cnt = nsb;
        pc.row_end = true;
    } else {
        int64_t per_unit = (int64_t)R * ppr;
        pc.unit = u0 + p / per_unit;
        int rem = (int)(p % per_unit);
        pc.half = rem / ppr;
        int pir = rem % ppr;
        pc.sb0 = kPieceSB * pir;
        pc.cnt = min(kPieceSB, nsb - pc.sb0);
        pc.rows = 1;
        pc.row_end = (pir == ppr - 1);
    }
    return pc;
}

__device__ __forceinline__ int seg_of(const Args &a, int64_t unit)
{
    int k = 0;
    while (k + 1 < a.nseg && unit >= a.seg_begin[k + 1]) ++k;
    return k;
}

template <int EPI>
__device__ __forceinline__ const uint8_t *row_src(const Args &a, int64_t unit, int half)
{
    if (EPI == EPI_SWIGLU) return a.w[half] + unit * a.row_bytes;
    int k = seg_of(a, unit);
    return a.w[k] + (unit - a.seg_begin[k]) * a.row_bytes;
}

// lane 0: arm the slot barrier and start the copies of piece pc
template <int EPI>
__device__ __forceinline__ void issue_piece(const Args &a, const Piece &pc, uint8_t *slot,
                                            uint64_t *bar)
{
    if (pc.rows > 1 || pc.cnt == a.nsb) {
        // whole rows: one copy per run of rows contiguous in one segment
        unsigned bytes = (unsigned)(pc.rows * a.row_bytes);
        mbar_arrive_expect_tx(bar, bytes);
        int r = 0;
        while (r < pc.rows) {
            int64_t u = pc.unit + r;
            int run = 1;
            if (EPI != EPI_SWIGLU) {
                int k = seg_of(a, u);
                int64_t left = a.seg_begin[k + 1] - u;
                run = (int)min((int64_t)(pc.rows - r), left);
            }
            bulk_g2s(slot + (int64_t)r * a.row_bytes, row_src<EPI>(a, u, pc.half),
                     (unsigned)(run * a.row_bytes), bar);
            r += run;
        }
    } else {
        unsigned bytes = (unsigned)(pc.cnt * kSB);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(slot, row_src<EPI>(a, pc.unit, pc.half) + (int64_t)pc.sb0 * kSB, bytes, bar);
    }
}

// Accumulate one super-block (shared memory at `blk`, row super-block index sb)
// into acc[t] for every token; lane owns 32-byte quant chunk c = lane & 3.
template <int MT>
__device__ __forceinline__ void sb_accumulate(const Args &a, const uint8_t *blk, int sb, int c,
                                              float (&acc)[MT])
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    const float d = h2f((uint16_t)(hdr.x & 0xffffu));
    const float dmin = h2f((uint16_t)(hdr.x >> 16));

    // 6-bit scale and min of sub-blocks j0 = 2c and j1 = 2c + 1
    const int k0 = (2 * c) & 3, k1 = (2 * c + 1) & 3;
    const uint32_t a0 = (hdr.y >> (8 * k0)) & 0xffu, a1 = (hdr.y >> (8 * k1)) & 0xffu;
    const uint32_t b0 = (hdr.z >> (8 * k0)) & 0xffu, b1 = (hdr.z >> (8 * k1)) & 0xffu;
    uint32_t sc0, sc1, m0, m1;
    if (c < 2) {
        sc0 = a0 & 63u;
        sc1 = a1 & 63u;
        m0 = b0 & 63u;
        m1 = b1 & 63u;
    } else {
        const uint32_t c0 = (hdr.w >> (8 * k0)) & 0xffu, c1 = (hdr.w >> (8 * k1)) & 0xffu;
        sc0 = (c0 & 15u) | ((a0 >> 6) << 4);
        sc1 = (c1 & 15u) | ((a1 >> 6) << 4);
        m0 = (c0 >> 4) | ((b0 >> 6) << 4);
        m1 = (c1 >> 4) | ((b1 >> 6) << 4);
    }
    const float dsc0 = d * (float)sc0, dsc1 = d * (float)sc1;
    const float dm0 = dmin * (float)m0, dm1 = dmin * (float)m1;

    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    int lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo[i] = (int)(q[i] & 0x0f0f0f0fu);
        hi[i] = (int)((q[i] >> 4) & 0x0f0f0f0fu);
    }

    const int64_t nb = a.in_dim / 32;
    const int64_t jb = (int64_t)sb * 8 + 2 * c;  // Q8_1 block of sub-block j0
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < a.m) {
            const int4 *xp = reinterpret_cast<const int4 *>(a.xq + t * a.in_dim + jb * 32);
            const int4 x0 = __ldg(xp), x1 = __ldg(xp + 1), x2 = __ldg(xp + 2), x3 = __ldg(xp + 3);
            const float2 d8 = __ldg(reinterpret_cast<const float2 *>(a.xd + t * nb + jb));
            const float2 s8 = __ldg(reinterpret_cast<const float2 *>(a.xs + t * nb + jb));
            int i0 = 0, i1 = 0;
            i0 = __dp4a(lo[0], x0.x, i0);
            i0 = __dp4a(lo[1], x0.y, i0);
            i0 = __dp4a(lo[2], x0.z, i0);
            i0 = __dp4a(lo[3], x0.w, i0);
            i0 = __dp4a(lo[4], x1.x, i0);
            i0 = __dp4a(lo[5], x1.y, i0);
            i0 = __dp4a(lo[6], x1.z, i0);
            i0 = __dp4a(lo[7], x1.w, i0);
            i1 = __dp4a(hi[0], x2.x, i1);
            i1 = __dp4a(hi[1], x2.y, i1);
            i1 = __dp4a(hi[2], x2.z, i1);
            i1 = __dp4a(hi[3], x2.w, i1);
            i1 = __dp4a(hi[4], x3.x, i1);
            i1 = __dp4a(hi[5], x3.y, i1);
            i1 = __dp4a(hi[6], x3.z, i1);
            i1 = __dp4a(hi[7], x3.w, i1);
            const float dot = dsc0 * (d8.x * (float)i0) + dsc1 * (d8.y * (float)i1);
            const float mins = dm0 * s8.x + dm1 * s8.y;
            acc[t] += dot - mins;
        }
    }
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g / (1.0f + expf(-g)) * u;
}

template <int MT, int EPI>
__device__ __forceinline__ void write_unit(const Args &a, int64_t unit, const float (&v)[MT],
                                           const float (&gate)[MT], int lane)
{
    int k = (EPI == EPI_SWIGLU) ? 0 : seg_of(a, unit);
    const int64_t rows = a.seg_begin[k + 1] - a.seg_begin[k];
    const int64_t lr = unit - a.seg_begin[k];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < a.m && lane == (t & 31)) {
            float out = v[t];
            if (EPI == EPI_RESID) out = a.res[k][t * rows + lr] + out;
            if (EPI == EPI_SWIGLU) out = silu_mul(gate[t], v[t]);
            a.y[k][t * rows + lr] = out;
        }
    }
}

template <int MT, int EPI>
__global__ void __launch_bounds__(kThreads, 2) q4k_gemv_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t *ring = smem + warp * kWarpSmem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kWarps * kWarpSmem) + warp * kSlots;

    // units of this CTA, then of this warp (balanced contiguous ranges)
    const int64_t G = gridDim.x;
    const int64_t c0 = a.units * blockIdx.x / G, c1 = a.units * (blockIdx.x + 1) / G;
    const int64_t u0 = c0 + (c1 - c0) * warp / kWarps;
    const int64_t u1 = c0 + (c1 - c0) * (warp + 1) / kWarps;

    const int R = (EPI == EPI_SWIGLU) ? 2 : 1;
    const int rpp = (EPI != EPI_SWIGLU && a.nsb < kPieceSB && kPieceSB % a.nsb == 0)
                        ? kPieceSB / a.nsb : 1;
    const int ppr = (a.nsb + kPieceSB - 1) / kPieceSB;
    const int64_t nu = u1 - u0;
    const int64_t npieces = (rpp > 1) ? (nu + rpp - 1) / rpp : nu * R * ppr;

    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // prologue: weights do not depend on the previous kernel
    if (lane == 0) {
        for (int64_t p = 0; p < npieces && p < kSlots; ++p)
            issue_piece<EPI>(a, piece_of(p, u0, u1, rpp, ppr, R, a.nsb), ring + p * kPieceBytes,
                             &bars[p]);
    }
    pdl_launch_dependents();
    pdl_wait();  // activations come from the previous kernel

    const int g = lane >> 2, c = lane & 3;
    float acc[MT], gate[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = gate[t] = 0.0f;

    for (int64_t p = 0; p < npieces; ++p) {
        const int s = (int)(p % kSlots);
        const unsigned parity = (unsigned)((p / kSlots) & 1);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[s], parity));
        if (!ok) {
            if (lane == 0) {
                set_error(a.err, DEV_TIMEOUT_GEMV);
                for (int64_t q = p; q < npieces && q < p + kSlots; ++q)
                    if (!mbar_wait(&bars[q % kSlots], (unsigned)((q / kSlots) & 1)))
                        set_error(a.err, DEV_TIMEOUT_DRAIN);
            }
            return;
        }
        const Piece pc = piece_of(p, u0, u1, rpp, ppr, R, a.nsb);
        const uint8_t *slot = ring + s * kPieceBytes;

        if (rpp > 1) {
            // several whole rows: group g -> row g / nsb, super-block g % nsb
            const int rip = g / a.nsb;
            float pacc[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) pacc[t] = 0.0f;
            if (rip < pc.rows) sb_accumulate<MT>(a, slot + g * kSB, g % a.nsb, c, pacc);
            const int seg = 4 * a.nsb;  // lanes per row: 4, 8 or 16
#pragma unroll
            for (int t = 0; t < MT; ++t)
                for (int o = 1; o < seg; o <<= 1) pacc[t] += __shfl_xor_sync(0xffffffffu, pacc[t], o);
            if ((lane % seg) == 0 && rip < pc.rows) {
                const int64_t unit = pc.unit + rip;
                const int k = seg_of(a, unit);
                const int64_t rows = a.seg_begin[k + 1] - a.seg_begin[k];
                const int64_t lr = unit - a.seg_begin[k];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t < a.m) {
                        float out = pacc[t];
                        if (EPI == EPI_RESID) out = a.res[k][t * rows + lr] + out;
                        a.y[k][t * rows + lr] = out;
                    }
                }
            }
        } else {
            if (g < pc.cnt) sb_accumulate<MT>(a, slot + g * kSB, pc.sb0 + g, c, acc);
            if (pc.row_end) {
#pragma unroll
                for (int t = 0; t < MT; ++t) acc[t] = warp_sum(acc[t]);
                if (EPI == EPI_SWIGLU && pc.half == 0) {
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        gate[t] = acc[t];
                        acc[t] = 0.0f;
                    }
                } else {
                    write_unit<MT, EPI>(a, pc.unit, acc, gate, lane);
#pragma unroll
                    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
                }
            }
        }

        // refill this slot with piece p + kSlots
        __syncwarp();
        if (lane == 0 && p + kSlots < npieces) {
            fence_proxy_async_smem();
            issue_piece<EPI>(a, piece_of(p + kSlots, u0, u1, rpp, ppr, R, a.nsb),
                             ring + s * kPieceBytes, &bars[s]);
        }
    }
}

// --------------------------------------------------------------------------
// Exact integer sub-block dots (checking aid): one thread per (row, sub-block).
__global__ void q4k_subblock_dots_kernel(const uint8_t *w, const int8_t *xq, int32_t *I,
                                         int64_t out_dim, int64_t in_dim)
{
    const int64_t nsub = in_dim / 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= out_dim * nsub) return;
    const int64_t r = idx / nsub, k = idx % nsub;
    const int64_t b = k / 8;
    const int j = (int)(k % 8);
    const uint8_t *blk = w + (r * (in_dim / 256) + b) * kSB;
    const uint8_t *qs = blk + 16 + 32 * (j / 2);
    const int8_t *xb = xq + k * 32;
    int acc = 0;
    for (int i = 0; i < 32; ++i) {
        const int q = (j & 1) ? (qs[i] >> 4) : (qs[i] & 15);
        acc += q * (int)xb[i];
    }
    I[idx] = acc;
}

template <int MT, int EPI>
cudaError_t launch_t(const Args &a, int grid, cudaStream_t s)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_gemv_kernel<MT, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4k_gemv_kernel<MT, EPI>, a);
}

template <int EPI>
cudaError_t launch_epi(const Args &a, int grid, cudaStream_t s)
{
    if (a.m <= 1) return launch_t<1, EPI>(a, grid, s);
    if (a.m <= 2) return launch_t<2, EPI>(a, grid, s);
    if (a.m <= 4) return launch_t<4, EPI>(a, grid, s);
    if (a.m <= 8) return launch_t<8, EPI>(a, grid, s);
    return launch_t<16, EPI>(a, grid, s);
}

}  // namespace

cudaError_t launch_q4k_gemv(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                            int64_t m, int64_t in_dim, cudaStream_t s)
{
    Args a = {};
    a.nseg = nseg;
    int64_t units = 0;
    for (int k = 0; k < nseg; ++k) {
        a.w[k] = static_cast<const uint8_t *>(seg[k].w);
        a.y[k] = seg[k].y;
        a.res[k] = seg[k].res;
        a.seg_begin[k] = (epilogue == EPI_SWIGLU) ? 0 : units;
        if (epilogue != EPI_SWIGLU) units += seg[k].rows;
    }
    if (epilogue == EPI_SWIGLU) {
        units = seg[0].rows;
        a.nseg = 1;  // outputs indexed by unit through segment 0
        a.seg_begin[1] = units;
    } else {
        a.seg_begin[nseg] = units;
    }
    a.units = units;
    a.nsb = (int)(in_dim / 256);
    a.row_bytes = (int64_t)a.nsb * kSB;
    a.m = (int)m;
    a.in_dim = in_dim;
    a.xq = static_cast<const int8_t *>(q8);
    a.xd = reinterpret_cast<const float *>(static_cast<const uint8_t *>(q8) + m * in_dim);
    a.xs = a.xd + m * (in_dim / 32);
    a.err = dev_error_word();

    const int sms = dev_info().sm_count;
    int64_t grid = (units + kWarps - 1) / kWarps;
    if (grid > 2 * sms) grid = 2 * sms;
    if (grid < 1) grid = 1;
    switch (epilogue) {
    case EPI_STORE: return launch_epi<EPI_STORE>(a, (int)grid, s);
    case EPI_RESID: return launch_epi<EPI_RESID>(a, (int)grid, s);
    default: return launch_epi<EPI_SWIGLU>(a, (int)grid, s);
    }
}

cudaError_t launch_q4k_subblock_dots(const void *w, const void *q8, int32_t *I, int64_t out_dim,
                                     int64_t in_dim, cudaStream_t s)
{
    const int64_t n = out_dim * (in_dim / 32);
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    q4k_subblock_dots_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<const uint8_t *>(w), static_cast<const int8_t *>(q8), I, out_dim, in_dim);
    return cudaGetLastError();
}

}  // namespace rz
