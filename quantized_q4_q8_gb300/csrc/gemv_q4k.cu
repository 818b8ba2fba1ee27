// gemv_q4k.cu -- Q4_K weight x Q8_1 activation GEMV for decode (m <= 16 tokens).
//
// Operation (q4k_q8_gemv_async of realizar 0.8.5 src/cuda/executor/cached.rs,
// transformer_layer_gpu_true_dp4a): for every output row r and token t
//   y[t][r] = sum_b d_b * sum_j sc_bj * d8_tbj * I_tbj - dmin_b * sum_j m_bj * s_tbj,
// I_tbj the exact int32 dot of the 32 4-bit codes of sub-block j with the 32
// int8 codes of the matching Q8_1 block.
//
// GB300 design.  The kernel streams 144-byte super-blocks from HBM; compute is
// a few dp4a per byte.  One CTA per SM owns a contiguous range of rows.  A
// producer warp keeps a ring of ~16 KB shared-memory stages full with the 1-D
// bulk copy engine (cp.async.bulk, completion counted on an mbarrier), so the
// bytes in flight live in shared memory, not registers, and it prefetches the
// rest of the CTA's rows into L2 (cp.async.bulk.prefetch.L2) at once.  A stage
// holds whole "packs" (one row, or 8/nsb rows when a row has fewer than 8
// super-blocks); sixteen consumer warps take packs round-robin, each waiting only on the stage
// of its own pack and releasing it with one mbarrier arrival, so warps run ahead
// of each other across stages and the ring stays full.  Within a pack each
// group of 4 lanes takes a super-block (two at a time for independent work) and
// each lane one 32-byte chunk of its quants (two sub-blocks: low and high
// nibbles), so every 32-element integer dot completes inside one lane (dp4a of
// unsigned nibbles with signed int8); only the f32 combination crosses lanes,
// once per row, in a fixed order (deterministic results).  The Q8_1 codes are
// staged in shared memory once per CTA when they fit, in padded 288-byte slots
// per super-block so that the activation reads are free of bank conflicts.
// The weight prologue is issued before waiting on the previous kernel
// (programmatic dependent launch), so it overlaps that kernel's tail.  Every
// wait is bounded; on expiry the kernel records an error code and drains its
// outstanding copies instead of trapping.
#include <algorithm>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kSB = 144;
constexpr int kCtaSmem = 200 * 1024;
constexpr int kStageTarget = 16 * 1024;
constexpr int kXSmemMax = 48 * 1024;
constexpr int kMaxStages = 16;

__host__ __device__ inline int64_t x_smem_bytes(int64_t m, int64_t in_dim)
{
    return m * (in_dim / 256) * 288 + 8 * m * (in_dim / 32);
}

struct Args {
    const uint8_t *w[3];
    float *y[3];
    const float *res[3];
    int64_t ldy[3], ldr[3];
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
    int rpp;               // rows per pack (8/nsb when nsb divides 8 and is < 8, else 1)
    int PS;                // packs per stage
    int NS;                // stages in the ring
    int stage_bytes;       // PS * rpp * R * row_bytes
    int x_smem;            // activations staged (swizzled) in shared memory
    // f32 input quantised in the kernel (XIN_NORM / XIN_F32)
    const float *xf;
    int64_t ldxf;
    const float *gamma;
    int64_t norm_n;
    float eps;
    unsigned *err;
};

enum XIn { XIN_Q8 = 0, XIN_NORM = 1, XIN_F32 = 2 };

__device__ __forceinline__ int seg_of(const Args &a, int64_t unit)
{
    int k = 0;
    while (k + 1 < a.nseg && unit >= a.seg_begin[k + 1]) ++k;
    return k;
}

// Shared-memory copy of the Q8_1 codes.  Super-block sb of token t occupies a
// 288-byte slot; the 64 bytes that lane chunk c reads (sub-blocks 2c, 2c+1) sit at
// 64c + 16(c >> 1) inside it.  With this padding the 8 lanes of a shared-memory
// phase (2 consecutive super-blocks x 4 chunks) hit 8 different bank groups, and
// every address is a lane constant plus a multiple of the super-block index.
constexpr int kXSlot = 288;

__device__ __forceinline__ int x_chunk_off(int c) { return 64 * c + 16 * (c >> 1); }

// Per-lane constants of the scale/min decode.  Lane chunk c owns sub-blocks
// j0 = 2c and j1 = 2c + 1; the two 6-bit scales (and mins) are built for both
// sub-blocks at once, one per byte, from the 16-bit windows A = s[k], s[k+1],
// B = s[4+k], s[5+k], C = s[8+k], s[9+k] with k = j0 & 3:
//   j < 4 : sc = A & 63,                    m = B & 63
//   j >= 4: sc = (C & 15) | (A >> 6) << 4,  m = (C >> 4) | (B >> 6) << 4
struct LaneConst {
    uint32_t sh;       // 8 * k
    uint32_t mask_lo;  // 0x3f3f for j < 4, else 0
    uint32_t mask_c;   // 0x0f0f for j >= 4, else 0
    uint32_t mask_hi;  // 0x3030 for j >= 4, else 0
};

__device__ __forceinline__ LaneConst lane_const(int c)
{
    LaneConst L;
    L.sh = 8u * (uint32_t)((2 * c) & 3);
    const bool hi = c >= 2;
    L.mask_lo = hi ? 0u : 0x3f3fu;
    L.mask_c = hi ? 0x0f0fu : 0u;
    L.mask_hi = hi ? 0x3030u : 0u;
    return L;
}

struct XSrc {
    uint32_t q;        // shared-memory byte address of the codes (token 0) (smem copy)
    uint32_t ds;       // shared-memory byte address of d (token 0); s follows at + m*nb*4
    const int8_t *gq;  // global copies (when the activations stay in global memory)
    const float *gd;
    const float *gs;
    int64_t in_dim, nb;
    int m;
};

__device__ __forceinline__ int4 lds128(uint32_t addr)
{
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// Accumulate one super-block at shared address `blk`, super-block index sb of
// its row, into acc[t]; the lane owns quant chunk c (sub-blocks 2c, 2c+1).
template <int MT, bool XS>
__device__ __forceinline__ void sb_accumulate(const XSrc &x, uint32_t blk, int sb, int c,
                                              const LaneConst &L, float (&acc)[MT])
{
    const int4 hdr = lds128(blk);
    const int4 qa = lds128(blk + 16 + 32 * c);
    const int4 qb = lds128(blk + 32 + 32 * c);
    const float d = h2f((uint16_t)((uint32_t)hdr.x & 0xffffu));
    const float dmin = h2f((uint16_t)((uint32_t)hdr.x >> 16));

    const uint32_t A = (uint32_t)hdr.y >> L.sh, B = (uint32_t)hdr.z >> L.sh, C = (uint32_t)hdr.w >> L.sh;
    const uint32_t scp = (A & L.mask_lo) | (C & L.mask_c) | ((A >> 2) & L.mask_hi);
    const uint32_t mnp = (B & L.mask_lo) | ((C >> 4) & L.mask_c) | ((B >> 2) & L.mask_hi);
    const int sc0 = (int)(scp & 0xffu), sc1 = (int)((scp >> 8) & 0xffu);
    const float dm0 = dmin * (float)(mnp & 0xffu), dm1 = dmin * (float)((mnp >> 8) & 0xffu);

    const uint32_t q[8] = {(uint32_t)qa.x, (uint32_t)qa.y, (uint32_t)qa.z, (uint32_t)qa.w,
                           (uint32_t)qb.x, (uint32_t)qb.y, (uint32_t)qb.z, (uint32_t)qb.w};
    int lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo[i] = (int)(q[i] & 0x0f0f0f0fu);
        hi[i] = (int)((q[i] >> 4) & 0x0f0f0f0fu);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < x.m) {
            int4 x0, x1, x2, x3;
            float2 d8, s8;
            if (XS) {
                const uint32_t xa = x.q + (uint32_t)(t * (x.in_dim / 256) + sb) * kXSlot + x_chunk_off(c);
                x0 = lds128(xa);
                x1 = lds128(xa + 16);
                x2 = lds128(xa + 32);
                x3 = lds128(xa + 48);
                const uint32_t da = x.ds + (uint32_t)(t * x.nb + sb * 8 + 2 * c) * 4u;
                d8 = lds64f(da);
                s8 = lds64f(da + (uint32_t)(x.m * x.nb) * 4u);
            } else {
                const int64_t jb = (int64_t)sb * 8 + 2 * c;
                const int4 *xp = reinterpret_cast<const int4 *>(x.gq + t * x.in_dim + jb * 32);
                x0 = __ldg(xp);
                x1 = __ldg(xp + 1);
                x2 = __ldg(xp + 2);
                x3 = __ldg(xp + 3);
                d8 = __ldg(reinterpret_cast<const float2 *>(x.gd + t * x.nb + jb));
                s8 = __ldg(reinterpret_cast<const float2 *>(x.gs + t * x.nb + jb));
            }
            // four independent dp4a chains (two per sub-block)
            int a0 = __dp4a(lo[0], x0.x, 0), a1 = __dp4a(lo[4], x1.x, 0);
            int b0 = __dp4a(hi[0], x2.x, 0), b1 = __dp4a(hi[4], x3.x, 0);
            a0 = __dp4a(lo[1], x0.y, a0);
            a1 = __dp4a(lo[5], x1.y, a1);
            b0 = __dp4a(hi[1], x2.y, b0);
            b1 = __dp4a(hi[5], x3.y, b1);
            a0 = __dp4a(lo[2], x0.z, a0);
            a1 = __dp4a(lo[6], x1.z, a1);
            b0 = __dp4a(hi[2], x2.z, b0);
            b1 = __dp4a(hi[6], x3.z, b1);
            a0 = __dp4a(lo[3], x0.w, a0);
            a1 = __dp4a(lo[7], x1.w, a1);
            b0 = __dp4a(hi[3], x2.w, b0);
            b1 = __dp4a(hi[7], x3.w, b1);
            // sc * I is exact in int32; one conversion per sub-block
            const float t0 = (float)(sc0 * (a0 + a1)) * d8.x;
            const float t1 = (float)(sc1 * (b0 + b1)) * d8.y;
            acc[t] = fmaf(d, t0 + t1, acc[t]) - (dm0 * s8.x + dm1 * s8.y);
        }
    }
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g / (1.0f + expf(-g)) * u;
}

__device__ __forceinline__ void prefetch_l2(const void *src, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <int MT, int EPI, bool XS, int XIN>
__global__ void __launch_bounds__(kThreads, 1) q4k_gemv_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *xsm = smem + (int64_t)a.NS * a.stage_bytes;
    const int64_t xbytes = XS ? x_smem_bytes(a.m, a.in_dim) : 0;
    uint64_t *full = reinterpret_cast<uint64_t *>(xsm + xbytes + 96);  // 96 B: norm reduction
    uint64_t *empty = full + a.NS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = (EPI == EPI_SWIGLU) ? 2 : 1;
    const int64_t G = gridDim.x;
    const int64_t r0 = a.units * blockIdx.x / G, r1 = a.units * (blockIdx.x + 1) / G;
    const int64_t npacks = (r1 - r0 + a.rpp - 1) / a.rpp;
    const int64_t nstages = (npacks + a.PS - 1) / a.PS;
    const int64_t pack_bytes = (int64_t)a.rpp * a.row_bytes;  // one half (gate or up)

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.PS);  // one arrival per pack
        }
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel may become resident now: its weights stream while we drain
    pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // everything beyond the first NS stages goes to L2 right away, so HBM
            // stays busy even while the ring is full
            for (int64_t k = a.NS; k < nstages; ++k) {
                const int64_t u0 = r0 + k * a.PS * a.rpp;
                const int n = (int)min((int64_t)a.PS * a.rpp, r1 - u0);
                if (EPI == EPI_SWIGLU) {
                    prefetch_l2(a.w[0] + u0 * a.row_bytes, (unsigned)(n * a.row_bytes));
                    prefetch_l2(a.w[1] + u0 * a.row_bytes, (unsigned)(n * a.row_bytes));
                } else {
                    int r = 0;
                    while (r < n) {
                        const int64_t u = u0 + r;
                        const int kseg = seg_of(a, u);
                        const int run = (int)min((int64_t)(n - r), a.seg_begin[kseg + 1] - u);
                        prefetch_l2(a.w[kseg] + (u - a.seg_begin[kseg]) * a.row_bytes,
                                    (unsigned)(run * a.row_bytes));
                        r += run;
                    }
                }
            }
            int64_t k = 0;
            bool ok = true;
            for (; k < nstages; ++k) {
                const int s = (int)(k % a.NS);
                if (k >= a.NS && !mbar_wait(&empty[s], (unsigned)(((k / a.NS) - 1) & 1))) {
                    set_error(a.err, DEV_TIMEOUT_GEMV);
                    ok = false;
                    break;
                }
                const int64_t u0 = r0 + k * a.PS * a.rpp;
                const int n = (int)min((int64_t)a.PS * a.rpp, r1 - u0);  // rows in this stage
                uint8_t *dst = ring + (int64_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], (unsigned)(R * n * a.row_bytes));
                if (EPI == EPI_SWIGLU) {
                    // stage layout: pack p -> [gate rows | up rows]
                    for (int p = 0; p * a.rpp < n; ++p) {
                        const int nr = min(a.rpp, n - p * a.rpp);
                        const int64_t u = u0 + (int64_t)p * a.rpp;
                        uint8_t *pd = dst + (int64_t)p * 2 * pack_bytes;
                        bulk_g2s(pd, a.w[0] + u * a.row_bytes, (unsigned)(nr * a.row_bytes), &full[s]);
                        bulk_g2s(pd + pack_bytes, a.w[1] + u * a.row_bytes, (unsigned)(nr * a.row_bytes),
                                 &full[s]);
                    }
                } else {
                    int r = 0;
                    while (r < n) {
                        const int64_t u = u0 + r;
                        const int kseg = seg_of(a, u);
                        const int run = (int)min((int64_t)(n - r), a.seg_begin[kseg + 1] - u);
                        bulk_g2s(dst + (int64_t)r * a.row_bytes,
                                 a.w[kseg] + (u - a.seg_begin[kseg]) * a.row_bytes,
                                 (unsigned)(run * a.row_bytes), &full[s]);
                        r += run;
                    }
                }
            }
            // drain: stages issued but possibly not complete must land before exit
            if (!ok) {
                for (int64_t q = (k > a.NS ? k - a.NS : 0); q < k; ++q)
                    if (!mbar_wait(&full[q % a.NS], (unsigned)((q / a.NS) & 1)))
                        set_error(a.err, DEV_TIMEOUT_DRAIN);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();  // activations and the output buffers belong to the previous kernel
    XSrc x;
    x.in_dim = a.in_dim;
    x.nb = a.in_dim / 32;
    x.m = a.m;
    x.gq = a.xq;
    x.gd = a.xd;
    x.gs = a.xs;
    if (XS && XIN == XIN_Q8) {
        // codes: 16-byte chunk i of super-block sbg (all tokens) -> padded slot layout
        const int64_t nsbx = (int64_t)a.m * (a.in_dim / 256);
        const int4 *src = reinterpret_cast<const int4 *>(a.xq);
        for (int64_t i = threadIdx.x; i < nsbx * 16; i += kConsumerWarps * 32) {
            const int64_t sbg = i >> 4;
            const int ch = (int)(i & 15), cc = ch >> 2;
            *reinterpret_cast<int4 *>(xsm + sbg * kXSlot + x_chunk_off(cc) + 16 * (ch & 3)) = src[i];
        }
        // d and s, unchanged
        const int64_t nds = 2LL * a.m * x.nb / 4;
        const int4 *dsrc = reinterpret_cast<const int4 *>(a.xd);
        int4 *ddst = reinterpret_cast<int4 *>(xsm + nsbx * kXSlot);
        for (int64_t i = threadIdx.x; i < nds; i += kConsumerWarps * 32) ddst[i] = dsrc[i];
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    }
    if (XS && XIN != XIN_Q8) {
        // quantise the f32 input (RMS-normalised first for XIN_NORM) straight into
        // the padded slot layout: warp per Q8_1 block, as the standalone kernels do
        const int64_t nsbx = (int64_t)a.m * (a.in_dim / 256);
        float *dsm = reinterpret_cast<float *>(xsm + nsbx * kXSlot);
        float *ssm = dsm + (int64_t)a.m * x.nb;
        float *red = reinterpret_cast<float *>(full) - 24;  // 17 floats below the barriers
        auto sync = [] { asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory"); };
        for (int t = 0; t < a.m; ++t) {
            // loads unrolled eight blocks at a time, so they are in flight together
            const float *xrow = a.xf + t * a.ldxf;
            const int64_t nval = XIN == XIN_NORM ? a.norm_n : a.in_dim;
            float scale = 1.0f;
            if (XIN == XIN_NORM) scale = rms_scale(row_sumsq(xrow, x.nb, nval, warp, lane, red, sync), a.norm_n, a.eps);
            for (int k0 = 0; k0 < kRowBlocksPerWarp; k0 += 8) {
                if (warp + (int64_t)kRowWarps * k0 >= x.nb) break;
                RowBatch rb;
                row_batch(xrow, XIN == XIN_NORM ? a.gamma : nullptr, x.nb, nval, warp, lane, k0, rb);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t b = warp + (int64_t)kRowWarps * (k0 + u);
                    if (b >= x.nb) break;
                    const int64_t i = b * 32 + lane;
                    float v = rb.v[u];
                    if (XIN == XIN_NORM) v = (i < a.norm_n) ? __fmul_rn(__fmul_rn(v, scale), rb.g[u]) : 0.0f;
                    const float amax = warp_max(fabsf(v));
                    const float dq = __fdiv_rn(amax, 127.0f);
                    const int qi = q8_code(v, dq);
                    const int sum = warp_sum_int(qi);
                    const int64_t sb = b >> 3;
                    const int j = (int)(b & 7);
                    xsm[(t * (a.in_dim / 256) + sb) * kXSlot + x_chunk_off(j >> 1) + 32 * (j & 1) + lane] =
                        (uint8_t)(int8_t)qi;
                    if (lane == 0) {
                        dsm[t * x.nb + b] = dq;
                        ssm[t * x.nb + b] = __fmul_rn(dq, (float)sum);
                    }
                }
            }
        }
        sync();
    }
    if (XS) {
        const int64_t nsbx = (int64_t)a.m * (a.in_dim / 256);
        x.q = smem_u32(xsm);
        x.ds = smem_u32(xsm + nsbx * kXSlot);
    }

    const int g = lane >> 2, c = lane & 3;
    const LaneConst Lc = lane_const(c);
    const int seg_lanes = (a.rpp > 1) ? 4 * a.nsb : 32;
    const int rip = (a.rpp > 1) ? g / a.nsb : 0;  // row of the pack this group works on
    const int leader = lane % seg_lanes == 0;
    const uint32_t ring_s = smem_u32(ring);

    for (int64_t i = warp; i < npacks; i += kConsumerWarps) {
        const int64_t k = i / a.PS;
        const int s = (int)(k % a.NS);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (unsigned)((k / a.NS) & 1)));
        if (!ok) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_GEMV);
            return;
        }
        const int64_t pack0 = r0 + i * a.rpp;
        const int pack_rows = (int)min((int64_t)a.rpp, r1 - pack0);
        const uint32_t pk = ring_s + (uint32_t)(s * a.stage_bytes + (i % a.PS) * R * pack_bytes);
        float acc[2][MT], acc2[2][MT];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[h][t] = acc2[h][t] = 0.0f;
#pragma unroll
        for (int h = 0; h < R; ++h) {
            const uint32_t half = pk + (uint32_t)(h * pack_bytes);
            if (a.rpp > 1) {
                if (rip < pack_rows)
                    sb_accumulate<MT, XS>(x, half + g * kSB, g % a.nsb, c, Lc, acc[h]);
            } else {
                int sb = g;
                if (MT <= 2) {
                    for (; sb + 8 < a.nsb; sb += 16) {  // two independent super-blocks per step
                        sb_accumulate<MT, XS>(x, half + sb * kSB, sb, c, Lc, acc[h]);
                        sb_accumulate<MT, XS>(x, half + (sb + 8) * kSB, sb + 8, c, Lc, acc2[h]);
                    }
                }
                for (; sb < a.nsb; sb += 8) sb_accumulate<MT, XS>(x, half + sb * kSB, sb, c, Lc, acc[h]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the slot's bytes are no longer read
        // reduce over the lanes of each row (fixed order)
#pragma unroll
        for (int h = 0; h < R; ++h)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                acc[h][t] += acc2[h][t];
                for (int o = 1; o < seg_lanes; o <<= 1) acc[h][t] += __shfl_xor_sync(0xffffffffu, acc[h][t], o);
            }
        if (rip < pack_rows) {
            const int64_t unit = pack0 + rip;
            const int kseg = (EPI == EPI_SWIGLU) ? 0 : seg_of(a, unit);
            const int64_t lr = unit - a.seg_begin[kseg];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                // spread the token stores over the lanes of the row
                if (t < a.m && ((seg_lanes == 32) ? lane == (t & 31) : leader)) {
                    float out = acc[0][t];
                    if (EPI == EPI_RESID) out = a.res[kseg][t * a.ldr[kseg] + lr] + out;
                    if (EPI == EPI_SWIGLU) out = silu_mul(acc[0][t], acc[1][t]);
                    a.y[kseg][t * a.ldy[kseg] + lr] = out;
                }
            }
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

size_t smem_bytes(const Args &a)
{
    const int64_t xbytes = a.x_smem ? x_smem_bytes(a.m, a.in_dim) : 0;
    return (size_t)a.NS * a.stage_bytes + (size_t)xbytes + 96 + 2 * 8 * (size_t)a.NS;
}

template <int MT, int EPI, bool XS, int XIN>
cudaError_t launch_t(const Args &a, int grid, cudaStream_t s)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    const size_t smem = smem_bytes(a);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_gemv_kernel<MT, EPI, XS, XIN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
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
    return cudaLaunchKernelEx(&cfg, q4k_gemv_kernel<MT, EPI, XS, XIN>, a);
}

template <int MT, int EPI>
cudaError_t launch_x(const Args &a, int grid, cudaStream_t s, int xin)
{
    if (xin == XIN_NORM) {
        if constexpr (EPI != EPI_RESID) return launch_t<MT, EPI, true, XIN_NORM>(a, grid, s);
        return cudaErrorInvalidValue;
    }
    if (xin == XIN_F32) {
        if constexpr (EPI == EPI_RESID) return launch_t<MT, EPI, true, XIN_F32>(a, grid, s);
        return cudaErrorInvalidValue;
    }
    return a.x_smem ? launch_t<MT, EPI, true, XIN_Q8>(a, grid, s) : launch_t<MT, EPI, false, XIN_Q8>(a, grid, s);
}

template <int EPI>
cudaError_t launch_epi(const Args &a, int grid, cudaStream_t s, int xin)
{
    if (a.m <= 1) return launch_x<1, EPI>(a, grid, s, xin);
    if (a.m <= 2) return launch_x<2, EPI>(a, grid, s, xin);
    if (a.m <= 4) return launch_x<4, EPI>(a, grid, s, xin);
    if (a.m <= 8) return launch_x<8, EPI>(a, grid, s, xin);
    return launch_x<16, EPI>(a, grid, s, xin);
}

static cudaError_t launch_common(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                                 const F32Input *f32in, int64_t m, int64_t in_dim, cudaStream_t s)
{
    Args a = {};
    int64_t units = 0;
    for (int k = 0; k < nseg; ++k) {
        a.w[k] = static_cast<const uint8_t *>(seg[k].w);
        a.y[k] = seg[k].y;
        a.res[k] = seg[k].res;
        a.ldy[k] = seg[k].ldy ? seg[k].ldy : seg[k].rows;
        a.ldr[k] = seg[k].ldr ? seg[k].ldr : seg[k].rows;
        if (epilogue != EPI_SWIGLU) {
            a.seg_begin[k] = units;
            units += seg[k].rows;
        }
    }
    if (epilogue == EPI_SWIGLU) {
        units = seg[0].rows;
        a.nseg = 1;  // outputs indexed by unit through segment 0
        a.seg_begin[0] = 0;
        a.seg_begin[1] = units;
    } else {
        a.nseg = nseg;
        a.seg_begin[nseg] = units;
    }
    const int R = (epilogue == EPI_SWIGLU) ? 2 : 1;
    a.units = units;
    a.nsb = (int)(in_dim / 256);
    a.row_bytes = (int64_t)a.nsb * kSB;
    a.m = (int)m;
    a.in_dim = in_dim;
    if (q8) {
        a.xq = static_cast<const int8_t *>(q8);
        a.xd = reinterpret_cast<const float *>(static_cast<const uint8_t *>(q8) + m * in_dim);
        a.xs = a.xd + m * (in_dim / 32);
    }
    int xin = XIN_Q8;
    if (f32in) {
        a.xf = f32in->x;
        a.ldxf = f32in->ldx;
        a.gamma = f32in->gamma;
        a.norm_n = f32in->norm_n;
        a.eps = f32in->eps;
        xin = f32in->gamma ? XIN_NORM : XIN_F32;
    }
    a.err = dev_error_word();
    a.rpp = (a.nsb < 8 && 8 % a.nsb == 0) ? 8 / a.nsb : 1;
    const int64_t pack = (int64_t)R * a.rpp * a.row_bytes;
    a.PS = (int)std::max<int64_t>(1, kStageTarget / pack);
    a.stage_bytes = (int)(a.PS * pack);
    const int64_t xbytes = x_smem_bytes(m, in_dim);
    a.x_smem = (xbytes <= kXSmemMax || f32in) ? 1 : 0;
    const int64_t budget = (int64_t)kCtaSmem - (a.x_smem ? xbytes : 0) - 1024;
    int64_t ns = budget / a.stage_bytes;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 2) {
        // wide rows: fall back to stages of one pack
        a.PS = 1;
        a.stage_bytes = (int)pack;
        ns = std::min<int64_t>(kMaxStages, budget / a.stage_bytes);
    }
    if (ns < 2) return cudaErrorInvalidConfiguration;  // excluded by q4k_gemv_supported
    a.NS = (int)ns;
    if ((int64_t)smem_bytes(a) > (int64_t)dev_info().smem_optin) return cudaErrorInvalidConfiguration;

    const int sms = dev_info().sm_count;
    int64_t grid = units < sms ? units : sms;
    if (grid < 1) grid = 1;
    switch (epilogue) {
    case EPI_STORE: return launch_epi<EPI_STORE>(a, (int)grid, s, xin);
    case EPI_RESID: return launch_epi<EPI_RESID>(a, (int)grid, s, xin);
    default: return launch_epi<EPI_SWIGLU>(a, (int)grid, s, xin);
    }
}

}  // namespace

cudaError_t launch_q4k_gemv(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                            int64_t m, int64_t in_dim, cudaStream_t s)
{
    return launch_common(seg, nseg, epilogue, q8, nullptr, m, in_dim, s);
}

bool q4k_gemv_f32_input_ok(int64_t m, int64_t in_dim)
{
    return x_smem_bytes(m, in_dim) <= kXSmemMax && in_dim <= 32LL * kRowWarps * kRowBlocksPerWarp;
}

cudaError_t launch_q4k_gemv_f32(const Q4kSegment *seg, int nseg, int epilogue, const F32Input &in,
                                int64_t m, int64_t in_dim, cudaStream_t s)
{
    if (!q4k_gemv_f32_input_ok(m, in_dim)) return cudaErrorInvalidValue;
    return launch_common(seg, nseg, epilogue, nullptr, &in, m, in_dim, s);
}




bool q4k_gemv_supported(int64_t m, int64_t in_dim, int epilogue)
{
    const int R = (epilogue == EPI_SWIGLU) ? 2 : 1;
    const int64_t nsb = in_dim / 256;
    const int64_t rpp = (nsb < 8 && 8 % nsb == 0) ? 8 / nsb : 1;
    const int64_t pack = R * rpp * nsb * kSB;
    const int64_t xbytes = x_smem_bytes(m, in_dim);
    const int64_t budget = (int64_t)kCtaSmem - (xbytes <= kXSmemMax ? xbytes : 0) - 1024;
    return budget / pack >= 2;
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
