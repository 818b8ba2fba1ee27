// gemv_q4k_mma.cu -- Q4_K weight x Q8_1 activation GEMV for several tokens
// (batched decode, 4..16 tokens per launch) on the tensor cores.
//
// Operation: the one of gemv_q4k.cu (q4k_q8_gemv_async of realizar 0.8.5
// src/cuda/executor/cached.rs, transformer_layer_gpu_true_dp4a), for every row r
// and token t
//   y[t][r] = sum_b d_b * sum_j sc_bj * d8_tbj * I_tbrj - dmin_b * sum_j m_bj * s_tbj.
//
// With several tokens the dp4a form spends most of its issue slots re-reading the
// activations and combining sub-block dots; here the per-sub-block integer dots
// of 16 rows x 8 tokens come out of mma.sync.m16n8k16 with f16 operands and f32
// accumulation (two MMAs cover the 32 values of a sub-block):
//   A (16 rows x 16 k)  = sc_j * q, the 4-bit code times the row's 6-bit scale,
//                         an integer <= 945, exact in f16 (folded with one
//                         HFMA2 from the 1024 + q bit pattern);
//   B (16 k x 8 tokens) = the int8 Q8_1 code, exact in f16 (from its offset-
//                         binary byte, 1152 + q, minus 1152);
//   D                   = sc_j * I_j exactly: every product is below 2^17 and the
//                         32-term sum below 2^22.
// The f32 epilogue of each sub-block scales D by the token's d8, the min term
// sum_j m_j s_j is accumulated beside it, and each super-block ends with
// acc += d_b * (...) - dmin_b * (...).  The f16 MMA rate of this part is four
// times its int8 rate, which is why the integer dots run as f16.
//
// Structure.  The rows of each weight matrix are split over CTAs in equal
// ranges of rpc rows (a CTA never straddles two matrices), cut into tiles of 16
// rows.  A producer warp streams stages through a ring with the tensor-memory-
// access engine: a stage is one 2-D box of a TMA tensor map -- the CTA's rpc rows
// over a slice of S super-blocks (S = 6, 2 or 1 so that the tiles x S units of a
// stage fill at most the 15 consumer warps; for the SwiGLU pair one box of gate
// rows and one of up rows) -- landing densely with a row pitch of S x 144 bytes
// (864 and 288 are 96 and 32 mod 128: conflict-free fragment loads).  One tensor
// copy per stage keeps the copy engine streaming; copies of single rows cost
// far more to issue than they move.  Consumer warp w always takes unit w (half,
// tile, super-block of the slice), so each warp accumulates one tile over the
// whole row in registers with no synchronisation but the ring's.  At the end the
// warps add their partials through shared memory in a fixed order
// (deterministic) and run the epilogue (store, + bias, + residual, or
// silu(gate) * up).  Activations are staged once per CTA: the codes of every
// token -- as f16 already in B-fragment order when that still leaves two ring
// stages (Q8_1 input; the warps' partial sums then reuse the idle ring), else as
// int8 in offset binary that every warp converts per fragment -- and per
// sub-block and lane group the d8 and s of the four tokens that lane group's
// accumulator columns hold.  When even the int8 codes of a Q8_1 input do not fit
// beside two stages (16 tokens at in_dim 11008 or 14336), they are staged one
// phase of K at a time (a multiple of 6 super-blocks, so no slice straddles two
// phases; the tables of the whole row stay resident): at each boundary the
// consumer warps meet, restage, and go on while the producer keeps the ring
// full.  f32 input runs in token groups instead.  Every wait is bounded.
#include <cuda_bf16.h>

#include <algorithm>

#include "mma_f16.cuh"
#include "q4k_dot.cuh"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

// 15 consumer warps and the producer make 16 warps, four per SM sub-partition:
// a thread may hold 128 registers (with 16 consumers, five warps on one
// sub-partition cap it at 96).
constexpr int kMW = 15;                    // consumer warps
constexpr int kMThreads = (kMW + 1) * 32;  // + 1 producer warp
constexpr int kMSmem = 224 * 1024;         // shared-memory budget of a CTA
constexpr int kMTile = 16;                 // rows per MMA tile

struct MArgs {
    CUtensorMap map[3];   // weight matrices (segments, or gate and up)
    float *y[3];
    const float *res[3];  // residual (EPI_RESID), bias (EPI_STORE, ldr 0) or nullptr
    int64_t ldy[3], ldr[3];
    int64_t seg_rows[3];
    int cta_begin[4];     // first CTA of each segment; cta_begin[nseg] = grid
    int rpc[3];           // rows per CTA (the box height) of each segment
    int nseg;
    int nsb;              // super-blocks per row
    int m;                // tokens of this launch (<= 8 * NT)
    int64_t in_dim;
    const int8_t *xq;     // Q8_1 input: codes [m][in_dim], d, s [m][in_dim / 32]
    const float *xd, *xs;
    const float *xf;      // or f32 input [m][ldxf], RMS-normalised first when gamma
    int64_t ldxf;
    const float *gamma;
    int64_t norm_n;
    float eps;
    int NS;               // stages in the ring
    int stage_bytes;      // bytes of a ring slot (the largest stage of any CTA)
    int xph;              // super-blocks of codes staged at a time (a multiple of 6, or nsb)
    unsigned *err;
    int stall_stage;      // test aid (rz_debug_stall_next_gemv), -1 otherwise
    uint32_t wait_limit;
    float *zy;            // zero padding of segment 0's output (last CTA), or nullptr
    int64_t zy_ld, zy_from, zy_cnt;
};

enum MXIn { MX_Q8 = 0, MX_NORM = 1, MX_F32 = 2 };

// Shared-memory layout of the activations (T = 8 NT token slots):
//   codes  uint8 [m][in_dim + 32]: q + 128 (offset binary)
//   d8     float [in_dim / 32][4 lane groups][2 NT]: for lane group i the d8 of
//          tokens 2i, 2i + 1 (then 2i + 8, 2i + 9): the columns of its accumulators
//   spc    uint32 [in_dim / 256][T][4 lane groups][4]: s of sub-blocks 2i, 2i + 1
//          of a token in three bf16 pieces (hi, mid, lo pairs; then 0), the B
//          fragments of the min-term MMA
// Token pitch of the codes in bytes: int8 codes, or (xh) the codes as f16 in
// B-fragment order (each group of eight x0..x7 stored as x0 x2 x1 x3 x4 x6 x5 x7,
// so that a lane's two fragments of a sub-block are one 16-byte load); 32 and 64
// mod 128, so that the 8 lanes of a load phase (two tokens) hit distinct banks.
__host__ __device__ inline int64_t mma_code_pitch(int64_t in_dim, bool xh) { return xh ? 2 * in_dim + 64 : in_dim + 32; }
__host__ __device__ inline int64_t mma_codes_bytes(int m, int64_t in_dim, bool xh)
{
    return ((int64_t)m * mma_code_pitch(in_dim, xh) + 127) & ~int64_t(127);
}
__host__ __device__ inline int64_t mma_d8_bytes(int64_t in_dim, int nt) { return (in_dim / 32) * 4 * 2 * nt * 4; }
__host__ __device__ inline int64_t mma_spc_bytes(int64_t in_dim, int nt) { return (in_dim / 256) * 8 * nt * 4 * 16; }
// kdim: values of each token's codes staged at a time (in_dim, or a phase of it)
__host__ __device__ inline int64_t mma_x_bytes(int m, int64_t in_dim, int nt, bool xh, int64_t kdim)
{
    return mma_codes_bytes(m, kdim, xh) + mma_d8_bytes(in_dim, nt) + mma_spc_bytes(in_dim, nt);
}
__host__ __device__ inline int64_t mma_red_bytes(int nt) { return (int64_t)kMW * 32 * 4 * nt * 4; }
// Super-blocks per stage for a CTA of `tiles` tiles (R halves): 6 or 2 (row
// pitches conflict-free for the fragment loads), else 1, so that the units of a
// stage, R x tiles x S, fit the consumer warps.
__host__ __device__ inline int mma_slice_sb(int tiles, int R, int nsb)
{
    const int u = R * tiles;
    const int S = 6 * u <= kMW ? 6 : (2 * u <= kMW ? 2 : 1);
    return S < nsb ? S : nsb;
}
__host__ __device__ inline int mma_half_bytes(int tiles, int S) { return (tiles * 16 * S * 144 + 127) / 128 * 128; }


constexpr uint32_t kF16x2_1024 = 0x64006400u;  // (1024, 1024)
constexpr uint32_t kF16x2_1152 = 0x64806480u;  // (1152, 1152)

// The byte (j & 3) of a packed word of four 6-bit values v as the f16 pair
// (v, v) (1024 + v in both halves, minus 1024: exact).
__device__ __forceinline__ uint32_t scale_splat(uint32_t packed, int j)
{
    const uint32_t sel = (uint32_t)(j & 3) | 0x4040u | ((uint32_t)(j & 3) << 8);  // bytes: b, 0, b, 0
    uint32_t v;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(v) : "r"(packed), "r"(sel));
    return hsub2u(v | kF16x2_1024, kF16x2_1024);
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The fold of a nibble pair into the MMA operand: with the nibble at bits 0-3 of
// each half, (1024 + q) v - 1024 v = q v; at bits 4-7, (1024 + 16 q) (v / 16) -
// 64 v = q v (no shift needed).  One rounding of an exact result either way.
struct ScaleFold {
    uint32_t m, c;  // multiplier and addend pairs
};
__device__ __forceinline__ ScaleFold fold_lo(uint32_t v2) { return {v2, hmul2u(v2, 0xE400E400u /* -1024 */)}; }
__device__ __forceinline__ ScaleFold fold_hi(uint32_t v2)
{
    return {hmul2u(v2, 0x2C002C00u /* 1/16 */), hmul2u(v2, 0xD400D400u /* -64 */)};
}

// Mins 2i, 2i + 1 of a packed set of eight (words lo = m0..3, hi = m4..7) as an
// exact bf16 pair: 128 + m in bf16 from the bit pattern, minus 128.
__device__ __forceinline__ uint32_t min_pair_bf16(uint32_t lo, uint32_t hi, int i)
{
    const uint32_t w = i < 2 ? lo : hi;
    const uint32_t b = (uint32_t)(2 * i) & 3u;
    const uint32_t sel = b | 0x4040u | ((b + 1) << 8);  // bytes: m_2i, 0, m_2i+1, 0
    uint32_t v, d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(v) : "r"(w), "r"(sel));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v | 0x43004300u), "r"(0x43004300u));
    return d;
}

// Offset-binary codes (1152 + q in f16 after the OR) of bytes 0, 2 and 1, 3 of a
// word, minus 1152: the int8 codes as exact f16 pairs.
__device__ __forceinline__ uint32_t code_pair(uint32_t w)
{
    return hsub2u(lop_and_or(w, 0x00FF00FFu, kF16x2_1024), kF16x2_1152);
}

// The six-bit scales and mins of a super-block header (words A, B, C = bytes
// 4-7, 8-11, 12-15) as four packed words of four values each.
__device__ __forceinline__ void unpack_scales(uint32_t A, uint32_t B, uint32_t C, uint32_t &sc03, uint32_t &sc47,
                                              uint32_t &mn03, uint32_t &mn47)
{
    sc03 = A & 0x3F3F3F3Fu;
    mn03 = B & 0x3F3F3F3Fu;
    sc47 = (C & 0x0F0F0F0Fu) | ((A >> 2) & 0x30303030u);
    mn47 = ((C >> 4) & 0x0F0F0F0Fu) | ((B >> 2) & 0x30303030u);
}


// One super-block of rows g and g + 8 of a tile (shared addresses blkA, blkB)
// against every token, accumulated into acc[nt][e]: e = 0, 1 row g with tokens
// 2i, 2i + 1 (+ 8 nt); e = 2, 3 row g + 8.  xrow: this lane's B-fragment row of
// codes for n-tile 0 (and + xstep for n-tile 1) at this super-block; d8a, spa:
// this lane's entries of the d8 table and the s pieces at this super-block.
template <int NT, bool XH>
__device__ __forceinline__ void mma_superblock(uint32_t blkA, uint32_t blkB, uint32_t xrow, uint32_t xstep,
                                               uint32_t d8a, uint32_t spa, int i, float (&acc)[NT][4])
{
    const uint4 hA = lds_u4(blkA), hB = lds_u4(blkB);
    uint32_t scA[2], scB[2], mnA[2], mnB[2];
    unpack_scales(hA.y, hA.z, hA.w, scA[0], scA[1], mnA[0], mnA[1]);
    unpack_scales(hB.y, hB.z, hB.w, scB[0], scB[1], mnB[0], mnB[1]);

    float tb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) tb[nt][e] = 0.0f;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};

#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint2 wA = lds_u2(blkA + 16 + 32 * c + 8 * i);
        const uint2 wB = lds_u2(blkB + 16 + 32 * c + 8 * i);
        // bytes 1 and 3 of each word moved to 0 and 2 (shared by both nibble halves)
        const uint32_t wAx8 = wA.x >> 8, wAy8 = wA.y >> 8, wBx8 = wB.x >> 8, wBy8 = wB.y >> 8;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int j = 2 * c + half;  // sub-block: low nibbles 2c, high nibbles 2c + 1
            const uint32_t mask = half ? 0x00F000F0u : 0x000F000Fu;
            const uint32_t vA = scale_splat(scA[j >> 2], j), vB = scale_splat(scB[j >> 2], j);
            const ScaleFold fA = half ? fold_hi(vA) : fold_lo(vA), fB = half ? fold_hi(vB) : fold_lo(vB);
            uint32_t a0[4], a1[4];
            // k slots 2i, 2i+1 <- elements e0, e0 + 2; 2i+8, 2i+9 <- e0 + 1, e0 + 3 (e0 = 8i + 4h)
            a0[0] = hfma2u(lop_and_or(wA.x, mask, kF16x2_1024), fA.m, fA.c);
            a0[1] = hfma2u(lop_and_or(wB.x, mask, kF16x2_1024), fB.m, fB.c);
            a0[2] = hfma2u(lop_and_or(wAx8, mask, kF16x2_1024), fA.m, fA.c);
            a0[3] = hfma2u(lop_and_or(wBx8, mask, kF16x2_1024), fB.m, fB.c);
            a1[0] = hfma2u(lop_and_or(wA.y, mask, kF16x2_1024), fA.m, fA.c);
            a1[1] = hfma2u(lop_and_or(wB.y, mask, kF16x2_1024), fB.m, fB.c);
            a1[2] = hfma2u(lop_and_or(wAy8, mask, kF16x2_1024), fA.m, fA.c);
            a1[3] = hfma2u(lop_and_or(wBy8, mask, kF16x2_1024), fB.m, fB.c);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float d[4];
                if constexpr (XH) {
                    // both fragments of the sub-block, staged as f16 in fragment order
                    const uint4 X = lds_u4(xrow + nt * xstep + 64 * j);
                    mma16816(d, a0, X.x, X.y, zero);
                    mma16816(d, a1, X.z, X.w, d);
                } else {
                    const uint2 X = lds_u2(xrow + nt * xstep + 32 * j);
                    mma16816(d, a0, code_pair(X.x), code_pair(X.x >> 8), zero);
                    mma16816(d, a1, code_pair(X.y), code_pair(X.y >> 8), d);
                }
                // d8 of tokens 2i, 2i + 1 (+ 8 nt)
                const float2 v = lds_f2(d8a + (j * 4 * 2 * NT + 2 * nt) * 4);
                tb[nt][0] = fmaf(d[0], v.x, tb[nt][0]);
                tb[nt][1] = fmaf(d[1], v.y, tb[nt][1]);
                tb[nt][2] = fmaf(d[2], v.x, tb[nt][2]);
                tb[nt][3] = fmaf(d[3], v.y, tb[nt][3]);
            }
        }
    }
    // min term sum_j m_j s_j on the tensor cores: A = the eight mins of rows g,
    // g + 8 (bf16, exact), B = s in three bf16 pieces (hi, mid | lo, 0)
    const uint32_t pA = min_pair_bf16(mnA[0], mnA[1], i), pB = min_pair_bf16(mnB[0], mnB[1], i);
    const uint32_t am0[4] = {pA, pB, pA, pB}, am1[4] = {pA, pB, 0u, 0u};
    const float dA = h2f((uint16_t)(hA.x & 0xffffu)), dminA = h2f((uint16_t)(hA.x >> 16));
    const float dB = h2f((uint16_t)(hB.x & 0xffffu)), dminB = h2f((uint16_t)(hB.x >> 16));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint4 sp = lds_u4(spa + nt * 8 * 4 * 16);
        float mn[4];
        mma16816_bf16(mn, am0, sp.x, sp.y, zero);
        mma16816_bf16(mn, am1, sp.z, 0u, mn);
        acc[nt][0] = fmaf(dA, tb[nt][0], acc[nt][0]) - dminA * mn[0];
        acc[nt][1] = fmaf(dA, tb[nt][1], acc[nt][1]) - dminA * mn[1];
        acc[nt][2] = fmaf(dB, tb[nt][2], acc[nt][2]) - dminB * mn[2];
        acc[nt][3] = fmaf(dB, tb[nt][3], acc[nt][3]) - dminB * mn[3];
    }
}

// s in three bf16 pieces: hi = bf16(s), mid = bf16(s - hi), lo = bf16(the rest)
// (each difference exact in f32): hi + mid + lo equals s to within 2^-24 |s|.
__device__ __forceinline__ void bf16_pieces(float s, uint16_t &hi, uint16_t &mid, uint16_t &lo)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(s);
    const float r1 = s - __bfloat162float(h);
    const __nv_bfloat16 md = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(md);
    const __nv_bfloat16 l = __float2bfloat16_rn(r2);
    hi = __bfloat16_as_ushort(h);
    mid = __bfloat16_as_ushort(md);
    lo = __bfloat16_as_ushort(l);
}

// Store functor of the MMA activation layout for the f32 quantiser: codes in
// offset binary, d8 into the per-lane-group table, s into its bf16 pieces.
// Token t sits in lane group (t & 7) / 2, n-tile t / 8, column t & 1.
template <int NT>
struct MmaStore {
    uint8_t *xcodes;
    float *d8t;
    uint32_t *spc;
    int64_t cpitch;
    __device__ __forceinline__ void codes(int t, int64_t b, int e0, uint32_t word) const
    {
        *reinterpret_cast<uint32_t *>(xcodes + t * cpitch + b * 32 + e0) = word ^ 0x80808080u;
    }
    __device__ __forceinline__ void meta(int t, int64_t b, float d, float s) const
    {
        d8t[(b * 4 + ((t & 7) >> 1)) * 2 * NT + 2 * (t >> 3) + (t & 1)] = d;
        // sub-block j = b % 8 of super-block b / 8: lane group j / 2, half j % 2
        const int j = (int)(b & 7);
        uint16_t *w = reinterpret_cast<uint16_t *>(spc + (((b >> 3) * 8 * NT + t) * 4 + (j >> 1)) * 4);
        uint16_t hi, mid, lo;
        bf16_pieces(s, hi, mid, lo);
        w[0 + (j & 1)] = hi;
        w[2 + (j & 1)] = mid;
        w[4 + (j & 1)] = lo;
    }
};

template <int EPI, int XIN, int NT, bool XH>
__global__ void __launch_bounds__(kMThreads, 1) q4k_gemv_mma_kernel(const __grid_constant__ MArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = (EPI == EPI_SWIGLU) ? 2 : 1;
    uint8_t *ring = smem;
    uint8_t *xcodes = ring + (int64_t)a.NS * a.stage_bytes;
    static_assert(!XH || XIN == MX_Q8, "f16 activations are staged from Q8_1 input only");
    // Q8_1 input whose codes do not fit beside the ring is staged in phases of
    // a.xph super-blocks (the d8 and s tables for the whole row stay resident)
    const bool phased = !XH && XIN == MX_Q8 && a.xph < a.nsb;
    const int64_t kdim = phased ? (int64_t)a.xph * 256 : a.in_dim;
    const int64_t cpitch = mma_code_pitch(kdim, XH);
    float *d8t = reinterpret_cast<float *>(xcodes + mma_codes_bytes(a.m, kdim, XH));
    uint32_t *spc = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(d8t) + mma_d8_bytes(a.in_dim, NT));
    const int64_t nb = a.in_dim / 32;
    // the partial sums of the warps: after the tables, or (XH) in the ring, idle
    // by then (every consumer warp has waited for every stage it reads)
    uint8_t *tables_end = reinterpret_cast<uint8_t *>(spc) + mma_spc_bytes(a.in_dim, NT);
    float *red = XH ? reinterpret_cast<float *>(ring) : reinterpret_cast<float *>(tables_end);
    float *nred = XH ? reinterpret_cast<float *>(tables_end) : red + mma_red_bytes(NT) / 4;  // 32 floats: the norm reduction
    uint64_t *full = reinterpret_cast<uint64_t *>(nred + 32);
    uint64_t *empty = full + a.NS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's segment (weight matrix) and rows
    int k = 0;
    while (k + 1 < a.nseg && (int)blockIdx.x >= a.cta_begin[k + 1]) ++k;
    const int rpc = a.rpc[k];
    const int64_t lr0 = (int64_t)(blockIdx.x - a.cta_begin[k]) * rpc;  // first row in the segment
    const int rows = (int)min((int64_t)rpc, a.seg_rows[k] - lr0);
    const int ntiles = (rpc + kMTile - 1) / kMTile;
    const int S = mma_slice_sb(ntiles, R, a.nsb), pitch = S * 144;
    const int hs = mma_half_bytes(ntiles, S);
    const int nslice = (a.nsb + S - 1) / S;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    // the stall test aid (rz_debug_stall_next_gemv) applies to CTA 0 only
    const int stall = (blockIdx.x == 0) ? a.stall_stage : -1;
    const uint32_t lim = (stall >= 0) ? a.wait_limit : kWaitLimit;

    if (warp == kMW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            for (int h = 0; h < R; ++h) tma_prefetch_desc(&a.map[R == 2 ? h : k]);
            const unsigned box_bytes = (unsigned)rpc * (unsigned)pitch;
            int64_t q = 0;
            bool ok = true;
            RingPos rp{0, 0u};
            for (; q < nslice; ++q, ring_next(rp, a.NS)) {
                const int s = rp.s;
                if (q >= a.NS && !mbar_wait(&empty[s], rp.par ^ 1u, lim)) {
                    set_error(a.err, DEV_TIMEOUT_GEMV);
                    ok = false;
                    break;
                }
                if (q == stall) continue;  // never issued: the consumers' wait runs out
                uint8_t *dst = ring + (int64_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], R * box_bytes);
                for (int h = 0; h < R; ++h)
                    tma_load_2d(dst + h * hs, &a.map[R == 2 ? h : k], (int)q * S * 36, (int)lr0, &full[s], pol);
            }
            if (!ok || stall >= 0) {
                for (int64_t p = (q > a.NS ? q - a.NS : 0); p < q; ++p)
                    if (p != stall && !mbar_wait(&full[p % a.NS], (unsigned)((p / a.NS) & 1)))
                        set_error(a.err, DEV_TIMEOUT_DRAIN);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();
    auto csync = [] { asm volatile("bar.sync 1, %0;" ::"r"(kMW * 32) : "memory"); };
    const int tid = threadIdx.x;
    if (a.zy && blockIdx.x == gridDim.x - 1)
        for (int64_t i = tid; i < (int64_t)a.m * a.zy_cnt; i += kMW * 32)
            a.zy[(i / a.zy_cnt) * a.zy_ld + a.zy_from + i % a.zy_cnt] = 0.0f;
    {
        // the d8 table and the s pieces start at zero: token slots past m contribute 0
        const int64_t n16 = (mma_d8_bytes(a.in_dim, NT) + mma_spc_bytes(a.in_dim, NT)) / 16;
        for (int64_t q = tid; q < n16; q += kMW * 32) reinterpret_cast<uint4 *>(d8t)[q] = make_uint4(0u, 0u, 0u, 0u);
        csync();
    }
    MmaStore<NT> st{xcodes, d8t, spc, cpitch};
    // codes of super-blocks [sb0, sb1) of every token (offset binary, or f16 in
    // fragment order), 16 bytes at a time.  Each thread issues all its loads
    // before its first store (one round trip to L2 rather than one per element).
    constexpr int kQ = 8;  // int4s per thread and round (16 tokens x 4096 codes: one round)
    auto stage_codes = [&](int sb0, int sb1) {
        const int n16 = (sb1 - sb0) * 16, nq = a.m * n16;
        for (int q0 = 0; q0 < nq; q0 += kQ * kMW * 32) {
            int4 v[kQ];
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kMW * 32 + tid;
                if (q < nq) {
                    const int t = q / n16;
                    v[u] = __ldg(reinterpret_cast<const int4 *>(a.xq + t * a.in_dim + (int64_t)sb0 * 256) + (q - t * n16));
                }
            }
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kMW * 32 + tid;
                if (q < nq) {
                    const int t = q / n16;
                    const uint32_t w0 = (uint32_t)v[u].x ^ 0x80808080u, w1 = (uint32_t)v[u].y ^ 0x80808080u;
                    const uint32_t w2 = (uint32_t)v[u].z ^ 0x80808080u, w3 = (uint32_t)v[u].w ^ 0x80808080u;
                    if constexpr (XH) {
                        // 16 codes -> two groups of eight f16 in fragment order
                        uint8_t *dst = xcodes + t * cpitch + (int64_t)(q - t * n16) * 32;
                        *reinterpret_cast<uint4 *>(dst) =
                            make_uint4(code_pair(w0), code_pair(w0 >> 8), code_pair(w1), code_pair(w1 >> 8));
                        *reinterpret_cast<uint4 *>(dst + 16) =
                            make_uint4(code_pair(w2), code_pair(w2 >> 8), code_pair(w3), code_pair(w3 >> 8));
                    } else {
                        *reinterpret_cast<uint4 *>(xcodes + t * cpitch + (int64_t)(q - t * n16) * 16) =
                            make_uint4(w0, w1, w2, w3);
                    }
                }
            }
        }
    };
    if (XIN == MX_Q8) {
        stage_codes(0, phased ? a.xph : a.nsb);
        // d and s of the whole row into the tables
        const int nbi = (int)nb, nm = a.m * nbi;
        for (int q0 = 0; q0 < nm; q0 += kQ * kMW * 32) {
            float dv[kQ], sv[kQ];
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kMW * 32 + tid;
                dv[u] = q < nm ? __ldg(a.xd + q) : 0.f;  // d and s are [m][nb], token-major
                sv[u] = q < nm ? __ldg(a.xs + q) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = q0 + u * kMW * 32 + tid;
                if (q < nm) st.meta(q / nbi, q % nbi, dv[u], sv[u]);
            }
        }
        csync();
    } else {
        stage_x_f32_to<false, XIN == MX_NORM, kMW>(st, a.xf, a.ldxf, a.gamma, a.norm_n, a.eps, a.m, a.in_dim, nred,
                                                   warp, lane, csync);
    }

    const int g = lane >> 2, i = lane & 3;
    // this lane's shared addresses at super-block 0: its B-fragment row of codes
    // (token g, clamped into the staged tokens; n-tile 1 is xstep further), its
    // d8 entries and its s pieces
    const uint32_t ring_s = smem_u32(ring);
    const uint32_t xrow0 = smem_u32(xcodes) + (uint32_t)(min(g, a.m - 1) * cpitch) + (XH ? 16u : 8u) * i;
    const uint32_t xstep = (uint32_t)((min(g + 8, a.m - 1) - min(g, a.m - 1)) * cpitch);
    const uint32_t d8a0 = smem_u32(d8t) + (uint32_t)i * (2 * NT * 4);
    const uint32_t spa0 = smem_u32(spc) + (uint32_t)(g * 4 + i) * 16u;
    const int nunits = R * ntiles * S;  // (half, tile, super-block) units of a stage, <= 16
    // this warp's unit: half h, tile tl, super-block js of every slice
    const int h = warp / (ntiles * S), tl = (warp / S) % ntiles, js = warp % S;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
    // A warp whose wait runs out records the error and stops reading and
    // releasing stages, but still meets the others at the final barriers; the
    // producer then runs out of its own wait and drains the copies it issued
    // before the CTA exits.
    bool failed = false;
    RingPos rp{0, 0u};
    for (int sl = 0; sl < nslice; ++sl, ring_next(rp, a.NS)) {
        const int s = rp.s;
        if (phased && sl > 0 && (sl * S) % a.xph == 0) {
            // the next phase of the codes: every warp is past the slices of the
            // last one (a.xph is a multiple of S, so no slice straddles two)
            csync();
            stage_codes(sl * S, min(a.nsb, sl * S + a.xph));
            csync();
        }
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(&full[s], rp.par, lim))) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_GEMV);
            failed = true;
        }
        const int sbs = min(S, a.nsb - sl * S);
        if (!failed && warp < nunits && js < sbs) {
            const uint32_t base = smem_after(ring_s);  // ordered after the wait
            const uint32_t t0 = base + (uint32_t)(s * a.stage_bytes + h * hs + (tl * kMTile) * pitch + js * 144);
            const int sbg = sl * S + js;
            const int sbx = phased ? sbg - (sl * S / a.xph) * a.xph : sbg;  // super-block within the staged codes
            const uint32_t off = base - ring_s;  // 0, carries the ordering to the other tables
            mma_superblock<NT, XH>(t0 + g * pitch, t0 + (g + 8) * pitch, xrow0 + off + (uint32_t)sbx * (XH ? 512u : 256u), xstep,
                               d8a0 + off + (uint32_t)sbg * (8 * 4 * 2 * NT * 4),
                               spa0 + off + (uint32_t)sbg * (8 * NT * 4 * 16), i, acc);
        }
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(&empty[s]);
    }
    // every unit done: partials -> fixed-order sums -> epilogue
    if constexpr (XH) csync();  // the partials overwrite the ring: every warp is past its last stage
    float *rw = red + (warp * 32 + lane) * 4 * NT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4 *>(rw + 4 * nt) = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    csync();
    const int nout = ntiles * kMTile * 8 * NT;  // (row, token) outputs
    for (int o = tid; o < nout; o += kMW * 32) {
        const int r = o % (ntiles * kMTile), t = o / (ntiles * kMTile);  // row of the CTA, token
        const int tile = r >> 4, rr = r & 15;
        const int ln = 4 * (rr & 7) + ((t & 7) >> 1);
        const int e = ((rr >> 3) << 1) + (t & 1), nt = t >> 3;
        if (r < rows && t < a.m) {
            float v[2] = {0.f, 0.f};
#pragma unroll
            for (int hh = 0; hh < R; ++hh)
                for (int jj = 0; jj < S; ++jj) {
                    const int w = (hh * ntiles + tile) * S + jj;
                    v[hh] += red[((w * 32 + ln) * NT + nt) * 4 + e];
                }
            const int64_t lr = lr0 + r;
            float out = v[0];
            if (EPI == EPI_RESID || (EPI == EPI_STORE && a.res[k])) out = a.res[k][t * a.ldr[k] + lr] + out;
            if (EPI == EPI_SWIGLU) out = silu_mul(v[0], v[1]);
            a.y[k][t * a.ldy[k] + lr] = out;
        }
    }
}

int64_t mma_smem_bytes(int m, int64_t in_dim, int nt, int NS, int stage_bytes, bool xh, int64_t kdim)
{
    return (int64_t)NS * stage_bytes + mma_x_bytes(m, in_dim, nt, xh, kdim) + (xh ? 0 : mma_red_bytes(nt)) + 32 * 4 +
           2 * 8 * NS;
}

template <int EPI, int XIN, int NT, bool XH = false>
cudaError_t mma_launch_t(const MArgs &a, int grid, cudaStream_t s, size_t smem)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_gemv_mma_kernel<EPI, XIN, NT, XH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4k_gemv_mma_kernel<EPI, XIN, NT, XH>, a);
}

template <int EPI, int NT>
cudaError_t mma_launch_x(const MArgs &a, int grid, cudaStream_t s, size_t smem, int xin, bool xh)
{
    if (xh) return xin == MX_Q8 ? mma_launch_t<EPI, MX_Q8, NT, true>(a, grid, s, smem) : cudaErrorInvalidValue;
    if (xin == MX_NORM) {
        if constexpr (EPI != EPI_RESID) return mma_launch_t<EPI, MX_NORM, NT>(a, grid, s, smem);
        return cudaErrorInvalidValue;
    }
    if (xin == MX_F32) {
        if constexpr (EPI == EPI_RESID) return mma_launch_t<EPI, MX_F32, NT>(a, grid, s, smem);
        return cudaErrorInvalidValue;
    }
    return mma_launch_t<EPI, MX_Q8, NT>(a, grid, s, smem);
}

// Rows per CTA of each segment, CTAs per segment: every segment gets CTAs in
// proportion to its rows (at least one, at most the SM count in total unless a
// CTA would hold more than 256 / R rows), each CTA an equal range.
struct MmaPlan {
    int nseg;
    int cta_begin[4];
    int rpc[3];
    int stage_bytes;  // largest stage of any CTA
};

MmaPlan mma_plan(const int64_t *rows, int nseg, int R, int nsb)
{
    MmaPlan p{};
    p.nseg = nseg;
    const int sms = dev_info().sm_count;
    int64_t U = 0;
    for (int k = 0; k < nseg; ++k) U += rows[k];
    int c0 = 0;
    for (int k = 0; k < nseg; ++k) {
        int64_t c = std::max<int64_t>(1, rows[k] * sms / U);
        int64_t rpc = (rows[k] + c - 1) / c;
        const int64_t cap = 16 * (kMW / R);  // R x tiles <= kMW
        if (rpc > cap) rpc = cap;
        c = (rows[k] + rpc - 1) / rpc;
        p.cta_begin[k] = c0;
        p.rpc[k] = (int)rpc;
        c0 += (int)c;
        const int tiles = (int)((rpc + 15) / 16);
        const int S = mma_slice_sb(tiles, R, nsb);
        p.stage_bytes = std::max(p.stage_bytes, R * mma_half_bytes(tiles, S));
    }
    p.cta_begin[nseg] = c0;
    return p;
}

// Ring stages that fit next to the activations of mt tokens (0 if fewer than
// two).  xh: the codes as f16, the partial sums in the ring (which must hold them).
int mma_stages(int mt, int64_t in_dim, int stage_bytes, bool xh = false, int64_t kdim = 0)
{
    const int nt = mt > 8 ? 2 : 1;
    const int64_t fixed = mma_x_bytes(mt, in_dim, nt, xh, kdim ? kdim : in_dim) + (xh ? 0 : mma_red_bytes(nt)) +
                          32 * 4 + 1024;
    const int64_t ns = ((int64_t)std::min<int64_t>(kMSmem, dev_info().smem_optin) - fixed) / (stage_bytes + 16);
    if (ns < 2 || (xh && ns * stage_bytes < mma_red_bytes(nt))) return 0;
    return (int)std::min<int64_t>(ns, 8);
}

// Super-blocks of int8 codes per phase for mt tokens of Q8_1 input: nsb when the
// whole row fits beside two stages, else the first of nsb / 2, nsb / 3, ... (up
// to eight phases, rounded up to a multiple of 6 -- of every slice length) that
// does; 0 when none does.
int mma_phase_sb(int mt, int64_t in_dim, int stage_bytes)
{
    const int nsb = (int)(in_dim / 256);
    if (mma_stages(mt, in_dim, stage_bytes) >= 2) return nsb;
    for (int P = 2; P <= 8; ++P) {
        const int ph = ((nsb + P - 1) / P + 5) / 6 * 6;
        if (ph >= nsb) continue;
        if (mma_stages(mt, in_dim, stage_bytes, false, (int64_t)ph * 256) >= 2) return ph;
    }
    return 0;
}

// The largest ring slot any plan can need: R x the largest half over tile counts.
int mma_stage_bound(int R, int nsb)
{
    int mx = 0;
    for (int tiles = 1; tiles <= 16 / R; ++tiles)
        mx = std::max(mx, R * mma_half_bytes(tiles, mma_slice_sb(tiles, R, nsb)));
    return mx;
}

}  // namespace

// Largest token count per launch whose activations leave room for two stages
// (of the largest stage any CTA can have); Q8_1 input may stage its codes in
// phases, f32 input stages the whole row.
int q4k_gemv_mma_group(int64_t m, int64_t in_dim, int epilogue, bool q8_input)
{
    const int R = (epilogue == EPI_SWIGLU) ? 2 : 1;
    const int sb = mma_stage_bound(R, (int)(in_dim / 256));
    int64_t mt = std::min<int64_t>(m, 16);
    while (mt > 0 && (q8_input ? mma_phase_sb((int)mt, in_dim, sb) : mma_stages((int)mt, in_dim, sb)) == 0) --mt;
    return (int)mt;
}

// One launch of the tensor-core GEMV for m <= 16 tokens (m > 8: two n-tiles):
// Q8_1 input (xq codes [m][in_dim], xd and xs [m][in_dim / 32]) or f32 input.
cudaError_t launch_q4k_gemv_mma(const Q4kSegment *seg, int nseg, int epilogue, const int8_t *xq, const float *xd,
                                const float *xs, const F32Input *f32in, int64_t m, int64_t in_dim, cudaStream_t s)
{
    MArgs a = {};
    const int R = (epilogue == EPI_SWIGLU) ? 2 : 1;
    const int nsb = (int)(in_dim / 256);
    const int64_t row_bytes = (int64_t)nsb * 144;
    int64_t rows[3];
    const int nplan = (R == 2) ? 1 : nseg;
    for (int k = 0; k < nseg; ++k) {
        a.y[k] = seg[k].y;
        a.res[k] = seg[k].res;
        a.ldy[k] = seg[k].ldy ? seg[k].ldy : seg[k].rows;
        a.ldr[k] = seg[k].ldr ? seg[k].ldr : seg[k].rows;
        if (epilogue == EPI_STORE) {
            a.res[k] = seg[k].bias;
            a.ldr[k] = 0;
        }
        rows[k] = seg[k].rows;
        a.seg_rows[k] = seg[k].rows;
    }
    const MmaPlan plan = mma_plan(rows, nplan, R, nsb);
    a.nseg = nplan;
    for (int k = 0; k <= nplan; ++k) a.cta_begin[k] = plan.cta_begin[k];
    for (int k = 0; k < nplan; ++k) a.rpc[k] = plan.rpc[k];
    // tensor maps: one per weight matrix, box = (S super-blocks, rpc rows)
    for (int k = 0; k < nseg; ++k) {
        const int kp = (R == 2) ? 0 : k;
        const int tiles = (plan.rpc[kp] + 15) / 16;
        const int S = mma_slice_sb(tiles, R, nsb);
        const cudaError_t e = encode_tensor_map_2d(&a.map[k], seg[k].w, 4, (uint64_t)row_bytes / 4,
                                                   (uint64_t)seg[k].rows, (uint64_t)row_bytes, (uint32_t)(S * 36),
                                                   (uint32_t)plan.rpc[kp]);
        if (e != cudaSuccess) return e;
    }
    a.nsb = nsb;
    a.m = (int)m;
    a.in_dim = in_dim;
    int xin = MX_Q8;
    if (f32in) {
        a.xf = f32in->x;
        a.ldxf = f32in->ldx;
        a.gamma = f32in->gamma;
        a.norm_n = f32in->norm_n;
        a.eps = f32in->eps;
        xin = f32in->gamma ? MX_NORM : MX_F32;
    } else {
        a.xq = xq;
        a.xd = xd;
        a.xs = xs;
    }
    a.err = dev_error_word();
    if (seg[0].zero_to > seg[0].rows) {
        a.zy = seg[0].y;
        a.zy_ld = seg[0].ldy ? seg[0].ldy : seg[0].rows;
        a.zy_from = seg[0].rows;
        a.zy_cnt = seg[0].zero_to - seg[0].rows;
    }
    a.stall_stage = -1;
    a.wait_limit = kWaitLimit;
    if (g_stall_next_gemv) {
        a.stall_stage = 0;
        a.wait_limit = g_stall_next_gemv;
        g_stall_next_gemv = 0;
    }
    a.stage_bytes = plan.stage_bytes;
    const int nt = m > 8 ? 2 : 1;
    // Q8_1 input: the codes staged as f16 in fragment order when two stages still fit
    // beside them (each warp then loads its B fragments instead of converting them)
    const bool xh = !f32in && mma_stages((int)m, in_dim, a.stage_bytes, true) >= 2;
    a.xph = (xh || f32in) ? nsb : mma_phase_sb((int)m, in_dim, a.stage_bytes);
    if (a.xph < 1) return cudaErrorInvalidConfiguration;
    const int64_t kdim = (int64_t)a.xph * 256;
    a.NS = mma_stages((int)m, in_dim, a.stage_bytes, xh, kdim);
    if (a.NS < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)mma_smem_bytes((int)m, in_dim, nt, a.NS, a.stage_bytes, xh, kdim);
    if (smem > dev_info().smem_optin) return cudaErrorInvalidConfiguration;
    const int grid = plan.cta_begin[nplan];
    switch (epilogue) {
    case EPI_STORE: return nt == 1 ? mma_launch_x<EPI_STORE, 1>(a, grid, s, smem, xin, xh)
                                   : mma_launch_x<EPI_STORE, 2>(a, grid, s, smem, xin, xh);
    case EPI_RESID: return nt == 1 ? mma_launch_x<EPI_RESID, 1>(a, grid, s, smem, xin, xh)
                                   : mma_launch_x<EPI_RESID, 2>(a, grid, s, smem, xin, xh);
    default: return nt == 1 ? mma_launch_x<EPI_SWIGLU, 1>(a, grid, s, smem, xin, xh)
                            : mma_launch_x<EPI_SWIGLU, 2>(a, grid, s, smem, xin, xh);
    }
}

}  // namespace rz
