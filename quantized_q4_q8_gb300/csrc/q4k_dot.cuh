// q4k_dot.cuh -- the Q4_K x Q8_1 dot-product core of the GEMV kernels: the padded
// shared-memory layout of the Q8_1 activations, the super-block accumulation of
// one lane, the packing of rows into ring stages, and the staging of activations
// (copy of Q8_1 codes, or quantisation of f32 values, optionally RMS-normalised
// first) into that layout.
//
// Super-block layout (block_q4_K of GGML's k-quants): f16 d, f16 dmin, 12 bytes
// of packed 6-bit scales and mins, 128 bytes of 4-bit codes; element e sits in
// byte 32 (e / 64) + e % 32, low nibble when e % 64 < 32.  Value of element e of
// sub-block j: d * sc_j * q - dmin * m_j.
#pragma once

#include "rz_common.cuh"

namespace rz {
namespace {

constexpr int kSB = 144;

// Shared-memory copy of the Q8_1 codes.  Super-block sb of token t occupies a
// 288-byte slot; the 64 bytes that lane chunk c reads (sub-blocks 2c, 2c+1) sit at
// 64c + 16(c >> 1) inside it.  With this padding the 8 lanes of a shared-memory
// phase (2 consecutive super-blocks x 4 chunks) hit 8 different bank groups, and
// every address is a lane constant plus a multiple of the super-block index.
// The f32 scales d then the f32 sums s of all tokens follow the slots.
constexpr int kXSlot = 288;

__device__ __forceinline__ int x_chunk_off(int c) { return 64 * c + 16 * (c >> 1); }

__host__ __device__ inline int64_t x_smem_bytes(int64_t m, int64_t in_dim)
{
    return m * (in_dim / 256) * kXSlot + 8 * m * (in_dim / 32);
}

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

// Weight super-block fields a lane needs: d, dmin, its two 6-bit scales and
// mins (as products), and its 32 quant bytes: the low nibbles masked down
// (0..15) and the high nibbles masked in place (16 x 0..15).
struct SbLane {
    float d, dm0, dm1;
    int sc0, sc1;
    uint32_t lo[8], hi16[8];
};

// dot of four unsigned bytes with four signed bytes, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ void sb_lane_load(uint32_t blk, int c, const LaneConst &L, SbLane &w)
{
    const int4 hdr = lds128(blk);
    const int4 qa = lds128(blk + 16 + 32 * c);
    const int4 qb = lds128(blk + 32 + 32 * c);
    w.d = h2f((uint16_t)((uint32_t)hdr.x & 0xffffu));
    const float dmin = h2f((uint16_t)((uint32_t)hdr.x >> 16));
    const uint32_t A = (uint32_t)hdr.y >> L.sh, B = (uint32_t)hdr.z >> L.sh, C = (uint32_t)hdr.w >> L.sh;
    const uint32_t scp = (A & L.mask_lo) | (C & L.mask_c) | ((A >> 2) & L.mask_hi);
    const uint32_t mnp = (B & L.mask_lo) | ((C >> 4) & L.mask_c) | ((B >> 2) & L.mask_hi);
    w.sc0 = (int)(scp & 0xffu);
    w.sc1 = (int)((scp >> 8) & 0xffu);
    w.dm0 = dmin * (float)(mnp & 0xffu);
    w.dm1 = dmin * (float)((mnp >> 8) & 0xffu);
    const uint32_t q[8] = {(uint32_t)qa.x, (uint32_t)qa.y, (uint32_t)qa.z, (uint32_t)qa.w,
                           (uint32_t)qb.x, (uint32_t)qb.y, (uint32_t)qb.z, (uint32_t)qb.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w.lo[i] = q[i] & 0x0f0f0f0fu;
        w.hi16[i] = q[i] & 0xf0f0f0f0u;
    }
}

// acc += the lane's share of one super-block (same value as sb_accumulate: the
// high-nibble dot comes out 16 times too large, exactly, and is shifted back)
__device__ __forceinline__ void sb_lane_dot(const SbLane &w, const int4 &x0, const int4 &x1, const int4 &x2,
                                            const int4 &x3, const float2 &d8, const float2 &s8, float &acc)
{
    int a0 = dp4a_us(w.lo[0], x0.x, 0), a1 = dp4a_us(w.lo[4], x1.x, 0);
    int b0 = dp4a_us(w.hi16[0], x2.x, 0), b1 = dp4a_us(w.hi16[4], x3.x, 0);
    a0 = dp4a_us(w.lo[1], x0.y, a0);
    a1 = dp4a_us(w.lo[5], x1.y, a1);
    b0 = dp4a_us(w.hi16[1], x2.y, b0);
    b1 = dp4a_us(w.hi16[5], x3.y, b1);
    a0 = dp4a_us(w.lo[2], x0.z, a0);
    a1 = dp4a_us(w.lo[6], x1.z, a1);
    b0 = dp4a_us(w.hi16[2], x2.z, b0);
    b1 = dp4a_us(w.hi16[6], x3.z, b1);
    a0 = dp4a_us(w.lo[3], x0.w, a0);
    a1 = dp4a_us(w.lo[7], x1.w, a1);
    b0 = dp4a_us(w.hi16[3], x2.w, b0);
    b1 = dp4a_us(w.hi16[7], x3.w, b1);
    const float t0 = (float)(w.sc0 * (a0 + a1)) * d8.x;
    const float t1 = (float)(w.sc1 * ((b0 + b1) >> 4)) * d8.y;  // |16 I| < 2^31: exact
    acc = fmaf(w.d, t0 + t1, acc) - (w.dm0 * s8.x + w.dm1 * s8.y);
}

// Two rows at once (one token, activations in shared memory): super-block sb of
// row A at blkA and of row B at blkB share one load of the activations.  No
// branch between the rows, so their dependency chains interleave (a missing row
// B is passed as a copy of row A and its result dropped by the caller).
__device__ __forceinline__ void sb_accumulate_pair(const XSrc &x, uint32_t blkA, uint32_t blkB, int sb, int c,
                                                   const LaneConst &L, float &accA, float &accB)
{
    const uint32_t xa = x.q + (uint32_t)sb * kXSlot + x_chunk_off(c);
    const int4 x0 = lds128(xa), x1 = lds128(xa + 16), x2 = lds128(xa + 32), x3 = lds128(xa + 48);
    const uint32_t da = x.ds + (uint32_t)(sb * 8 + 2 * c) * 4u;
    const float2 d8 = lds64f(da), s8 = lds64f(da + (uint32_t)x.nb * 4u);
    SbLane wa, wb;
    sb_lane_load(blkA, c, L, wa);
    sb_lane_load(blkB, c, L, wb);
    sb_lane_dot(wa, x0, x1, x2, x3, d8, s8, accA);
    sb_lane_dot(wb, x0, x1, x2, x3, d8, s8, accB);
}

// Two packs of one row each (rows with 8 or more super-blocks), one token.  On
// return the totals of row A are in lane 0 (acc[h][0]) and those of row B in
// lane 16 (acc[h][1]).  Reduction: one exchange across the half-warps (lanes
// below 16 keep row A, the others row B), then the xor butterfly 8, 4, 2, 1 within
// each half: a fixed order, so the result is deterministic.
__device__ __forceinline__ void pack_pair_accumulate(const XSrc &x, uint32_t pkA, uint32_t pkB, bool hasB, int R,
                                                     uint32_t pack_bytes, int nsb, int lane, float (&acc)[2][2])
{
    const int g = lane >> 2, c = lane & 3;
    const LaneConst Lc = lane_const(c);
    float a[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) a[h][0] = a[h][1] = 0.0f;
#pragma unroll 1
    for (int h = 0; h < R; ++h) {
        const uint32_t hA = pkA + (uint32_t)h * pack_bytes;
        const uint32_t hB = (hasB ? pkB : pkA) + (uint32_t)h * pack_bytes;
        for (int sb = g; sb < nsb; sb += 8)
            sb_accumulate_pair(x, hA + sb * kSB, hB + sb * kSB, sb, c, Lc, a[h][0], a[h][1]);
    }
    const bool upper = lane & 16;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float rA = a[h][0], rB = a[h][1];
        const float keep = upper ? rB : rA, send = upper ? rA : rB;
        float v = keep + __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[h][0] = acc[h][1] = v;  // row A in lanes 0-15, row B in lanes 16-31
    }
}

// Two packs of one row each (rows with 8 or more super-blocks), tokens t0 ..
// t0 + TG - 1 (those below x.m), activations in shared memory: each activation
// load feeds both rows, so shared-memory traffic per token is about half that
// of one row at a time.  On return acc[h][i] holds, for token t0 + i, the total
// of row A in lanes 0-15 and that of row B in lanes 16-31 (the reduction of
// pack_pair_accumulate, per token).
template <int TG>
__device__ __forceinline__ void pack_pair_accumulate_tg(const XSrc &x, uint32_t pkA, uint32_t pkB, bool hasB, int R,
                                                        uint32_t pack_bytes, int nsb, int t0, int lane,
                                                        float (&acc)[2][TG])
{
    const int g = lane >> 2, c = lane & 3;
    const LaneConst Lc = lane_const(c);
    const int nt = min(TG, x.m - t0);
    const int nsbx = (int)(x.in_dim / 256);
    float a[2][2][TG];  // [half][row][token]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < TG; ++i) a[h][0][i] = a[h][1][i] = 0.0f;
#pragma unroll 1
    for (int h = 0; h < R; ++h) {
        const uint32_t hA = pkA + (uint32_t)h * pack_bytes;
        const uint32_t hB = (hasB ? pkB : pkA) + (uint32_t)h * pack_bytes;
        for (int sb = g; sb < nsb; sb += 8) {
            SbLane wa, wb;
            sb_lane_load(hA + sb * kSB, c, Lc, wa);
            sb_lane_load(hB + sb * kSB, c, Lc, wb);
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                if (i < nt) {
                    const int t = t0 + i;
                    const uint32_t xa = x.q + (uint32_t)(t * nsbx + sb) * kXSlot + x_chunk_off(c);
                    const int4 x0 = lds128(xa), x1 = lds128(xa + 16), x2 = lds128(xa + 32), x3 = lds128(xa + 48);
                    const uint32_t da = x.ds + (uint32_t)(t * x.nb + sb * 8 + 2 * c) * 4u;
                    const float2 d8 = lds64f(da), s8 = lds64f(da + (uint32_t)(x.m * x.nb) * 4u);
                    sb_lane_dot(wa, x0, x1, x2, x3, d8, s8, a[h][0][i]);
                    sb_lane_dot(wb, x0, x1, x2, x3, d8, s8, a[h][1][i]);
                }
            }
        }
    }
    const bool upper = lane & 16;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < TG; ++i) {
            const float rA = a[h][0][i], rB = a[h][1][i];
            const float keep = upper ? rB : rA, send = upper ? rA : rB;
            float v = keep + __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[h][i] = v;
        }
}

// Rows per pack: a warp takes a whole pack; rows with fewer than 8 super-blocks
// are packed 8 / nsb to a warp so that every lane group has a super-block.
__host__ __device__ inline int pack_rows_for(int nsb) { return (nsb < 8 && 8 % nsb == 0) ? 8 / nsb : 1; }

// One pack at shared address pk (R halves of pack_bytes each: gate then up for
// the SwiGLU pair) against the staged activations; the per-row results end up
// reduced over the lanes of the row in acc[h][t] (fixed order: deterministic).
// Lane layout: group g = lane / 4 takes super-blocks g, g + 8, ... of its row
// (row rip = g / nsb of the pack when rows are packed), lane c = lane % 4 one
// 32-byte quant chunk of each.
template <int MT, int R, bool XS>
__device__ __forceinline__ void pack_accumulate(const XSrc &x, uint32_t pk, uint32_t pack_bytes, int nsb,
                                                int rpp, int rip, int pack_rows, int lane,
                                                float (&acc)[2][MT])
{
    const int g = lane >> 2, c = lane & 3;
    const LaneConst Lc = lane_const(c);
    float acc2[2][MT];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[h][t] = acc2[h][t] = 0.0f;
#pragma unroll
    for (int h = 0; h < R; ++h) {
        const uint32_t half = pk + (uint32_t)h * pack_bytes;
        if (rpp > 1) {
            if (rip < pack_rows) sb_accumulate<MT, XS>(x, half + g * kSB, g % nsb, c, Lc, acc[h]);
        } else {
            int sb = g;
            if (MT <= 2) {
                for (; sb + 8 < nsb; sb += 16) {  // two independent super-blocks per step
                    sb_accumulate<MT, XS>(x, half + sb * kSB, sb, c, Lc, acc[h]);
                    sb_accumulate<MT, XS>(x, half + (sb + 8) * kSB, sb + 8, c, Lc, acc2[h]);
                }
            }
            for (; sb < nsb; sb += 8) sb_accumulate<MT, XS>(x, half + sb * kSB, sb, c, Lc, acc[h]);
        }
    }
    const int seg_lanes = (rpp > 1) ? 4 * nsb : 32;
#pragma unroll
    for (int h = 0; h < R; ++h)
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            acc[h][t] += acc2[h][t];
            for (int o = 1; o < seg_lanes; o <<= 1) acc[h][t] += __shfl_xor_sync(0xffffffffu, acc[h][t], o);
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

// ---------------------------------------------------------------- activation staging
// Both helpers run on the 32 * NW threads of NW warps (thread index tid, warp,
// lane) and end with `sync` over them.

// Q8_1 codes of m rows of in_dim ([m][in_dim]) and their d and s ([m][in_dim/32]
// each) -> slot layout.
template <bool CG, int NW = kRowWarps, typename Sync>
__device__ __forceinline__ void stage_x_q8(uint8_t *xsm, const int8_t *xq, const float *xd, const float *xs,
                                           int m, int64_t in_dim, int tid, Sync sync)
{
    const int64_t nsbx = (int64_t)m * (in_dim / 256);
    const int4 *src = reinterpret_cast<const int4 *>(xq);
    for (int64_t i = tid; i < nsbx * 16; i += NW * 32) {
        const int64_t sbg = i >> 4;
        const int ch = (int)(i & 15), cc = ch >> 2;
        const int4 v = CG ? __ldcg(src + i) : src[i];
        *reinterpret_cast<int4 *>(xsm + sbg * kXSlot + x_chunk_off(cc) + 16 * (ch & 3)) = v;
    }
    // d, then s, unchanged
    const int64_t nd = (int64_t)m * (in_dim / 32) / 4;  // int4 of each
    const int4 *dsrc = reinterpret_cast<const int4 *>(xd);
    const int4 *ssrc = reinterpret_cast<const int4 *>(xs);
    int4 *ddst = reinterpret_cast<int4 *>(xsm + nsbx * kXSlot);
    for (int64_t i = tid; i < 2 * nd; i += NW * 32) {
        const int4 *src = i < nd ? dsrc + i : ssrc + (i - nd);
        ddst[i] = CG ? __ldcg(src) : *src;
    }
    sync();
}

// f32 rows x[t * ldx + i] quantised into the slot layout: RMS-normalised over
// their first norm_n values with gamma first when NORM, else as they are.
// Layout: thread j of the NT = 32 NW threads takes float4 number j, j + NT, ...
// (KF of them at most), so the 32 float4s of a warp are 128 consecutive values,
// four Q8_1 blocks of eight lanes each.  All loads are issued at once (one round
// trip to memory); a block's max |x| and code sum take three shuffles within its
// eight lanes, and each lane stores its four codes as one word.  The sum of
// squares runs in a fixed order (per thread over its float4s in order, then the
// xor butterfly of each warp, then the warp sums in order), so every CTA
// computes the same bits.  `red`: NW + 1 floats of shared memory.
// Store functor of the padded-slot layout above: codes(t, b, e0, word) writes the
// four codes e0..e0+3 of Q8_1 block b of token t, meta(t, b, d, s) its d and s.
struct SlotStore {
    uint8_t *xsm;
    float *dsm, *ssm;
    int64_t nb, nsb;
    __device__ __forceinline__ void codes(int t, int64_t b, int e0, uint32_t word) const
    {
        const int j = (int)(b & 7);
        *reinterpret_cast<uint32_t *>(xsm + (t * nsb + (b >> 3)) * kXSlot + x_chunk_off(j >> 1) + 32 * (j & 1) + e0) =
            word;
    }
    __device__ __forceinline__ void meta(int t, int64_t b, float d, float s) const
    {
        dsm[t * nb + b] = d;
        ssm[t * nb + b] = s;
    }
};

struct NoWait {
    __device__ void operator()() const {}
};

template <bool CG, bool NORM, int KF, int NW, typename Store, typename Sync, typename PreWait>
__device__ __forceinline__ void stage_x_f32_kf(const Store &st, const float *xf, int64_t ldx, const float *gamma,
                                               int64_t norm_n, float eps, int m, int64_t in_dim, float *red,
                                               int warp, int lane, Sync sync, PreWait prewait)
{
    constexpr int NT = 32 * NW;
    const int64_t n4 = in_dim / 4;
    const int tid = warp * 32 + lane;
    auto load_gamma = [&](int64_t f) {
        // gamma holds norm_n values (not padded): no read past them
        const int64_t i0 = f * 4;
        float4 g;
        if (i0 + 3 < norm_n) {
            g = __ldg(reinterpret_cast<const float4 *>(gamma) + f);
        } else {
            g.x = i0 < norm_n ? __ldg(gamma + i0) : 0.f;
            g.y = i0 + 1 < norm_n ? __ldg(gamma + i0 + 1) : 0.f;
            g.z = i0 + 2 < norm_n ? __ldg(gamma + i0 + 2) : 0.f;
            g.w = 0.f;
        }
        return g;
    };
    // Short rows keep their gammas in registers, loaded once for every token and
    // before `prewait` (the wait on the kernel that writes xf: gamma is a weight,
    // and read cold it would otherwise arrive from HBM behind the weight stream
    // after the values); long rows fetch them after the reduction.
    constexpr bool kEarly = NORM && KF <= 4;
    float4 gm[kEarly ? KF : 1];
    if constexpr (kEarly) {
#pragma unroll
        for (int k = 0; k < KF; ++k) {
            const int64_t f = (int64_t)k * NT + tid;
            gm[k] = f < n4 ? load_gamma(f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    prewait();
    for (int t = 0; t < m; ++t) {
        const float4 *xrow = reinterpret_cast<const float4 *>(xf + t * ldx);
        float4 v[KF];
#pragma unroll
        for (int k = 0; k < KF; ++k) {
            const int64_t f = (int64_t)k * NT + tid;  // validity is uniform over a warp
            if (f < n4) {
                if constexpr (CG)
                    v[k] = __ldcg(xrow + f);
                else
                    v[k] = __ldg(xrow + f);
            } else {
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if constexpr (NORM) {
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < KF; ++k) {
                const int64_t i0 = ((int64_t)k * NT + tid) * 4;
                // values at or past norm_n are padding
                const float x0 = i0 < norm_n ? v[k].x : 0.f, x1 = i0 + 1 < norm_n ? v[k].y : 0.f;
                const float x2 = i0 + 2 < norm_n ? v[k].z : 0.f, x3 = i0 + 3 < norm_n ? v[k].w : 0.f;
                v[k] = make_float4(x0, x1, x2, x3);
                ss = fmaf(x0, x0, ss);
                ss = fmaf(x1, x1, ss);
                ss = fmaf(x2, x2, ss);
                ss = fmaf(x3, x3, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) red[warp] = ss;
            sync();
            if (warp == 0) {
                float r = 0.0f;
                for (int w = 0; w < NW; ++w) r += red[w];  // every lane, same order
                if (lane == 0) red[NW] = r;
            }
            sync();
            const float scale = rms_scale(red[NW], norm_n, eps);
            sync();  // red is reused by the next token
#pragma unroll
            for (int k = 0; k < KF; ++k) {
                const int64_t f = (int64_t)k * NT + tid;
                float4 g;
                if constexpr (kEarly)
                    g = gm[k];
                else
                    g = (f < n4) ? load_gamma(f) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[k].x = __fmul_rn(__fmul_rn(v[k].x, scale), g.x);
                v[k].y = __fmul_rn(__fmul_rn(v[k].y, scale), g.y);
                v[k].z = __fmul_rn(__fmul_rn(v[k].z, scale), g.z);
                v[k].w = __fmul_rn(__fmul_rn(v[k].w, scale), g.w);
            }
        }
#pragma unroll
        for (int k = 0; k < KF; ++k) {
            const int64_t f = (int64_t)k * NT + tid;
            if ((int64_t)k * NT + warp * 32 >= n4) break;  // warp-uniform
            float am = fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w)));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            const float d = __fdiv_rn(am, 127.0f);
            const Q8Scale sc = q8_scale(d);
            const int q0 = q8_code(v[k].x, sc), q1 = q8_code(v[k].y, sc);
            const int q2 = q8_code(v[k].z, sc), q3 = q8_code(v[k].w, sc);
            int sum = q0 + q1 + q2 + q3;
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            const int64_t b = f >> 3;  // Q8_1 block
            const int e0 = (int)(f & 7) * 4;
            const uint32_t word = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) |
                                  ((uint32_t)(q2 & 0xff) << 16) | ((uint32_t)(q3 & 0xff) << 24);
            st.codes(t, b, e0, word);
            if ((lane & 7) == 0) st.meta(t, b, d, __fmul_rn(d, (float)sum));
        }
    }
    sync();
}

// Dispatch on the float4s per thread the row needs (rows up to 16384 values:
// 16 warps x 8 float4s, or 8 warps x 16).  `prewait` runs once, after the loads
// that do not depend on xf and before the first load of xf.
template <bool CG, bool NORM, int NW = kRowWarps, typename Store, typename Sync, typename PreWait = NoWait>
__device__ __forceinline__ void stage_x_f32_to(const Store &st, const float *xf, int64_t ldx, const float *gamma,
                                               int64_t norm_n, float eps, int m, int64_t in_dim, float *red,
                                               int warp, int lane, Sync sync, PreWait prewait = PreWait())
{
    const int64_t kf = (in_dim / 4 + 32 * NW - 1) / (32 * NW);
    if (kf <= 2)
        stage_x_f32_kf<CG, NORM, 2, NW>(st, xf, ldx, gamma, norm_n, eps, m, in_dim, red, warp, lane, sync, prewait);
    else if (kf <= 4)
        stage_x_f32_kf<CG, NORM, 4, NW>(st, xf, ldx, gamma, norm_n, eps, m, in_dim, red, warp, lane, sync, prewait);
    else if (kf <= 8 || NW >= 16)
        stage_x_f32_kf<CG, NORM, 8, NW>(st, xf, ldx, gamma, norm_n, eps, m, in_dim, red, warp, lane, sync, prewait);
    else
        stage_x_f32_kf<CG, NORM, 16, NW>(st, xf, ldx, gamma, norm_n, eps, m, in_dim, red, warp, lane, sync, prewait);
}

// The same into the padded-slot layout.
template <bool CG, bool NORM, int NW = kRowWarps, typename Sync, typename PreWait = NoWait>
__device__ __forceinline__ void stage_x_f32(uint8_t *xsm, const float *xf, int64_t ldx, const float *gamma,
                                            int64_t norm_n, float eps, int m, int64_t in_dim, float *red,
                                            int warp, int lane, Sync sync, PreWait prewait = PreWait())
{
    SlotStore st;
    st.xsm = xsm;
    st.nb = in_dim / 32;
    st.nsb = in_dim / 256;
    st.dsm = reinterpret_cast<float *>(xsm + (int64_t)m * st.nsb * kXSlot);
    st.ssm = st.dsm + (int64_t)m * st.nb;
    stage_x_f32_to<CG, NORM, NW>(st, xf, ldx, gamma, norm_n, eps, m, in_dim, red, warp, lane, sync, prewait);
}

}  // namespace
}  // namespace rz
