// rz_common.cuh -- shared device helpers for the librz kernels (sm_103a).
//
// PTX wrappers for mbarriers and the 1-D bulk copy engine (cp.async.bulk),
// the device error word protocol, and small numeric helpers.  Every wait on an
// mbarrier is bounded: when the bound runs out the kernel records an error
// code in the device error word and stops, it never traps.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rz {

// ---------------------------------------------------------------- error word
enum DevErr : unsigned {
    DEV_OK = 0,
    DEV_TIMEOUT_GEMV = 0x101,   // bulk-copy wait in a GEMV gave up
    DEV_TIMEOUT_Q40 = 0x102,
    DEV_TIMEOUT_ATTN = 0x104,   // the V-row copy wait of the attention kernel gave up
    DEV_TIMEOUT_GEMM = 0x108,   // a wait of the tensor-core many-token GEMM gave up
    DEV_TIMEOUT_DRAIN = 0x1ff,  // draining outstanding copies gave up
    DEV_BAD_POSITION = 0x201,   // a device-resident position outside [0, max_seq)
    DEV_ATTN_GEOMETRY = 0x202,  // an attention work split outgrew its records or tables (skipped)
};

__device__ __forceinline__ void set_error(unsigned *err, unsigned code)
{
    if (err) atomicCAS(err, 0u, code);   // first error wins
}

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy accesses of shared memory before later async-proxy
// (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrival that counts `count` times (the phase completes when the arrivals of
// the phase add up to the count given at initialisation).
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, uint32_t limit = kWaitLimit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policy for data read once per step (the weight stream): its lines are
// evicted first, so streaming gigabytes through L2 does not push out what is
// reused (kernel code, activations, norm weights, the KV rows just written).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// bulk_g2s with an L2 cache policy (from createpolicy) for the source lines
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, unsigned bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
// The same with the destination as a shared-memory address.
__device__ __forceinline__ void bulk_g2s_u32(uint32_t dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled tensor copy (TMA) global -> shared: the box of the tensor map at
// element coordinates (x inner, y outer), completion counted on `bar` in bytes
// (the whole box, out-of-range parts zero-filled).  dst 128-byte aligned; the
// map a __grid_constant__ kernel parameter (or in global / constant memory).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// The same for a 3-D box at (x, y, z), without a cache hint.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Position in a ring of n slots, advanced one stage at a time: the slot and the
// parity of the slot's current phase (no division in the loops that walk it).
struct RingPos {
    int s;
    unsigned par;
};

__device__ __forceinline__ RingPos ring_pos(int64_t k, int n)
{
    return RingPos{(int)(k % n), (unsigned)((k / n) & 1)};
}

__device__ __forceinline__ void ring_next(RingPos &r, int n)
{
    if (++r.s == n) {
        r.s = 0;
        r.par ^= 1u;
    }
}

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: wait for the preceding kernel in the stream
// (no-op when launched without the attribute).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float h2f(uint16_t h)
{
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Q8_1 code of one value of a block with scale d: round half away from zero of
// the IEEE f32 quotient fl(x / d), clamped to [-127, 127]; 0 when d == 0 --
// exactly, without a division and without a branch.
//   y = |x| * rd (rd = rcp_approx(d), within 1 ulp of 1/d) lies within
//   127 (2^-22 + 2^-24) < 8e-5 of fl(|x| / d), because d = max|x| / 127 bounds the
//   quotient by 127 (1 + 2^-24).  So with k = floor(y) the code is k or k + 1 (the
//   quotient lies in (k - 1e-4, k + 1 + 1e-4)), and it is k + 1 exactly when
//   fl(|x| / d) >= h = k + 1/2.  Rounding is monotonic and h is a float whose last
//   significand bit is 0, so that holds exactly when |x| / d >= m = h - ulp(h) / 2
//   (at |x| / d == m the even neighbour, h, is chosen), i.e. when
//   t = |x| - h d >= -u, u = ulp(h) / 2 * d = d 2^(E - 24), E = floor(log2 h).
//   h d has at most 8 + 24 significant bits, so whenever t lies within a few u of
//   -u it is a small multiple of the grid of |x| and h d and the fused
//   multiply-add computes it exactly; further away its rounding cannot move it
//   across -u.  u is d scaled by a power of two (exact).
// Blocks with d < 2^-64 (1/d could overflow) scale x and d by 2^64 first: exact,
// and the quotient is unchanged.  Non-finite values give +-127.
// (An earlier form took rint(y) and formed the IEEE quotient out of line for the
// values next to a half-integer; the call in the loop cost the activation staging
// of a decode layer about 1.5 us, and an inline branch cost more.)

__device__ __forceinline__ float rcp_approx(float d)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

struct Q8Scale {
    float ds, rds, s;  // d * s, rcp_approx(d * s), s = 2^64 when d < 2^-64 else 1
    bool live;         // d != 0
};

__device__ __forceinline__ Q8Scale q8_scale(float d)
{
    Q8Scale q;
    q.live = d != 0.0f;
    q.s = d < 0x1p-64f ? 0x1p64f : 1.0f;
    q.ds = d * q.s;
    q.rds = rcp_approx(q.ds);
    return q;
}

__device__ __forceinline__ int q8_code(float x, const Q8Scale &q)
{
    const float ax = fabsf(x) * q.s;
    const float k = floorf(__fmul_rn(ax, q.rds));
    const float h = k + 0.5f;
    const float pw = __int_as_float((__float_as_int(h) & 0x7f800000) - (24 << 23));  // 2^(E - 24)
    const float u = __fmul_rn(q.ds, pw);
    const float t = __fmaf_rn(-h, q.ds, ax);
    const float c = fminf(t >= -u ? k + 1.0f : k, 127.0f);
    return q.live ? static_cast<int>(copysignf(c, x)) : 0;
}

// One activation row walked by 16 warps (512 threads): warp w owns the Q8_1
// blocks b = w, w + 16, w + 32, ... (at most kRowBlocksPerWarp of them) and lane l
// element 32 b + l of each.  Values at or beyond `n_valid` count as 0.  Loads are
// unrolled eight at a time so they are in flight together.
constexpr int kRowWarps = 16;
constexpr int kRowBlocksPerWarp = 32;  // rows up to 16384 values

// Activation loads.  CG = false takes the read-only path (data written before the
// kernel started); CG = true reads through L2 only, for data that other CTAs of
// the same kernel wrote (a persistent kernel after a grid barrier).
template <bool CG>
__device__ __forceinline__ float ld_act(const float *p)
{
    if constexpr (CG)
        return __ldcg(p);
    else
        return __ldg(p);
}

template <bool CG = false>
__device__ __forceinline__ float row_value(const float *x, int64_t nb, int64_t n_valid, int warp, int lane,
                                           int k)
{
    const int64_t b = warp + (int64_t)kRowWarps * k;
    const int64_t i = b * 32 + lane;
    return (b < nb && i < n_valid) ? ld_act<CG>(x + i) : 0.0f;
}

// Sum of squares of the row in a fixed order: per thread over its blocks in
// ascending block order, then the xor butterfly of each warp, then the butterfly
// over the 16 warp sums.  `red` holds 17 floats of shared memory; `sync`
// synchronises the 512 participating threads.  Every thread returns the total.
template <bool CG = false, typename Sync>
__device__ __forceinline__ float row_sumsq(const float *x, int64_t nb, int64_t n_valid, int warp, int lane,
                                           float *red, Sync sync)
{
    float ss = 0.0f;
#pragma unroll 8
    for (int k = 0; k < kRowBlocksPerWarp; ++k) {
        const float v = row_value<CG>(x, nb, n_valid, warp, lane, k);
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    sync();
    if (warp == 0) {
        float v = (lane < kRowWarps) ? red[lane] : 0.0f;
        v = warp_sum(v);
        if (lane == 0) red[kRowWarps] = v;
    }
    sync();
    const float total = red[kRowWarps];
    sync();  // red may be reused right after
    return total;
}

// RMSNorm scale 1 / sqrt(sum x^2 / n + eps) (rms_norm_inplace)
__device__ __forceinline__ float rms_scale(float sumsq, int64_t n, float eps)
{
    return 1.0f / sqrtf(sumsq / (float)n + eps);
}

}  // namespace rz
