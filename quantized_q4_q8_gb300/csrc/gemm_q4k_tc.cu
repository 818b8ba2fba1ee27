// gemm_q4k_tc.cu -- the Q4_K x Q8_1 projection of many tokens at once (the
// prompt of GpuModelQ4::forward in realizar 0.8.4 src/gpu/adapters/using.rs
// arrives as a sequence of token ids) on the fifth-generation tensor cores:
// tcgen05.mma, accumulators in tensor memory, operands in shared memory.
//
// The product is the one of the decode GEMV (q4k_q8_gemv_async in realizar 0.8.5
// src/cuda/executor/cached.rs, transformer_layer_gpu_true_dp4a):
//   y[t][r] = sum_b [ d_b sum_j sc_bj d8_tbj I_tbrj - dmin_b sum_j m_bj s_tbj ]
// with I the exact integer dot of the 32 codes of sub-block j.
//
// Exactness on the tensor cores.  A holds the activation codes (|q8| <= 127) as
// f16 and B the products sc * q (<= 63 * 15 = 945) as f16, both exact; one
// sub-block (K = 32) sums to at most 945 * 127 * 32 < 2^24, so the f32 accumulator
// holds sc_bj * I_tbrj exactly.  d8 changes with the token and the sub-block, so
// every sub-block is accumulated into a region of its own and scaled on the CUDA
// cores as it drains.  The min term sum_j m_bj s_tbj is a ninth product per
// super-block in bf16: the 6-bit mins against s split exactly into three bf16
// pieces (s = s1 + s2 + s3, 8 significant bits each).
//
// Tile: 128 tokens (MMA M = tensor-memory lanes) x 128 weight rows (MMA N =
// columns); K walks the super-blocks, nine regions of K = 32 each (region
// g = 9 sb + j).  Every synchronising instruction (an mbarrier wait, an MMA
// issue, a commit) costs a warp on the order of a hundred cycles here while one
// region is 128 cycles of tensor work, so the work of a region is spread over
// warps that run side by side, each region's steps on its own warp:
//   warps 0-2    MMA: warp b issues the regions g = b mod 3 into tensor-memory
//                buffer b and frees the region's operand slots by a commit
//                (warp 0 also allocates tensor memory)
//   warp 3       copies: the bulk copy of every region's activation operand and
//                the TMA load of every raw Q4_K tile (one per super-block)
//   warps 4-7    conversion: warp c converts the regions g = c mod 4 (all 128
//                rows, four in flight per lane) into the B operand
//   warps 8-23   drain: region -> registers, times d8 (sub-block) and d, dmin
//                (super-block); the running sums stay in tensor memory
// Shared-memory operand layout: K-major core matrices of 8 rows x 16 bytes, no
// swizzle; the two core matrices along K 128 bytes apart, 8-row groups 512 bytes
// apart (one 128 x 32 operand = 8 KiB).  Within every 4 consecutive K slots both
// operands hold elements (0, 2, 1, 3) of the sub-block: the order in which a
// 32-bit word of packed nibbles unpacks into two f16 pairs; the dot is the same.
//
// Every wait is bounded; on a timeout the CTA records DEV_TIMEOUT_GEMM, every
// role stops, the copies and MMAs in flight are waited for (bounded), tensor
// memory is freed and the CTA exits.
#include <algorithm>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kTM = 128;                  // tokens per tile
constexpr int kTN = 128;                  // weight rows per tile
constexpr int kRegions = 9;               // per super-block: 8 sub-blocks + the min term
constexpr int kOpBytes = 8192;            // one 128 x 32 operand of 16-bit values
constexpr int kStages = 8;                // operand slots (A and B each), region g in slot g % 8
constexpr int kStagesW = 3;               // raw Q4_K tiles
constexpr int kStagesH = 2;               // d, dmin of the tile's rows
constexpr int kTBufs = 3;                 // region buffers in tensor memory = MMA warps
constexpr int kAccCol = kTBufs * kTN;     // columns 384..511: the running sums
constexpr int kMmaWarps = kTBufs;
constexpr int kLoadWarp = kMmaWarps;      // warp 3
constexpr int kFirstConv = kLoadWarp + 1; // warps 4-7
constexpr int kConvWarps = 4;
constexpr int kFirstDrain = kFirstConv + kConvWarps;  // warps 8-23
constexpr int kDrainWarps = 16;
constexpr int kThreads = 32 * (kFirstDrain + kDrainWarps);
constexpr int kWBytes = 144 * kTN;        // raw Q4_K of one super-block of the tile

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kOpBytes;
constexpr int kOffW = kOffB + kStages * kOpBytes;
constexpr int kOffH = kOffW + kStagesW * kWBytes;
constexpr int kOffBar = kOffH + kStagesH * kTN * 8;
constexpr int kNumBars = 3 * kStages + 2 * kStagesW + 2 * kTBufs + 2 * kStagesH + kMmaWarps;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack

static_assert(kOffW % 1024 == 0 && kWBytes % 128 == 0, "TMA destinations 128-byte aligned");
static_assert(kStages % kConvWarps == 0, "a conversion warp's regions cycle through its own slots");

// instruction descriptors (kind::f16): D f32 (bits 4-5 = 1), A and B K-major,
// N >> 3 at bits 17-22, M >> 4 at bits 24-28; bf16 operands: bits 7-9 and 10-12 = 1
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(kTN >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
constexpr uint32_t kIdescBF16 = kIdescF16 | (1u << 7) | (1u << 10);

struct GemmArgs {
    CUtensorMap wmap;     // Q4_K bytes [out_dim][row_bytes], box 144 x 128
    const uint8_t *pack;  // activation operands [token tiles][regions][8 KiB]
    const float *d8;      // Q8_1 block scales [m][in_dim / 32]
    float *y;
    int64_t ldy;
    int m, out_dim, nsb;
    unsigned *err;
    uint32_t wait_limit;
};

// ---------------------------------------------------------------- tcgen05 wrappers
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr)
{
    // start address >> 4 (bits 0-13), leading byte offset 128 >> 4 (bits 16-29),
    // stride byte offset 512 >> 4 (bits 32-45), descriptor version 1 (bit 46),
    // base offset 0, no swizzle
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(512 >> 4) << 32) |
           (1ull << 46);
}

__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define RZ_R16(b)                                                                                                    \
    "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), \
        "=r"(r[b + 7]), "=r"(r[b + 8]), "=r"(r[b + 9]), "=r"(r[b + 10]), "=r"(r[b + 11]), "=r"(r[b + 12]),          \
        "=r"(r[b + 13]), "=r"(r[b + 14]), "=r"(r[b + 15])

// Consecutive columns of this warp's 32 lanes (one value per thread and column),
// waited for inside the same statement so no use can move above the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : RZ_R16(0)
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
        : "memory");
}

// a += b * c on two f32 lanes at once (fma.rn.f32x2)
__device__ __forceinline__ void fma2(float &a0, float &a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\tmov.b64 rc, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, rb, rc, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// mbarrier wait that lets the thread sleep until the phase completes (or the
// 20 us hint runs out), instead of spinning on the barrier
__device__ __forceinline__ bool try_wait_sleep(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase: issued early, its result is read later, so its
// latency overlaps other work.
__device__ __forceinline__ bool test_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Warp-wide bounded wait: every lane waits, the verdict is made uniform.  A
// timeout, or an abort raised by another role, returns false.  Each try lasts
// at most the 20 us hint, so the bound is a 64th of the poll limit in tries.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, unsigned par, const GemmArgs &a, volatile int *abort_flag)
{
    bool ok = false;
    for (uint32_t i = 0; i < (a.wait_limit >> 6); ++i) {
        if (try_wait_sleep(bar, par)) {
            ok = true;
            break;
        }
        if (*abort_flag) break;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0 && !*abort_flag) {
        *abort_flag = 1;
        set_error(a.err, DEV_TIMEOUT_GEMM);
    }
    return ok;
}

// byte offset of row `row`, 16-byte chunk `kk` (K slots 8 kk .. 8 kk + 7) of an operand
__device__ __forceinline__ int op_offset(int row, int kk) { return (row >> 3) * 512 + kk * 128 + (row & 7) * 16; }

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// 6-bit scale / min of sub-block j from header bytes 4-15 (s0-3 in y, s4-7 in z,
// s8-11 in w)
__device__ __forceinline__ int q4k_scale(const uint4 &h, int j)
{
    const int k = j & 3;
    const int b0 = (int)((h.y >> (8 * k)) & 0xFFu), b8 = (int)((h.w >> (8 * k)) & 0xFFu);
    return j < 4 ? (b0 & 63) : ((b8 & 15) | ((b0 >> 6) << 4));
}
__device__ __forceinline__ int q4k_min(const uint4 &h, int j)
{
    const int k = j & 3;
    const int b4 = (int)((h.z >> (8 * k)) & 0xFFu), b8 = (int)((h.w >> (8 * k)) & 0xFFu);
    return j < 4 ? (b4 & 63) : ((b8 >> 4) | ((b4 >> 6) << 4));
}

__global__ void __launch_bounds__(kThreads, 1) q4k_gemm_tc_kernel(const __grid_constant__ GemmArgs a)
{
    extern __shared__ uint8_t gsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *full_a = bars, *full_b = full_a + kStages, *empty_ab = full_b + kStages;
    uint64_t *full_w = empty_ab + kStages, *empty_w = full_w + kStagesW;
    uint64_t *full_t = empty_w + kStagesW, *empty_t = full_t + kTBufs;
    uint64_t *full_h = empty_t + kTBufs, *empty_h = full_h + kStagesH;
    uint64_t *done_bar = empty_h + kStagesH;  // one per MMA warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    float *hdr = reinterpret_cast<float *>(sm + kOffH);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * kTN, tile_t = blockIdx.y;
    const int nsb = a.nsb, G = nsb * kRegions;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_a[i], 1);    // the bulk copy's arrive.expect_tx
            mbar_init(&full_b[i], 1);    // the converting warp
            mbar_init(&empty_ab[i], 1);  // the commit after the region's MMAs
        }
        for (int i = 0; i < kStagesW; ++i) {
            mbar_init(&full_w[i], 1);
            mbar_init(&empty_w[i], kRegions);  // one arrival per region converted from it
        }
        for (int i = 0; i < kTBufs; ++i) {
            mbar_init(&full_t[i], 1);
            mbar_init(&empty_t[i], kDrainWarps);
        }
        for (int i = 0; i < kStagesH; ++i) {
            mbar_init(&full_h[i], 1);
            mbar_init(&empty_h[i], kDrainWarps);
        }
        for (int i = 0; i < kMmaWarps; ++i) mbar_init(&done_bar[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&a.wmap);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kMmaWarps) {
        // ------------------------------------------------------------ MMA issue
        const int b = warp;
        const uint32_t d = tmem + (uint32_t)(b * kTN);
        int issued = 0;
        for (int g = b; g < G; g += kTBufs) {
            const RingPos ps = ring_pos(g, kStages);
            const RingPos pt = ring_pos(g / kTBufs, 1);  // parity of this buffer's use
            // the three phases tested together (one latency); only a phase not yet
            // complete is waited for
            const bool ra = test_wait(&full_a[ps.s], ps.par);
            const bool rb = test_wait(&full_b[ps.s], ps.par);
            const bool rt = test_wait(&empty_t[b], pt.par ^ 1u);
            if (!__all_sync(0xffffffffu, ra && rb && rt)) {
                if (!warp_wait(&full_a[ps.s], ps.par, a, abort_flag)) break;
                if (!warp_wait(&full_b[ps.s], ps.par, a, abort_flag)) break;
                if (!warp_wait(&empty_t[b], pt.par ^ 1u, a, abort_flag)) break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sa = smem_u32(sm + kOffA + ps.s * kOpBytes);
                const uint32_t sb_ = smem_u32(sm + kOffB + ps.s * kOpBytes);
                const uint32_t idesc = (g % kRegions == 8) ? kIdescBF16 : kIdescF16;
#pragma unroll
                for (int h = 0; h < 2; ++h)  // K = 16 each: core matrices 2h, 2h + 1 along K
                    mma_issue(d, kmajor_desc(sa + 256u * h), kmajor_desc(sb_ + 256u * h), idesc, (uint32_t)h);
                mma_commit(&empty_ab[ps.s]);
                mma_commit(&full_t[b]);
            }
            __syncwarp();
            ++issued;
        }
        // every MMA this warp issued has completed once this arrives
        if (lane == 0) {
            mma_commit(&done_bar[b]);
            mbar_wait(&done_bar[b], 0, a.wait_limit);
        }
        __syncwarp();
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------ copies
        const uint64_t pol = l2_evict_first_policy();
        const uint8_t *pack_tile = a.pack + (int64_t)tile_t * G * kOpBytes;
        int w_issued = 0, a_issued = 0;
        auto issue_w = [&](int sbk) {  // raw tile sbk into slot sbk % 3 once its regions are converted
            const RingPos p = ring_pos(sbk, kStagesW);
            if (!warp_wait(&empty_w[p.s], p.par ^ 1u, a, abort_flag)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full_w[p.s], kWBytes);
                tma_load_2d(sm + kOffW + p.s * kWBytes, &a.wmap, sbk * 144, r0, &full_w[p.s], pol);
            }
            __syncwarp();
            ++w_issued;
            return true;
        };
        bool ok = true;
        for (int k = 0; k < min(kStagesW - 1, nsb) && ok; ++k) ok = issue_w(k);
        for (int g = 0; g < G && ok; ++g) {
            // the raw tile two super-blocks ahead, at the first region of each super-block
            if (g % kRegions == 0 && w_issued < nsb && !(ok = issue_w(w_issued))) break;
            const RingPos p = ring_pos(g, kStages);
            if (!warp_wait(&empty_ab[p.s], p.par ^ 1u, a, abort_flag)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full_a[p.s], kOpBytes);
                bulk_g2s(sm + kOffA + p.s * kOpBytes, pack_tile + (int64_t)g * kOpBytes, kOpBytes, &full_a[p.s]);
            }
            __syncwarp();
            ++a_issued;
        }
        // copies in flight must land before the CTA exits: the last phase issued
        // into every slot
        if (lane == 0) {
            for (int k = max(0, w_issued - kStagesW); k < w_issued; ++k) {
                const RingPos p = ring_pos(k, kStagesW);
                mbar_wait(&full_w[p.s], p.par, a.wait_limit);
            }
            for (int k = max(0, a_issued - kStages); k < a_issued; ++k) {
                const RingPos p = ring_pos(k, kStages);
                mbar_wait(&full_a[p.s], p.par, a.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp < kFirstDrain) {
        // ------------------------------------------------------------ conversion
        const int c = warp - kFirstConv;
        for (int g = c; g < G; g += kConvWarps) {
            const int sbk = g / kRegions, j = g - kRegions * sbk;
            const RingPos pw = ring_pos(sbk, kStagesW);
            const RingPos ps = ring_pos(g, kStages);
            if (!warp_wait(&full_w[pw.s], pw.par, a, abort_flag)) break;
            if (!warp_wait(&empty_ab[ps.s], ps.par ^ 1u, a, abort_flag)) break;
            const uint8_t *wtile = sm + kOffW + pw.s * kWBytes;
            uint8_t *dst = sm + kOffB + ps.s * kOpBytes;
            if (j < 8) {
                // sub-block j: the low (j even) or high (j odd) nibbles of bytes
                // 32 (j / 2) .. + 31; q * sc exactly as (1024 + q) * sc - 1024 * sc, or
                // (1024 + 16 q) * (sc / 16) - 64 * sc, one rounding of an exact small
                // integer
                const int hi = j & 1;
                const uint32_t mask = hi ? 0x00F000F0u : 0x000F000Fu;
#pragma unroll
                for (int rr = 0; rr < kTN / 32; ++rr) {
                    const int row = 32 * rr + lane;
                    const uint8_t *raw = wtile + row * 144;
                    const uint4 h0 = *reinterpret_cast<const uint4 *>(raw);
                    const uint4 qa = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * (j >> 1));
                    const uint4 qb = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * (j >> 1));
                    const int s6 = q4k_scale(h0, j);
                    const __half2 mul = __float2half2_rn(hi ? (float)s6 * 0.0625f : (float)s6);
                    const __half2 add = __float2half2_rn(hi ? -64.0f * (float)s6 : -1024.0f * (float)s6);
                    const uint32_t wv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t o[4];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint32_t wi = wv[2 * kk + u];
                            const uint32_t e02 = (wi & mask) | 0x64006400u;         // elements 4i, 4i + 2
                            const uint32_t e13 = ((wi >> 8) & mask) | 0x64006400u;  // elements 4i + 1, 4i + 3
                            o[2 * u] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&e02), mul, add));
                            o[2 * u + 1] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&e13), mul, add));
                        }
                        *reinterpret_cast<uint4 *>(dst + op_offset(row, kk)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            } else {
                // the min-term operand: m_0..7 in K slots 0-7, 8-15 and 16-23 (against
                // the three bf16 pieces of s), zeros in 24-31; and d, dmin of every
                // row for the drain
                const RingPos ph = ring_pos(sbk, kStagesH);
                if (!warp_wait(&empty_h[ph.s], ph.par ^ 1u, a, abort_flag)) break;
#pragma unroll 1
                for (int rr = 0; rr < kTN / 32; ++rr) {
                    const int row = 32 * rr + lane;
                    const uint4 h0 = *reinterpret_cast<const uint4 *>(wtile + row * 144);
                    uint32_t mm[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)  // bf16 of a 6-bit integer: the top half of its f32
                        mm[i] = (__float_as_uint((float)q4k_min(h0, 2 * i)) >> 16) |
                                (__float_as_uint((float)q4k_min(h0, 2 * i + 1)) & 0xFFFF0000u);
#pragma unroll
                    for (int kk = 0; kk < 3; ++kk)
                        *reinterpret_cast<uint4 *>(dst + op_offset(row, kk)) = make_uint4(mm[0], mm[1], mm[2], mm[3]);
                    *reinterpret_cast<uint4 *>(dst + op_offset(row, 3)) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<float2 *>(hdr + ph.s * kTN * 2 + row * 2) =
                        make_float2(h2f((uint16_t)(h0.x & 0xffffu)), h2f((uint16_t)(h0.x >> 16)));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full_h[ph.s]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_b[ps.s]);
                mbar_arrive(&empty_w[pw.s]);
            }
        }
    } else {
        // ------------------------------------------------------------ drain
        const int q = warp & 3;                      // tensor-memory lanes 32q .. 32q + 31
        const int cg = (warp - kFirstDrain) >> 2;    // columns 32cg .. 32cg + 31 of a region
        const int tl = 32 * q + lane;                // token within the tile
        const int64_t t = (int64_t)tile_t * kTM + tl;
        const bool tok = t < a.m;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t acc_addr = tmem + lane_base + (uint32_t)(kAccCol + 32 * cg);
        const float *d8row = a.d8 + (tok ? t : 0) * (int64_t)(nsb * 8);
        float acc_sb[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc_sb[i] = 0.0f;
        RingPos pt{0, 0}, ph{0, 0};
        bool ok = true, ready = false;  // ready: region g known complete
        int g = 0;
        for (int sbk = 0; sbk < nsb && ok; ++sbk) {
            float4 dn0 = make_float4(0.f, 0.f, 0.f, 0.f), dn1 = dn0;
            if (tok) {
                dn0 = __ldg(reinterpret_cast<const float4 *>(d8row + 8 * sbk));
                dn1 = __ldg(reinterpret_cast<const float4 *>(d8row + 8 * sbk + 4));
            }
            const float d8[8] = {dn0.x, dn0.y, dn0.z, dn0.w, dn1.x, dn1.y, dn1.z, dn1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (!ready && !warp_wait(&full_t[pt.s], pt.par, a, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t src = tmem + lane_base + (uint32_t)(pt.s * kTN + 32 * cg);
                const float dj = d8[j];
                RingPos pn = pt;
                ring_next(pn, kTBufs);
                float v[16];
                tmem_ld16(src, v);
                const bool nxt = test_wait(&full_t[pn.s], pn.par);  // region g + 1, read at the end
#pragma unroll
                for (int i = 0; i < 16; i += 2) fma2(acc_sb[i], acc_sb[i + 1], v[i], v[i + 1], dj, dj);
                tmem_ld16(src + 16, v);
#pragma unroll
                for (int i = 0; i < 16; i += 2) fma2(acc_sb[16 + i], acc_sb[16 + i + 1], v[i], v[i + 1], dj, dj);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_t[pt.s]);
                pt = pn;
                ++g;
                ready = __all_sync(0xffffffffu, nxt);
            }
            if (!ok) break;
            // the min-term region: acc += d * acc_sb - dmin * mins, the running sums in
            // tensor memory
            if ((!ready && !warp_wait(&full_t[pt.s], pt.par, a, abort_flag)) ||
                !warp_wait(&full_h[ph.s], ph.par, a, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *hrow = hdr + ph.s * kTN * 2 + 64 * cg;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                float mins[8], accv[8];
                tmem_ld8(tmem + lane_base + (uint32_t)(pt.s * kTN + 32 * cg + 8 * qq), mins);
                if (sbk > 0) {
                    tmem_ld8(acc_addr + 8 * qq, accv);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) accv[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const float4 hd = *reinterpret_cast<const float4 *>(hrow + 2 * (8 * qq + i));
                    fma2(accv[i], accv[i + 1], acc_sb[8 * qq + i], acc_sb[8 * qq + i + 1], hd.x, hd.z);
                    fma2(accv[i], accv[i + 1], mins[i], mins[i + 1], -hd.y, -hd.w);
                }
                tmem_st8(acc_addr + 8 * qq, accv);
            }
            RingPos pn = pt;
            ring_next(pn, kTBufs);
            const bool nxt = test_wait(&full_t[pn.s], pn.par);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty_t[pt.s]);
                mbar_arrive(&empty_h[ph.s]);
            }
            pt = pn;
            ring_next(ph, kStagesH);
            ++g;
            ready = __all_sync(0xffffffffu, nxt);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc_sb[i] = 0.0f;
        }
        if (ok && !*abort_flag) {
            // epilogue: y[t][r0 + 32cg + c]
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float accv[16];
                tmem_ld16(acc_addr + 16 * half, accv);
                const int rb = r0 + 32 * cg + 16 * half;
                if (tok) {
                    float *yr = a.y + t * a.ldy + rb;
                    if (rb + 16 <= a.out_dim && ((reinterpret_cast<uintptr_t>(yr) & 15) == 0)) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(yr + i) = make_float4(accv[i], accv[i + 1], accv[i + 2], accv[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (rb + i < a.out_dim) yr[i] = accv[i];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// Activation operands: region g = 9 sb + j of token tile T is 8 KiB at
// pack + (T * G + g) * 8 KiB in the operand layout above.  j < 8: the codes of
// block 8 sb + j as f16 in the K order (0, 2, 1, 3) per 4; j = 8: the three bf16
// pieces of s of the super-block's 8 blocks in K slots 0-7, 8-15, 16-23, zeros
// after.  Tokens beyond m are zero.
__global__ void __launch_bounds__(128) q8_pack_tc_kernel(const int8_t *__restrict__ q, const float *__restrict__ s,
                                                         uint8_t *__restrict__ pack, int m, int in_dim, int G)
{
    const int g = blockIdx.x, tile = blockIdx.y, tl = threadIdx.x;
    const int sb = g / kRegions, j = g - kRegions * sb;
    const int64_t t = (int64_t)tile * kTM + tl;
    const int nb = in_dim / 32;
    uint8_t *out = pack + ((int64_t)tile * G + g) * kOpBytes;
    uint32_t o[16];
    if (j < 8) {
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        if (t < m) {
            const uint4 *src = reinterpret_cast<const uint4 *>(q + t * in_dim + (int64_t)(sb * 8 + j) * 32);
            c0 = __ldg(src);
            c1 = __ldg(src + 1);
        }
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b0 = (int)(int8_t)(w[i] & 0xFFu), b1 = (int)(int8_t)((w[i] >> 8) & 0xFFu);
            const int b2 = (int)(int8_t)((w[i] >> 16) & 0xFFu), b3 = (int)(int8_t)(w[i] >> 24);
            o[2 * i] = h2_bits(__halves2half2(__int2half_rn(b0), __int2half_rn(b2)));
            o[2 * i + 1] = h2_bits(__halves2half2(__int2half_rn(b1), __int2half_rn(b3)));
        }
    } else {
        uint32_t p1[8], p2[8], p3[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float sv = (t < m) ? __ldg(s + t * nb + sb * 8 + i) : 0.0f;
            // s = s1 + s2 + s3 exactly: the top 8 significant bits, the next 8, the rest
            const uint32_t u1 = __float_as_uint(sv) & 0xFFFF0000u;
            const float r1 = sv - __uint_as_float(u1);
            const uint32_t u2 = __float_as_uint(r1) & 0xFFFF0000u;
            const float r2 = r1 - __uint_as_float(u2);
            p1[i] = u1 >> 16;
            p2[i] = u2 >> 16;
            p3[i] = __float_as_uint(r2) >> 16;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[i] = p1[2 * i] | (p1[2 * i + 1] << 16);
            o[4 + i] = p2[2 * i] | (p2[2 * i + 1] << 16);
            o[8 + i] = p3[2 * i] | (p3[2 * i + 1] << 16);
            o[12 + i] = 0u;
        }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        *reinterpret_cast<uint4 *>(out + op_offset(tl, kk)) = make_uint4(o[4 * kk], o[4 * kk + 1], o[4 * kk + 2], o[4 * kk + 3]);
}

}  // namespace

int64_t q4k_gemm_tc_workspace_bytes(int64_t m, int64_t in_dim)
{
    return ((m + kTM - 1) / kTM) * (in_dim / 256) * kRegions * (int64_t)kOpBytes;
}

int q4k_gemm_tc_launch_count() { return 2; }

cudaError_t launch_q4k_gemm_tc(const void *w, const void *q8, float *y, int64_t ldy, int64_t m, int64_t out_dim,
                               int64_t in_dim, void *workspace, cudaStream_t s)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    if ((size_t)kSmemBytes > dev_info().smem_optin) return cudaErrorInvalidConfiguration;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const int nsb = (int)(in_dim / 256);
    const int G = nsb * kRegions;
    const int tiles_t = (int)((m + kTM - 1) / kTM);
    const int8_t *xq = static_cast<const int8_t *>(q8);
    const float *xd = reinterpret_cast<const float *>(static_cast<const uint8_t *>(q8) + m * in_dim);
    const float *xs = xd + m * (in_dim / 32);
    uint8_t *pack = static_cast<uint8_t *>(workspace);

    q8_pack_tc_kernel<<<dim3(G, tiles_t), 128, 0, s>>>(xq, xs, pack, (int)m, (int)in_dim, G);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    GemmArgs a = {};
    const int64_t row_bytes = (int64_t)nsb * 144;
    e = encode_tensor_map_2d(&a.wmap, w, 1, (uint64_t)row_bytes, (uint64_t)out_dim, (uint64_t)row_bytes, 144u,
                             (uint32_t)kTN);
    if (e != cudaSuccess) return e;
    a.pack = pack;
    a.d8 = xd;
    a.y = y;
    a.ldy = ldy;
    a.m = (int)m;
    a.out_dim = (int)out_dim;
    a.nsb = nsb;
    a.err = dev_error_word();
    a.wait_limit = kWaitLimit;
    const dim3 grid((unsigned)((out_dim + kTN - 1) / kTN), (unsigned)tiles_t);
    q4k_gemm_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace rz

