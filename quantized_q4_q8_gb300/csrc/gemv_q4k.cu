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
// producer warp keeps a ring of two shared-memory stages (each about half of
// what the activations leave) full with the 1-D bulk copy engine
// (cp.async.bulk in copies of at most 12 KB, completion counted on an
// mbarrier), so the bytes in flight live in shared memory, not registers.  (Prefetching the rest
// of the CTA's rows into L2 up front was measured slower: it queues ahead of
// the ring's own copies and of the activation loads.)  A stage
// holds whole "packs" (one row, or 8/nsb rows when a row has fewer than 8
// super-blocks); pack i goes to consumer warp i % 15.  Every consumer warp
// passes every stage in order -- waits for it, works its own packs in it,
// releases the slot with one arrival -- so no warp can get a ring length ahead
// of a stage that has not been filled (the parity waits stay unambiguous), and
// a stage is refilled once all fifteen have passed it.  Within a pack each
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

#include "q4k_dot.cuh"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

// Consumer warps and shared-memory budget per CTA, for several tokens and for one
// (a one-token CTA of 8 warps in <= 110 KB, two per SM so that the next kernel's
// CTA streams its weights beside this one, measured slower: 9.8 us against 8.9
// for 4096 x 14336, 2.32 ms against 1.71 for the decode step).  15 consumer warps
// and the producer make 16 warps, four per SM sub-partition, so that a thread may
// hold 128 registers; with 16 consumers one sub-partition holds five warps and
// the limit is 96 (the staging loops spilled there; decode step 1.491 -> 1.478 ms).
// One token on CTAs whose work splits better over 16 warps (16 packs of short
// rows: the Qwen2-shaped gate/up, 26.9 -> 25.8 us per layer) takes a 16-warp
// instantiation instead (nw_for below).
constexpr int kConsumerWarps = 15;
constexpr int kCtaSmem = 200 * 1024;
constexpr int kCtaSmem1 = 200 * 1024;
constexpr int kXSmemMax = 128 * 1024;  // activations staged up to this size (the ring keeps >= 70 KB)
constexpr int kMaxStages = 16;
// Bytes per bulk copy of a stage's rows (whole rows, at least one; the row
// count is worked out on the host: left as a 64-bit division inside the
// producer loop, it slowed the step by 9%).  Measured on the 32-layer decode step against
// one copy per contiguous run of rows (about 90 KB per stage): rows of 2304
// bytes copied 5 at a time and rows of 6192 bytes one at a time, 1.471 -> 1.406
// ms; 2, 3 or 4 rows of 2304 bytes at a time (the 6192-byte rows one at a
// time): +5.2%, -0.4%, -3.7%; 6192-byte rows two or three at a time (the short
// rows five at a time): -0.2%, +0.8%.  A CTA whose rows fit one stage (the
// 4096 x 4096 projection: 27 rows) copies them whole: 1.408 -> 1.402 ms.
// The SwiGLU pair keeps a copy per row and half: its gate and up rows
// interleaved pack by pack beat both halves laid out in blocks of rows, copied
// whole (+1.7%) or 8-16 KB at a time (+2.8%).
constexpr int64_t kCopyBytes = 12 * 1024;

struct Args {
    const uint8_t *w[3];
    float *y[3];
    const float *res[3];   // residual (EPI_RESID), or bias (EPI_STORE, ldr 0), or nullptr
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
    int copy_rows;         // rows per bulk copy (kCopyBytes of whole rows, at least one)
    int x_smem;            // activations staged (swizzled) in shared memory
    // f32 input quantised in the kernel (XIN_NORM / XIN_F32)
    const float *xf;
    int64_t ldxf;
    const float *gamma;
    int64_t norm_n;
    float eps;
    unsigned *err;
    // test aid (rz_debug_stall_next_gemv): in CTA 0 the stage stall_stage is never
    // issued and every wait polls at most wait_limit times; -1 / unused otherwise
    int stall_stage;
    uint32_t wait_limit;
    // zero padding of the output: y[0][t * zy_ld + zy_from + j] = 0 for j < zy_cnt,
    // written by the last CTA (segment 0 only)
    float *zy;
    int64_t zy_ld, zy_from, zy_cnt;
};

enum XIn { XIN_Q8 = 0, XIN_NORM = 1, XIN_F32 = 2 };

__device__ __forceinline__ int seg_of(const Args &a, int64_t unit)
{
    int k = 0;
    while (k + 1 < a.nseg && unit >= a.seg_begin[k + 1]) ++k;
    return k;
}

// PR: several tokens with the rows in pairs (a separate instantiation, so that
// its register allocation does not touch the one-row-per-warp path)
template <int MT, int EPI, bool XS, int XIN, bool PR, int NW>
__global__ void __launch_bounds__((NW + 1) * 32, 1) q4k_gemv_kernel(const Args a)
{
    constexpr int kConsumerWarps = NW;
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
            mbar_init(&empty[s], kConsumerWarps);  // one arrival per consumer warp
        }
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel may become resident now: its weights stream while we drain
    pdl_launch_dependents();

    // the stall test aid applies to CTA 0 only; every other CTA runs as usual
    const int stall = (blockIdx.x == 0) ? a.stall_stage : -1;
    const uint32_t lim = (stall >= 0) ? a.wait_limit : kWaitLimit;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int64_t k = 0;
            bool ok = true;
            RingPos rp{0, 0u};
            // rows per copy; a CTA whose rows fit one stage copies each run whole
            const int crows = nstages == 1 ? 0x7fffffff : a.copy_rows;
            for (; k < nstages; ++k, ring_next(rp, a.NS)) {
                const int s = rp.s;
                if (k >= a.NS && !mbar_wait(&empty[s], rp.par ^ 1u, lim)) {
                    set_error(a.err, DEV_TIMEOUT_GEMV);
                    ok = false;
                    break;
                }
                if (k == stall) continue;  // never issued: the consumers' wait runs out
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
                        bulk_g2s_hint(pd, a.w[0] + u * a.row_bytes, (unsigned)(nr * a.row_bytes), &full[s], pol);
                        bulk_g2s_hint(pd + pack_bytes, a.w[1] + u * a.row_bytes, (unsigned)(nr * a.row_bytes),
                                 &full[s], pol);
                    }
                } else {
                    int r = 0;
                    while (r < n) {
                        const int64_t u = u0 + r;
                        const int kseg = seg_of(a, u);
                        const int run = (int)min((int64_t)min(n - r, crows), a.seg_begin[kseg + 1] - u);
                        bulk_g2s_hint(dst + (int64_t)r * a.row_bytes,
                                 a.w[kseg] + (u - a.seg_begin[kseg]) * a.row_bytes,
                                 (unsigned)(run * a.row_bytes), &full[s], pol);
                        r += run;
                    }
                }
            }
            // drain: stages issued but possibly not complete must land before exit
            // (the consumers may have given up on them)
            if (!ok || stall >= 0) {
                for (int64_t q = (k > a.NS ? k - a.NS : 0); q < k; ++q)
                    if (q != stall && !mbar_wait(&full[q % a.NS], (unsigned)((q / a.NS) & 1)))
                        set_error(a.err, DEV_TIMEOUT_DRAIN);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // activations and the output buffers belong to the previous kernel: wait for
    // it (inside the f32 staging, after its loads of the weights it needs)
    constexpr bool kF32Stage = XS && XIN != XIN_Q8;
    if (!kF32Stage) pdl_wait();
    XSrc x;
    x.in_dim = a.in_dim;
    x.nb = a.in_dim / 32;
    x.m = a.m;
    x.gq = a.xq;
    x.gd = a.xd;
    x.gs = a.xs;
    auto csync = [] { asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory"); };
    if (XS && XIN == XIN_Q8)
        stage_x_q8<false, kConsumerWarps>(xsm, a.xq, a.xd, a.xs, a.m, a.in_dim, threadIdx.x, csync);
    if (XS && XIN != XIN_Q8) {
        // quantise the f32 input (RMS-normalised first for XIN_NORM) straight into
        // the padded slot layout
        float *red = reinterpret_cast<float *>(full) - 24;  // 17 floats below the barriers
        stage_x_f32<false, XIN == XIN_NORM, kConsumerWarps>(xsm, a.xf, a.ldxf, a.gamma, a.norm_n, a.eps, a.m,
                                                            a.in_dim, red, warp, lane, csync, [] { pdl_wait(); });
    }
    if (a.zy && blockIdx.x == gridDim.x - 1)
        for (int64_t i = threadIdx.x; i < (int64_t)a.m * a.zy_cnt; i += kConsumerWarps * 32)
            a.zy[(i / a.zy_cnt) * a.zy_ld + a.zy_from + i % a.zy_cnt] = 0.0f;
    if (XS) {
        const int64_t nsbx = (int64_t)a.m * (a.in_dim / 256);
        x.q = smem_u32(xsm);
        x.ds = smem_u32(xsm + nsbx * kXSlot);
    }

    const int g = lane >> 2;
    const int seg_lanes = (a.rpp > 1) ? 4 * a.nsb : 32;
    const int rip = (a.rpp > 1) ? g / a.nsb : 0;  // row of the pack this group works on
    const int leader = lane % seg_lanes == 0;
    const uint32_t ring_s = smem_u32(ring);

    // Every consumer warp passes every stage in order (waits for it, takes its own
    // packs -- pack i goes to warp i % 15 -- and releases the slot once), so no
    // warp can run a ring length ahead of a stage that is not filled yet and the
    // parity waits stay unambiguous.
    RingPos rp{0, 0u};
    const int npk = (int)npacks, PS = a.PS, pps = (PS + 1) / 2;  // packs and pairs per stage
    int prot = 0, rot = 0;  // pairs / packs of the earlier stages, modulo the warp count
    for (int k = 0; k < (int)nstages; ++k, ring_next(rp, a.NS)) {
        const int s = rp.s;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], rp.par, lim));
        if (!ok) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_GEMV);
            return;
        }
        const int first = k * PS, end = min(first + PS, npk);
        const uint32_t slot = ring_s + (uint32_t)(s * a.stage_bytes);
        const int q0 = (warp - prot + kConsumerWarps) % kConsumerWarps, i0 = (warp - rot + kConsumerWarps) % kConsumerWarps;
        prot += pps;
        while (prot >= kConsumerWarps) prot -= kConsumerWarps;
        rot += PS;
        while (rot >= kConsumerWarps) rot -= kConsumerWarps;
        if (MT == 1 && XS && a.rpp == 1) {
            // rows in pairs: pair q of the stage (packs first + 2q, first + 2q + 1)
            // goes to warp (pairs of earlier stages + q) % 15
            const int npair = (end - first + 1) / 2;
            for (int q = q0; q < npair; q += kConsumerWarps) {
                const int iA = first + 2 * q;
                const bool hasB = iA + 1 < end;
                const uint32_t pkA = slot + (uint32_t)(2 * q * R * pack_bytes);
                float acc[2][2];
                pack_pair_accumulate(x, pkA, pkA + (uint32_t)(R * pack_bytes), hasB, R, (uint32_t)pack_bytes, a.nsb,
                                     lane, acc);
                if (lane == 0 || (lane == 16 && hasB)) {
                    const int64_t unit = r0 + iA + (lane >> 4);
                    const int kseg = (EPI == EPI_SWIGLU) ? 0 : seg_of(a, unit);
                    const int64_t lr = unit - a.seg_begin[kseg];
                    float out = acc[0][0];
                    if (EPI == EPI_RESID || (EPI == EPI_STORE && a.res[kseg])) out = a.res[kseg][lr] + out;
                    if (EPI == EPI_SWIGLU) out = silu_mul(acc[0][0], acc[1][0]);
                    a.y[kseg][lr] = out;
                }
            }
        } else if constexpr (PR) {
            // several tokens (at least four rows per consumer warp): rows in pairs as
            // above, tokens in groups of TG, each activation load shared by the two
            // rows
            constexpr int TG = MT < 4 ? MT : 4;
            const int npair = (end - first + 1) / 2;
            for (int q = q0; q < npair; q += kConsumerWarps) {
                const int iA = first + 2 * q;
                const bool hasB = iA + 1 < end;
                const uint32_t pkA = slot + (uint32_t)(2 * q * R * pack_bytes);
                for (int t0 = 0; t0 < a.m; t0 += TG) {
                    float acc[2][TG];
                    pack_pair_accumulate_tg<TG>(x, pkA, pkA + (uint32_t)(R * pack_bytes), hasB, R,
                                                (uint32_t)pack_bytes, a.nsb, t0, lane, acc);
                    if (lane == 0 || (lane == 16 && hasB)) {
                        const int64_t unit = r0 + iA + (lane >> 4);
                        const int kseg = (EPI == EPI_SWIGLU) ? 0 : seg_of(a, unit);
                        const int64_t lr = unit - a.seg_begin[kseg];
#pragma unroll
                        for (int i = 0; i < TG; ++i) {
                            const int t = t0 + i;
                            if (t < a.m) {
                                float out = acc[0][i];
                                if (EPI == EPI_RESID || (EPI == EPI_STORE && a.res[kseg]))
                                    out = a.res[kseg][t * a.ldr[kseg] + lr] + out;
                                if (EPI == EPI_SWIGLU) out = silu_mul(acc[0][i], acc[1][i]);
                                a.y[kseg][t * a.ldy[kseg] + lr] = out;
                            }
                        }
                    }
                }
            }
        } else {
            for (int i = first + i0; i < end; i += kConsumerWarps) {
                const int64_t pack0 = r0 + (int64_t)i * a.rpp;
                const int pack_rows = (int)min((int64_t)a.rpp, r1 - pack0);
                const uint32_t pk = slot + (uint32_t)((i - first) * R * pack_bytes);
                float acc[2][MT];
                pack_accumulate<MT, R, XS>(x, pk, (uint32_t)pack_bytes, a.nsb, a.rpp, rip, pack_rows, lane, acc);
                if (rip < pack_rows) {
                    const int64_t unit = pack0 + rip;
                    const int kseg = (EPI == EPI_SWIGLU) ? 0 : seg_of(a, unit);
                    const int64_t lr = unit - a.seg_begin[kseg];
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        // spread the token stores over the lanes of the row
                        if (t < a.m && ((seg_lanes == 32) ? lane == (t & 31) : leader)) {
                            float out = acc[0][t];
                            if (EPI == EPI_RESID || (EPI == EPI_STORE && a.res[kseg]))
                                out = a.res[kseg][t * a.ldr[kseg] + lr] + out;
                            if (EPI == EPI_SWIGLU) out = silu_mul(acc[0][t], acc[1][t]);
                            a.y[kseg][t * a.ldy[kseg] + lr] = out;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp no longer reads the slot
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

template <int MT, int EPI, bool XS, int XIN, bool PR, int NW>
cudaError_t launch_t(const Args &a, int grid, cudaStream_t s)
{
    static bool attr_done[64] = {};
    const int dev = dev_info().device;
    const size_t smem = smem_bytes(a);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(q4k_gemv_kernel<MT, EPI, XS, XIN, PR, NW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((NW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, q4k_gemv_kernel<MT, EPI, XS, XIN, PR, NW>, a);
}

template <int MT, int EPI, bool PR, int NW = kConsumerWarps>
cudaError_t launch_x(const Args &a, int grid, cudaStream_t s, int xin)
{
    if (xin == XIN_NORM) {
        if constexpr (EPI != EPI_RESID) return launch_t<MT, EPI, true, XIN_NORM, PR, NW>(a, grid, s);
        return cudaErrorInvalidValue;
    }
    if (xin == XIN_F32) {
        if constexpr (EPI == EPI_RESID) return launch_t<MT, EPI, true, XIN_F32, PR, NW>(a, grid, s);
        return cudaErrorInvalidValue;
    }
    if (a.x_smem) return launch_t<MT, EPI, true, XIN_Q8, PR, NW>(a, grid, s);
    if constexpr (PR) return cudaErrorInvalidValue;  // the pair path wants the activations staged
    return launch_t<MT, EPI, false, XIN_Q8, false, NW>(a, grid, s);
}

// Consumer warps of a one-token launch: 16 when a CTA's work -- row pairs, or
// packs of short rows -- gives some warp one unit fewer than over 15 warps, else
// 15 (more registers a thread).
int nw_for(const Args &a, int grid)
{
    const int64_t rows = (a.units + grid - 1) / grid;
    const int64_t work = a.rpp > 1 ? (rows + a.rpp - 1) / a.rpp : (rows + 1) / 2;
    return (work + 15) / 16 < (work + 14) / 15 ? 16 : 15;
}

// One to three tokens (from kMmaMinTokens on, the tensor-core kernel of
// gemv_q4k_mma.cu runs instead).  Several tokens take the row-pair kernels when
// each consumer warp gets at least four rows.
template <int EPI>
cudaError_t launch_epi(const Args &a, int grid, cudaStream_t s, int xin)
{
    static_assert(kMmaMinTokens <= 4, "the dp4a kernels cover fewer than four tokens");
    const bool pr = a.m > 1 && a.rpp == 1 && a.x_smem && a.units / grid >= 4 * kConsumerWarps;
    if (a.m <= 1)
        return nw_for(a, grid) == 16 ? launch_x<1, EPI, false, 16>(a, grid, s, xin) : launch_x<1, EPI, false>(a, grid, s, xin);
    if (a.m <= 2) return pr ? launch_x<2, EPI, true>(a, grid, s, xin) : launch_x<2, EPI, false>(a, grid, s, xin);
    if (a.m <= 4) return pr ? launch_x<4, EPI, true>(a, grid, s, xin) : launch_x<4, EPI, false>(a, grid, s, xin);
    return cudaErrorInvalidValue;
}

}  // namespace
namespace {

// Q8_1 activations of m tokens: codes [m][in_dim], then d [m][in_dim/32], then s.
struct Q8Src {
    const int8_t *q;
    const float *d, *s;
};

static cudaError_t launch_core(const Q4kSegment *seg, int nseg, int epilogue, const Q8Src *q8,
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
        if (epilogue == EPI_STORE) {
            a.res[k] = seg[k].bias;  // the same bias row for every token
            a.ldr[k] = 0;
        }
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
        a.xq = q8->q;
        a.xd = q8->d;
        a.xs = q8->s;
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
        g_stall_next_gemv = 0;  // one launch only
    }
    a.rpp = (a.nsb < 8 && 8 % a.nsb == 0) ? 8 / a.nsb : 1;
    a.copy_rows = (int)std::max<int64_t>(1, kCopyBytes / a.row_bytes);
    const int64_t pack = (int64_t)R * a.rpp * a.row_bytes;
    // Two stages (four in one case, below), each half of the shared memory left
    // beside the activations.  Every consumer warp waits on every stage (a few hundred cycles per wait on
    // this GPU) and a small stage leaves most warps without a row pair in it, so
    // fewer, larger stages win even though the first one lands later; the bytes
    // in flight (one stage, ~90 KB per SM) still cover the HBM latency.
    const int64_t xbytes = x_smem_bytes(m, in_dim);
    a.x_smem = (xbytes <= kXSmemMax || f32in) ? 1 : 0;
    const int64_t budget = (int64_t)(m == 1 ? kCtaSmem1 : kCtaSmem) - (a.x_smem ? xbytes : 0) - 1024;
    // The stand-alone product of one token (Q8_1 in, plain store out) streams
    // best through four stages when a CTA's rows do not fit the ring at once
    // (4096 x 14336: 8.85 -> 8.16 us, 14336 x 4096: 8.46 -> 7.89 us); the fused
    // launches of the decode step keep two (four there: O +0.45%, gate/up
    // +0.7%, down +1.8% per step).
    const int64_t cta_rows = (units + dev_info().sm_count - 1) / dev_info().sm_count;
    const bool four = m == 1 && xin == XIN_Q8 && epilogue == EPI_STORE && cta_rows * R * a.row_bytes > budget;
    const int64_t tgt = budget / (four ? 4 : 2);
    a.PS = (int)std::max<int64_t>(1, tgt / pack);
    if (a.rpp == 1 && (a.PS & 1) && a.PS > 1) a.PS -= 1;  // row pairs: an even pack count per stage
    a.stage_bytes = (int)(a.PS * pack);
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

// Several tokens: the tensor-core kernel, in equal groups of tokens whose
// activations fit in shared memory beside its stage ring (one launch each).
static cudaError_t launch_mma_groups(const Q4kSegment *seg, int nseg, int epilogue, const Q8Src *x,
                                     const F32Input *f32in, int64_t m, int64_t in_dim, cudaStream_t s)
{
    const int64_t ng = q4k_gemv_launch_count(m, in_dim, epilogue, f32in == nullptr);
    const int64_t mc = (m + ng - 1) / ng;
    const int64_t nb = in_dim / 32;
    for (int64_t t0 = 0; t0 < m; t0 += mc) {
        const int64_t n = std::min(mc, m - t0);
        Q4kSegment part[3];
        for (int k = 0; k < nseg; ++k) {
            part[k] = seg[k];
            const int64_t ldy = seg[k].ldy ? seg[k].ldy : seg[k].rows;
            const int64_t ldr = seg[k].ldr ? seg[k].ldr : seg[k].rows;
            part[k].ldy = ldy;
            part[k].ldr = ldr;
            part[k].y = seg[k].y + t0 * ldy;
            part[k].res = seg[k].res ? seg[k].res + t0 * ldr : nullptr;
        }
        cudaError_t e;
        if (f32in) {
            F32Input in = *f32in;
            in.x = f32in->x + t0 * f32in->ldx;
            e = launch_q4k_gemv_mma(part, nseg, epilogue, nullptr, nullptr, nullptr, &in, n, in_dim, s);
        } else {
            e = launch_q4k_gemv_mma(part, nseg, epilogue, x->q + t0 * in_dim, x->d + t0 * nb, x->s + t0 * nb,
                                    nullptr, n, in_dim, s);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

static cudaError_t launch_common(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                                 const F32Input *f32in, int64_t m, int64_t in_dim, cudaStream_t s)
{
    Q8Src x{};
    if (q8) {
        const int64_t nb = in_dim / 32;
        x.q = static_cast<const int8_t *>(q8);
        x.d = reinterpret_cast<const float *>(x.q + m * in_dim);
        x.s = x.d + m * nb;
    }
    if (m >= kMmaMinTokens) return launch_mma_groups(seg, nseg, epilogue, q8 ? &x : nullptr, f32in, m, in_dim, s);
    return launch_core(seg, nseg, epilogue, q8 ? &x : nullptr, f32in, m, in_dim, s);
}

}  // namespace

cudaError_t launch_q4k_gemv(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                            int64_t m, int64_t in_dim, cudaStream_t s)
{
    return launch_common(seg, nseg, epilogue, q8, nullptr, m, in_dim, s);
}

int q4k_gemv_launch_count(int64_t m, int64_t in_dim, int epilogue, bool q8_input)
{
    if (m < kMmaMinTokens) return 1;
    const int64_t mt = q4k_gemv_mma_group(m, in_dim, epilogue, q8_input);
    return mt < 1 ? 0 : (int)((m + mt - 1) / mt);
}

bool q4k_gemv_f32_input_ok(int64_t m, int64_t in_dim)
{
    if (in_dim > 32LL * kRowWarps * kRowBlocksPerWarp) return false;
    // several tokens: each token group of the tensor-core kernel normalises and
    // quantises its own tokens
    if (m >= kMmaMinTokens) return q4k_gemv_mma_group(m, in_dim, EPI_SWIGLU, false) >= 1;
    return x_smem_bytes(m, in_dim) <= kXSmemMax;
}

bool q4k_gemv_f32_input_preferred(int64_t m, int64_t in_dim)
{
    // Several tokens (the tensor-core kernel) would stage their input one token
    // after another in every CTA, each token a round trip and a block reduction: at
    // 16 tokens that was most of the launch (Q|K|V 54 us, down 2 x 37 us).  The
    // separate norm / quantise kernels do all tokens at once, so from
    // kMmaMinTokens on a layer passes the GEMV its input as Q8_1.
    return m < kMmaMinTokens && q4k_gemv_f32_input_ok(m, in_dim);
}

cudaError_t launch_q4k_gemv_f32(const Q4kSegment *seg, int nseg, int epilogue, const F32Input &in,
                                int64_t m, int64_t in_dim, cudaStream_t s)
{
    if (!q4k_gemv_f32_input_ok(m, in_dim)) return cudaErrorInvalidValue;
    return launch_common(seg, nseg, epilogue, nullptr, &in, m, in_dim, s);
}




bool q4k_gemv_supported(int64_t m, int64_t in_dim, int epilogue)
{
    if (m >= kMmaMinTokens) return q4k_gemv_mma_group(m, in_dim, epilogue, true) >= 1;
    const int R = (epilogue == EPI_SWIGLU) ? 2 : 1;
    const int64_t nsb = in_dim / 256;
    const int64_t rpp = (nsb < 8 && 8 % nsb == 0) ? 8 / nsb : 1;
    const int64_t pack = R * rpp * nsb * kSB;
    const int64_t xbytes = x_smem_bytes(m, in_dim);
    const int64_t budget = (int64_t)(m == 1 ? kCtaSmem1 : kCtaSmem) - (xbytes <= kXSmemMax ? xbytes : 0) - 1024;
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
