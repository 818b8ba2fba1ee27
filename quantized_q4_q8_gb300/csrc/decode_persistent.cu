// decode_persistent.cu -- the decode step of a stack of Q4_K layers (m = 1) as
// ONE persistent kernel: one CTA per SM for the whole step.
//
// Same operations and order as the launch sequence in layer.cu (the layer of
// transformer_layer_gpu_true_dp4a, realizar 0.8.5 src/cuda/executor/cached.rs):
// per layer, RMSNorm -> Q8_1 -> fused Q|K|V GEMV; RoPE, KV append and split-
// sequence attention with the Q8_1 of its output; O GEMV + residual; RMSNorm ->
// Q8_1 -> gate/up GEMV with silu(gate) * up; Q8_1 of h -> down GEMV + residual.
//
// Why one kernel.  A decode step streams every weight byte once, and at batch 1
// the work per byte is a few integer dot instructions, so the step is bound by
// HBM -- but only if HBM never idles.  As separate launches each GEMV pays a ramp
// (CTAs start, compute the activation prologue, fill their pipeline) and a tail
// (the last CTAs finish alone), and with 9-51 MB per matrix those fixed costs are
// as long as the transfer itself.  Here the weights never stop flowing: in every
// CTA a producer warp walks the whole step's list of byte ranges -- the CTA's
// share of each layer's Q|K|V rows, its attention units' K and V cache rows, its
// O rows, gate/up rows and down rows, layer after layer -- and keeps a ring of
// shared-memory slots full with the 1-D bulk copy engine (cp.async.bulk on
// mbarriers), plus an L2 prefetch window further ahead.  None of those bytes
// depend on the step's activations (the cache rows read are those of earlier
// tokens), so the producer never waits for anything but a free slot.  Sixteen
// consumer warps follow the same list.  Between dependent phases (Q|K|V ->
// attention -> O -> gate/up -> down -> next layer) the consumers meet at a grid
// barrier; meanwhile the ring and the L2 window keep filling with the next
// phase's weights, so the barrier and the activation prologue hide behind HBM
// traffic instead of adding to it.
//
// Grid barriers need every CTA resident: the kernel is launched cooperatively
// (the launch fails rather than run with CTAs missing).  Every wait is bounded
// and also gives up as soon as any CTA has recorded an error, so a failure
// ends the kernel with an error code instead of hanging the GPU.
//
// Attention runs one warp per unit (token, kv head, chunk of CL cache rows);
// the unit's K and V rows arrive in one ring slot.  The warp rotates the query
// heads of its kv head with a per-CTA RoPE table, scores the chunk, applies the
// chunk softmax and the weighted values, and leaves a partial record; the last
// warp to finish a (token, kv head) -- an atomic counter, no spinning -- merges
// the chunks (log-sum-exp rule) and writes the Q8_1 of the merged heads.  The
// warp whose chunk holds the token's own row rotates k, appends k and v to the
// cache and uses them from registers.  Lane l holds elements 32 e + l of a head.
#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "q4k_dot.cuh"
#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {

bool g_use_persistent = false;

namespace {

// 15 consumer warps + 1 producer warp: 16 warps, 4 per SM sub-partition, which
// leaves 128 registers per thread (a 17th warp would cut that to 96).
constexpr int kPWarps = 15;                    // consumer warps
constexpr int kPThreads = (kPWarps + 1) * 32;  // + the producer warp
constexpr int kPMaxRow = kPWarps * 32 * 32;    // activation rows the staging helpers take
constexpr int kPMaxLayers = 32;                // layers per launch (kernel parameter space)
constexpr int kMaxSlots = 32;
constexpr int kAttnUnitBytes = 16384;          // K rows + V rows of one attention unit
constexpr int kMaxG = 8;                       // query heads per kv head
constexpr double kTwoPi = 6.283185307179586476925286766559;

enum Kind { K_QKV = 0, K_O = 1, K_GU = 2, K_DN = 3, K_ATT = 4 };
constexpr int kPhases = 5;
__device__ __forceinline__ int phase_kind(int p)
{
    return p == 0 ? K_QKV : p == 1 ? K_ATT : p == 2 ? K_O : p == 3 ? K_GU : K_DN;
}

struct PLayer {
    const uint8_t *w[7];  // q, k, v, o, gate, up, down
    const float *attn_gamma, *ffn_gamma;
    float *kc, *vc;
};

struct PArgs {
    PLayer L[kPMaxLayers];
    int n_layers, m;
    int hidden, hidden_pad, n_heads, n_kv_heads, head_dim, inter, group, q_dim, q_pad, kv_dim;
    float eps, rope_theta;
    int rope_mode;
    int64_t seq_stride;
    int max_seq;
    const int32_t *positions;
    int position;
    int chunk_len, n_chunks;  // attention rows per unit; chunks covering max_seq
    int slot_bytes, n_slots, pf_stages;
    int x_region;
    int ps[4];  // packs per stage of each GEMV kind
    const float *input;
    float *output;
    float *xbuf[2];
    float *qkv, *part, *res1, *h;
    int8_t *a8;
    int *counters;
    unsigned *gbar;
    unsigned *err;
};

// ---------------------------------------------------------------- per-CTA plan
struct GemvShape {
    int64_t units, in_dim, row_bytes;
    int nsb, R, rpp, ps;
};

__host__ __device__ inline void gemv_dims(int kind, int q_dim, int kv_dim, int hidden, int hidden_pad, int q_pad,
                                          int inter, int64_t &units, int64_t &in_dim, int &R)
{
    R = 1;
    if (kind == K_QKV) {
        units = q_dim + 2 * (int64_t)kv_dim;
        in_dim = hidden_pad;
    } else if (kind == K_O) {
        units = hidden;
        in_dim = q_pad;
    } else if (kind == K_GU) {
        units = inter;
        in_dim = hidden_pad;
        R = 2;
    } else {
        units = hidden;
        in_dim = inter;
    }
}

__device__ __forceinline__ GemvShape gemv_shape(const PArgs &a, int kind)
{
    GemvShape g;
    gemv_dims(kind, a.q_dim, a.kv_dim, a.hidden, a.hidden_pad, a.q_pad, a.inter, g.units, g.in_dim, g.R);
    g.nsb = (int)(g.in_dim / 256);
    g.row_bytes = (int64_t)g.nsb * kSB;
    g.rpp = pack_rows_for(g.nsb);
    g.ps = a.ps[kind];
    return g;
}

struct Plan {
    int64_t r0[4], r1[4];    // this CTA's rows of each GEMV kind
    int64_t nst[kPhases];    // stages of each kind (indexed by Kind)
    int64_t au0, au1;        // this CTA's attention units
    int pos[4];              // positions of the tokens (m <= 4)
    int nc[4];               // chunks of each token
};
constexpr int kPlanBytes = 256;
static_assert(sizeof(Plan) <= kPlanBytes, "plan");

__device__ __forceinline__ int token_pos(const PArgs &a, int t)
{
    return a.positions ? a.positions[t] : a.position;
}

__device__ __forceinline__ bool pos_valid(const PArgs &a, int p) { return p >= 0 && p < a.max_seq; }

__device__ __forceinline__ void make_plan(const PArgs &a, Plan &p)
{
    const int64_t G = gridDim.x, b = blockIdx.x;
    for (int k = 0; k < 4; ++k) {
        const GemvShape g = gemv_shape(a, k);
        p.r0[k] = g.units * b / G;
        p.r1[k] = g.units * (b + 1) / G;
        const int64_t npacks = (p.r1[k] - p.r0[k] + g.rpp - 1) / g.rpp;
        p.nst[k] = (npacks + g.ps - 1) / g.ps;
    }
    int64_t U = 0;
    for (int t = 0; t < a.m; ++t) {
        p.pos[t] = token_pos(a, t);
        p.nc[t] = pos_valid(a, p.pos[t]) ? min(a.n_chunks, p.pos[t] / a.chunk_len + 1) : 1;
        U += (int64_t)a.n_kv_heads * p.nc[t];
    }
    p.au0 = U * b / G;
    p.au1 = U * (b + 1) / G;
    p.nst[K_ATT] = p.au1 - p.au0;
}

// attention unit u -> (token, kv head, chunk)
// (32-bit: at most m * n_kv_heads * 4096 units)
__device__ __forceinline__ void unit_coords(const PArgs &a, const Plan &p, int64_t u64, int &t, int &kvh, int &chunk)
{
    int u = (int)u64;
    t = 0;
    while (t + 1 < a.m && u >= a.n_kv_heads * p.nc[t]) {
        u -= a.n_kv_heads * p.nc[t];
        ++t;
    }
    const int nc = p.nc[t];
    kvh = u / nc;
    chunk = u - kvh * nc;
}

__device__ __forceinline__ int unit_rows(const PArgs &a, const Plan &p, int t, int chunk)
{
    const int pos = p.pos[t];
    if (!pos_valid(a, pos)) return 0;
    return max(0, min(a.chunk_len, pos + 1 - chunk * a.chunk_len));
}

__device__ __forceinline__ const uint8_t *seg_weight(const PArgs &a, int l, int kind, int seg)
{
    const PLayer &L = a.L[l];
    switch (kind) {
    case K_QKV: return L.w[seg];
    case K_O: return L.w[3];
    case K_GU: return L.w[4 + seg];
    default: return L.w[6];
    }
}

// ---------------------------------------------------------------- producer
// The whole producer warp walks the step phase by phase.  Per phase it works out
// the phase's geometry once; per stage it then needs a few additions: lane 0
// waits for the slot, arms the full barrier with the stage's byte count, and the
// stage's byte ranges (one run per Q|K|V matrix, a gate and an up range per pack,
// a K and a V row per cache row) are spread over the lanes.  A copy may land
// before the barrier is armed: the transaction count goes negative and the phase
// still cannot complete before lane 0's arrival.  When a phase starts, the next
// phase's byte ranges are prefetched into L2 (64 KB pieces over the lanes), so
// the ring's copies mostly read L2.

// Byte ranges of this CTA's share of phase (l, kind), for the L2 prefetch.
__device__ __forceinline__ void prefetch_phase(const PArgs &a, const Plan &p, int l, int kind, int lane)
{
    if (kind == K_ATT) {
        const unsigned rb = (unsigned)a.head_dim * 4u;
        const int nunits = (int)(p.au1 - p.au0);
        const int rows = nunits * a.chunk_len;
        for (int j = lane; j < rows; j += 32) {
            const int i = j / a.chunk_len, r = j - i * a.chunk_len;
            int t, kvh, chunk;
            unit_coords(a, p, p.au0 + i, t, kvh, chunk);
            if (r < unit_rows(a, p, t, chunk)) {
                const int64_t off = (int64_t)t * a.seq_stride + ((int64_t)chunk * a.chunk_len + r) * a.kv_dim +
                                    (int64_t)kvh * a.head_dim;
                prefetch_l2(a.L[l].kc + off, rb);
                prefetch_l2(a.L[l].vc + off, rb);
            }
        }
        return;
    }
    const GemvShape g = gemv_shape(a, kind);
    const int64_t r0 = p.r0[kind], r1 = p.r1[kind];
    if (r1 <= r0) return;
    // up to three contiguous row ranges (Q|K|V: one per matrix; gate/up: two)
    const uint8_t *src[3];
    int64_t len[3];
    int nr = 0;
    if (kind == K_QKV) {
        const int64_t bnd[4] = {0, a.q_dim, a.q_dim + (int64_t)a.kv_dim, a.q_dim + 2 * (int64_t)a.kv_dim};
        for (int sgi = 0; sgi < 3; ++sgi) {
            const int64_t lo = max(r0, bnd[sgi]), hi = min(r1, bnd[sgi + 1]);
            if (hi > lo) {
                src[nr] = a.L[l].w[sgi] + (lo - bnd[sgi]) * g.row_bytes;
                len[nr++] = (hi - lo) * g.row_bytes;
            }
        }
    } else {
        for (int h = 0; h < g.R; ++h) {
            src[nr] = seg_weight(a, l, kind, h) + r0 * g.row_bytes;
            len[nr++] = (r1 - r0) * g.row_bytes;
        }
    }
    constexpr int64_t kPiece = 64 * 1024;
    int piece = 0;
    for (int q = 0; q < nr; ++q)
        for (int64_t off = 0; off < len[q]; off += kPiece, ++piece)
            if ((piece & 31) == lane) prefetch_l2(src[q] + off, (unsigned)min(kPiece, len[q] - off));
}

__device__ __forceinline__ void producer(const PArgs &a, const Plan &p, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                         int lane)
{
    const int NS = a.n_slots;
    const uint32_t ring_s = smem_u32(ring);
    // The RMSNorm gammas are read by every CTA right after a grid barrier, when
    // HBM is busiest: each CTA brings a 1 KB slice of the next one into L2 a phase
    // ahead (attention gamma of layer l + 1 with layer l's down rows, FFN gamma of
    // layer l with its O rows).
    const unsigned gbytes = (unsigned)a.hidden * 4u & ~15u, goff = blockIdx.x * 1024u;
    auto prefetch_gamma = [&](const float *gm) {
        if (lane == 0 && goff < gbytes) prefetch_l2(reinterpret_cast<const uint8_t *>(gm) + goff, min(1024u, gbytes - goff));
    };
    prefetch_gamma(a.L[0].attn_gamma);
    prefetch_phase(a, p, 0, K_QKV, lane);
    int64_t K = 0;
    RingPos rp{0, 0u};
    bool ok = true;
    for (int l = 0; l < a.n_layers && ok; ++l) {
        for (int ph = 0; ph < kPhases && ok; ++ph) {
            const int kind = phase_kind(ph);
            if (ph == 2) prefetch_gamma(a.L[l].ffn_gamma);
            if (ph == 4 && l + 1 < a.n_layers) prefetch_gamma(a.L[l + 1].attn_gamma);
            if (ph + 1 < kPhases)
                prefetch_phase(a, p, l, phase_kind(ph + 1), lane);
            else if (l + 1 < a.n_layers)
                prefetch_phase(a, p, l + 1, K_QKV, lane);
            const int64_t nst = p.nst[kind];
            // phase geometry
            GemvShape g{};
            const uint8_t *w0 = nullptr, *w1 = nullptr, *w2 = nullptr;
            int64_t r0 = 0, r1 = 0, stage_rows = 0, pack_bytes = 0;
            if (kind != K_ATT) {
                g = gemv_shape(a, kind);
                r0 = p.r0[kind];
                r1 = p.r1[kind];
                stage_rows = (int64_t)g.ps * g.rpp;
                pack_bytes = (int64_t)g.rpp * g.row_bytes;
                w0 = seg_weight(a, l, kind, 0);
                w1 = seg_weight(a, l, kind, 1);
                w2 = seg_weight(a, l, kind, 2);
            }
            for (int64_t k = 0; k < nst; ++k, ++K, ring_next(rp, NS)) {
                const int s = rp.s;
                if (K >= NS) {
                    // the slot's previous stage (one ring length back) is released
                    const bool got = __all_sync(0xffffffffu, mbar_wait_abortable(&empty[s], rp.par ^ 1u, a.err,
                                                                                 DEV_TIMEOUT_STEP));
                    if (!got) {
                        ok = false;
                        break;
                    }
                }
                const uint32_t dst = ring_s + (uint32_t)s * (uint32_t)a.slot_bytes;
                unsigned bytes = 0;
                if (kind == K_ATT) {
                    int t, kvh, chunk;
                    unit_coords(a, p, p.au0 + k, t, kvh, chunk);
                    const int n = unit_rows(a, p, t, chunk);
                    const unsigned rb = (unsigned)a.head_dim * 4u;
                    bytes = 2u * (unsigned)n * rb;
                    const int64_t base = (int64_t)t * a.seq_stride + (int64_t)chunk * a.chunk_len * a.kv_dim +
                                         (int64_t)kvh * a.head_dim;
                    for (int j = lane; j < 2 * n; j += 32) {
                        const int r = j >> 1;
                        const float *src = ((j & 1) ? a.L[l].vc : a.L[l].kc) + base + (int64_t)r * a.kv_dim;
                        bulk_g2s_u32(dst + (uint32_t)((j & 1) * a.chunk_len + r) * rb, src, rb, &full[s]);
                    }
                } else {
                    const int64_t u0 = r0 + k * stage_rows;
                    const int n = (int)min(stage_rows, r1 - u0);
                    bytes = (unsigned)(g.R * n * g.row_bytes);
                    if (g.R == 2) {
                        const int npk = (n + g.rpp - 1) / g.rpp;
                        for (int j = lane; j < 2 * npk; j += 32) {
                            const int q = j >> 1, h = j & 1;
                            const int nr = min(g.rpp, n - q * g.rpp);
                            const uint8_t *src = (h ? w1 : w0) + (u0 + (int64_t)q * g.rpp) * g.row_bytes;
                            bulk_g2s_u32(dst + (uint32_t)((2 * q + h) * pack_bytes), src, (unsigned)(nr * g.row_bytes),
                                         &full[s]);
                        }
                    } else if (kind == K_QKV) {
                        if (lane < 3) {
                            const int64_t bnd[4] = {0, a.q_dim, a.q_dim + (int64_t)a.kv_dim,
                                                    a.q_dim + 2 * (int64_t)a.kv_dim};
                            const int64_t lo = max(u0, bnd[lane]), hi = min(u0 + n, bnd[lane + 1]);
                            if (hi > lo)
                                bulk_g2s_u32(dst + (uint32_t)((lo - u0) * g.row_bytes),
                                             (lane == 0 ? w0 : lane == 1 ? w1 : w2) + (lo - bnd[lane]) * g.row_bytes,
                                             (unsigned)((hi - lo) * g.row_bytes), &full[s]);
                        }
                    } else if (lane == 0) {
                        bulk_g2s_u32(dst, w0 + u0 * g.row_bytes, bytes, &full[s]);
                    }
                }
                if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
            }
        }
    }
    // stages issued but perhaps not landed must land before the CTA exits
    if (!ok && lane == 0) {
        for (int64_t q = (K > NS ? K - NS : 0); q < K; ++q)
            if (!mbar_wait(&full[q % NS], (unsigned)((q / NS) & 1))) set_error(a.err, DEV_TIMEOUT_DRAIN);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- consumers
struct CCtx {
    uint32_t ring_s;
    uint64_t *full, *empty;
    uint8_t *xsm;
    float *red;
    const float *rope;  // [m][head_dim / 2][2] cos, sin
    int warp, lane, tid;
};

__device__ __forceinline__ void csync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(kPWarps * 32) : "memory");
}

// All consumer warps of every CTA: after it, every global write made by any CTA
// before it is visible.  `idx`: barriers passed so far in this launch.
__device__ __forceinline__ void grid_barrier(const PArgs &a, const CCtx &c, unsigned idx)
{
    csync();
    if (c.warp == 0) {
        if (c.lane == 0) {
            unsigned *ctr = a.gbar;
            const unsigned target = gridDim.x * (idx + 1);
            __threadfence();
            atomicAdd(ctr, 1u);
            bool done = false;
            for (uint32_t i = 0; i < kWaitLimit; ++i) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
                if (v >= target) {
                    done = true;
                    break;
                }
                if ((i & 15u) == 15u && *reinterpret_cast<volatile unsigned *>(a.err) != 0u) break;
                __nanosleep(64);
            }
            if (!done && *reinterpret_cast<volatile unsigned *>(a.err) == 0u) set_error(a.err, DEV_TIMEOUT_GRID);
            __threadfence();
        }
        __syncwarp();
    }
    csync();
}

// One GEMV phase: the CTA's packs, warp w taking packs w, w + 16, ...
// One GEMV phase of the consumers (kind K_QKV, K_O, K_GU or K_DN).  Called from
// one place for all four kinds: with a copy per kind the kernel's code outgrew
// the instruction caches and instruction fetch became the first stall.
__device__ __forceinline__ void gemv_phase(const PArgs &a, const Plan &p, const CCtx &cc, int kind, int64_t K0,
                                           const float *res, float *y)
{
    const CCtx c = cc;
    const int R = kind == K_GU ? 2 : 1;
    const GemvShape g = gemv_shape(a, kind);
    const int64_t r0 = p.r0[kind], r1 = p.r1[kind];
    const int64_t npacks = (r1 - r0 + g.rpp - 1) / g.rpp;
    const uint32_t pack_bytes = (uint32_t)(g.rpp * g.row_bytes);
    const int n_slots = a.n_slots, slot_bytes = a.slot_bytes, q_dim = a.q_dim, kv_dim = a.kv_dim;
    unsigned *const err = a.err;
    XSrc x;
    x.in_dim = g.in_dim;
    x.nb = g.in_dim / 32;
    x.m = 1;
    x.q = smem_u32(c.xsm);
    x.ds = smem_u32(c.xsm + (g.in_dim / 256) * kXSlot);
    x.gq = nullptr;
    x.gd = x.gs = nullptr;
    const int gl = c.lane >> 2;
    const int seg_lanes = (g.rpp > 1) ? 4 * g.nsb : 32;
    const int rip = (g.rpp > 1) ? gl / g.nsb : 0;
    const int leader = c.lane % seg_lanes == 0;

    // epilogue of one output row
    auto store_row = [&](int64_t unit, float v0, float v1) {
        int64_t lr = unit;
        float *yk = y;
        if (kind == K_QKV) {
            const int seg = unit < q_dim ? 0 : unit < q_dim + kv_dim ? 1 : 2;
            const int64_t base = seg == 0 ? 0 : seg == 1 ? q_dim : (int64_t)q_dim + kv_dim;
            lr = unit - base;
            yk = y + base;
        }
        float out = v0;
        if (kind == K_O || kind == K_DN) out = __ldcg(res + lr) + out;
        if (kind == K_GU) out = silu_mul(v0, v1);
        yk[lr] = out;
    };
    // Every warp passes every stage of the phase in order (waits for it, takes its
    // own packs in it, releases it), so no warp can run a ring length ahead of a
    // stage that is not filled yet: the parity waits stay unambiguous.
    const int nst = (int)p.nst[kind];
    const int npk = (int)npacks, ps = g.ps, pps = (ps + 1) / 2;  // packs and pairs per stage
    RingPos rp = ring_pos(K0, n_slots);
    int prot = 0, rot = 0;  // pairs / packs of the earlier stages, modulo the warp count
    for (int k = 0; k < nst; ++k, ring_next(rp, n_slots)) {
        const int s = rp.s;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_abortable(&c.full[s], rp.par, err, DEV_TIMEOUT_STEP));
        const int first = k * ps, end = min(first + ps, npk);
        const uint32_t slot = c.ring_s + (uint32_t)(s * slot_bytes);
        if (ok && g.rpp == 1) {
            // rows in pairs: pair q of the stage (packs first + 2q, first + 2q + 1)
            // goes to warp (pairs of earlier stages + q) % 15
            const int npair = (end - first + 1) / 2;
            for (int q = (c.warp - prot + kPWarps) % kPWarps; q < npair; q += kPWarps) {
                const int iA = first + 2 * q;
                const bool hasB = iA + 1 < end;
                const uint32_t pkA = slot + (uint32_t)(2 * q) * R * pack_bytes;
                float acc[2][2];
                pack_pair_accumulate(x, pkA, pkA + R * pack_bytes, hasB, R, pack_bytes, g.nsb, c.lane, acc);
                if (c.lane == 0 || (c.lane == 16 && hasB))
                    store_row(r0 + iA + (c.lane >> 4), acc[0][0], acc[1][0]);
            }
        } else if (ok) {
            for (int i = first + (c.warp - rot + kPWarps) % kPWarps; i < end; i += kPWarps) {
                const int64_t pack0 = r0 + (int64_t)i * g.rpp;
                const int pack_rows = (int)min((int64_t)g.rpp, r1 - pack0);
                const uint32_t pk = slot + (uint32_t)(i - first) * R * pack_bytes;
                float acc[2][1];
                if (R == 2)
                    pack_accumulate<1, 2, true>(x, pk, pack_bytes, g.nsb, g.rpp, rip, pack_rows, c.lane, acc);
                else
                    pack_accumulate<1, 1, true>(x, pk, pack_bytes, g.nsb, g.rpp, rip, pack_rows, c.lane, acc);
                if (rip < pack_rows && leader) store_row(pack0 + rip, acc[0][0], acc[1][0]);
            }
        }
        prot += pps;
        while (prot >= kPWarps) prot -= kPWarps;
        rot += ps;
        while (rot >= kPWarps) rot -= kPWarps;
        if (!ok) continue;
        __syncwarp();
        if (c.lane == 0) mbar_arrive(&c.empty[s]);  // this warp is done with the slot
    }
}

// Activation staging of the consumers (one call site for the same reason).
__device__ __forceinline__ void stage_f32(uint8_t *xsm, const float *xf, int64_t ldx, const float *gamma,
                                          int64_t norm_n, float eps, int64_t in_dim, float *red, int warp, int lane)
{
    auto sync = [] { csync(); };
    if (gamma)
        stage_x_f32<true, true, kPWarps>(xsm, xf, ldx, gamma, norm_n, eps, 1, in_dim, red, warp, lane, sync);
    else
        stage_x_f32<true, false, kPWarps>(xsm, xf, ldx, nullptr, 0, 0.0f, 1, in_dim, red, warp, lane, sync);
}

// RoPE of one head held lane-strided (v[e] = element 32 e + lane) with the
// token's table.  Mode 0 pairs (2i, 2i + 1): partner in lane ^ 1, same e.
// Mode 1 pairs (i, i + hd/2): partner in the same lane, e +- CPT/2.
template <int CPT>
__device__ __forceinline__ void rope_lanes(float (&v)[CPT], const float *tab, int mode, int lane)
{
    if (mode == 0) {
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
            const int d = 32 * e + lane;
            const float cs = tab[2 * (d >> 1)], sn = tab[2 * (d >> 1) + 1];
            const float other = __shfl_xor_sync(0xffffffffu, v[e], 1);
            v[e] = (lane & 1) ? other * sn + v[e] * cs : v[e] * cs - other * sn;
        }
    } else {
        constexpr int H = CPT / 2;
#pragma unroll
        for (int e = 0; e < H; ++e) {
            const int i = 32 * e + lane;
            const float cs = tab[2 * i], sn = tab[2 * i + 1];
            const float x0 = v[e], x1 = v[e + H];
            v[e] = x0 * cs - x1 * sn;
            v[e + H] = x0 * sn + x1 * cs;
        }
    }
}

// Partial record [max, sum, o[head_dim]] of one query head: first for one
// chunk, then (at the run's first chunk) for a run of chunks one CTA worked.
__device__ __forceinline__ float *part_rec(const PArgs &a, int t, int kvh, int chunk, int g)
{
    const int64_t idx = (((int64_t)t * a.n_kv_heads + kvh) * a.n_chunks + chunk) * a.group + g;
    return a.part + idx * (a.head_dim + 2);
}

// Log-sum-exp combination of records [m_k, l_k, o_k] in the order given, as a
// running (M, L, O): for each non-empty record, M' = max(M, m_k) and
// L, O <- L, O * exp(M - M') + l_k, o_k * exp(m_k - M').  Four records' loads are
// in flight at a time.  GLOBAL: the records are in global memory, written by
// other CTAs (read through L2); else in shared memory.  Lane-strided o.
template <int CPT, bool GLOBAL, typename Rec>
__device__ __forceinline__ void lse_combine(int n, Rec rec, int lane, float &M, float &L, float (&O)[CPT])
{
    auto ld = [](const float *q) { return GLOBAL ? __ldcg(q) : *q; };
    M = -INFINITY;
    L = 0.0f;
#pragma unroll
    for (int e = 0; e < CPT; ++e) O[e] = 0.0f;
    for (int k0 = 0; k0 < n; k0 += 4) {
        float mk[4], lk[4], ov[4][CPT];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            lk[u] = 0.0f;
            mk[u] = -INFINITY;
            if (k0 + u < n) {
                const float *r = rec(k0 + u);
                mk[u] = ld(r);
                lk[u] = ld(r + 1);
#pragma unroll
                for (int e = 0; e < CPT; ++e) ov[u][e] = ld(r + 2 + 32 * e + lane);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (lk[u] > 0.0f) {
                const float Mn = fmaxf(M, mk[u]);
                const float sa = (L > 0.0f) ? expf(M - Mn) : 0.0f;
                const float sb = expf(mk[u] - Mn);
                L = fmaf(L, sa, lk[u] * sb);
#pragma unroll
                for (int e = 0; e < CPT; ++e) O[e] = fmaf(O[e], sa, ov[u][e] * sb);
                M = Mn;
            }
        }
    }
}

// CTA owning attention unit u (the units are split evenly over the grid)
__device__ __forceinline__ int unit_owner(int u, int U, int G)
{
    int b = (int)((int64_t)u * G / U);
    while (b + 1 < G && (int64_t)U * (b + 1) / G <= u) ++b;
    while (b > 0 && (int64_t)U * b / G > u) --b;
    return b;
}

// Query heads of kv head kvh for token t, lane-strided (not yet rotated).
template <int CPT, int GM>
__device__ __forceinline__ void load_q(const PArgs &a, int t, int kvh, int lane, float (&qv)[GM][CPT])
{
    const int64_t ld_qkv = a.q_dim + 2 * (int64_t)a.kv_dim;
    const float *qrow = a.qkv + (int64_t)t * ld_qkv + (int64_t)kvh * a.group * a.head_dim;
#pragma unroll
    for (int g = 0; g < GM; ++g)
        if (g < a.group)
#pragma unroll
            for (int e = 0; e < CPT; ++e) qv[g][e] = __ldcg(qrow + g * a.head_dim + 32 * e + lane);
}

// Step 2 of the attention phase, after every chunk record of the CTA is
// written: the CTA's consecutive units of one (token, kv head) are combined into
// one record at the run's first chunk (warp r % 16 takes run r); the run then
// arrives on the head's counter with its chunk count, and the run that completes
// the head merges the runs of all CTAs in chunk order and writes the Q8_1 of the
// head's output.  srec: the chunk records in shared memory, or nullptr.
template <int CPT>
__device__ __forceinline__ void attention_runs(const PArgs &a, const Plan &p, const float *srec, int warp, int lane)
{
    const int hd = a.head_dim, G = a.group;
    int U = 0, ubase[4];
    for (int t = 0; t < a.m; ++t) {
        ubase[t] = U;
        U += a.n_kv_heads * p.nc[t];
    }
    const int au0 = (int)p.au0, au1 = (int)p.au1;
    int rw = 0;  // warp of the current run
    for (int u = au0; u < au1; rw = rw + 1 == kPWarps ? 0 : rw + 1) {
        int t, kvh, chunk;
        unit_coords(a, p, u, t, kvh, chunk);
        const int nc = p.nc[t];
        const int head0 = ubase[t] + kvh * nc;  // unit of chunk 0
        const int run_end = min(au1, head0 + nc);
        const int len = run_end - u;
        if (rw == warp) {
            for (int g = 0; g < G; ++g) {
                float M, L, O[CPT];
                if (srec)
                    lse_combine<CPT, false>(len, [&](int k) { return srec + ((int64_t)(u - au0 + k) * G + g) * (hd + 2); },
                                            lane, M, L, O);
                else
                    lse_combine<CPT, true>(len, [&](int k) { return part_rec(a, t, kvh, chunk + k, g); }, lane, M,
                                           L, O);
                __syncwarp();  // every lane has read the first record before it is overwritten
                float *rec = part_rec(a, t, kvh, chunk, g);
                if (lane == 0) {
                    rec[0] = M;
                    rec[1] = L;
                }
#pragma unroll
                for (int e = 0; e < CPT; ++e) rec[2 + 32 * e + lane] = O[e];
            }
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                int *cnt = a.counters + (int64_t)t * a.n_kv_heads + kvh;
                const int prev = atomicAdd(cnt, len);
                last = (prev + len == nc);
                if (last) *cnt = 0;  // ready for the next layer
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                int8_t *q = a.a8;
                float *qd = reinterpret_cast<float *>(q + (int64_t)a.m * a.q_pad);
                float *qsum = qd + (int64_t)a.m * (a.q_pad / 32);
                const int Gd = gridDim.x;
                for (int g = 0; g < G; ++g) {
                    // run starts of this head in chunk order: run k starts at the first
                    // unit of the k-th CTA that holds units of the head
                    const int b0 = unit_owner(head0, U, Gd);
                    const int nrun = unit_owner(head0 + nc - 1, U, Gd) - b0 + 1;
                    float M, L, O[CPT];
                    lse_combine<CPT, true>(nrun, [&](int k) {
                        const int first = k == 0 ? head0 : (int)((int64_t)U * (b0 + k) / Gd);
                        return part_rec(a, t, kvh, first - head0, g);
                    }, lane, M, L, O);
                    const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;  // 0 only after a bad position
#pragma unroll
                    for (int e = 0; e < CPT; ++e) {
                        const float v = O[e] * inv;
                        const float amax = warp_max(fabsf(v));
                        const float dq = __fdiv_rn(amax, 127.0f);
                        const int qi = q8_code(v, dq, rcp_approx(dq));
                        const int sum = warp_sum_int(qi);
                        const int64_t blk = ((int64_t)(kvh * G + g) * hd) / 32 + e;
                        q[(int64_t)t * a.q_pad + blk * 32 + lane] = (int8_t)qi;
                        if (lane == 0) {
                            qd[(int64_t)t * (a.q_pad / 32) + blk] = dq;
                            qsum[(int64_t)t * (a.q_pad / 32) + blk] = __fmul_rn(dq, (float)sum);
                        }
                    }
                }
            }
        }
        u = run_end;
    }
}

template <int CPT, int GM>
__device__ __forceinline__ void attention_phase(const PArgs &a, const Plan &p, const CCtx &c, int l, int64_t K0)
{
    const int hd = a.head_dim, G = a.group, lane = c.lane;
    const float scale = 1.0f / sqrtf((float)hd);
    // Q8_1 padding columns q_dim .. q_pad of the attention output are zero
    if (blockIdx.x == 0 && c.warp == 0 && a.q_pad > a.q_dim) {
        float *qd = reinterpret_cast<float *>(a.a8 + (int64_t)a.m * a.q_pad);
        float *qsum = qd + (int64_t)a.m * (a.q_pad / 32);
        for (int t = 0; t < a.m; ++t) {
            for (int i = a.q_dim + lane; i < a.q_pad; i += 32) a.a8[(int64_t)t * a.q_pad + i] = 0;
            for (int b = a.q_dim / 32 + lane; b < a.q_pad / 32; b += 32) {
                qd[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
                qsum[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
            }
        }
    }
    const int nunits = (int)(p.au1 - p.au0);
    // chunk records in the (idle) activation region when they fit
    const int rec_floats = G * (hd + 2);
    float *srec = ((int64_t)nunits * rec_floats * 4 <= a.x_region) ? reinterpret_cast<float *>(c.xsm) : nullptr;

    // 1. chunks: every warp passes every unit's stage in order; unit i is worked by
    //    warp i % 16, which loads its query heads before it waits for the stage
    int mine = c.warp;
    float qv[GM][CPT];
    if (mine < nunits) {
        int t, kvh, chunk;
        unit_coords(a, p, p.au0 + mine, t, kvh, chunk);
        load_q<CPT, GM>(a, t, kvh, lane, qv);
    }
    RingPos rp = ring_pos(K0, a.n_slots);
    for (int i = 0; i < nunits; ++i, ring_next(rp, a.n_slots)) {
        const int s = rp.s;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_abortable(&c.full[s], rp.par, a.err, DEV_TIMEOUT_STEP));
        if (!ok) continue;
        if (i != mine) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.empty[s]);
            continue;
        }
        int t, kvh, chunk;
        unit_coords(a, p, p.au0 + i, t, kvh, chunk);
        const int pos = p.pos[t];
        const bool pos_ok = pos_valid(a, pos);
        const int n = unit_rows(a, p, t, chunk);
        const int c0 = chunk * a.chunk_len;
        const bool own = pos_ok && pos >= c0 && pos < c0 + a.chunk_len;
        if (!pos_ok && chunk == 0 && kvh == 0 && lane == 0) set_error(a.err, DEV_BAD_POSITION);
        const float *tab = c.rope + (int64_t)t * hd;  // hd / 2 pairs of (cos, sin)
#pragma unroll
        for (int g = 0; g < GM; ++g)
            if (g < G) rope_lanes<CPT>(qv[g], tab, a.rope_mode, lane);
        // the token's own k (rotated) and v, appended to the cache
        float kn[CPT], vn[CPT];
#pragma unroll
        for (int e = 0; e < CPT; ++e) kn[e] = vn[e] = 0.0f;
        if (own) {
            const int64_t ld_qkv = a.q_dim + 2 * (int64_t)a.kv_dim;
            const float *kr = a.qkv + (int64_t)t * ld_qkv + a.q_dim + (int64_t)kvh * hd;
            const float *vr = kr + a.kv_dim;
#pragma unroll
            for (int e = 0; e < CPT; ++e) {
                kn[e] = __ldcg(kr + 32 * e + lane);
                vn[e] = __ldcg(vr + 32 * e + lane);
            }
            rope_lanes<CPT>(kn, tab, a.rope_mode, lane);
            const int64_t row = (int64_t)t * a.seq_stride + (int64_t)pos * a.kv_dim + (int64_t)kvh * hd;
#pragma unroll
            for (int e = 0; e < CPT; ++e) {
                a.L[l].kc[row + 32 * e + lane] = kn[e];
                a.L[l].vc[row + 32 * e + lane] = vn[e];
            }
        }
        // scores, RJ rows at a time (independent reductions in flight); lane j
        // keeps row j's score of each head
        const uint32_t ks = c.ring_s + (uint32_t)(s * a.slot_bytes);
        const uint32_t vs = ks + (uint32_t)(a.chunk_len * hd * 4);
        constexpr int RJ = GM == 1 ? 4 : 2;
        float sc[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) sc[g] = -INFINITY;
        for (int j0 = 0; j0 < n; j0 += RJ) {
            float kj[RJ][CPT];
#pragma unroll
            for (int r = 0; r < RJ; ++r) {
                const int j = j0 + r;
                const bool me = (c0 + j == pos);
#pragma unroll
                for (int e = 0; e < CPT; ++e) {
                    float v = 0.0f;
                    if (j < n)
                        asm volatile("ld.shared.f32 %0, [%1];"
                                     : "=f"(v)
                                     : "r"(ks + (uint32_t)((j * hd + 32 * e + lane) * 4)));
                    kj[r][e] = me ? kn[e] : v;
                }
            }
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
                    float dot[RJ];
#pragma unroll
                    for (int r = 0; r < RJ; ++r) {
                        dot[r] = 0.0f;
#pragma unroll
                        for (int e = 0; e < CPT; ++e) dot[r] = fmaf(qv[g][e], kj[r][e], dot[r]);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int r = 0; r < RJ; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
#pragma unroll
                    for (int r = 0; r < RJ; ++r)
                        if (lane == j0 + r && j0 + r < n) sc[g] = dot[r] * scale;
                }
            }
        }
        // chunk softmax per head
        float pr[GM], mx[GM], sm[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g < G) {
                mx[g] = warp_max(sc[g]);
                pr[g] = lane < n ? expf(sc[g] - mx[g]) : 0.0f;
                sm[g] = warp_sum(pr[g]);
            }
        }
        // weighted values
        float o[GM][CPT];
#pragma unroll
        for (int g = 0; g < GM; ++g)
#pragma unroll
            for (int e = 0; e < CPT; ++e) o[g][e] = 0.0f;
#pragma unroll 4
        for (int j = 0; j < n; ++j) {
            float vj[CPT];
            const bool me = (c0 + j == pos);
#pragma unroll
            for (int e = 0; e < CPT; ++e) {
                float v;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(vs + (uint32_t)((j * hd + 32 * e + lane) * 4)));
                vj[e] = me ? vn[e] : v;
            }
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
                    const float pj = __shfl_sync(0xffffffffu, pr[g], j);
#pragma unroll
                    for (int e = 0; e < CPT; ++e) o[g][e] = fmaf(pj, vj[e], o[g][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.empty[s]);  // this warp is done with the slot
        // the next unit's query heads are on their way while this record is written
        mine += kPWarps;
        if (mine < nunits) {
            int t2, kvh2, chunk2;
            unit_coords(a, p, p.au0 + mine, t2, kvh2, chunk2);
            load_q<CPT, GM>(a, t2, kvh2, lane, qv);
        }
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g < G) {
                float *rec = srec ? srec + ((int64_t)i * G + g) * (hd + 2) : part_rec(a, t, kvh, chunk, g);
                if (lane == 0) {
                    rec[0] = n > 0 ? mx[g] : -INFINITY;
                    rec[1] = n > 0 ? sm[g] : 0.0f;
                }
#pragma unroll
                for (int e = 0; e < CPT; ++e) rec[2 + 32 * e + lane] = o[g][e];
            }
        }
    }
    csync();  // every chunk record of this CTA is written
    attention_runs<CPT>(a, p, srec, c.warp, lane);
}

template <int CPT, int GM>
__global__ void __launch_bounds__(kPThreads, 1) decode_persistent_kernel(const __grid_constant__ PArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *xsm = smem + (int64_t)a.n_slots * a.slot_bytes;
    float *rope = reinterpret_cast<float *>(xsm + a.x_region);
    float *red = rope + a.m * a.head_dim;
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 32);
    uint64_t *empty = full + a.n_slots;
    Plan &p = *reinterpret_cast<Plan *>(empty + a.n_slots);  // in shared memory: read often, indexed
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        make_plan(a, p);
        for (int s = 0; s < a.n_slots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPWarps);  // every consumer warp releases every stage
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kPWarps) {
        producer(a, p, ring, full, empty, lane);
    } else {
        // RoPE table of every token: angle reduced modulo 2 pi in double precision
        const int half = a.head_dim / 2;
        const double l2t = log2((double)a.rope_theta);
        for (int idx = threadIdx.x; idx < a.m * half; idx += kPWarps * 32) {
            const int t = idx / half, i = idx % half;
            const int pos = pos_valid(a, p.pos[t]) ? p.pos[t] : 0;
            const double inv_freq = exp2(-(2.0 * i / a.head_dim) * l2t);
            const double ang = (double)pos * inv_freq;
            const double rd = ang - kTwoPi * rint(ang / kTwoPi);
            float sn, cs;
            sincosf((float)rd, &sn, &cs);
            rope[(t * half + i) * 2] = cs;
            rope[(t * half + i) * 2 + 1] = sn;
        }
        CCtx c;
        c.ring_s = smem_u32(ring);
        c.full = full;
        c.empty = empty;
        c.xsm = xsm;
        c.red = red;
        c.rope = rope;
        c.warp = warp;
        c.lane = lane;
        c.tid = threadIdx.x;
        csync();

        unsigned nbar = 0;
        int64_t K = 0;
        auto sync = [] { csync(); };
        // The five phases of a layer run through one call site each for the
        // staging and the GEMV, so that their code exists once (see gemv_phase).
        for (int l = 0; l < a.n_layers; ++l) {
            const PLayer &L = a.L[l];
            const float *x_in = l == 0 ? a.input : a.xbuf[(l - 1) & 1];
            float *x_out = l == a.n_layers - 1 ? a.output : a.xbuf[l & 1];
            for (int ph = 0; ph < kPhases; ++ph) {
                const int kind = phase_kind(ph);
                if (kind == K_ATT) {
                    // 4-5: attention, Q8_1 of its output
                    attention_phase<CPT, GM>(a, p, c, l, K);
                } else {
                    // 1-3: RMSNorm -> Q8_1 -> Q|K|V; 6-7: O + residual; 8-9: RMSNorm ->
                    // Q8_1 -> gate/up, silu(gate) * up; 9-10: Q8_1 of h -> down + residual
                    if (kind == K_O) {
                        const float *a8d = reinterpret_cast<const float *>(a.a8 + a.q_pad);
                        stage_x_q8<true, kPWarps>(xsm, a.a8, a8d, a8d + a.q_pad / 32, 1, a.q_pad, threadIdx.x, sync);
                    } else {
                        const float *src = kind == K_QKV ? x_in : kind == K_GU ? a.res1 : a.h;
                        const int64_t n = kind == K_DN ? a.inter : a.hidden_pad;
                        const float *gamma = kind == K_QKV ? L.attn_gamma : kind == K_GU ? L.ffn_gamma : nullptr;
                        stage_f32(xsm, src, n, gamma, gamma ? a.hidden : 0, a.eps, n, red, warp, lane);
                    }
                    const float *res = kind == K_O ? x_in : kind == K_DN ? a.res1 : nullptr;
                    float *y = kind == K_QKV ? a.qkv : kind == K_O ? a.res1 : kind == K_GU ? a.h : x_out;
                    gemv_phase(a, p, c, kind, K, res, y);
                }
                K += p.nst[kind];
                if (kind == K_DN && blockIdx.x == 0 && a.hidden_pad > a.hidden) {
                    for (int i = a.hidden + threadIdx.x; i < a.hidden_pad; i += kPWarps * 32) x_out[i] = 0.0f;
                }
                if (ph + 1 < kPhases || l + 1 < a.n_layers) grid_barrier(a, c, nbar++);
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host planning
struct HostPlan {
    bool ok;
    int slot_bytes, n_slots, ps[4], x_region, chunk_len, n_chunks;
    size_t smem;
};

int env_int(const char *name, int dflt)
{
    const char *v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}

// Packs per slot.  With one row per pack the rows are worked in pairs, so an
// odd count above one drops to the even count below it (an odd count leaves the
// last pair with a single row, worked twice).
int64_t even_packs(int64_t per, bool one_row)
{
    return (one_row && per > 1 && (per & 1)) ? per - 1 : per;
}

HostPlan host_plan(const LayerDesc &L, int64_t m, int max_seq, size_t smem_optin)
{
    HostPlan h{};
    h.ok = false;
    const int q_dim = L.n_heads * L.head_dim, kv_dim = L.n_kv_heads * L.head_dim;
    const int q_pad = (q_dim + 255) / 256 * 256;
    int64_t pack[4];
    bool rpp1[4];
    int64_t xr = 0;
    for (int k = 0; k < 4; ++k) {
        int64_t units, in_dim;
        int R;
        gemv_dims(k, q_dim, kv_dim, L.hidden, L.hidden_pad, q_pad, L.inter, units, in_dim, R);
        const int nsb = (int)(in_dim / 256);
        rpp1[k] = pack_rows_for(nsb) == 1;
        pack[k] = (int64_t)R * pack_rows_for(nsb) * nsb * kSB;
        xr = std::max(xr, x_smem_bytes(m, in_dim));
    }
    h.x_region = (int)((xr + 127) / 128 * 128);
    h.chunk_len = kAttnUnitBytes / (2 * L.head_dim * 4);
    h.n_chunks = (max_seq + h.chunk_len - 1) / h.chunk_len;
    const int64_t fixed = h.x_region + (int64_t)m * L.head_dim * 4 + 32 * 4 + 2 * 8 * kMaxSlots + kPlanBytes;
    const int64_t budget = (int64_t)smem_optin - fixed;
    double best = 0.0;
    for (int S = kAttnUnitBytes; S <= 32768; S += 128) {
        const int ns = (int)std::min<int64_t>(kMaxSlots, budget / S);
        if (ns < 4) continue;
        double fill = 1.0;
        bool fits = true;
        for (int k = 0; k < 4; ++k) {
            if (pack[k] > S) {
                fits = false;
                break;
            }
            fill = std::min(fill, (double)(even_packs(S / pack[k], rpp1[k]) * pack[k]) / S);
        }
        if (!fits) continue;
        const double score = (double)ns * S * fill;
        if (score > best) {
            best = score;
            h.slot_bytes = S;
            h.n_slots = ns;
        }
    }
    if (best <= 0.0) return h;
    for (int k = 0; k < 4; ++k) h.ps[k] = (int)even_packs(h.slot_bytes / pack[k], rpp1[k]);
    h.smem = (size_t)h.n_slots * h.slot_bytes + (size_t)fixed;
    h.ok = h.smem <= smem_optin;
    return h;
}

const void *kernel_for(int head_dim, int group)
{
    if (head_dim == 128) return group == 1 ? (const void *)decode_persistent_kernel<4, 1>
                                           : (const void *)decode_persistent_kernel<4, 8>;
    return (const void *)decode_persistent_kernel<2, 8>;
}

}  // namespace

int persistent_chunk_len(int head_dim) { return kAttnUnitBytes / (2 * head_dim * 4); }

bool persistent_decode_ok(const LayerDesc &L, int64_t m, int max_seq)
{
    if (!g_use_persistent || m != 1) return false;
    if (L.head_dim != 64 && L.head_dim != 128) return false;
    if (L.n_heads % L.n_kv_heads != 0 || L.n_heads / L.n_kv_heads > kMaxG) return false;
    // activation rows walked by the staging helpers
    if (L.hidden_pad > kPMaxRow || L.inter > kPMaxRow) return false;
    const DevInfo &d = dev_info();
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, d.device) != cudaSuccess || !coop) return false;
    return host_plan(L, m, max_seq, d.smem_optin).ok;
}

cudaError_t launch_decode_persistent(const float *input, const LayerDesc *layers, const KvDesc *kvs, int n_layers,
                                     const int32_t *positions, int position, int64_t m, float *output,
                                     const PersistentWs &ws, cudaStream_t s)
{
    const LayerDesc &L0 = layers[0];
    const DevInfo &d = dev_info();
    const HostPlan hp = host_plan(L0, m, kvs[0].max_seq, d.smem_optin);
    if (!hp.ok) return cudaErrorInvalidConfiguration;
    const void *fn = kernel_for(L0.head_dim, L0.n_heads / L0.n_kv_heads);
    {
        static std::mutex mu;
        static bool attr_done[64][3] = {};
        std::lock_guard<std::mutex> lk(mu);
        const int which = L0.head_dim == 128 ? (L0.n_heads == L0.n_kv_heads ? 0 : 1) : 2;
        if (d.device < 64 && !attr_done[d.device][which]) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
            if (e != cudaSuccess) return e;
            attr_done[d.device][which] = true;
        }
    }
    const int pf_kb = env_int("RZ_L2_PREFETCH_KB", 384);
    const float *cur = input;
    for (int g0 = 0; g0 < n_layers; g0 += kPMaxLayers) {
        const int nl = std::min(kPMaxLayers, n_layers - g0);
        PArgs a{};
        for (int i = 0; i < nl; ++i) {
            const LayerDesc &L = layers[g0 + i];
            const void *w[7] = {L.wq, L.wk, L.wv, L.wo, L.wgate, L.wup, L.wdown};
            for (int k = 0; k < 7; ++k) a.L[i].w[k] = static_cast<const uint8_t *>(w[k]);
            a.L[i].attn_gamma = L.attn_gamma;
            a.L[i].ffn_gamma = L.ffn_gamma;
            a.L[i].kc = kvs[g0 + i].k;
            a.L[i].vc = kvs[g0 + i].v;
        }
        a.n_layers = nl;
        a.m = (int)m;
        a.hidden = L0.hidden;
        a.hidden_pad = L0.hidden_pad;
        a.n_heads = L0.n_heads;
        a.n_kv_heads = L0.n_kv_heads;
        a.head_dim = L0.head_dim;
        a.inter = L0.inter;
        a.group = L0.n_heads / L0.n_kv_heads;
        a.q_dim = L0.n_heads * L0.head_dim;
        a.q_pad = (a.q_dim + 255) / 256 * 256;
        a.kv_dim = L0.n_kv_heads * L0.head_dim;
        a.eps = L0.eps;
        a.rope_theta = L0.rope_theta;
        a.rope_mode = L0.rope_mode;
        a.seq_stride = kvs[0].seq_stride;
        a.max_seq = kvs[0].max_seq;
        a.positions = positions;
        a.position = position;
        a.chunk_len = hp.chunk_len;
        a.n_chunks = hp.n_chunks;
        a.slot_bytes = hp.slot_bytes;
        a.n_slots = hp.n_slots;
        a.pf_stages = std::max(0, pf_kb * 1024 / hp.slot_bytes);
        a.x_region = hp.x_region;
        for (int k = 0; k < 4; ++k) a.ps[k] = hp.ps[k];
        a.input = cur;
        const bool last_group = g0 + nl == n_layers;
        a.output = last_group ? output : ws.gbuf[(g0 / kPMaxLayers) & 1];
        a.xbuf[0] = ws.xbuf[0];
        a.xbuf[1] = ws.xbuf[1];
        a.qkv = ws.qkv;
        a.part = ws.part;
        a.res1 = ws.res1;
        a.h = ws.h;
        a.a8 = static_cast<int8_t *>(ws.a8);
        a.counters = ws.counters;
        a.gbar = ws.gbar;
        a.err = dev_error_word();
        // grid-barrier words and merge counters start at zero in every launch
        cudaError_t e = cudaMemsetAsync(ws.counters, 0, ((size_t)m * L0.n_kv_heads + 2) * sizeof(int), s);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)d.sm_count);
        cfg.blockDim = dim3(kPThreads);
        cfg.dynamicSmemBytes = hp.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        void *args[] = {&a};
        e = cudaLaunchKernelExC(&cfg, fn, args);
        if (e != cudaSuccess) return e;
        cur = a.output;
    }
    return cudaSuccess;
}

}  // namespace rz
