// attention.cu -- RoPE, KV-cache append and split-sequence decode attention.
//
// Semantics (forward_single_full_cuda_with_cache in realizar 0.8.4
// src/gguf/cuda/clone_layer_weights.rs; incremental_attention_async in
// transformer_layer_gpu_true_dp4a, realizar 0.8.5 src/cuda/executor/cached.rs):
// q and k are rotated at the token's position, k and v are stored in the cache
// row `position`, and every query head h attends over cache rows 0..position of
// kv head h / (n_heads / n_kv_heads) with softmax(q.k / sqrt(head_dim)).
//
// RoPE pairs (2i, 2i + 1) for mode 0 and (i, i + head_dim/2) for mode 1 turn by
// position * theta^(-2i/head_dim).  Every CTA forms the cosine and sine of its
// token's pair angles itself, one pair per thread: theta^(-2i/head_dim) is the
// i-th power of r = theta^(-2/head_dim) (computed on the host), taken by binary
// powering in double precision; the angle is formed and reduced modulo 2*pi in
// double precision (positions reach thousands of radians), then sin/cos are taken
// in single precision.  A dozen double operations per thread, no table kernel and
// no dependency on one.
//
// Attention is split over the sequence in chunks of 64 cache rows (flash-
// decoding style).  The grid is one wave: CTA (z, kv head, token) works chunks
// z, z + Z, ... in turn, Z sized so that every CTA is resident at once and the
// chunks are spread evenly.  It rotates its query heads once, and the CTA that
// works the chunk holding the token's own row rotates k, writes k and v to the
// cache and uses them from shared memory.  A chunk's K and V rows arrive in
// shared memory as one TMA tensor copy each (a box of one kv head's columns over
// 64 cache rows, 32 KB at head_dim 128), and each buffer is refilled with the
// CTA's next chunk as soon as it has been read, so the copies of the next chunk
// overlap the work on this one and HBM rather than latency or a second wave of
// CTAs bounds the kernel.  Each CTA leaves per chunk the max,
// exp-sum and unnormalised weighted values; the CTA that completes the last
// chunks of a (token, kv head) -- found with an atomic
// counter, no spinning -- merges the chunks with the log-sum-exp rule and writes
// the f32 output and its Q8_1 quantisation (head_dim is a multiple of 32, so Q8_1
// blocks never straddle heads) for the O projection.  The counter is reset by the
// merging CTA.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kChunk = 64;  // cache rows per CTA
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;

__device__ __forceinline__ int token_position(const AttnArgs &a, int t)
{
    return a.positions ? a.positions[t] : a.position;
}

// cos/sin of the pair angles of position pos into tabs[i] = (cos, sin), one pair
// per thread of the CTA
__device__ __forceinline__ void rope_angles(const AttnArgs &a, int pos, float *tabs, int tid, int nthreads)
{
    const int half = a.head_dim / 2;
    for (int i = tid; i < half; i += nthreads) {
        double f = 1.0, b = a.rope_r;  // f = r^i
        for (int e = i; e; e >>= 1) {
            if (e & 1) f *= b;
            b *= b;
        }
        const double ang = (double)pos * f;
        const double red = ang - kTwoPi * rint(ang * kInvTwoPi);
        float sn, cs;
        sincosf((float)red, &sn, &cs);
        tabs[2 * i] = cs;
        tabs[2 * i + 1] = sn;
    }
}

// rotate one head (hd values at src) into dst using the token's table
__device__ __forceinline__ void rope_head(const float *src, float *dst, const float *tab, int hd,
                                          int mode, int tid, int nthreads)
{
    const int half = hd / 2;
    for (int i = tid; i < half; i += nthreads) {
        const int ia = mode == 0 ? 2 * i : i;
        const int ib = mode == 0 ? 2 * i + 1 : i + half;
        const float cs = tab[2 * i], sn = tab[2 * i + 1];
        const float x0 = src[ia], x1 = src[ib];
        dst[ia] = x0 * cs - x1 * sn;
        dst[ib] = x0 * sn + x1 * cs;
    }
}

// Partial record of one chunk for one query head: [max, sum, o[head_dim]]
__device__ __forceinline__ float *part_rec(const AttnArgs &a, int t, int kvh, int chunk, int g)
{
    const int64_t idx = (((int64_t)t * a.n_kv_heads + kvh) * a.n_chunks + chunk) * a.group + g;
    return a.part + idx * (a.head_dim + 2);
}

// `cnt` consecutive floats at p (16-byte aligned when cnt >= 4) into r
template <int CNT>
__device__ __forceinline__ void load_cols(const float *p, float (&r)[CNT])
{
    if (CNT % 4 == 0) {
#pragma unroll
        for (int e = 0; e < CNT; e += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(p + e);
            r[e] = v.x;
            r[e + 1] = v.y;
            r[e + 2] = v.z;
            r[e + 3] = v.w;
        }
    } else if (CNT == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        r[0] = v.x;
        r[1] = v.y;
    } else {
        r[0] = p[0];
    }
}

// grid (n_kv_heads, m, Z), Z <= launch_chunks chunk slots; 256 threads; CPT =
// head_dim / 32.  A chunk's K and V rows are bulk-copied into shared memory (one
// copy per row, completion counted on two mbarriers, one phase per chunk): the copy engine
// keeps the whole chunk in flight, which per-thread loads cannot (the SM's limit
// on outstanding misses held them near 2 TB/s).  Scores: warp w takes rows w,
// w + 8, ..., lane l dims l + 32 e of each (conflict-free), with the rotated query
// heads in shared memory.
// shared memory: kbuf [64][hd] | vbuf [64][hd] | qs [G][hd] | kn [hd] | vn [hd] |
//                ps [G][64] | stat [G][2] + 2 (padded to 4) | red [8][G][hd] | flag | 2 mbarriers |
//                tabs [hd/2][2] (cos, sin of the token's pair angles)
// With att_bufs == 1 (every chunk has a CTA of its own) vbuf is kbuf: the V rows
// are copied in once the scores have read the K rows, and the smaller footprint
// lets more CTAs share an SM.
template <int CPT>
__global__ void __launch_bounds__(kAttnThreads, 4) attention_chunk_kernel(const __grid_constant__ AttnArgs a)
{
    extern __shared__ __align__(128) float sm[];
    const int kvh = blockIdx.x, t = blockIdx.y, chunk = blockIdx.z;
    const int hd = a.head_dim, G = a.group;
    const int nbuf = a.att_bufs;
    float *kbuf = sm;
    float *vbuf = kbuf + (nbuf - 1) * kChunk * hd;
    float *qs = kbuf + nbuf * kChunk * hd;
    float *kn = qs + G * hd;
    float *vn = kn + hd;
    float *ps = vn + hd;
    float *stat = ps + G * kChunk;
    float *red = stat + ((2 * G + 2 + 3) & ~3);  // 16-byte aligned for the float4 stores
    int *flag = reinterpret_cast<int *>(red + 8 * G * hd);
    uint64_t *kbar = reinterpret_cast<uint64_t *>(flag + 2);
    uint64_t *vbar = kbar + 1;
    float *tabs = reinterpret_cast<float *>(vbar + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    // With the position a host value, nothing before the rotation of q depends on
    // the previous kernel: the cache rows below the position were written by
    // earlier steps, so their copies start before the wait for this step's q, k
    // and v.  With device positions everything waits.  Every global write comes
    // after the wait.
    const bool early = a.positions == nullptr;
    if (!early) pdl_wait();

    const int pos = token_position(a, t);
    const bool pos_ok = pos >= 0 && pos < a.max_seq;
    // chunks holding rows of this token; after a bad position chunk 0 alone takes
    // part and the merge writes zeros
    const int nc = pos_ok ? min(a.n_chunks, pos / kChunk + 1) : 1;
    // this CTA works chunks chunk, chunk + Z, ... below nc, in that order
    const int Z = gridDim.z;
    const int mine = chunk < nc ? (nc - 1 - chunk) / Z + 1 : 0;
    if (mine == 0) return;
    if (!pos_ok && chunk == 0 && kvh == 0 && tid == 0) set_error(a.err, DEV_BAD_POSITION);
    const float *tab = tabs;
    const float scale = 1.0f / sqrtf((float)hd);
    const int64_t kv_base = (int64_t)t * a.seq_stride + (int64_t)kvh * hd;
    auto rows_of = [&](int c) { return pos_ok ? max(0, min(kChunk, pos + 1 - c * kChunk)) : 0; };
    const int own_chunk = pos / kChunk;  // the chunk holding the new row
    const bool own = pos_ok && own_chunk >= chunk && (own_chunk - chunk) % Z == 0;

    if (rows_of(chunk) > 0) {
        // K and V rows of chunk c on their way into kbuf / vbuf: one tensor copy each
        // (a box of this kv head's columns over the chunk's 64 rows; rows past the
        // cache read as zero, rows past the position are copied but unused; the
        // token's own row is taken from kn / vn: its cache copy is written by this
        // CTA).  A buffer is refilled for the CTA's next chunk as soon as every
        // thread is done with it, so the next chunk streams in meanwhile.
        auto issue_k = [&](int c) {
            if (tid == 0) {
                mbar_arrive_expect_tx(kbar, (unsigned)(kChunk * hd * 4));
                tma_load_3d(kbuf, &a.kmap, kvh * hd, c * kChunk, t, kbar);
            }
        };
        auto issue_v = [&](int c) {
            if (tid == 0) {
                mbar_arrive_expect_tx(vbar, (unsigned)(kChunk * hd * 4));
                tma_load_3d(vbuf, &a.vmap, kvh * hd, c * kChunk, t, vbar);
            }
        };
        if (tid == 0) {
            mbar_init(kbar, 1);
            mbar_init(vbar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        issue_k(chunk);
        if (nbuf == 2) issue_v(chunk);
        rope_angles(a, pos, tabs, tid, kAttnThreads);
        if (early) pdl_wait();  // q, k and v of this step come from the previous kernel
        __syncthreads();

        // rotated query heads of this kv head, and (owner) the new row
        for (int g = 0; g < G; ++g)
            rope_head(a.q + (int64_t)t * a.ld_qkv + (int64_t)(kvh * G + g) * hd, qs + g * hd, tab, hd, a.rope_mode,
                      tid, kAttnThreads);
        if (own) {
            const float *ks = a.k + (int64_t)t * a.ld_qkv + (int64_t)kvh * hd;
            const float *vs = a.v + (int64_t)t * a.ld_qkv + (int64_t)kvh * hd;
            rope_head(ks, kn, tab, hd, a.rope_mode, tid, kAttnThreads);
            for (int i = tid; i < hd; i += kAttnThreads) vn[i] = vs[i];
        }
        __syncthreads();
        if (own) {
            float *kd = a.kc + kv_base + (int64_t)pos * a.kv_dim;
            float *vd = a.vc + kv_base + (int64_t)pos * a.kv_dim;
            for (int i = tid; i < hd; i += kAttnThreads) {
                kd[i] = kn[i];
                vd[i] = vn[i];
            }
        }

        bool ok = true;
        for (int it = 0, c = chunk; it < mine && ok; ++it, c += Z) {
            const unsigned par = (unsigned)(it & 1);
            const int c0 = c * kChunk, n = rows_of(c);
            // the K rows have landed (bounded wait; on expiry the copies are waited
            // out again before the CTA may leave, and no further chunk is started)
            if (!mbar_wait(kbar, par)) {
                if (tid == 0) set_error(a.err, DEV_TIMEOUT_ATTN);
                if (!mbar_wait(kbar, par) && tid == 0) set_error(a.err, DEV_TIMEOUT_DRAIN);
                ok = false;
            }

            // ---- scores: warp w rows w + 8 r, lane l dims l + 32 e
            for (int g = 0; g < G; ++g) {
                float qv[CPT];
#pragma unroll
                for (int e = 0; e < CPT; ++e) qv[e] = qs[g * hd + 32 * e + lane];
                float dot[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int jj = warp + 8 * r;
                    const float *kr = (c0 + jj == pos) ? kn : kbuf + jj * hd;
                    dot[r] = 0.0f;
                    if (jj < n) {
#pragma unroll
                        for (int e = 0; e < CPT; ++e) dot[r] = fmaf(qv[e], kr[32 * e + lane], dot[r]);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int r = 0; r < 8; ++r) dot[r] += __shfl_xor_sync(0xffffffffu, dot[r], o);
                if (lane == 0) {
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        if (warp + 8 * r < n) ps[g * kChunk + warp + 8 * r] = dot[r] * scale;
                }
            }
            __syncthreads();
            if (nbuf == 1)
                issue_v(c);  // the K rows are read: the buffer takes the V rows
            else if (ok && it + 1 < mine)
                issue_k(c + Z);  // kbuf is free
            // ---- chunk softmax statistics (warp per query head)
            for (int g = warp; g < G; g += kAttnThreads / 32) {
                const float v0 = lane < n ? ps[g * kChunk + lane] : -INFINITY;
                const float v1 = lane + 32 < n ? ps[g * kChunk + lane + 32] : -INFINITY;
                const float mx = warp_max(fmaxf(v0, v1));
                const float p0 = lane < n ? expf(v0 - mx) : 0.0f;
                const float p1 = lane + 32 < n ? expf(v1 - mx) : 0.0f;
                ps[g * kChunk + lane] = p0;
                ps[g * kChunk + lane + 32] = p1;
                const float sum = warp_sum(p0 + p1);
                if (lane == 0) {
                    stat[2 * g] = mx;
                    stat[2 * g + 1] = sum;
                }
            }
            // the V rows have landed
            if (!mbar_wait(vbar, par)) {
                if (tid == 0) set_error(a.err, DEV_TIMEOUT_ATTN);
                if (!mbar_wait(vbar, par) && tid == 0) set_error(a.err, DEV_TIMEOUT_DRAIN);
                ok = false;
            }
            __syncthreads();
            // ---- weighted values: 8 row groups x 32 column threads, CPT columns each
            {
                const int rg = warp, col = lane;
                for (int g = 0; g < G; ++g) {
                    float o[CPT];
#pragma unroll
                    for (int e = 0; e < CPT; ++e) o[e] = 0.0f;
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int jj = rg + 8 * r;
                        if (jj < n) {
                            float vv[CPT];
                            load_cols<CPT>(((c0 + jj == pos) ? vn : vbuf + jj * hd) + col * CPT, vv);
                            const float p = ps[g * kChunk + jj];
#pragma unroll
                            for (int e = 0; e < CPT; ++e) o[e] = fmaf(p, vv[e], o[e]);
                        }
                    }
                    float *rd = red + (rg * G + g) * hd + col * CPT;
                    if (CPT % 4 == 0) {
#pragma unroll
                        for (int e = 0; e < CPT; e += 4)
                            *reinterpret_cast<float4 *>(rd + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < CPT; ++e) rd[e] = o[e];
                    }
                }
            }
            __syncthreads();
            if (ok && it + 1 < mine) {
                if (nbuf == 1)
                    issue_k(c + Z);  // the buffer is free again
                else
                    issue_v(c + Z);  // vbuf is free
            }
            // fixed-order sum over the 8 row groups -> partial record of chunk c
            for (int i = tid; i < G * hd; i += kAttnThreads) {
                const int g = i / hd, dd = i % hd;
                float s8 = 0.0f;
#pragma unroll
                for (int r = 0; r < 8; ++r) s8 += red[(r * G + g) * hd + dd];
                part_rec(a, t, kvh, c, g)[2 + dd] = s8;
            }
            for (int g = tid; g < G; g += kAttnThreads) {
                float *rec = part_rec(a, t, kvh, c, g);
                rec[0] = stat[2 * g];
                rec[1] = stat[2 * g + 1];
            }
            __syncthreads();  // ps, stat and red are reused by the next chunk
        }
    } else {
        if (early) pdl_wait();
        for (int g = tid; g < G; g += kAttnThreads) {
            float *rec = part_rec(a, t, kvh, chunk, g);
            rec[0] = -INFINITY;
            rec[1] = 0.0f;
        }
    }

    // ---- arrive; the last chunk of (t, kvh) merges
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int *cnt = a.counters + (int64_t)t * a.n_kv_heads + kvh;
        const int prev = atomicAdd(cnt, mine);
        const int last = (prev + mine == nc);
        if (last) *cnt = 0;  // ready for the next call
        *flag = last;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();

    // The records of (t, kvh) go to shared memory first (kbuf / vbuf are free
    // now), every load of a batch in flight at once: one round trip to L2 instead
    // of one per few chunks.  Records of a query head are rows of hd + 4 floats
    // (max, sum, o[hd], pad); as many heads per batch as fit in the K/V buffers
    // (one head always fits: nc <= 64 with two buffers, checked at launch with one).
    float *wts = ps;   // [G][kChunk]: chunk weights exp(m_c - M)
    float *outv = red;  // merged output [G][hd]
    float *rs = kbuf;
    const int rstride = hd + 4;
    const int gb = max(1, min(G, (nbuf * kChunk * hd) / (nc * rstride)));  // >= 1 head: checked at launch
    constexpr int kRecLanes = CPT + 1;  // 32 * kRecLanes >= hd + 2
    constexpr int kRecsInFlight = 4;    // per warp
    for (int g0 = 0; g0 < G; g0 += gb) {
        const int ng = min(gb, G - g0), nrec = ng * nc;
        for (int r0 = 0; r0 < nrec; r0 += kRecsInFlight * (kAttnThreads / 32)) {
            float v[kRecsInFlight][kRecLanes];
#pragma unroll
            for (int u = 0; u < kRecsInFlight; ++u) {
                const int r = r0 + warp + (kAttnThreads / 32) * u;
                const float *src = part_rec(a, t, kvh, r < nrec ? r % nc : 0, g0 + (r < nrec ? r / nc : 0));
#pragma unroll
                for (int k = 0; k < kRecLanes; ++k) {
                    const int e = lane + 32 * k;
                    v[u][k] = (r < nrec && e < hd + 2) ? __ldcg(src + e) : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < kRecsInFlight; ++u) {
                const int r = r0 + warp + (kAttnThreads / 32) * u;
                if (r < nrec) {
#pragma unroll
                    for (int k = 0; k < kRecLanes; ++k) {
                        const int e = lane + 32 * k;
                        if (e < hd + 2) rs[r * rstride + e] = v[u][k];
                    }
                }
            }
        }
        __syncthreads();
        // chunk statistics (warp per query head, lane per chunk), then the weights
        for (int gl = warp; gl < ng; gl += kAttnThreads / 32) {
            const int g = g0 + gl;
            float mc[2], lc[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = lane + 32 * h;
                mc[h] = c < nc ? rs[(gl * nc + c) * rstride] : -INFINITY;
                lc[h] = c < nc ? rs[(gl * nc + c) * rstride + 1] : 0.0f;
            }
            const float M = warp_max(fmaxf(mc[0], mc[1]));
            float lsum = 0.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = lane + 32 * h;
                const float w = (c < nc && lc[h] > 0.0f) ? expf(mc[h] - M) : 0.0f;
                if (c < kChunk) wts[g * kChunk + c] = w;
                lsum += w * lc[h];
            }
            lsum = warp_sum(lsum);
            if (lane == 0) stat[2 * g] = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;  // 0 only after a bad position
        }
        __syncthreads();
        // weighted sum over the chunks in chunk order (every record c < nc is
        // written and finite; a zero weight adds exactly nothing)
        for (int i = tid; i < ng * hd; i += kAttnThreads) {
            const int gl = i / hd, dd = i % hd, g = g0 + gl;
            const float *col = rs + gl * nc * rstride + 2 + dd;
            float acc = 0.0f;
            for (int c = 0; c < nc; ++c) acc = fmaf(col[c * rstride], wts[g * kChunk + c], acc);
            outv[g * hd + dd] = acc * stat[2 * g];
        }
        __syncthreads();
    }
    const int64_t col0 = (int64_t)kvh * G * hd;
    if (a.att) {
        for (int i = tid; i < G * hd; i += kAttnThreads) a.att[(int64_t)t * a.q_dim + col0 + i] = outv[i];
    }
    if (a.att_q8) {
        // Q8_1 of the merged output: warp per block of 32
        int8_t *q = static_cast<int8_t *>(a.att_q8);
        float *qd = reinterpret_cast<float *>(q + (int64_t)a.m * a.q_pad);
        float *qsum = qd + (int64_t)a.m * (a.q_pad / 32);
        const int nblk = G * hd / 32;
        for (int b = warp; b < nblk; b += kAttnThreads / 32) {
            const float v = outv[b * 32 + lane];
            const float amax = warp_max(fabsf(v));
            const float dq = __fdiv_rn(amax, 127.0f);
            const int qi = q8_code(v, dq, rcp_approx(dq));
            const int sum = warp_sum_int(qi);
            const int64_t blk = (col0 / 32) + b;
            q[(int64_t)t * a.q_pad + blk * 32 + lane] = (int8_t)qi;
            if (lane == 0) {
                qd[(int64_t)t * (a.q_pad / 32) + blk] = dq;
                qsum[(int64_t)t * (a.q_pad / 32) + blk] = __fmul_rn(dq, (float)sum);
            }
        }
        // zero padding blocks q_dim .. q_pad (written once per token)
        if (kvh == 0) {
            for (int64_t i = a.q_dim + tid; i < a.q_pad; i += kAttnThreads) q[(int64_t)t * a.q_pad + i] = 0;
            for (int64_t b = a.q_dim / 32 + tid; b < a.q_pad / 32; b += kAttnThreads) {
                qd[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
                qsum[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
            }
        }
    }
}

cudaError_t launch_ex(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// CTAs of kernel fn resident on the whole GPU at `smem` bytes of dynamic shared
// memory (cached: the first launch of each configuration asks the runtime).
int resident_ctas(const void *fn, size_t smem)
{
    struct Entry {
        const void *fn;
        size_t smem;
        int dev, n;
    };
    static Entry cache[16];
    static int used = 0;
    static std::mutex mu;
    const int dev = dev_info().device;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].smem == smem && cache[i].dev == dev) return cache[i].n;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kAttnThreads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    const int n = std::max(1, per_sm) * dev_info().sm_count;
    if (used < 16) cache[used++] = Entry{fn, smem, dev, n};
    return n;
}

}  // namespace

int attention_chunk_len(int, int, int) { return kChunk; }

size_t attention_smem_bytes_n(int group, int head_dim, int nbuf)
{
    return ((size_t)nbuf * kChunk * head_dim + (size_t)group * head_dim + 2 * (size_t)head_dim +
            (size_t)group * kChunk + ((2 * (size_t)group + 2 + 3) & ~(size_t)3) + 8 * (size_t)group * head_dim) *
               sizeof(float) +
           16 + 16 + (size_t)head_dim * sizeof(float);  // flag (+ pad), two mbarriers, the pair angles
}

size_t attention_smem_bytes(int group, int head_dim, int) { return attention_smem_bytes_n(group, head_dim, 2); }

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s)
{
    AttnArgs args = a;
    void *kargs[] = {&args};
    {
        // the caches as [m][max_seq][kv_dim] f32 tensors; a box is one head x 64 rows
        const uint64_t seq = a.m > 1 ? (uint64_t)a.seq_stride * 4 : (uint64_t)a.max_seq * a.kv_dim * 4;
        const uint64_t dims[3] = {(uint64_t)a.kv_dim, (uint64_t)a.max_seq, (uint64_t)a.m};
        const uint64_t strides[2] = {(uint64_t)a.kv_dim * 4, seq};
        const uint32_t box[3] = {(uint32_t)a.head_dim, (uint32_t)kChunk, 1u};
        cudaError_t e = encode_tensor_map(&args.kmap, a.kc, 4, 3, dims, strides, box);
        if (e == cudaSuccess) e = encode_tensor_map(&args.vmap, a.vc, 4, 3, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    const void *fn = a.head_dim == 32    ? (const void *)attention_chunk_kernel<1>
                     : a.head_dim == 64  ? (const void *)attention_chunk_kernel<2>
                     : a.head_dim == 128 ? (const void *)attention_chunk_kernel<4>
                                         : (const void *)attention_chunk_kernel<8>;
    if (attention_smem_bytes_n(a.group, a.head_dim, 2) > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
    }
    // One wave.  Else, when every chunk can have a resident CTA of its own with K
    // and V through one buffer (and the merge's records fit in it), that; else as many
    // chunk slots per (kv head, token) as resident CTAs allow with two buffers,
    // the chunks spread evenly over them (each CTA streams its chunks in turn).
    // With two buffers V streams in beside K; when every chunk can have a CTA of
    // its own that way (short positions, small grids), that comes first.
    const int per_z = a.n_kv_heads * a.m;
    const size_t smem1 = attention_smem_bytes_n(a.group, a.head_dim, 1);
    const bool two_all = resident_ctas(fn, attention_smem_bytes_n(a.group, a.head_dim, 2)) >= per_z * a.launch_chunks;
    const bool one = !two_all && resident_ctas(fn, smem1) >= per_z * a.launch_chunks &&
                     (size_t)a.n_chunks * (a.head_dim + 4) <= (size_t)kChunk * a.head_dim;
    args.att_bufs = one ? 1 : 2;
    const size_t smem = one ? smem1 : attention_smem_bytes_n(a.group, a.head_dim, 2);
    const int zcap = std::max(1, resident_ctas(fn, smem) / per_z);
    int Z = std::min(a.launch_chunks, zcap);
    const int per_cta = (a.launch_chunks + Z - 1) / Z;
    Z = (a.launch_chunks + per_cta - 1) / per_cta;
    return launch_ex(fn, dim3((unsigned)a.n_kv_heads, (unsigned)a.m, (unsigned)Z), dim3(kAttnThreads), smem, s,
                     kargs);
}

}  // namespace rz
