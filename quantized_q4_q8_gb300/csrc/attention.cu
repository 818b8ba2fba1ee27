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
// tokens' pair angles itself: theta^(-2i/head_dim) is the i-th power of r =
// theta^(-2/head_dim), taken on the host by binary powering in double precision
// and passed with the arguments; the angle is formed and reduced modulo 2*pi in
// double precision (positions reach thousands of radians), then sin/cos are taken
// in single precision.  Four double operations per pair, no table kernel and no
// dependency on one.
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

// cos and sin of pair i's angle at position pos
__device__ __forceinline__ void rope_pair(const AttnArgs &a, int pos, int i, float &cs, float &sn)
{
    const double ang = (double)pos * a.rope_f[i];
    const double red = ang - kTwoPi * rint(ang * kInvTwoPi);
    sincosf((float)red, &sn, &cs);
}

// cos/sin of the pair angles of position pos into tabs[i] = (cos, sin), one pair
// per thread of the CTA
__device__ __forceinline__ void rope_angles(const AttnArgs &a, int pos, float *tabs, int tid, int nthreads)
{
    const int half = a.head_dim / 2;
    for (int i = tid; i < half; i += nthreads) rope_pair(a, pos, i, tabs[2 * i], tabs[2 * i + 1]);
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

// The merged output of (token t, kv head kvh): the G query heads' hd values at
// outv, in shared memory.  Writes the f32 rows and the Q8_1 quantisation of them
// (a warp per block of 32; head_dim is a multiple of 32, so no block straddles
// two heads) and, once per token (kv head 0), the zero padding q_dim .. q_pad.
// Every thread of a 256-thread CTA takes part.
__device__ __forceinline__ void write_outputs(const AttnArgs &a, int t, int kvh, const float *outv, int tid,
                                              int warp, int lane)
{
    const int hd = a.head_dim, G = a.group;
    const int64_t col0 = (int64_t)kvh * G * hd;
    if (a.att) {
        for (int i = tid; i < G * hd; i += kAttnThreads) a.att[(int64_t)t * a.q_dim + col0 + i] = outv[i];
    }
    if (a.att_q8) {
        int8_t *q = static_cast<int8_t *>(a.att_q8);
        float *qd = reinterpret_cast<float *>(q + (int64_t)a.m * a.q_pad);
        float *qsum = qd + (int64_t)a.m * (a.q_pad / 32);
        const int nblk = G * hd / 32;
        for (int b = warp; b < nblk; b += kAttnThreads / 32) {
            const float v = outv[b * 32 + lane];
            const float amax = warp_max(fabsf(v));
            const float dq = __fdiv_rn(amax, 127.0f);
            const int qi = q8_code(v, q8_scale(dq));
            const int sum = warp_sum_int(qi);
            const int64_t blk = (col0 / 32) + b;
            q[(int64_t)t * a.q_pad + blk * 32 + lane] = (int8_t)qi;
            if (lane == 0) {
                qd[(int64_t)t * (a.q_pad / 32) + blk] = dq;
                qsum[(int64_t)t * (a.q_pad / 32) + blk] = __fmul_rn(dq, (float)sum);
            }
        }
        if (kvh == 0) {
            for (int64_t i = a.q_dim + tid; i < a.q_pad; i += kAttnThreads) q[(int64_t)t * a.q_pad + i] = 0;
            for (int64_t b = a.q_dim / 32 + tid; b < a.q_pad / 32; b += kAttnThreads) {
                qd[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
                qsum[(int64_t)t * (a.q_pad / 32) + b] = 0.0f;
            }
        }
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
    write_outputs(a, t, kvh, outv, tid, warp, lane);
}

// ---------------------------------------------------------------- streaming kernel
// For a decode step the rows to read -- for token t and kv head h, the cache rows
// 0 .. position_t of that head: a "segment" -- are cut into tiles of 8 rows (the
// last one of a segment may be short), the tiles laid end to end (token-major,
// then kv head) into one flat sequence of W tiles, and warp g of the PW warps of
// the grid takes tiles [g W / PW, (g + 1) W / PW).  Every SM reads the same
// number of rows (to a tile per warp) whatever the positions, the group size or
// the number of tokens.  A warp streams its tiles through a ring of its own (one
// TMA tensor copy for the K rows and one for the V rows of a tile, a few tiles in
// flight), keeps an online softmax per query head of the segment it is in
// (running maximum, exp-sum and weighted values), and leaves one record per
// segment piece it covered.  No warp waits for another until its CTA is done;
// then the CTA counts itself in for each segment it touched (an atomic counter
// per segment, one lane per segment, no spinning), and the CTA that completes a
// segment merges the segment's records with the log-sum-exp rule (each warp
// combines its share of the records in registers, then the warps' partials are
// combined in a fixed order) and writes the outputs.  The token's own row is
// taken from this step's projections: the warp holding the segment's last tile
// rotates the new k, stores k and v to the cache and puts them in the tile.
constexpr int kSW = 8;                 // warps of a CTA (the output writer wants 256 threads)
constexpr int kTR = 8;                 // cache rows per tile
constexpr int kMaxStreamWarps = 2048;  // record slots per segment are sized for this many warps in a grid
constexpr int kMaxSlots = 6;           // tiles in flight per warp
constexpr int kRecPad = 4;             // a record: max, exp-sum, 2 pad floats, then head_dim weighted values
constexpr int kMB = 8;                 // records a warp holds in registers at once while merging

__device__ __forceinline__ int token_rows(const AttnArgs &a, int t, bool &ok)
{
    const int p = token_position(a, t);
    ok = p >= 0 && p < a.max_seq;
    return ok ? p + 1 : 1;  // a bad position keeps one row, never read; its output is zero
}
__device__ __forceinline__ int seg_tiles(int n) { return (n + kTR - 1) / kTR; }

// Part g of the N equal parts of [0, W): [g W / N, (g + 1) W / N).
__device__ __forceinline__ int64_t part_start(int64_t g, int64_t W, int64_t N) { return g * W / N; }
// The part holding x.
__device__ __forceinline__ int64_t part_of(int64_t x, int64_t W, int64_t N)
{
    return min(N - 1, ((x + 1) * N + W - 1) / W - 1);
}
// The non-empty parts meeting [A, A + n): how many, and the rank of part g among them.
__device__ void cover(int64_t A, int64_t n, int64_t W, int64_t N, int64_t g, int &count, int &rank)
{
    const int64_t lo = part_of(A, W, N), hi = part_of(A + n - 1, W, N);
    if (W >= N) {  // no part is empty
        count = (int)(hi - lo + 1);
        rank = (int)(g - lo);
        return;
    }
    count = 0;
    rank = 0;
    for (int64_t p = lo; p <= hi; ++p)
        if (part_start(p + 1, W, N) > part_start(p, W, N)) {
            if (p < g) ++rank;
            ++count;
        }
}

// A segment: token t, kv head kvh, n rows in nt tiles from flat tile seg0.
struct Seg {
    int t, kvh, n, nt;
    bool ok;       // the token's position is valid
    int64_t seg0;
};
// Segment s (= t * n_kv_heads + kvh).
__device__ Seg seg_of(const AttnArgs &a, int s)
{
    Seg g;
    g.t = s / a.n_kv_heads;
    g.kvh = s % a.n_kv_heads;
    int64_t acc = 0;
    for (int t = 0; t < g.t; ++t) {
        bool ok;
        acc += (int64_t)a.n_kv_heads * seg_tiles(token_rows(a, t, ok));
    }
    g.n = token_rows(a, g.t, g.ok);
    g.nt = seg_tiles(g.n);
    g.seg0 = acc + (int64_t)g.kvh * g.nt;
    return g;
}
// The segment holding flat tile x.
__device__ int seg_at(const AttnArgs &a, int64_t x)
{
    int64_t acc = 0;
    for (int t = 0;; ++t) {
        bool ok;
        const int64_t nt = seg_tiles(token_rows(a, t, ok));
        if (t + 1 == a.m || x < acc + a.n_kv_heads * nt) return t * a.n_kv_heads + (int)((x - acc) / nt);
        acc += a.n_kv_heads * nt;
    }
}

// A walk over a range of flat tiles.
struct Cursor {
    Seg g;
    int j;           // tile of the segment
    int64_t x, end;  // flat tile, end of the range
};
struct Tile {
    int t, kvh, r0, cnt, n, seg;
    bool ok, last;   // last: the range's last tile of this segment
    int64_t seg0, nt;
};

__device__ void cursor_at(const AttnArgs &a, Cursor &c, int64_t x, int64_t end)
{
    c.g = seg_of(a, seg_at(a, x));
    c.j = (int)(x - c.g.seg0);
    c.x = x;
    c.end = end;
}

__device__ Tile cursor_next(const AttnArgs &a, Cursor &c)
{
    Tile tl;
    tl.t = c.g.t;
    tl.kvh = c.g.kvh;
    tl.seg = c.g.t * a.n_kv_heads + c.g.kvh;
    tl.n = c.g.n;
    tl.nt = c.g.nt;
    tl.ok = c.g.ok;
    tl.seg0 = c.g.seg0;
    tl.r0 = c.j * kTR;
    tl.cnt = min(kTR, c.g.n - tl.r0);
    ++c.j;
    ++c.x;
    tl.last = c.j == c.g.nt || c.x == c.end;
    if (c.j == c.g.nt && c.x < c.end) {  // on to the next segment
        c.j = 0;
        const int64_t next0 = c.g.seg0 + c.g.nt;
        if (++c.g.kvh == a.n_kv_heads) {
            c.g.kvh = 0;
            ++c.g.t;
            c.g.n = token_rows(a, c.g.t, c.g.ok);
            c.g.nt = seg_tiles(c.g.n);
        }
        c.g.seg0 = next0;
    }
    return tl;
}

// Sum over the 32 lanes of each of 8 values; lane l returns the sum of value
// (l >> 2) & 7.  Three halving exchanges (offsets 16, 8, 4) then a butterfly over
// the last two lane bits: 9 shuffles instead of 40.
__device__ __forceinline__ float reduce8(const float (&v)[kTR], int lane)
{
    constexpr unsigned kAll = 0xffffffffu;
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float h[4], q[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(kAll, b4 ? v[i] : v[i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) q[i] = (b3 ? h[i + 2] : h[i]) + __shfl_xor_sync(kAll, b3 ? h[i] : h[i + 2], 8);
    float s = (b2 ? q[1] : q[0]) + __shfl_xor_sync(kAll, b2 ? q[0] : q[1], 4);
    s += __shfl_xor_sync(kAll, s, 2);
    s += __shfl_xor_sync(kAll, s, 1);
    return s;
}

// Rotate this lane's CPT values (dims lane * CPT + e of one head) by the pair
// angles of tab ([head_dim / 2][cos, sin] of the token's position); the partner of
// a value sits in the same lane (mode 0, CPT >= 2) or in lane l ^ 1 (mode 0, CPT
// == 1) or l ^ 16 (mode 1).
template <int CPT>
__device__ __forceinline__ void rope_lane(float (&x)[CPT], const float *tab, int mode, int lane)
{
    constexpr unsigned kAll = 0xffffffffu;
    constexpr int half = CPT * 16;
    float xp[CPT];
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
        if (mode == 0)
            xp[e] = CPT == 1 ? __shfl_xor_sync(kAll, x[e], 1) : x[e ^ 1];
        else
            xp[e] = __shfl_xor_sync(kAll, x[e], 16);
    }
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
        const int d = lane * CPT + e;
        const int i = mode == 0 ? d >> 1 : (d < half ? d : d - half);
        const bool first = mode == 0 ? (d & 1) == 0 : d < half;
        const float cs = tab[2 * i], sn = tab[2 * i + 1];
        x[e] = first ? x[e] * cs - xp[e] * sn : xp[e] * sn + x[e] * cs;
    }
}

template <int CPT>
__device__ __forceinline__ void ld_lane(const float *p, float (&v)[CPT])
{
    if constexpr (CPT == 4) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
    } else if constexpr (CPT == 2) {
        const float2 u = *reinterpret_cast<const float2 *>(p);
        v[0] = u.x, v[1] = u.y;
    } else {
#pragma unroll
        for (int e = 0; e < CPT; ++e) v[e] = p[e];
    }
}
template <int CPT>
__device__ __forceinline__ void ldcg_lane(const float *p, float (&v)[CPT])
{
    if constexpr (CPT == 4) {
        const float4 u = __ldcg(reinterpret_cast<const float4 *>(p));
        v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
    } else if constexpr (CPT == 2) {
        const float2 u = __ldcg(reinterpret_cast<const float2 *>(p));
        v[0] = u.x, v[1] = u.y;
    } else {
#pragma unroll
        for (int e = 0; e < CPT; ++e) v[e] = __ldcg(p + e);
    }
}
template <int CPT>
__device__ __forceinline__ void st_lane(float *p, const float (&v)[CPT])
{
    if constexpr (CPT == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (CPT == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int e = 0; e < CPT; ++e) p[e] = v[e];
    }
}

// atomicAdd with acquire-release semantics at GPU scope (no separate fence).
__device__ __forceinline__ int atom_add_acq_rel(int *p, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Records of segment seg: rank k, query head g.
__device__ __forceinline__ float *stream_rec(const AttnArgs &a, int seg, int k, int g)
{
    return a.part + (((int64_t)seg * a.stream_kmax + k) * a.group + g) * (a.head_dim + kRecPad);
}

// Merge of segment sg by a whole CTA.  Warp w combines records w, w + 8, ... into
// a partial (max, exp-sum, weighted values) in registers -- the loads of up to kMB
// records in flight at once -- and the partials are combined in warp order.
template <int CPT>
__device__ void stream_merge(const AttnArgs &a, float *sm, const Seg &sg, int K, int tid, int warp, int lane)
{
    constexpr int hd = CPT * 32;
    const int G = a.group, seg = sg.t * a.n_kv_heads + sg.kvh;
    float *pacc = sm;                    // [kSW][G][hd]
    float *pml = pacc + kSW * G * hd;    // [kSW][G][2]: max, exp-sum
    float *outv = pml + kSW * G * 2;     // [G][hd]
    for (int g = 0; g < G; ++g) {
        float mw = -INFINITY, lw = 0.0f, acc[CPT];
#pragma unroll
        for (int e = 0; e < CPT; ++e) acc[e] = 0.0f;
        for (int k0 = warp; k0 < K; k0 += kSW * kMB) {
            float mk[kMB], lk[kMB], ov[kMB][CPT];
#pragma unroll
            for (int i = 0; i < kMB; ++i) {
                const int k = k0 + kSW * i;
                mk[i] = -INFINITY;
                lk[i] = 0.0f;
#pragma unroll
                for (int e = 0; e < CPT; ++e) ov[i][e] = 0.0f;
                if (k < K) {
                    const float *r = stream_rec(a, seg, k, g);
                    mk[i] = __ldcg(r);
                    lk[i] = __ldcg(r + 1);
                    ldcg_lane<CPT>(r + kRecPad + lane * CPT, ov[i]);
                }
            }
            float bm = mw;
#pragma unroll
            for (int i = 0; i < kMB; ++i)
                if (lk[i] > 0.0f) bm = fmaxf(bm, mk[i]);
            const float sc = lw > 0.0f ? expf(mw - bm) : 0.0f;
            lw *= sc;
#pragma unroll
            for (int e = 0; e < CPT; ++e) acc[e] *= sc;
#pragma unroll
            for (int i = 0; i < kMB; ++i) {
                const float w = lk[i] > 0.0f ? expf(mk[i] - bm) : 0.0f;  // an empty record adds nothing
                lw = fmaf(w, lk[i], lw);
#pragma unroll
                for (int e = 0; e < CPT; ++e) acc[e] = fmaf(w, ov[i][e], acc[e]);
            }
            mw = bm;
        }
        st_lane<CPT>(pacc + (warp * G + g) * hd + lane * CPT, acc);
        if (lane == 0) {
            pml[(warp * G + g) * 2] = mw;
            pml[(warp * G + g) * 2 + 1] = lw;
        }
    }
    __syncthreads();
    for (int i = tid; i < G * hd; i += kSW * 32) {
        const int g = i / hd;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSW; ++w)
            if (pml[(w * G + g) * 2 + 1] > 0.0f) M = fmaxf(M, pml[(w * G + g) * 2]);
        float v = 0.0f, L = 0.0f;
#pragma unroll
        for (int w = 0; w < kSW; ++w) {
            const float lw = pml[(w * G + g) * 2 + 1];
            const float sc = lw > 0.0f ? expf(pml[(w * G + g) * 2] - M) : 0.0f;
            v = fmaf(sc, pacc[(w * G + g) * hd + i % hd], v);
            L = fmaf(sc, lw, L);
        }
        outv[i] = v * (L > 0.0f ? 1.0f / L : 0.0f);  // L == 0 only after a bad position
    }
    __syncthreads();
    write_outputs(a, sg.t, sg.kvh, outv, tid, warp, lane);
}

// Tile tl into slot s of a warp's ring: one tensor copy for its K rows, one for its
// V rows (a tile holding only the token's own row needs none).  Lane 0 alone.
__device__ __forceinline__ void issue_tile(const AttnArgs &a, float *ring, uint64_t *bars, const Tile &tl, int s,
                                           int hd, int lane)
{
    if (lane == 0) {
        const bool copy = tl.ok && tl.r0 + 1 < tl.n;
        float *kd = ring + s * 2 * kTR * hd;
        mbar_arrive_expect_tx(&bars[s], copy ? (unsigned)(2 * kTR * hd * 4) : 0u);
        if (copy) {
            tma_load_3d(kd, &a.kmap, tl.kvh * hd, tl.r0, tl.t, &bars[s]);
            tma_load_3d(kd + kTR * hd, &a.vmap, tl.kvh * hd, tl.r0, tl.t, &bars[s]);
        }
    }
}

// Online-softmax state of one warp for the query heads of one segment.
template <int CPT, int GM>
struct WarpState {
    float q[GM][CPT], o[GM][CPT], m[GM], l[GM];
};

// The tile loop of one warp.  Tiles come from cursor cc; the copies run ahead
// through cursor ic (`issued` tiles issued so far) in the warp's NS ring slots.
// At the end of each segment piece emit(tile, state) is called.  tabs holds the
// angle tables of tokens t_a .. t_a + ntab - 1.  Returns false after a wait ran
// out (the copies in flight have been waited out again).
template <int CPT, int GM, typename Emit>
__device__ __forceinline__ bool warp_tiles(const AttnArgs &a, float *ring, uint64_t *bars, int NS, Cursor &ic,
                                           Cursor &cc, int issued, const float *tabs, int t_a, int ntab, int lane,
                                           Emit &&emit)
{
    constexpr int hd = CPT * 32;
    constexpr unsigned kAll = 0xffffffffu;
    constexpr int slot_f = 2 * kTR * hd;
    const int G = a.group;
    const float scale = 1.0f / sqrtf((float)hd);
    WarpState<CPT, GM> st;
    float kn[CPT], vn[CPT];  // the token's own k (rotated) and v
    bool own_seg = false;
    int cur = -1;            // segment of the running state
    for (int done = 0; cc.x < cc.end; ++done) {
        const Tile tl = cursor_next(a, cc);
        const int s = done % NS;
        const int tt = tl.t - t_a;
        const bool use = tl.ok && tt < ntab;
        const float *tab = tabs + (size_t)min(tt, max(ntab - 1, 0)) * hd;
        if (tl.seg != cur) {
            // a new segment: its query heads and, when the range ends the segment, the
            // token's own k and v -- every load issued before any is used
            cur = tl.seg;
            own_seg = use && tl.seg0 + tl.nt <= cc.end;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                st.m[g] = -INFINITY;
                st.l[g] = 0.0f;
#pragma unroll
                for (int e = 0; e < CPT; ++e) st.o[g][e] = st.q[g][e] = 0.0f;
                if (use && g < G)
                    ld_lane<CPT>(a.q + (int64_t)tl.t * a.ld_qkv + (int64_t)(tl.kvh * G + g) * hd + lane * CPT, st.q[g]);
            }
            if (own_seg) {
                const int64_t src = (int64_t)tl.t * a.ld_qkv + (int64_t)tl.kvh * hd + lane * CPT;
                ld_lane<CPT>(a.k + src, kn);
                ld_lane<CPT>(a.v + src, vn);
            }
#pragma unroll
            for (int g = 0; g < GM; ++g)
                if (use && g < G) rope_lane<CPT>(st.q[g], tab, a.rope_mode, lane);
            if (own_seg) {
                // k rotated; k and v stored to the cache row of the token's position
                rope_lane<CPT>(kn, tab, a.rope_mode, lane);
                const int64_t dst =
                    (int64_t)tl.t * a.seq_stride + (int64_t)(tl.n - 1) * a.kv_dim + (int64_t)tl.kvh * hd + lane * CPT;
                st_lane<CPT>(a.kc + dst, kn);
                st_lane<CPT>(a.vc + dst, vn);
            }
        }
        // the segment's last tile holds the token's own row
        const bool own = own_seg && tl.r0 + tl.cnt == tl.n;
        if (!__all_sync(kAll, mbar_wait(&bars[s], (unsigned)((done / NS) & 1)))) {
            if (lane == 0) set_error(a.err, DEV_TIMEOUT_ATTN);
            // the copies still in flight must land before the CTA may leave
            for (int j = done; j < issued; ++j)
                if (!__all_sync(kAll, mbar_wait(&bars[j % NS], (unsigned)((j / NS) & 1))) && lane == 0)
                    set_error(a.err, DEV_TIMEOUT_DRAIN);
            return false;
        }
        if (use) {
            float *kt = ring + s * slot_f, *vt = kt + kTR * hd;
            if (own) {
                // the token's own row goes into its place in the tile (the copy brought
                // the cache's old row); each lane writes and later reads only its columns
                st_lane<CPT>(kt + (tl.cnt - 1) * hd + lane * CPT, kn);
                st_lane<CPT>(vt + (tl.cnt - 1) * hd + lane * CPT, vn);
            }
            float kr[kTR][CPT], vr[kTR][CPT];
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                // rows past cnt are not the segment's: their scores are masked, their values skipped
                ld_lane<CPT>(kt + r * hd + lane * CPT, kr[r]);
                ld_lane<CPT>(vt + r * hd + lane * CPT, vr[r]);
            }
            const int rr = (lane >> 2) & 7;  // the row whose score this lane holds
            // every head slot of GM in one straight run (slots past the group hold q = 0 and
            // are never written out), so the heads' shuffle chains interleave
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float dot[kTR];
#pragma unroll
                for (int r = 0; r < kTR; ++r) {
                    dot[r] = 0.0f;
#pragma unroll
                    for (int e = 0; e < CPT; ++e) dot[r] = fmaf(st.q[g][e], kr[r][e], dot[r]);
                }
                const float full = reduce8(dot, lane);  // every lane takes part in the shuffles
                const float sc = rr < tl.cnt ? full * scale : -INFINITY;
                float mx = fmaxf(sc, __shfl_xor_sync(kAll, sc, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 16));
                const float mnew = fmaxf(st.m[g], mx);
                const float alpha = expf(st.m[g] - mnew);  // 0 on the segment's first tile
                const float p = rr < tl.cnt ? expf(sc - mnew) : 0.0f;
                float ps = p + __shfl_xor_sync(kAll, p, 4);
                ps += __shfl_xor_sync(kAll, ps, 8);
                ps += __shfl_xor_sync(kAll, ps, 16);
                st.l[g] = fmaf(st.l[g], alpha, ps);
                st.m[g] = mnew;
#pragma unroll
                for (int e = 0; e < CPT; ++e) st.o[g][e] *= alpha;
#pragma unroll
                for (int r = 0; r < kTR; ++r) {
                    const float pr = __shfl_sync(kAll, p, r * 4);
                    if (r < tl.cnt) {
#pragma unroll
                        for (int e = 0; e < CPT; ++e) st.o[g][e] = fmaf(pr, vr[r][e], st.o[g][e]);
                    }
                }
            }
        }
        // the slot is read: refill it with the range's next tile
        fence_proxy_async_smem();
        __syncwarp();
        if (ic.x < ic.end) {
            issue_tile(a, ring, bars, cursor_next(a, ic), s, hd, lane);
            ++issued;
        }
        if (tl.last) {
            emit(tl, st);
            cur = -1;
        }
    }
    return true;
}

// Angle tables of tokens t_a .. t_a + ntab - 1 into tabs, by every thread of the CTA.
__device__ __forceinline__ void stream_tables(const AttnArgs &a, float *tabs, int t_a, int ntab, int half, int tid,
                                              int nthreads)
{
    for (int i = tid; i < ntab * half; i += nthreads) {
        bool ok;
        const int n = token_rows(a, t_a + i / half, ok);
        rope_pair(a, ok ? n - 1 : 0, i % half, tabs[2 * i], tabs[2 * i + 1]);
    }
}

// grid P <= SMs CTAs of kSW warps, one CTA per SM; CPT = head_dim / 32; GM >= group.
// kmap / vmap: the caches with boxes of one head x kTR rows.
// shared memory: per warp stream_slots tiles [K rows | V rows] of kTR x head_dim
// floats | tabs [stream_tab_tokens][head_dim / 2][cos, sin] | kSW x stream_slots
// mbarriers | the segments to merge (32 flags).
template <int CPT, int GM>
__global__ void __launch_bounds__(kSW * 32, 1) attention_stream_kernel(const __grid_constant__ AttnArgs a)
{
    constexpr int hd = CPT * 32, half = hd / 2;
    constexpr unsigned kAll = 0xffffffffu;
    constexpr int slot_f = 2 * kTR * hd;
    extern __shared__ __align__(128) float sm[];
    const int NS = a.stream_slots, G = a.group, nkv = a.n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *ring = sm + (size_t)warp * NS * slot_f;
    float *tabs = sm + (size_t)kSW * NS * slot_f;
    uint64_t *bar0 = reinterpret_cast<uint64_t *>(tabs + (size_t)a.stream_tab_tokens * hd);
    uint64_t *bars = bar0 + warp * NS;
    unsigned *mflags = reinterpret_cast<unsigned *>(bar0 + kSW * NS);
    pdl_launch_dependents();
    // With the position a host value nothing before the rotation of q depends on
    // the previous kernel (the cache rows below the position were written by
    // earlier steps): the first tiles' copies and the angle table start before the
    // wait for this step's q, k and v.  With device positions everything waits.
    // Every global write comes after the wait.
    const bool early = a.positions == nullptr;
    if (!early) pdl_wait();

    if (tid == 0) {
        for (int i = 0; i < kSW * NS; ++i) mbar_init(&bar0[i], 1);
        fence_mbar_init();
    }
    int64_t W = 0;
    for (int t = 0; t < a.m; ++t) {
        bool ok;
        W += (int64_t)nkv * seg_tiles(token_rows(a, t, ok));
    }
    const int64_t P = gridDim.x, PW = P * kSW, gw = (int64_t)blockIdx.x * kSW + warp;
    const int64_t x0 = part_start(gw, W, PW), x1 = part_start(gw + 1, W, PW);
    const int64_t X0 = part_start(blockIdx.x, W, P), X1 = part_start(blockIdx.x + 1, W, P);
    __syncthreads();

    Cursor ic, cc;
    int issued = 0;
    if (x1 > x0) {
        cursor_at(a, ic, x0, x1);
        cc = ic;
        while (issued < NS && ic.x < ic.end) {
            issue_tile(a, ring, bars, cursor_next(a, ic), issued % NS, hd, lane);
            ++issued;
        }
    }
    // the angle table of the tokens the CTA's tiles belong to
    int t_a = 0, ntab = 0;
    if (X1 > X0) {
        t_a = seg_at(a, X0) / nkv;
        ntab = seg_at(a, X1 - 1) / nkv - t_a + 1;
        if (ntab > a.stream_tab_tokens) {
            if (tid == 0) set_error(a.err, DEV_ATTN_GEOMETRY);
            ntab = a.stream_tab_tokens;  // the tokens past the table are skipped
        }
    }
    stream_tables(a, tabs, t_a, ntab, half, tid, kSW * 32);
    __syncthreads();
    if (early) pdl_wait();  // q, k and v of this step come from the previous kernel

    if (x1 > x0) {
        warp_tiles<CPT, GM>(a, ring, bars, NS, ic, cc, issued, tabs, t_a, ntab, lane,
                            [&](const Tile &tl, const WarpState<CPT, GM> &st) {
                                // the record of this warp's piece of the segment
                                int count, rank;
                                cover(tl.seg0, tl.nt, W, PW, gw, count, rank);
                                if (rank >= a.stream_kmax) {
                                    if (lane == 0) set_error(a.err, DEV_ATTN_GEOMETRY);
                                    return;
                                }
#pragma unroll
                                for (int g = 0; g < GM; ++g) {
                                    if (g >= G) break;
                                    float *rec = stream_rec(a, tl.seg, rank, g);
                                    if (lane == 0) {
                                        rec[0] = st.m[g];
                                        rec[1] = st.l[g];
                                    }
                                    st_lane<CPT>(rec + kRecPad + lane * CPT, st.o[g]);
                                }
                            });
    }

    // ---- count in for every segment the CTA touched (warp 0, a lane per segment);
    // the CTA completing a segment merges it
    __syncthreads();
    if (X1 > X0) {
        const int s_first = seg_at(a, X0), s_last = seg_at(a, X1 - 1);
        for (int b0 = s_first; b0 <= s_last; b0 += 32) {
            if (warp == 0) {
                bool last = false;
                const int sg = b0 + lane;
                if (sg <= s_last) {
                    const Seg g = seg_of(a, sg);
                    int expect, rank;
                    cover(g.seg0, g.nt, W, P, blockIdx.x, expect, rank);
                    // release: the CTA's records (ordered before this by the barrier) become
                    // visible with the count; acquire: the merging CTA sees every record
                    int *cnt = a.counters + sg;
                    last = atom_add_acq_rel(cnt, 1) + 1 == expect;
                    if (last) *cnt = 0;  // ready for the next call
                }
                const unsigned bits = __ballot_sync(kAll, last);
                if (lane == 0) *mflags = bits;
            }
            __syncthreads();
            const unsigned bits = *mflags;  // the barrier orders the records' loads after the acquire
            for (unsigned mb = bits; mb; mb &= mb - 1) {
                const Seg g = seg_of(a, b0 + __ffs(mb) - 1);
                int K, rank;
                cover(g.seg0, g.nt, W, PW, 0, K, rank);
                stream_merge<CPT>(a, sm, g, min(K, a.stream_kmax), tid, warp, lane);
                if (!g.ok && g.kvh == 0 && tid == 0) set_error(a.err, DEV_BAD_POSITION);
                __syncthreads();  // the scratch is reused
            }
            __syncthreads();  // mflags is reused
        }
    }
}

// ---- thread-block clusters and distributed shared memory
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The generic address of p (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ float *cluster_ptr(float *p, unsigned rank)
{
    uint64_t r;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<float *>(r);
}

// grid C x n_segments CTAs in clusters of C = stream_cluster: cluster j works
// segment j (token j / n_kv_heads, kv head j % n_kv_heads) and CTA r of it the
// segment's tiles [r T / C, (r + 1) T / C), each warp an equal share of those.  The
// warps' states are combined in shared memory into the CTA's partial (max, exp-sum,
// weighted values per query head), which the CTA stores into CTA 0's shared
// memory (distributed shared memory) before a cluster barrier; CTA 0 then combines
// the C partials in rank order and writes the outputs.  No global records, no
// counters, no remote loads.
// shared memory: per warp stream_slots tiles | tabs [head_dim / 2][cos, sin] |
// kSW x stream_slots mbarriers | recv [C][group][head_dim + kRecPad] (CTA 0: the
// partials of the cluster).
template <int CPT, int GM>
__global__ void __launch_bounds__(kSW * 32, 1) attention_cluster_kernel(const __grid_constant__ AttnArgs a)
{
    constexpr int hd = CPT * 32, half = hd / 2;
    constexpr int slot_f = 2 * kTR * hd;
    extern __shared__ __align__(128) float sm[];
    const int NS = a.stream_slots, G = a.group, C = a.stream_cluster;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x / C, rank = blockIdx.x % C;
    float *ring = sm + (size_t)warp * NS * slot_f;
    float *tabs = sm + (size_t)kSW * NS * slot_f;
    uint64_t *bar0 = reinterpret_cast<uint64_t *>(tabs + hd);
    uint64_t *bars = bar0 + warp * NS;
    const bool early = a.positions == nullptr;  // as in the flat kernel
    if (!early) pdl_wait();

    float *recv = reinterpret_cast<float *>(bar0 + kSW * NS);
    cluster_arrive_relaxed();  // this CTA has started (waited on before any remote store)
    if (tid == 0) {
        for (int i = 0; i < kSW * NS; ++i) mbar_init(&bar0[i], 1);
        fence_mbar_init();
    }
    const Seg sg = seg_of(a, seg);
    const int c0 = rank * sg.nt / C, c1 = (rank + 1) * sg.nt / C;
    const int w0 = c0 + warp * (c1 - c0) / kSW, w1 = c0 + (warp + 1) * (c1 - c0) / kSW;
    __syncthreads();

    Cursor ic, cc;
    int issued = 0;
    if (w1 > w0) {
        ic.g = sg;
        ic.j = w0;
        ic.x = sg.seg0 + w0;
        ic.end = sg.seg0 + w1;
        cc = ic;
        while (issued < NS && ic.x < ic.end) {
            issue_tile(a, ring, bars, cursor_next(a, ic), issued % NS, hd, lane);
            ++issued;
        }
    }
    stream_tables(a, tabs, sg.t, 1, half, tid, kSW * 32);
    __syncthreads();
    if (early) pdl_wait();

    float wm[GM], wl[GM], wo[GM][CPT];  // this warp's state (empty without tiles)
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        wm[g] = -INFINITY;
        wl[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < CPT; ++e) wo[g][e] = 0.0f;
    }
    if (w1 > w0) {
        warp_tiles<CPT, GM>(a, ring, bars, NS, ic, cc, issued, tabs, sg.t, 1, lane,
                            [&](const Tile &, const WarpState<CPT, GM> &st) {
#pragma unroll
                                for (int g = 0; g < GM; ++g) {
                                    wm[g] = st.m[g];
                                    wl[g] = st.l[g];
#pragma unroll
                                    for (int e = 0; e < CPT; ++e) wo[g][e] = st.o[g][e];
                                }
                            });
    }
    // The next kernel may start only now: its CTAs would take the SMs this grid
    // leaves free and stream their weights against the K/V tiles (measured: the
    // step 1.568 -> 1.531 ms with the trigger here rather than at the start).
    pdl_launch_dependents();
    __syncthreads();  // the rings are idle: their space holds the partials now
    float *pacc = sm;                      // [kSW][G][hd] the warps' weighted values
    float *pml = pacc + kSW * G * hd;      // [kSW][G][2] their max and exp-sum
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
        st_lane<CPT>(pacc + (warp * G + g) * hd + lane * CPT, wo[g]);
        if (lane == 0) {
            pml[(warp * G + g) * 2] = wm[g];
            pml[(warp * G + g) * 2 + 1] = wl[g];
        }
    }
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
    // this CTA's partial (the warps combined in order) into CTA 0's recv[rank]
    const int rs = hd + kRecPad;
    float *dst = cluster_ptr(recv + rank * G * rs, 0);
    for (int i = tid; i < G * hd; i += kSW * 32) {
        const int g = i / hd;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSW; ++w)
            if (pml[(w * G + g) * 2 + 1] > 0.0f) M = fmaxf(M, pml[(w * G + g) * 2]);
        float v = 0.0f, L = 0.0f;
#pragma unroll
        for (int w = 0; w < kSW; ++w) {
            const float lw = pml[(w * G + g) * 2 + 1];
            const float sc = lw > 0.0f ? expf(pml[(w * G + g) * 2] - M) : 0.0f;
            v = fmaf(sc, pacc[(w * G + g) * hd + i % hd], v);
            L = fmaf(sc, lw, L);
        }
        dst[g * rs + kRecPad + i % hd] = v;
        if (i % hd == 0) {
            dst[g * rs] = M;
            dst[g * rs + 1] = L;
        }
    }
    cluster_arrive_release();  // the partials are in CTA 0
    cluster_wait_acquire();
    if (rank != 0) return;
    float *outv = pacc;  // [G][hd]
    for (int i = tid; i < G * hd; i += kSW * 32) {
        const float *rg = recv + (i / hd) * rs;  // rank r's partial of this head at rg + r * G * rs
        float mr[8], lr[8], vr[8], M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // C <= 8: every load of the C partials at once
            mr[r] = r < C ? rg[r * G * rs] : -INFINITY;
            lr[r] = r < C ? rg[r * G * rs + 1] : 0.0f;
            vr[r] = r < C ? rg[r * G * rs + kRecPad + i % hd] : 0.0f;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (lr[r] > 0.0f) M = fmaxf(M, mr[r]);
        float v = 0.0f, L = 0.0f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float w = lr[r] > 0.0f ? expf(mr[r] - M) : 0.0f;
            v = fmaf(w, vr[r], v);
            L = fmaf(w, lr[r], L);
        }
        outv[i] = v * (L > 0.0f ? 1.0f / L : 0.0f);  // L == 0 only after a bad position
    }
    __syncthreads();
    write_outputs(a, sg.t, sg.kvh, outv, tid, warp, lane);
    if (!sg.ok && sg.kvh == 0 && tid == 0) set_error(a.err, DEV_BAD_POSITION);
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

int stream_kmax(int n_kv_heads, int max_seq)
{
    // a segment's covering warps number at most PW / n_kv_heads + 2 (W >= n_kv_heads
    // x the segment's tiles) and at most its tiles (each holds one of them)
    return std::max(1, std::min(kMaxStreamWarps / n_kv_heads + 2, (max_seq + kTR - 1) / kTR));
}

template <int CPT>
const void *stream_fn_g(int G, bool cluster)
{
    if (cluster) {
        if (G == 1) return (const void *)attention_cluster_kernel<CPT, 1>;
        if (G <= 4) return (const void *)attention_cluster_kernel<CPT, 4>;
        return (const void *)attention_cluster_kernel<CPT, 8>;
    }
    if (G == 1) return (const void *)attention_stream_kernel<CPT, 1>;
    if (G <= 4) return (const void *)attention_stream_kernel<CPT, 4>;
    return (const void *)attention_stream_kernel<CPT, 8>;
}
const void *stream_fn(int hd, int G, bool cluster)
{
    return hd == 32 ? stream_fn_g<1>(G, cluster) : hd == 64 ? stream_fn_g<2>(G, cluster) : stream_fn_g<4>(G, cluster);
}

// Shapes and pointers the tiled kernels take: head_dim 32, 64 or 128, at most 8
// query heads per kv head, 16-byte aligned rows.
bool tiled_ok(const AttnArgs &a)
{
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (a.group > 8 || (a.head_dim != 32 && a.head_dim != 64 && a.head_dim != 128)) return false;
    if (!al16(a.q) || !al16(a.k) || !al16(a.v)) return false;
    return !(a.m > 1 && a.ld_qkv % 4);
}

// Ring slots per warp and the tensor maps (boxes of one head x kTR rows).
cudaError_t tiled_setup(AttnArgs &args, const AttnArgs &a)
{
    const size_t slot_b = (size_t)2 * kTR * a.head_dim * 4;
    args.stream_slots = (int)std::min<size_t>(kMaxSlots, std::max<size_t>(2, (24 * 1024) / slot_b));
    const uint64_t seq = a.m > 1 ? (uint64_t)a.seq_stride * 4 : (uint64_t)a.max_seq * a.kv_dim * 4;
    const uint64_t dims[3] = {(uint64_t)a.kv_dim, (uint64_t)a.max_seq, (uint64_t)a.m};
    const uint64_t strides[2] = {(uint64_t)a.kv_dim * 4, seq};
    const uint32_t box[3] = {(uint32_t)a.head_dim, (uint32_t)kTR, 1u};
    cudaError_t e = encode_tensor_map(&args.kmap, a.kc, 4, 3, dims, strides, box);
    if (e == cudaSuccess) e = encode_tensor_map(&args.vmap, a.vc, 4, 3, dims, strides, box);
    return e;
}

cudaError_t launch_tiled(const void *fn, const AttnArgs &args, int grid, int cluster, size_t smem, cudaStream_t s)
{
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    AttnArgs local = args;
    void *kargs[] = {&local};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kSW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (g_use_pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, fn, kargs);
}

// Clusters that can be resident at once for fn with `cluster` CTAs each (cached).
int resident_clusters(const void *fn, int cluster, size_t smem)
{
    struct Entry {
        const void *fn;
        int cluster, dev;
        size_t smem;
        int n;
    };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;
    const int dev = dev_info().device;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].fn == fn && cache[i].cluster == cluster && cache[i].smem == smem && cache[i].dev == dev)
            return cache[i].n;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kSW * 32);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (used < 32) cache[used++] = Entry{fn, cluster, dev, smem, n};
    return n;
}

// The cluster kernel: while every (token, kv head) segment can have a cluster of
// its own resident at once (up to 8 CTAs per segment, one CTA per SM).
bool launch_cluster(const AttnArgs &a, cudaStream_t s, cudaError_t &err)
{
    if (!tiled_ok(a)) return false;
    const int nseg = a.m * a.n_kv_heads, sms = dev_info().sm_count;
    if (nseg > sms) return false;
    AttnArgs args = a;
    err = tiled_setup(args, a);
    if (err != cudaSuccess) return true;
    const int hd = a.head_dim, G = a.group;
    const void *fn = stream_fn(hd, G, true);
    auto smem_for = [&](int c) {
        return (size_t)kSW * args.stream_slots * 2 * kTR * hd * 4 + (size_t)hd * 4 +
               (size_t)kSW * args.stream_slots * 8 + (size_t)c * G * (hd + kRecPad) * 4;
    };
    int C = std::min(8, sms / nseg);
    while (C > 1 && (smem_for(C) > dev_info().smem_optin || resident_clusters(fn, C, smem_for(C)) < nseg)) --C;
    const size_t smem = smem_for(C);
    if (smem > dev_info().smem_optin) return false;
    args.stream_cluster = C;
    err = launch_tiled(fn, args, C * nseg, C, smem, s);
    return true;
}

// The flat kernel: any number of segments, every SM the same share of tiles.
bool launch_stream(const AttnArgs &a, cudaStream_t s, cudaError_t &err)
{
    if (!tiled_ok(a)) return false;
    const int hd = a.head_dim, nkv = a.n_kv_heads;
    const int sms = dev_info().sm_count;
    // tiles as the host sees them: exact for a host position, an upper bound else
    const int64_t n_host =
        a.positions ? a.max_seq : ((a.position >= 0 && a.position < a.max_seq) ? a.position + 1 : 1);
    const int64_t tok_tiles = (int64_t)nkv * ((n_host + kTR - 1) / kTR);  // tiles of one token
    const int64_t W = (int64_t)a.m * tok_tiles;
    const int64_t pw = std::min<int64_t>((int64_t)sms * kSW, std::max<int64_t>(kSW, W));
    const int P = (int)std::min<int64_t>((pw + kSW - 1) / kSW, kMaxStreamWarps / kSW);
    // tokens whose angles a CTA tabulates: exact for a host position
    int tab_tokens = a.m;
    if (!a.positions) {
        tab_tokens = 1;
        for (int c = 0; c < P; ++c) {
            const int64_t x0 = (int64_t)c * W / P, x1 = (int64_t)(c + 1) * W / P;
            if (x1 > x0) tab_tokens = std::max<int64_t>(tab_tokens, (x1 - 1) / tok_tiles - x0 / tok_tiles + 1);
        }
    }
    AttnArgs args = a;
    err = tiled_setup(args, a);
    if (err != cudaSuccess) return true;
    const size_t smem = (size_t)kSW * args.stream_slots * 2 * kTR * hd * 4 + (size_t)tab_tokens * hd * 4 +
                        (size_t)kSW * args.stream_slots * 8 + 16;
    if (smem > dev_info().smem_optin) return false;
    args.stream_tab_tokens = tab_tokens;
    args.stream_kmax = stream_kmax(nkv, a.max_seq);
    err = launch_tiled(stream_fn(hd, a.group, false), args, P, 1, smem, s);
    return true;
}

}  // namespace

int attention_chunk_len(int, int, int) { return kChunk; }

size_t attention_part_bytes(int64_t m, int n_kv_heads, int group, int head_dim, int max_seq)
{
    const size_t n_chunks = (size_t)(max_seq + kChunk - 1) / kChunk;
    const size_t chunk_b = (size_t)m * n_kv_heads * n_chunks * group * (head_dim + 2) * 4;
    const size_t stream_b =
        (size_t)m * n_kv_heads * stream_kmax(n_kv_heads, max_seq) * group * (head_dim + kRecPad) * 4;
    return std::max(chunk_b, stream_b);
}

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
    {
        cudaError_t e = cudaSuccess;
        if (launch_cluster(a, s, e) || launch_stream(a, s, e)) return e;  // else the chunk kernel below
    }
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
