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
// position * theta^(-2i/head_dim).  A small kernel builds, per token, the cosine
// and sine of every pair's angle: the angle is formed and reduced modulo 2*pi in
// double precision (positions reach thousands of radians), then sin/cos are taken
// in single precision.  The table depends only on the positions, so the layer
// stack builds it once per step and every layer reuses it.
//
// Attention is split over the sequence in chunks of 64 cache rows (flash-
// decoding style).  CTA (chunk, kv head, token) rotates its query heads, and the
// CTA whose chunk holds the token's own row rotates k, writes k and v to the
// cache and uses them from shared memory.  The scores and the weighted values are
// computed with every load of the chunk issued before it is used (32 KB of K,
// then 32 KB of V in flight per CTA at head_dim 128), so HBM rather than latency
// bounds the kernel.  Each CTA leaves its chunk max, exp-sum and unnormalised
// weighted values; the last CTA of each (token, kv head) -- found with an atomic
// counter, no spinning -- merges the chunks with the log-sum-exp rule and writes
// the f32 output and its Q8_1 quantisation (head_dim is a multiple of 32, so Q8_1
// blocks never straddle heads) for the O projection.  The counter is reset by the
// merging CTA.
#include <math.h>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kChunk = 64;  // cache rows per CTA
constexpr double kTwoPi = 6.283185307179586476925286766559;

__device__ __forceinline__ int token_position(const AttnArgs &a, int t)
{
    return a.positions ? a.positions[t] : a.position;
}

// cos/sin of every pair angle, per token: tab[t][i] = (cos, sin)
__global__ void rope_table_kernel(const AttnArgs a)
{
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x;
    const int half = a.head_dim / 2;
    const int pos = token_position(a, t);
    const double l2t = log2((double)a.rope_theta);
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv_freq = exp2(-(2.0 * i / a.head_dim) * l2t);
        const double ang = (double)pos * inv_freq;
        const double red = ang - kTwoPi * rint(ang / kTwoPi);
        float sn, cs;
        sincosf((float)red, &sn, &cs);
        a.rope_tab[((int64_t)t * half + i) * 2] = cs;
        a.rope_tab[((int64_t)t * half + i) * 2 + 1] = sn;
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

// grid (n_kv_heads, m, launch_chunks), chunk-major so that low chunks (needed by
// every token) are scheduled first; 256 threads; CPT = head_dim / 32.
// The chunk's K and V rows are bulk-copied into shared memory (one copy per row,
// completion counted on two mbarriers) as soon as the CTA starts: the copy engine
// keeps the whole chunk in flight, which per-thread loads cannot (the SM's limit
// on outstanding misses held them near 2 TB/s).  Scores: warp w takes rows w,
// w + 8, ..., lane l dims l + 32 e of each (conflict-free), with the rotated query
// heads in shared memory.
// shared memory: kbuf [64][hd] | vbuf [64][hd] | qs [G][hd] | kn [hd] | vn [hd] |
//                ps [G][64] | stat [G][2] + 2 (padded to 4) | red [8][G][hd] | flag | 2 mbarriers
template <int CPT>
__global__ void __launch_bounds__(kAttnThreads) attention_chunk_kernel(const AttnArgs a)
{
    extern __shared__ __align__(16) float sm[];
    const int kvh = blockIdx.x, t = blockIdx.y, chunk = blockIdx.z;
    const int hd = a.head_dim, G = a.group;
    float *kbuf = sm;
    float *vbuf = kbuf + kChunk * hd;
    float *qs = vbuf + kChunk * hd;
    float *kn = qs + G * hd;
    float *vn = kn + hd;
    float *ps = vn + hd;
    float *stat = ps + G * kChunk;
    float *red = stat + ((2 * G + 2 + 3) & ~3);  // 16-byte aligned for the float4 stores
    int *flag = reinterpret_cast<int *>(red + 8 * G * hd);
    uint64_t *kbar = reinterpret_cast<uint64_t *>(flag + 2);
    uint64_t *vbar = kbar + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    pdl_wait();

    const int pos = token_position(a, t);
    const bool pos_ok = pos >= 0 && pos < a.max_seq;
    // chunks holding rows of this token; after a bad position chunk 0 alone takes
    // part and the merge writes zeros
    const int nc = pos_ok ? min(a.n_chunks, pos / kChunk + 1) : 1;
    if (chunk >= nc) return;
    const int c0 = chunk * kChunk;
    const int n = pos_ok ? max(0, min(kChunk, pos + 1 - c0)) : 0;
    const bool own = pos_ok && pos >= c0 && pos < c0 + kChunk;  // this chunk holds the new row
    if (!pos_ok && chunk == 0 && kvh == 0 && tid == 0) set_error(a.err, DEV_BAD_POSITION);
    const float *tab = a.rope_tab + (int64_t)t * (hd / 2) * 2;
    const float scale = 1.0f / sqrtf((float)hd);
    const int64_t kv_base = (int64_t)t * a.seq_stride + (int64_t)kvh * hd;

    if (n > 0) {
        // K and V rows on their way into shared memory (the token's own row is taken
        // from kn / vn below: its cache copy is written by this CTA)
        if (tid == 0) {
            mbar_init(kbar, 1);
            mbar_init(vbar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(kbar, (unsigned)(n * hd * 4));
            mbar_arrive_expect_tx(vbar, (unsigned)(n * hd * 4));
        }
        if (tid < n)
            bulk_g2s(kbuf + tid * hd, a.kc + kv_base + (int64_t)(c0 + tid) * a.kv_dim, (unsigned)(hd * 4), kbar);
        else if (tid >= kChunk && tid - kChunk < n)
            bulk_g2s(vbuf + (tid - kChunk) * hd, a.vc + kv_base + (int64_t)(c0 + tid - kChunk) * a.kv_dim,
                     (unsigned)(hd * 4), vbar);

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
        // the K rows have landed (bounded wait; on expiry the copies are waited
        // out again before the CTA may leave)
        if (!mbar_wait(kbar, 0)) {
            if (tid == 0) set_error(a.err, DEV_TIMEOUT_ATTN);
            if (!mbar_wait(kbar, 0) && tid == 0) set_error(a.err, DEV_TIMEOUT_DRAIN);
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
        if (!mbar_wait(vbar, 0)) {
            if (tid == 0) set_error(a.err, DEV_TIMEOUT_ATTN);
            if (!mbar_wait(vbar, 0) && tid == 0) set_error(a.err, DEV_TIMEOUT_DRAIN);
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
        // fixed-order sum over the 8 row groups -> partial record
        for (int i = tid; i < G * hd; i += kAttnThreads) {
            const int g = i / hd, dd = i % hd;
            float s8 = 0.0f;
#pragma unroll
            for (int r = 0; r < 8; ++r) s8 += red[(r * G + g) * hd + dd];
            part_rec(a, t, kvh, chunk, g)[2 + dd] = s8;
        }
        for (int g = tid; g < G; g += kAttnThreads) {
            float *rec = part_rec(a, t, kvh, chunk, g);
            rec[0] = stat[2 * g];
            rec[1] = stat[2 * g + 1];
        }
    } else {
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
        const int prev = atomicAdd(cnt, 1);
        const int last = (prev == nc - 1);
        if (last) *cnt = 0;  // ready for the next call
        *flag = last;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();

    // chunk statistics in parallel (thread per (head, chunk)), then the weights
    float *wts = ps;  // [G][kChunk] reused: chunk weights exp(m_c - M)
    for (int g = warp; g < G; g += kAttnThreads / 32) {
        float mc[2], lc[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = lane + 32 * h;
            mc[h] = c < nc ? __ldcg(part_rec(a, t, kvh, c, g)) : -INFINITY;
            lc[h] = c < nc ? __ldcg(part_rec(a, t, kvh, c, g) + 1) : 0.0f;
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
    float *outv = red;  // merged output [G][hd]
    for (int i = tid; i < G * hd; i += kAttnThreads) {
        const int g = i / hd, dd = i % hd;
        float acc = 0.0f;
        // eight records' loads in flight at a time (every record c < nc is written and
        // finite; a zero weight adds exactly nothing), summed in chunk order
        int c = 0;
        for (; c + 8 <= nc; c += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(part_rec(a, t, kvh, c + u, g) + 2 + dd);
#pragma unroll
            for (int u = 0; u < 8; ++u) acc = fmaf(v[u], wts[g * kChunk + c + u], acc);
        }
        for (; c < nc; ++c) acc = fmaf(__ldcg(part_rec(a, t, kvh, c, g) + 2 + dd), wts[g * kChunk + c], acc);
        outv[g * hd + dd] = acc * stat[2 * g];
    }
    __syncthreads();
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

}  // namespace

int attention_chunk_len(int, int, int) { return kChunk; }

size_t attention_smem_bytes(int group, int head_dim, int)
{
    return (2 * (size_t)kChunk * head_dim + (size_t)group * head_dim + 2 * (size_t)head_dim +
            (size_t)group * kChunk + ((2 * (size_t)group + 2 + 3) & ~(size_t)3) + 8 * (size_t)group * head_dim) *
               sizeof(float) +
           16 + 16;  // flag (+ pad), two mbarriers
}

cudaError_t launch_rope_table(const AttnArgs &a, cudaStream_t s)
{
    AttnArgs args = a;
    void *kargs[] = {&args};
    return launch_ex((const void *)rope_table_kernel, dim3((unsigned)a.m), dim3(64), 0, s, kargs);
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s)
{
    AttnArgs args = a;
    void *kargs[] = {&args};
    if (a.make_table) {
        cudaError_t e = launch_rope_table(a, s);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = attention_smem_bytes(a.group, a.head_dim, kChunk);
    const void *fn = a.head_dim == 32    ? (const void *)attention_chunk_kernel<1>
                     : a.head_dim == 64  ? (const void *)attention_chunk_kernel<2>
                     : a.head_dim == 128 ? (const void *)attention_chunk_kernel<4>
                                         : (const void *)attention_chunk_kernel<8>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dev_info().smem_optin);
        if (e != cudaSuccess) return e;
    }
    return launch_ex(fn, dim3((unsigned)a.n_kv_heads, (unsigned)a.m, (unsigned)a.launch_chunks),
                     dim3(kAttnThreads), smem, s, kargs);
}

}  // namespace rz
