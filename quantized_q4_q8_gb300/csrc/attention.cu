// attention.cu -- RoPE, KV-cache append and split-sequence decode attention.
//
// Semantics (forward_single_full_cuda_with_cache in realizar 0.8.4
// src/gguf/cuda/clone_layer_weights.rs; incremental_attention_async in
// transformer_layer_gpu_true_dp4a, realizar 0.8.5 src/cuda/executor/cached.rs):
// q and k are rotated at the token's position, k and v are stored in the cache
// row `position`, and every query head h attends over cache rows 0..position of
// kv head h / (n_heads / n_kv_heads) with softmax(q.k / sqrt(head_dim)).
//
// RoPE pairs (i, i + 1) for mode 0 and (i, i + head_dim/2) for mode 1 turn by
// position * theta^(-2i/head_dim).  The angle is formed and reduced modulo 2*pi
// in double precision (positions reach thousands of radians), then rotated with
// single-precision sin/cos of the reduced angle.
//
// Attention is split over the sequence (flash-decoding style): CTA (token, kv
// head, chunk) scores its chunk of cache rows for all query heads of the group,
// keeps the chunk max, the exp-sum and the unnormalised weighted sum of values,
// and the last CTA of each (token, kv head) -- found with an atomic counter, no
// spinning -- merges the chunks with the log-sum-exp rule, writes the f32 output
// and its Q8_1 quantisation (head_dim is a multiple of 32, so Q8_1 blocks never
// straddle heads) for the O projection.  The counter is reset by the merging CTA.
#include <math.h>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {
namespace {

constexpr int kAttnThreads = 128;
constexpr double kTwoPi = 6.283185307179586476925286766559;

__device__ __forceinline__ int token_position(const AttnArgs &a, int t)
{
    return a.positions ? a.positions[t] : a.position;
}

// rotate pair (x0, x1) of dimension index i at position pos
__device__ __forceinline__ void rope_pair(float &x0, float &x1, int i, int head_dim, int pos,
                                          double log2_theta)
{
    const double inv_freq = exp2(-(2.0 * i / head_dim) * log2_theta);
    const double ang = (double)pos * inv_freq;
    const double red = ang - kTwoPi * rint(ang / kTwoPi);
    float sn, cs;
    sincosf((float)red, &sn, &cs);
    const float a = x0, b = x1;
    x0 = a * cs - b * sn;
    x1 = a * sn + b * cs;
}

// One CTA per (token, head) of q and of k: rotate; k and v go to the cache row.
__global__ void rope_append_kernel(const AttnArgs a)
{
    pdl_wait();
    const int t = blockIdx.y;
    const int head = blockIdx.x;  // [0, n_heads) q heads, then kv heads
    const int pos = token_position(a, t);
    const int hd = a.head_dim, half = hd / 2;
    if (pos < 0 || pos >= a.max_seq) {
        if (threadIdx.x == 0) set_error(a.err, DEV_BAD_POSITION);
        return;
    }
    const double l2t = log2((double)a.rope_theta);
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const int ia = a.rope_mode == 0 ? 2 * i : i;
        const int ib = a.rope_mode == 0 ? 2 * i + 1 : i + half;
        if (head < a.n_heads) {
            const float *src = a.q + (int64_t)t * a.ld_qkv + (int64_t)head * hd;
            float *dst = a.q_rot + (int64_t)t * a.q_dim + (int64_t)head * hd;
            float x0 = src[ia], x1 = src[ib];
            rope_pair(x0, x1, i, hd, pos, l2t);
            dst[ia] = x0;
            dst[ib] = x1;
        } else {
            const int kh = head - a.n_heads;
            const float *ks = a.k + (int64_t)t * a.ld_qkv + (int64_t)kh * hd;
            const float *vs = a.v + (int64_t)t * a.ld_qkv + (int64_t)kh * hd;
            float *kd = a.kc + (int64_t)t * a.seq_stride + (int64_t)pos * a.kv_dim + (int64_t)kh * hd;
            float *vd = a.vc + (int64_t)t * a.seq_stride + (int64_t)pos * a.kv_dim + (int64_t)kh * hd;
            float x0 = ks[ia], x1 = ks[ib];
            rope_pair(x0, x1, i, hd, pos, l2t);
            kd[ia] = x0;
            kd[ib] = x1;
            vd[ia] = vs[ia];
            vd[ib] = vs[ib];
        }
    }
}

// Partial record of one chunk for one query head: [max, sum, o[head_dim]]
__device__ __forceinline__ float *part_rec(const AttnArgs &a, int t, int kvh, int chunk, int g)
{
    const int64_t idx = (((int64_t)t * a.n_kv_heads + kvh) * a.n_chunks + chunk) * a.group + g;
    return a.part + idx * (a.head_dim + 2);
}

// grid (n_chunks, n_kv_heads, m); dynamic smem: q [group][hd] + p [group][chunk_len]
__global__ void __launch_bounds__(kAttnThreads) attention_chunk_kernel(const AttnArgs a)
{
    extern __shared__ float sm[];
    const int chunk = blockIdx.x, kvh = blockIdx.y, t = blockIdx.z;
    const int hd = a.head_dim, G = a.group, L = a.chunk_len;
    float *qs = sm;                 // [G][hd]
    float *ps = sm + G * hd;        // [G][L]
    float *stat = ps + G * L;       // [G][2] and a flag
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = kAttnThreads / 32;
    pdl_wait();

    const int pos = token_position(a, t);
    const bool pos_ok = pos >= 0 && pos < a.max_seq;
    const int c0 = chunk * L;
    const int c1 = pos_ok ? min(c0 + L, pos + 1) : c0;
    const int n = max(0, c1 - c0);
    const float scale = 1.0f / sqrtf((float)hd);

    if (n > 0) {
        for (int i = tid; i < G * hd; i += kAttnThreads)
            qs[i] = a.q_rot[(int64_t)t * a.q_dim + (int64_t)(kvh * G) * hd + i];
        __syncthreads();
        const float *kbase = a.kc + (int64_t)t * a.seq_stride + (int64_t)kvh * hd;
        // scores: each warp takes 4 positions at a time (loads first, then the
        // dot products), lanes over head_dim
        const int per = hd / 32;  // 1..8 values per lane
        for (int j0 = warp * 4; j0 < n; j0 += nwarps * 4) {
            float kv[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float *kr = kbase + (int64_t)(c0 + j0 + u) * a.kv_dim;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    kv[u][e] = (e < per && j0 + u < n) ? kr[e * 32 + lane] : 0.0f;
            }
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float dot = 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e < per) dot = fmaf(qs[g * hd + e * 32 + lane], kv[u][e], dot);
                    dot = warp_sum(dot);
                    if (lane == 0 && j0 + u < n) ps[g * L + j0 + u] = dot * scale;
                }
            }
        }
        __syncthreads();
        // chunk softmax statistics per query head (warp per head)
        for (int g = warp; g < G; g += nwarps) {
            float mx = -INFINITY;
            for (int j = lane; j < n; j += 32) mx = fmaxf(mx, ps[g * L + j]);
            mx = warp_max(mx);
            float sum = 0.0f;
            for (int j = lane; j < n; j += 32) {
                const float p = expf(ps[g * L + j] - mx);
                ps[g * L + j] = p;
                sum += p;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                stat[2 * g] = mx;
                stat[2 * g + 1] = sum;
            }
        }
        __syncthreads();
        // weighted values: thread per head_dim element, loop over positions
        const float *vbase = a.vc + (int64_t)t * a.seq_stride + (int64_t)kvh * hd;
        for (int dd = tid; dd < hd; dd += kAttnThreads) {
            float o[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) o[g] = 0.0f;
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const float v = vbase[(int64_t)(c0 + j) * a.kv_dim + dd];
#pragma unroll
                for (int g = 0; g < 16; ++g)
                    if (g < G) o[g] = fmaf(ps[g * L + j], v, o[g]);
            }
#pragma unroll
            for (int g = 0; g < 16; ++g)
                if (g < G) part_rec(a, t, kvh, chunk, g)[2 + dd] = o[g];
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
    int *flag = reinterpret_cast<int *>(stat + 2 * G);
    if (tid == 0) {
        int *cnt = a.counters + (int64_t)t * a.n_kv_heads + kvh;
        const int prev = atomicAdd(cnt, 1);
        const int last = (prev == a.n_chunks - 1);
        if (last) *cnt = 0;  // ready for the next call
        *flag = last;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();

    float *outv = qs;  // reuse: merged output [G][hd]
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
        for (int c = 0; c < a.n_chunks; ++c) M = fmaxf(M, __ldcg(part_rec(a, t, kvh, c, g)));
        float Lsum = 0.0f;
        for (int c = 0; c < a.n_chunks; ++c) {
            const float *rec = part_rec(a, t, kvh, c, g);
            const float l = __ldcg(rec + 1);
            if (l > 0.0f) Lsum += l * expf(__ldcg(rec) - M);
        }
        for (int dd = tid; dd < hd; dd += kAttnThreads) {
            float acc = 0.0f;
            for (int c = 0; c < a.n_chunks; ++c) {
                const float *rec = part_rec(a, t, kvh, c, g);
                const float l = __ldcg(rec + 1);
                if (l > 0.0f) acc += __ldcg(rec + 2 + dd) * expf(__ldcg(rec) - M);
            }
            outv[g * hd + dd] = (Lsum > 0.0f) ? acc / Lsum : 0.0f;  // 0 only after a bad position
        }
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
        for (int b = warp; b < nblk; b += nwarps) {
            const float v = outv[b * 32 + lane];
            const float amax = warp_max(fabsf(v));
            const float dq = __fdiv_rn(amax, 127.0f);
            const int qi = q8_code(v, dq);
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

int attention_chunk_len(int max_seq, int n_kv_heads, int m)
{
    // enough CTAs to cover the GPU about twice at the longest sequence
    const int sms = dev_info().sm_count;
    int L = 64;
    while (L > 16 && (int64_t)((max_seq + L - 1) / L) * n_kv_heads * m < 2 * sms) L /= 2;
    return L;
}

size_t attention_smem_bytes(int group, int head_dim, int chunk_len)
{
    return ((size_t)group * head_dim + (size_t)group * chunk_len + 2 * (size_t)group + 4) * sizeof(float);
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s)
{
    AttnArgs args = a;
    void *kargs[] = {&args};
    cudaError_t e = launch_ex((const void *)rope_append_kernel,
                              dim3((unsigned)(a.n_heads + a.n_kv_heads), (unsigned)a.m),
                              dim3(64), 0, s, kargs);
    if (e != cudaSuccess) return e;
    const size_t smem = attention_smem_bytes(a.group, a.head_dim, a.chunk_len);
    return launch_ex((const void *)attention_chunk_kernel,
                     dim3((unsigned)a.n_chunks, (unsigned)a.n_kv_heads, (unsigned)a.m),
                     dim3(kAttnThreads), smem, s, kargs);
}

}  // namespace rz
