/*
 * rz_oracle.c -- plain single-threaded CPU oracle for the Q4_K x Q8_1 decode path.
 *
 * TEST INFRASTRUCTURE ONLY: used by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.  Compile without fast-math and with
 * -ffp-contract=off so that every f32 operation is the IEEE-754 one written.
 *
 * Sources followed (page titles are the docs.rs source pages of realizar):
 *   - realizar 0.8.5 src/cuda/executor/cached.rs, transformer_layer_gpu_true_dp4a:
 *     the step order of the decode layer (norm -> one Q8_1 quantisation shared
 *     by Q/K/V -> integer GEMVs -> incremental attention -> Q8_1 of the
 *     attention output -> O GEMV -> residual -> norm -> SwiGLU FFN -> residual).
 *   - realizar 0.8.4 src/gguf/cuda/clone_layer_weights.rs,
 *     forward_single_full_cuda_with_cache and cuda_swiglu_ffn: RoPE on q and k,
 *     GQA head mapping, first-token attention, SiLU(gate) * up.
 *   - realizar 0.8.4 src/gpu/adapters/using.rs, rms_norm_inplace: the RMSNorm
 *     formula; GpuModelQ4::forward: output norm then Q4_0 LM head on f32 input.
 *   - realizar 0.8.5 src/cuda/executor/layers/forward_utils.rs,
 *     pad_and_upload_input: zero padding of the hidden vector to a multiple of 256.
 */
#include "rz_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the row loops use: 1 in the plain build, the OpenMP team size in the
   all-core build that only the CPU baseline loads. */
int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16, written from the standard's definition:                 */
/* value = (-1)^s * 2^(e-15) * (1 + f/1024) for 0 < e < 31,                   */
/*         (-1)^s * 2^-14 * (f/1024)      for e == 0 (subnormal).            */
/* ------------------------------------------------------------------------- */
double orc_f16_to_f64(uint16_t h)
{
    int s = h >> 15;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

uint16_t orc_f32_to_f16(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    if (isinf(x))
        return (uint16_t)(sign | 0x7c00u);
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    /* The largest finite half is 65504; 65520 lies halfway to 2^16 and rounds
       to the even neighbour, which is the overflow to infinity. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: a = k * 2^-24; k == 1024 encodes the smallest normal */
        double k = nearbyint(ldexp(a, 24)); /* default mode: ties to even */
        return (uint16_t)(sign | (uint16_t)k);
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;           /* a = (2m) * 2^E, 2m in [1, 2) */
    double frac = nearbyint((2.0 * m - 1.0) * 1024.0);
    if (frac == 1024.0) {
        frac = 0.0;
        E += 1;
    }
    return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | (int)frac));
}

void orc_f32_to_f16_array(const float *x, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f32_array(const uint16_t *h, float *x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        x[i] = (float)orc_f16_to_f64(h[i]);
}

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr_u16(uint8_t *p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xff);
    p[1] = (uint8_t)(v >> 8);
}

/* ------------------------------------------------------------------------- */
/* Q4_K super-block (256 weights, 144 bytes).                                 */
/* Sub-block j (32 weights) has a 6-bit scale sc_j and a 6-bit min m_j:       */
/*   j < 4 : sc_j = s[j] & 63,                m_j = s[j+4] & 63                */
/*   j >= 4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4,                        */
/*           m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4                         */
/* Weight e (0..255): byte qs[32*(e/64) + e%32], low nibble when e%64 < 32,   */
/* high nibble otherwise.  Dequantised value: d*sc_j*q - dmin*m_j, j = e/32.  */
/* ------------------------------------------------------------------------- */
void orc_q4k_unpack(const uint8_t *blk, uint16_t *d, uint16_t *dmin,
                    uint8_t sc[8], uint8_t mn[8], uint8_t q[256])
{
    const uint8_t *s = blk + 4;
    const uint8_t *qs = blk + 16;
    *d = rd_u16(blk);
    *dmin = rd_u16(blk + 2);
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        mn[j] = s[j + 4] & 63;
    }
    for (int j = 4; j < 8; ++j) {
        sc[j] = (uint8_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
        mn[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
    }
    for (int e = 0; e < 256; ++e) {
        int chunk = e / 64, t = e % 64;
        uint8_t byte = qs[32 * chunk + t % 32];
        q[e] = (t < 32) ? (byte & 15) : (byte >> 4);
    }
}

void orc_q4k_pack(uint16_t d, uint16_t dmin, const uint8_t sc[8], const uint8_t mn[8],
                  const uint8_t q[256], uint8_t *blk)
{
    uint8_t *s = blk + 4;
    uint8_t *qs = blk + 16;
    wr_u16(blk, d);
    wr_u16(blk + 2, dmin);
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((mn[j] & 63) | ((mn[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
    }
    memset(qs, 0, 128);
    for (int e = 0; e < 256; ++e) {
        int chunk = e / 64, t = e % 64;
        uint8_t *byte = &qs[32 * chunk + t % 32];
        if (t < 32)
            *byte = (uint8_t)((*byte & 0xf0) | (q[e] & 15));
        else
            *byte = (uint8_t)((*byte & 0x0f) | ((q[e] & 15) << 4));
    }
}

void orc_q4k_dequantize(const uint8_t *w, int64_t n_blocks, double *out)
{
    uint16_t d, dmin;
    uint8_t sc[8], mn[8], q[256];
    for (int64_t b = 0; b < n_blocks; ++b) {
        orc_q4k_unpack(w + b * ORC_Q4K_BYTES, &d, &dmin, sc, mn, q);
        double dd = orc_f16_to_f64(d), dm = orc_f16_to_f64(dmin);
        for (int e = 0; e < 256; ++e) {
            int j = e / 32;
            out[b * 256 + e] = dd * sc[j] * q[e] - dm * mn[j];
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Q4_0 block (32 weights, 18 bytes): weight i < 16 is the low nibble of      */
/* qs[i], weight i + 16 the high nibble; value d * (q - 8).                   */
/* ------------------------------------------------------------------------- */
void orc_q4_0_unpack(const uint8_t *blk, uint16_t *d, uint8_t q[32])
{
    *d = rd_u16(blk);
    for (int i = 0; i < 16; ++i) {
        q[i] = blk[2 + i] & 15;
        q[i + 16] = blk[2 + i] >> 4;
    }
}

void orc_q4_0_pack(uint16_t d, const uint8_t q[32], uint8_t *blk)
{
    wr_u16(blk, d);
    for (int i = 0; i < 16; ++i)
        blk[2 + i] = (uint8_t)((q[i] & 15) | ((q[i + 16] & 15) << 4));
}

void orc_q4_0_dequantize(const uint8_t *w, int64_t n_blocks, double *out)
{
    uint16_t d;
    uint8_t q[32];
    for (int64_t b = 0; b < n_blocks; ++b) {
        orc_q4_0_unpack(w + b * ORC_Q4_0_BYTES, &d, q);
        double dd = orc_f16_to_f64(d);
        for (int i = 0; i < 32; ++i)
            out[b * 32 + i] = dd * ((int)q[i] - 8);
    }
}

/* ------------------------------------------------------------------------- */
/* Q8_1 (blocks of 32 activations).  Per block: d = max|x| / 127 (f32),       */
/* q_i = round(x_i / d) half away from zero, clamped to [-127, 127]           */
/* (all zero when d == 0), s = d * sum(q) in f32.  Buffer for m rows of n:    */
/* int8 q[m][n] | f32 d[m][n/32] | f32 s[m][n/32]  (structure of arrays).    */
/* ------------------------------------------------------------------------- */
static const float *q8_d(const uint8_t *q8, int64_t m, int64_t n)
{
    return (const float *)(q8 + m * n);
}
static const float *q8_s(const uint8_t *q8, int64_t m, int64_t n)
{
    return (const float *)(q8 + m * n) + m * (n / ORC_QK8);
}

void orc_q8_1_quantize(const float *x, uint8_t *out, int64_t m, int64_t n)
{
    int64_t nb = n / ORC_QK8;
    float *dout = (float *)(out + m * n);
    float *sout = dout + m * nb;
    for (int64_t t = 0; t < m; ++t) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + t * n + b * ORC_QK8;
            int8_t *qb = (int8_t *)(out + t * n + b * ORC_QK8);
            float amax = 0.0f;
            for (int i = 0; i < ORC_QK8; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < ORC_QK8; ++i) {
                int qi = 0;
                if (d != 0.0f) {
                    float v = xb[i] / d;
                    float r = roundf(v);
                    if (r > 127.0f)
                        r = 127.0f;
                    if (r < -127.0f)
                        r = -127.0f;
                    qi = (int)r;
                }
                qb[i] = (int8_t)qi;
                sum += qi;
            }
            dout[t * nb + b] = d;
            sout[t * nb + b] = d * (float)sum;
        }
    }
}

void orc_q8_1_dequantize(const uint8_t *q8, double *out, int64_t m, int64_t n)
{
    const float *d = q8_d(q8, m, n);
    for (int64_t i = 0; i < m * n; ++i)
        out[i] = (double)d[i / ORC_QK8] * (double)((const int8_t *)q8)[i];
}

/* ------------------------------------------------------------------------- */
/* Q4_K x Q8_1.  For super-block b of row r and sub-block j, the integer dot  */
/*   I_bj = sum_k q4[32j+k] * q8_bj[k]   (exact in int32)                      */
/* and the row output                                                          */
/*   y_r = sum_b [ d_b * sum_j sc_bj * d8_bj * I_bj - dmin_b * sum_j m_bj * s_bj ] */
/* which is the dot of the dequantised row with the dequantised activation,  */
/* with the activation sum term taken from the stored s.  Accumulated in f64. */
/* ------------------------------------------------------------------------- */
static int32_t subblock_dot(const uint8_t q[256], int j, const int8_t *x8blk)
{
    int32_t acc = 0;
    for (int k = 0; k < 32; ++k)
        acc += (int32_t)q[32 * j + k] * (int32_t)x8blk[k];
    return acc;
}

void orc_q4k_q8_subblock_dots(const uint8_t *w, const uint8_t *x8, int32_t *I,
                              int64_t out_dim, int64_t in_dim)
{
    int64_t nsb = in_dim / ORC_QK_K;
    const int8_t *xq = (const int8_t *)x8;
    uint16_t d, dmin;
    uint8_t sc[8], mn[8], q[256];
    for (int64_t r = 0; r < out_dim; ++r)
        for (int64_t b = 0; b < nsb; ++b) {
            orc_q4k_unpack(w + (r * nsb + b) * ORC_Q4K_BYTES, &d, &dmin, sc, mn, q);
            for (int j = 0; j < 8; ++j)
                I[r * nsb * 8 + b * 8 + j] = subblock_dot(q, j, xq + (b * 8 + j) * ORC_QK8);
        }
}

void orc_q4k_q8_gemv(const uint8_t *w, const uint8_t *x8, float *y,
                     int64_t m, int64_t out_dim, int64_t in_dim)
{
    int64_t nsb = in_dim / ORC_QK_K;
    int64_t nb8 = in_dim / ORC_QK8;
    const float *xd = q8_d(x8, m, in_dim);
    const float *xs = q8_s(x8, m, in_dim);
    for (int64_t t = 0; t < m; ++t) {
        const int8_t *xq = (const int8_t *)x8 + t * in_dim;
        /* rows are independent: the all-core build (-fopenmp, the CPU baseline)
           splits them over threads; each row's sum keeps this order */
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < out_dim; ++r) {
            uint16_t d, dmin;
            uint8_t sc[8], mn[8], q[256];
            double acc = 0.0;
            for (int64_t b = 0; b < nsb; ++b) {
                orc_q4k_unpack(w + (r * nsb + b) * ORC_Q4K_BYTES, &d, &dmin, sc, mn, q);
                double dd = orc_f16_to_f64(d), dm = orc_f16_to_f64(dmin);
                for (int j = 0; j < 8; ++j) {
                    int64_t blk = b * 8 + j;
                    double d8 = xd[t * nb8 + blk];
                    double s8 = xs[t * nb8 + blk];
                    int32_t I = subblock_dot(q, j, xq + blk * ORC_QK8);
                    acc += dd * sc[j] * d8 * (double)I - dm * mn[j] * s8;
                }
            }
            y[t * out_dim + r] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Q4_K x f32 (no activation quantisation; q4k_gemv_cached_async in          */
/* transformer_layer_gpu_cached): y_r = sum_e w_re * x_e with the dequantised */
/* weight w = d * sc_j * q - dmin * m_j, accumulated in f64.                  */
/* ------------------------------------------------------------------------- */
void orc_q4k_f32_gemv(const uint8_t *w, const float *x, float *y,
                      int64_t m, int64_t out_dim, int64_t in_dim)
{
    int64_t nsb = in_dim / ORC_QK_K;
    for (int64_t t = 0; t < m; ++t)
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < out_dim; ++r) {
            uint16_t d, dmin;
            uint8_t sc[8], mn[8], q[256];
            double acc = 0.0;
            for (int64_t b = 0; b < nsb; ++b) {
                orc_q4k_unpack(w + (r * nsb + b) * ORC_Q4K_BYTES, &d, &dmin, sc, mn, q);
                double dd = orc_f16_to_f64(d), dm = orc_f16_to_f64(dmin);
                const float *xb = x + t * in_dim + b * ORC_QK_K;
                for (int e = 0; e < 256; ++e) {
                    int j = e / 32;
                    acc += (dd * sc[j] * q[e] - dm * mn[j]) * (double)xb[e];
                }
            }
            y[t * out_dim + r] = (float)acc;
        }
}

void orc_q4_0_gemv(const uint8_t *w, const float *x, float *y,
                   int64_t m, int64_t out_dim, int64_t in_dim)
{
    int64_t nb = in_dim / ORC_QK4_0;
    for (int64_t t = 0; t < m; ++t)
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < out_dim; ++r) {
            uint16_t d;
            uint8_t q[32];
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                orc_q4_0_unpack(w + (r * nb + b) * ORC_Q4_0_BYTES, &d, q);
                double dd = orc_f16_to_f64(d);
                const float *xb = x + t * in_dim + b * ORC_QK4_0;
                for (int i = 0; i < 32; ++i)
                    acc += dd * ((int)q[i] - 8) * (double)xb[i];
            }
            y[t * out_dim + r] = (float)acc;
        }
}

/* ------------------------------------------------------------------------- */
/* RMSNorm (rms_norm_inplace): rms = sqrt(sum x^2 / n + eps), y = x/rms * g.  */
/* The mean runs over the logical n; the padding [n, n_pad) is written as 0.  */
/* ------------------------------------------------------------------------- */
void orc_rmsnorm(const float *x, const float *gamma, float *y,
                 int64_t m, int64_t n, int64_t n_pad, float eps)
{
    for (int64_t t = 0; t < m; ++t) {
        const float *xr = x + t * n_pad;
        float *yr = y + t * n_pad;
        double ss = 0.0;
        for (int64_t i = 0; i < n; ++i)
            ss += (double)xr[i] * (double)xr[i];
        double rms = sqrt(ss / (double)n + (double)eps);
        double scale = 1.0 / rms;
        for (int64_t i = 0; i < n; ++i)
            yr[i] = (float)((double)xr[i] * scale * (double)gamma[i]);
        for (int64_t i = n; i < n_pad; ++i)
            yr[i] = 0.0f;
    }
}

void orc_residual_add(const float *a, const float *b, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)((double)a[i] + (double)b[i]);
}

double orc_silu(double x) { return x / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* RoPE: pair (a, b) of head dimension index i < head_dim/2 turns by          */
/* angle pos * theta^(-2i/head_dim).  Mode 0 pairs (2i, 2i+1); mode 1 pairs    */
/* (i, i + head_dim/2).                                                        */
/* ------------------------------------------------------------------------- */
void orc_rope(float *v, int64_t n_heads, int64_t head_dim, int64_t pos, double theta, int mode)
{
    int64_t half = head_dim / 2;
    for (int64_t h = 0; h < n_heads; ++h) {
        float *hv = v + h * head_dim;
        for (int64_t i = 0; i < half; ++i) {
            double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)head_dim);
            double c = cos(ang), s = sin(ang);
            int64_t ia = mode == 0 ? 2 * i : i;
            int64_t ib = mode == 0 ? 2 * i + 1 : i + half;
            double a = hv[ia], b = hv[ib];
            hv[ia] = (float)(a * c - b * s);
            hv[ib] = (float)(a * s + b * c);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Decode attention over cache rows 0..pos (the new token's k, v already at   */
/* row pos).  GQA: q head h reads kv head h / (n_heads / n_kv_heads).         */
/* ------------------------------------------------------------------------- */
void orc_attention(const float *q, const float *kc, const float *vc, int64_t pos,
                   int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float *out)
{
    int64_t kv_dim = n_kv_heads * head_dim;
    int64_t group = n_heads / n_kv_heads;
    int64_t T = pos + 1;
    double inv = 1.0 / sqrt((double)head_dim);
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n_heads; ++h) {
        double *sc = (double *)malloc((size_t)T * sizeof(double));
        double *acc = (double *)malloc((size_t)head_dim * sizeof(double));
        int64_t kvh = h / group;
        const float *qh = q + h * head_dim;
        double mx = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            const float *kt = kc + t * kv_dim + kvh * head_dim;
            double dot = 0.0;
            for (int64_t d = 0; d < head_dim; ++d)
                dot += (double)qh[d] * (double)kt[d];
            sc[t] = dot * inv;
            if (sc[t] > mx)
                mx = sc[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            sc[t] = exp(sc[t] - mx);
            z += sc[t];
        }
        for (int64_t d = 0; d < head_dim; ++d)
            acc[d] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const float *vt = vc + t * kv_dim + kvh * head_dim;
            for (int64_t d = 0; d < head_dim; ++d)
                acc[d] += sc[t] * (double)vt[d];
        }
        for (int64_t d = 0; d < head_dim; ++d)
            out[h * head_dim + d] = (float)(acc[d] / z);
        free(sc);
        free(acc);
    }
}

/* ------------------------------------------------------------------------- */
/* Layer pieces.                                                               */
/* ------------------------------------------------------------------------- */
static int64_t pad256(int64_t n) { return (n + 255) / 256 * 256; }

void orc_swiglu_ffn(const float *x, const float *gamma, const uint8_t *wgate,
                    const uint8_t *wup, const uint8_t *wdown, float *out,
                    int64_t hidden, int64_t hidden_pad, int64_t inter, float eps)
{
    float *normed = (float *)malloc((size_t)hidden_pad * sizeof(float));
    uint8_t *x8 = (uint8_t *)malloc((size_t)ORC_Q8_1_SIZE(1, hidden_pad));
    float *g = (float *)malloc((size_t)inter * sizeof(float));
    float *u = (float *)malloc((size_t)inter * sizeof(float));
    float *h = (float *)malloc((size_t)inter * sizeof(float));
    uint8_t *h8 = (uint8_t *)malloc((size_t)ORC_Q8_1_SIZE(1, inter));
    float *dn = (float *)malloc((size_t)hidden * sizeof(float));

    orc_rmsnorm(x, gamma, normed, 1, hidden, hidden_pad, eps);
    orc_q8_1_quantize(normed, x8, 1, hidden_pad);
    orc_q4k_q8_gemv(wgate, x8, g, 1, inter, hidden_pad);
    orc_q4k_q8_gemv(wup, x8, u, 1, inter, hidden_pad);
    for (int64_t i = 0; i < inter; ++i)
        h[i] = (float)(orc_silu((double)g[i]) * (double)u[i]);
    orc_q8_1_quantize(h, h8, 1, inter);
    orc_q4k_q8_gemv(wdown, h8, dn, 1, hidden, inter);
    orc_residual_add(x, dn, out, hidden);
    for (int64_t i = hidden; i < hidden_pad; ++i)
        out[i] = 0.0f;

    free(normed);
    free(x8);
    free(g);
    free(u);
    free(h);
    free(h8);
    free(dn);
}

void orc_decode_layer(const float *input, const orc_layer *L, float *kc, float *vc,
                      int64_t pos, float *output)
{
    int64_t hidden = L->hidden, hp = L->hidden_pad;
    int64_t q_dim = L->n_heads * L->head_dim;
    int64_t kv_dim = L->n_kv_heads * L->head_dim;
    int64_t q_pad = pad256(q_dim);

    float *normed = (float *)malloc((size_t)hp * sizeof(float));
    uint8_t *x8 = (uint8_t *)malloc((size_t)ORC_Q8_1_SIZE(1, hp));
    float *q = (float *)malloc((size_t)q_dim * sizeof(float));
    float *k = (float *)malloc((size_t)kv_dim * sizeof(float));
    float *v = (float *)malloc((size_t)kv_dim * sizeof(float));
    float *att = (float *)calloc((size_t)q_pad, sizeof(float));
    uint8_t *a8 = (uint8_t *)malloc((size_t)ORC_Q8_1_SIZE(1, q_pad));
    float *o = (float *)malloc((size_t)hidden * sizeof(float));
    float *res1 = (float *)malloc((size_t)hp * sizeof(float));

    orc_rmsnorm(input, L->attn_gamma, normed, 1, hidden, hp, L->eps);
    orc_q8_1_quantize(normed, x8, 1, hp);
    orc_q4k_q8_gemv(L->wq, x8, q, 1, q_dim, hp);
    orc_q4k_q8_gemv(L->wk, x8, k, 1, kv_dim, hp);
    orc_q4k_q8_gemv(L->wv, x8, v, 1, kv_dim, hp);
    /* projection biases (Qwen2's QKV bias, preload_qkv_bias in realizar 0.8.5
       cached.rs): one f32 add per output, before RoPE */
    if (L->bq)
        orc_residual_add(q, L->bq, q, q_dim);
    if (L->bk)
        orc_residual_add(k, L->bk, k, kv_dim);
    if (L->bv)
        orc_residual_add(v, L->bv, v, kv_dim);
    orc_rope(q, L->n_heads, L->head_dim, pos, L->rope_theta, L->rope_mode);
    orc_rope(k, L->n_kv_heads, L->head_dim, pos, L->rope_theta, L->rope_mode);
    memcpy(kc + pos * kv_dim, k, (size_t)kv_dim * sizeof(float));
    memcpy(vc + pos * kv_dim, v, (size_t)kv_dim * sizeof(float));
    orc_attention(q, kc, vc, pos, L->n_heads, L->n_kv_heads, L->head_dim, att);
    orc_q8_1_quantize(att, a8, 1, q_pad);
    orc_q4k_q8_gemv(L->wo, a8, o, 1, hidden, q_pad);
    orc_residual_add(input, o, res1, hidden);
    for (int64_t i = hidden; i < hp; ++i)
        res1[i] = 0.0f;
    orc_swiglu_ffn(res1, L->ffn_gamma, L->wgate, L->wup, L->wdown, output,
                   hidden, hp, L->inter, L->eps);

    free(normed);
    free(x8);
    free(q);
    free(k);
    free(v);
    free(att);
    free(a8);
    free(o);
    free(res1);
}

void orc_decode_stack(const float *input, const orc_layer *layers, int64_t n_layers,
                      float *const *kcs, float *const *vcs, int64_t pos,
                      const float *out_gamma, const uint8_t *lm_head, const float *lm_bias, int64_t vocab,
                      int64_t hidden, int64_t hidden_pad, float eps,
                      float *hidden_out, float *logits)
{
    float *a = (float *)malloc((size_t)hidden_pad * sizeof(float));
    float *b = (float *)malloc((size_t)hidden_pad * sizeof(float));
    memcpy(a, input, (size_t)hidden_pad * sizeof(float));
    for (int64_t l = 0; l < n_layers; ++l) {
        orc_decode_layer(a, &layers[l], kcs[l], vcs[l], pos, b);
        float *t = a;
        a = b;
        b = t;
    }
    memcpy(hidden_out, a, (size_t)hidden_pad * sizeof(float));
    orc_rmsnorm(a, out_gamma, b, 1, hidden, hidden_pad, eps);
    orc_q4_0_gemv(lm_head, b, logits, 1, vocab, hidden);
    if (lm_bias) /* the LM-head bias (preload_lm_head_bias in cached.rs): one f32 add */
        orc_residual_add(logits, lm_bias, logits, vocab);
    free(a);
    free(b);
}

/* ------------------------------------------------------------------------- */
/* Q4_0 whole-model layer (GpuModelQ4::forward_layer, realizar 0.8.4          */
/* src/gpu/adapters/using.rs): RMSNorm -> fused QKV Q4_0 GEMV -> RoPE q, k ->  */
/* attention over the cache -> output Q4_0 GEMV -> residual -> RMSNorm ->     */
/* FFN -> residual.  The FFN is ffn_swiglu_gpu (silu(gate) * up, then down)   */
/* when a gate matrix is given, else ffn_standard_gpu (up, GELU, down).       */
/* Every intermediate is an f32 buffer, as in the page.                       */
/* ------------------------------------------------------------------------- */
double orc_gelu(double x)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

void orc_decode_layer_q4_0(const float *input, const orc_layer_q4_0 *L, float *kc, float *vc,
                           int64_t pos, float *output)
{
    int64_t hidden = L->hidden;
    int64_t q_dim = L->n_heads * L->head_dim;
    int64_t kv_dim = L->n_kv_heads * L->head_dim;
    int64_t qkv_dim = q_dim + 2 * kv_dim;
    float *normed = (float *)malloc((size_t)hidden * sizeof(float));
    float *qkv = (float *)malloc((size_t)qkv_dim * sizeof(float));
    float *att = (float *)malloc((size_t)q_dim * sizeof(float));
    float *o = (float *)malloc((size_t)hidden * sizeof(float));
    float *res1 = (float *)malloc((size_t)hidden * sizeof(float));
    float *n2 = (float *)malloc((size_t)hidden * sizeof(float));
    float *u = (float *)malloc((size_t)L->inter * sizeof(float));
    float *g = (float *)malloc((size_t)L->inter * sizeof(float));
    float *h = (float *)malloc((size_t)L->inter * sizeof(float));
    float *dn = (float *)malloc((size_t)hidden * sizeof(float));

    orc_rmsnorm(input, L->attn_gamma, normed, 1, hidden, hidden, L->eps);
    orc_q4_0_gemv(L->wqkv, normed, qkv, 1, qkv_dim, hidden);
    float *q = qkv, *k = qkv + q_dim, *v = qkv + q_dim + kv_dim;
    orc_rope(q, L->n_heads, L->head_dim, pos, L->rope_theta, L->rope_mode);
    orc_rope(k, L->n_kv_heads, L->head_dim, pos, L->rope_theta, L->rope_mode);
    memcpy(kc + pos * kv_dim, k, (size_t)kv_dim * sizeof(float));
    memcpy(vc + pos * kv_dim, v, (size_t)kv_dim * sizeof(float));
    orc_attention(q, kc, vc, pos, L->n_heads, L->n_kv_heads, L->head_dim, att);
    orc_q4_0_gemv(L->wo, att, o, 1, hidden, q_dim);
    orc_residual_add(input, o, res1, hidden);
    orc_rmsnorm(res1, L->ffn_gamma, n2, 1, hidden, hidden, L->eps);
    orc_q4_0_gemv(L->wup, n2, u, 1, L->inter, hidden);
    if (L->wgate) {
        orc_q4_0_gemv(L->wgate, n2, g, 1, L->inter, hidden);
        for (int64_t i = 0; i < L->inter; ++i)
            h[i] = (float)(orc_silu((double)g[i]) * (double)u[i]);
    } else {
        for (int64_t i = 0; i < L->inter; ++i)
            h[i] = (float)orc_gelu((double)u[i]);
    }
    orc_q4_0_gemv(L->wdown, h, dn, 1, hidden, L->inter);
    orc_residual_add(res1, dn, output, hidden);

    free(normed);
    free(qkv);
    free(att);
    free(o);
    free(res1);
    free(n2);
    free(u);
    free(g);
    free(h);
    free(dn);
}
