/*
 * rz_oracle.h -- plain single-threaded CPU oracle for the Q4_K x Q8_1 decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the librz CUDA library
 * and its Python binding) includes, links or calls this code; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg do.  It shares no
 * code, header, table or constant generator with the GPU path.
 *
 * Precision: every step is computed in double and rounded to float where the
 * method hands an f32 buffer to the next step (GpuBuffer<f32> between the calls
 * of realizar 0.8.5 src/cuda/executor/cached.rs, transformer_layer_gpu_true_dp4a).
 * Quantisation decisions (Q8_1 codes) are taken in f32, as the format defines.
 *
 * Byte formats (GGML convention; the pages name the types but do not print
 * their layouts, so the layouts follow the workload definition of the
 * super-block: fp16 d and dmin, eight 6-bit scales and eight 6-bit mins packed
 * GGML-style into 12 bytes, 256 4-bit quants):
 *   Q4_K super-block, 144 B:  [0,2) d f16 | [2,4) dmin f16 | [4,16) scales[12] | [16,144) qs[128]
 *   Q4_0 block,        18 B:  [0,2) d f16 | [2,18) qs[16]
 *   Q8_1 activations, m rows of n (n % 32 == 0), structure of arrays:
 *       int8 q[m][n] | f32 d[m][n/32] | f32 s[m][n/32]     (1.25 bytes per value)
 *   The pages name Q8_1 without fixing how d and s are stored; f32 keeps s = d*sum(q)
 *   finite for activations whose block maximum exceeds what fp16 can hold times 32.
 */
#ifndef RZ_ORACLE_H
#define RZ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_QK_K 256
#define ORC_Q4K_BYTES 144
#define ORC_QK8 32
#define ORC_Q8_1_SIZE(m, n) ((m) * (n) + 8 * (m) * ((n) / 32))
#define ORC_QK4_0 32
#define ORC_Q4_0_BYTES 18

/* Threads of the row loops: 1, or the OpenMP team size in the all-core build. */
int orc_threads(void);

/* ---- IEEE-754 binary16 <-> binary32/64 (round to nearest, ties to even) ---- */
uint16_t orc_f32_to_f16(float x);
double orc_f16_to_f64(uint16_t h);
void orc_f32_to_f16_array(const float *x, uint16_t *h, int64_t n);
void orc_f16_to_f32_array(const uint16_t *h, float *x, int64_t n);

/* ---- Q4_K ---- */
void orc_q4k_unpack(const uint8_t *blk, uint16_t *d, uint16_t *dmin,
                    uint8_t sc[8], uint8_t mn[8], uint8_t q[256]);
void orc_q4k_pack(uint16_t d, uint16_t dmin, const uint8_t sc[8], const uint8_t mn[8],
                  const uint8_t q[256], uint8_t *blk);
/* n_blocks super-blocks -> 256*n_blocks doubles */
void orc_q4k_dequantize(const uint8_t *w, int64_t n_blocks, double *out);

/* ---- Q4_0 ---- */
void orc_q4_0_unpack(const uint8_t *blk, uint16_t *d, uint8_t q[32]);
void orc_q4_0_pack(uint16_t d, const uint8_t q[32], uint8_t *blk);
void orc_q4_0_dequantize(const uint8_t *w, int64_t n_blocks, double *out);

/* ---- Q8_1 ---- */
/* x: m rows of n floats (n % 32 == 0) -> ORC_Q8_1_SIZE(m, n) bytes */
void orc_q8_1_quantize(const float *x, uint8_t *out, int64_t m, int64_t n);
void orc_q8_1_dequantize(const uint8_t *q8, double *out, int64_t m, int64_t n);

/* ---- GEMVs ---- */
/* I[r][k] = sum over the 32 elements of sub-block k of q4 * q8 (int32, exact);
   x8 holds one row (m = 1). */
void orc_q4k_q8_subblock_dots(const uint8_t *w, const uint8_t *x8, int32_t *I,
                              int64_t out_dim, int64_t in_dim);
/* y[t][r] for t < m tokens; w row-major [out_dim][in_dim/256] super-blocks,
   x8 the Q8_1 buffer of m rows of in_dim. */
void orc_q4k_q8_gemv(const uint8_t *w, const uint8_t *x8, float *y,
                     int64_t m, int64_t out_dim, int64_t in_dim);
/* Q4_K weights against f32 activations (no Q8_1): y[t][r] = sum_e w[r][e] x[t][e]
   with the dequantised weights, accumulated in f64. */
void orc_q4k_f32_gemv(const uint8_t *w, const float *x, float *y,
                      int64_t m, int64_t out_dim, int64_t in_dim);
/* y[t][r] = sum_i w[r][i] * x[t][i]; w row-major [out_dim][in_dim/32] Q4_0 blocks */
void orc_q4_0_gemv(const uint8_t *w, const float *x, float *y,
                   int64_t m, int64_t out_dim, int64_t in_dim);

/* ---- elementwise / normalisation ---- */
/* y[0,n) = x * (1/sqrt(sum x^2 / n + eps)) * gamma; y[n, n_pad) = 0 */
void orc_rmsnorm(const float *x, const float *gamma, float *y,
                 int64_t m, int64_t n, int64_t n_pad, float eps);
void orc_residual_add(const float *a, const float *b, float *out, int64_t n);
double orc_silu(double x);
/* rotate n_heads heads of head_dim in place at position pos.
   mode 0: adjacent pairs (2i, 2i+1); mode 1: halves (i, i + head_dim/2). */
void orc_rope(float *v, int64_t n_heads, int64_t head_dim, int64_t pos, double theta, int mode);
/* out[n_heads*head_dim] = softmax over t = 0..pos of q.k_t / sqrt(head_dim), times v_t,
   K/V caches [*][kv_dim] with row stride kv_dim; kv head of q head h is h / (n_heads/n_kv_heads). */
void orc_attention(const float *q, const float *kc, const float *vc, int64_t pos,
                   int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float *out);

/* ---- layer / stack ---- */
typedef struct {
    const uint8_t *wq, *wk, *wv, *wo, *wgate, *wup, *wdown; /* Q4_K */
    const float *attn_gamma, *ffn_gamma;                     /* [hidden] */
    int64_t hidden, hidden_pad, n_heads, n_kv_heads, head_dim, inter;
    float eps;
    double rope_theta;
    int rope_mode;
    const float *bq, *bk, *bv; /* optional projection biases (NULL: none) */
} orc_layer;

/* out[hidden_pad] = x + down(q8(silu(gate.q8(norm x)) * up.q8(norm x))) */
void orc_swiglu_ffn(const float *x, const float *gamma, const uint8_t *wgate,
                    const uint8_t *wup, const uint8_t *wdown, float *out,
                    int64_t hidden, int64_t hidden_pad, int64_t inter, float eps);
/* One decode step of one token at `pos` (0-based).  kc/vc: [max_seq][kv_dim]
   f32, written at row pos, read at rows 0..pos.  A non-NULL bias is added (f32)
   to its projection's output before RoPE. */
void orc_decode_layer(const float *input, const orc_layer *L, float *kc, float *vc,
                      int64_t pos, float *output);
/* layers, then output RMSNorm, then Q4_0 LM head (+ lm_bias, when not NULL) -> logits[vocab]. */
void orc_decode_stack(const float *input, const orc_layer *layers, int64_t n_layers,
                      float *const *kcs, float *const *vcs, int64_t pos,
                      const float *out_gamma, const uint8_t *lm_head, const float *lm_bias, int64_t vocab,
                      int64_t hidden, int64_t hidden_pad, float eps,
                      float *hidden_out, float *logits);

/* ---- Q4_0 whole-model layer (GpuModelQ4::forward_layer of realizar 0.8.4
   src/gpu/adapters/using.rs): every projection Q4_0 against f32 activations. */
/* GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
double orc_gelu(double x);
typedef struct {
    const uint8_t *wqkv;   /* Q4_0 [q_dim + 2 kv_dim][hidden]: Q rows, then K, then V */
    const uint8_t *wo;     /* Q4_0 [hidden][q_dim] */
    const uint8_t *wgate;  /* Q4_0 [inter][hidden], or NULL: the GELU FFN (up -> GELU -> down) */
    const uint8_t *wup;    /* Q4_0 [inter][hidden] */
    const uint8_t *wdown;  /* Q4_0 [hidden][inter] */
    const float *attn_gamma, *ffn_gamma; /* [hidden] */
    int64_t hidden, n_heads, n_kv_heads, head_dim, inter;
    float eps;
    double rope_theta;
    int rope_mode;
} orc_layer_q4_0;
/* One decode step of one token at `pos`; kc/vc [max_seq][kv_dim], written at row pos. */
void orc_decode_layer_q4_0(const float *input, const orc_layer_q4_0 *L, float *kc, float *vc,
                           int64_t pos, float *output);

#ifdef __cplusplus
}
#endif
#endif
