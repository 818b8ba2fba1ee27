/*
 * rz.h -- C ABI of librz, the GB300 (sm_103a) Q4_K x Q8_1 single-token decode path.
 *
 * The operations follow the dp4a decode layer of realizar 0.8.5
 * src/cuda/executor/cached.rs (transformer_layer_gpu_true_dp4a), the Q4_0 model
 * forward of realizar 0.8.4 src/gpu/adapters/using.rs (GpuModelQ4::forward,
 * q4_0_gemv_into, rms_norm_inplace), the GPU-resident stack of realizar 0.8.5
 * src/cuda/executor/layers/forward_utils.rs (forward_all_layers_gpu_to_logits)
 * and the single-token semantics of realizar 0.8.4
 * src/gguf/cuda/clone_layer_weights.rs (forward_single_full_cuda_with_cache).
 *
 * Conventions for every entry point
 *   - Pointers named w, x, y, q8, gamma, out, input, output, workspace, k, v are
 *     DEVICE pointers owned by the caller.  librz never allocates device memory,
 *     never synchronises the stream and never copies between host and device
 *     (except rz_check_device_error, which reads one word back).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and returns immediately.  Launches are stream-ordered and can be captured
 *     into a CUDA graph.
 *   - Every shape, alignment and range check runs on the host before anything is
 *     launched.  A failed check returns a non-zero rz_status, launches nothing and
 *     sets a message readable with rz_last_error() (thread-local).
 *   - Weights must be 16-byte aligned; f32 and Q8_1 buffers 16-byte aligned.
 *   - Device-side conditions that the host cannot see (a position read from device
 *     memory outside the cache, a bounded wait that ran out) never trap: the kernel
 *     records a code in a device error word and skips the access; the host reads
 *     and clears it with rz_check_device_error().
 *
 * Data formats (GGML convention for the weights; the pages name the types but do
 * not print their layouts):
 *   Q4_K  super-block of 256 weights in 144 bytes: f16 d | f16 dmin | 12 bytes of
 *         eight 6-bit scales and eight 6-bit mins | 128 bytes of 4-bit quants.
 *         weight = d * sc_j * q - dmin * m_j for sub-block j = e / 32; weight e is
 *         nibble (e % 64 < 32 ? low : high) of qs[32 * (e / 64) + e % 32].
 *         A matrix [out_dim][in_dim] is row-major: out_dim rows of in_dim / 256
 *         consecutive super-blocks.
 *   Q4_0  block of 32 weights in 18 bytes: f16 d | 16 bytes of 4-bit quants;
 *         weight i = d * (q_i - 8), q_i the low nibble of byte i (i < 16) or the
 *         high nibble of byte i - 16.  Row-major like Q4_K.
 *   Q8_1  activations quantised in blocks of 32: d = max|x| / 127 (f32 division),
 *         q = round-half-away(x / d) clamped to [-127, 127] (0 when d == 0),
 *         s = d * sum(q).  A buffer for m rows of n values (n % 32 == 0) holds
 *         int8 q[m][n], then f32 d[m][n/32], then f32 s[m][n/32]:
 *         RZ_Q8_1_BYTES(m, n) bytes.  (d and s are f32 so that s stays finite for
 *         block maxima beyond fp16 range / 32.)
 */
#ifndef RZ_H
#define RZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RZ_OK = 0,
    RZ_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad enum */
    RZ_ERR_SHAPE = 2,       /* dimension not a multiple of the block size, m > RZ_MAX_BATCH, ... */
    RZ_ERR_ALIGN = 3,       /* pointer not 16-byte aligned */
    RZ_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has the CUDA error) */
    RZ_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (rz_check_device_error) */
    RZ_ERR_UNSUPPORTED = 6, /* no sm_103a device, or a configuration this build does not handle */
    RZ_ERR_DEVICE = 7       /* a device-side range check failed (rz_check_device_error) */
} rz_status;

typedef void *rz_stream; /* cudaStream_t */

#define RZ_Q4K_BLOCK_BYTES 144
#define RZ_Q4K_BLOCK_WEIGHTS 256
#define RZ_Q4_0_BLOCK_BYTES 18
#define RZ_Q4_0_BLOCK_WEIGHTS 32
#define RZ_Q8_1_BLOCK 32
#define RZ_Q8_1_BYTES(m, n) ((m) * (n) + 8 * (m) * ((n) / 32))
#define RZ_MAX_BATCH 16

/* Message of the last failed call on this thread ("" if none). */
const char *rz_last_error(void);
/* Library version string. */
const char *rz_version(void);

/*
 * rz_q8_1_quantize -- Q8_1 quantisation of activations (q8_quantize_async in
 * transformer_layer_gpu_true_dp4a, steps 2 and 5).
 *   x    f32 [m][n], row-major.            q8  RZ_Q8_1_BYTES(m, n) bytes (output).
 *   1 <= m, n % 32 == 0.  Bit-exact with the format definition above.
 */
rz_status rz_q8_1_quantize(const float *x, void *q8, int64_t m, int64_t n, rz_stream stream);

/*
 * rz_q4k_q8_gemv -- y = W x for Q4_K weights and Q8_1 activations, the integer
 * GEMV behind every Q/K/V/O and FFN projection (q4k_q8_gemv_async in
 * transformer_layer_gpu_true_dp4a, steps 3 and 6).
 *   For token t < m and row r:
 *     y[t][r] = sum_b d_b * sum_j sc_bj * d8_tbj * I_tbrj - dmin_b * sum_j m_bj * s_tbj
 *   with I the exact int32 dot of the 32 codes of sub-block j.
 *   w   Q4_K [out_dim][in_dim]     q8  Q8_1 of m rows of in_dim     y  f32 [m][out_dim]
 *   1 <= m <= RZ_MAX_BATCH, in_dim % 256 == 0, out_dim >= 1.  Weights are read once
 *   for all m tokens.  f32 combination order differs from a sequential sum
 *   (deterministic run to run).
 */
rz_status rz_q4k_q8_gemv(const void *w, const void *q8, float *y, int64_t m, int64_t out_dim,
                         int64_t in_dim, rz_stream stream);

/*
 * rz_q4k_q8_subblock_dots -- the integer sub-block dots alone, for exact checks:
 *   I[r][k] = sum_{i<32} q4[r][32k + i] * q8[32k + i]   (one activation row)
 *   I  int32 [out_dim][in_dim/32] (output).  in_dim % 256 == 0.
 */
rz_status rz_q4k_q8_subblock_dots(const void *w, const void *q8, int32_t *I, int64_t out_dim,
                                  int64_t in_dim, rz_stream stream);

/*
 * rz_q4k_q8_gemv_ex -- the same GEMV with an epilogue:
 *     y[t][r] = (W x_t)_r + bias[r]           (bias != NULL; the QKV and head biases
 *                                              of preload_qkv_bias in cached.rs)
 *     y[t][r] = (W x_t)_r + residual[t][r]    (residual != NULL; steps 6-7 and 9-10 of
 *                                              transformer_layer_gpu_true_dp4a)
 *     y[t][r] = (W x_t)_r                     (both NULL)
 *   bias f32 [out_dim] (4-byte aligned); residual, y f32 [m][ld] with row stride ld
 *   (0 = out_dim; ld >= out_dim); y may alias residual.  A bias and a residual in
 *   one call: RZ_ERR_UNSUPPORTED.  Other arguments and checks as rz_q4k_q8_gemv.
 */
rz_status rz_q4k_q8_gemv_ex(const void *w, const void *q8, const float *bias, const float *residual, float *y,
                            int64_t ld, int64_t m, int64_t out_dim, int64_t in_dim, rz_stream stream);

/*
 * rz_q4k_q8_gemm -- the same product for many tokens at once (a prompt's prefill:
 * GpuModelQ4::forward of realizar 0.8.4 src/gpu/adapters/using.rs takes a sequence
 * of token ids), on the tensor cores (tcgen05.mma):
 *     y[t][r] = sum_b d_b * sum_j sc_bj * d8_tbj * I_tbrj - dmin_b * sum_j m_bj * s_tbj
 *   for every token t < m, with the integer sub-block dots I exact, as
 *   rz_q4k_q8_gemv.  Each 128 x 128 tile of (tokens, rows) reads its weights once.
 *   w          Q4_K [out_dim][in_dim]         q8  Q8_1 of m rows of in_dim
 *   y          f32 [m][ldy] (ldy 0 = out_dim; ldy >= out_dim), 4-byte aligned
 *   workspace  device scratch of at least rz_q4k_q8_gemm_workspace_bytes(m, in_dim)
 *              bytes, 16-byte aligned (the activations re-laid out as tensor-core
 *              operands); contents need no initialisation and are not kept.
 *   1 <= m (any; tokens beyond a multiple of 128 are padding inside the kernel),
 *   in_dim % 256 == 0, out_dim >= 1.  Two launches.  f32 combination order
 *   differs from rz_q4k_q8_gemv's (deterministic run to run).  A bounded wait that
 *   runs out records RZ_ERR_TIMEOUT for rz_check_device_error.
 */
size_t rz_q4k_q8_gemm_workspace_bytes(int64_t m, int64_t in_dim);
rz_status rz_q4k_q8_gemm(const void *w, const void *q8, float *y, int64_t ldy, int64_t m, int64_t out_dim,
                         int64_t in_dim, void *workspace, size_t ws_bytes, rz_stream stream);

/*
 * rz_rmsnorm_q4k_gemv -- steps 1-3 of transformer_layer_gpu_true_dp4a in one
 * launch: RMSNorm of x over its first n values with gamma (zero padding after n),
 * Q8_1 quantisation of the normed row (bit-identical to rz_rmsnorm's q8 output),
 * then up to three Q4_K GEMVs against that one Q8_1 activation, their outputs
 * side by side in y (the Q | K | V projections):
 *     y[t][off_k + r] = (W_k q8(norm(x_t)))_r (+ bias[k][r]),  off_k = rows[0] + ... + rows[k-1]
 *   x      f32 [m][ldx], in_dim values per row are read (ldx >= in_dim)
 *   gamma  f32 [n]; n <= in_dim; in_dim % 256 == 0
 *   w      host array of n_mats (1..3) device pointers to Q4_K [rows[k]][in_dim]
 *   bias   host array of n_mats device pointers (each may be NULL), or NULL
 *   y      f32 [m][ldy], ldy >= rows[0] + ... + rows[n_mats-1]
 *   x, gamma, y 16-byte aligned, ldx and ldy multiples of 4.  Every CTA normalises and
 *   quantises the whole row (m * in_dim * 1.25 B of shared memory must fit, else
 *   RZ_ERR_UNSUPPORTED).
 */
rz_status rz_rmsnorm_q4k_gemv(const float *x, int64_t ldx, const float *gamma, int64_t n, float eps, int32_t n_mats,
                              const void *const *w, const int64_t *rows, const float *const *bias, float *y,
                              int64_t ldy, int64_t m, int64_t in_dim, rz_stream stream);

/*
 * rz_q4k_q8_gemv_multi -- up to three Q4_K GEMVs against one Q8_1 activation in one
 * launch (the Q | K | V projections of transformer_layer_gpu_true_dp4a, realizar
 * 0.8.5 src/cuda/executor/cached.rs, with the activation quantised beforehand, as
 * a layer does from four tokens on):
 *     y[t][off_k + r] = (W_k q8_t)_r (+ bias[k][r]),  off_k = rows[0] + ... + rows[k-1]
 *   q8     Q8_1 of m rows of in_dim values (the layout of rz_q8_1_quantize), 16-byte aligned
 *   w      host array of n_mats (1..3) device pointers to Q4_K [rows[k]][in_dim], 16-byte aligned
 *   bias   host array of n_mats device pointers (each may be NULL), or NULL
 *   y      f32 [m][ldy], ldy >= rows[0] + ... + rows[n_mats-1], 4-byte aligned
 *   1 <= m <= RZ_MAX_BATCH, in_dim % 256 == 0.  The same results as one
 *   rz_q4k_q8_gemv_ex per matrix.
 */
rz_status rz_q4k_q8_gemv_multi(const void *q8, int32_t n_mats, const void *const *w, const int64_t *rows,
                               const float *const *bias, float *y, int64_t ldy, int64_t m, int64_t in_dim,
                               rz_stream stream);

/*
 * rz_q4k_f32_gemv -- y = W x (+ bias) for Q4_K weights and f32 activations, with no
 * Q8_1 quantisation of x (q4k_gemv_cached_async in transformer_layer_gpu_cached,
 * realizar 0.8.5 src/cuda/executor/cached.rs):
 *     y[t][r] = sum_e (d * sc_j * q_e - dmin * m_j) x[t][e]   (+ bias[r])
 *   w Q4_K [out_dim][in_dim]   x f32 [m][in_dim]   y f32 [m][out_dim]   bias f32 [out_dim] or NULL
 *   1 <= m <= RZ_MAX_BATCH, in_dim % 256 == 0; w and x 16-byte aligned, y and bias
 *   4-byte aligned.  f32 products and sums (order differs from a sequential sum;
 *   deterministic run to run).
 */
rz_status rz_q4k_f32_gemv(const void *w, const float *x, const float *bias, float *y, int64_t m, int64_t out_dim,
                          int64_t in_dim, rz_stream stream);

/*
 * rz_q4_0_gemv -- y = W x for Q4_0 weights and f32 activations (the LM head of
 * GpuModelQ4::forward, q4_0_gemv_into; step 5 of that function).
 *   w  Q4_0 [out_dim][in_dim]   x  f32 [m][in_dim]   y  f32 [m][out_dim]
 *   in_dim % 32 == 0, 1 <= m <= RZ_MAX_BATCH.  Only w needs 16-byte alignment of
 *   its base; rows of 18-byte blocks may start anywhere.  When in_dim % 256 == 0
 *   and x is 16-byte aligned the products run on the tensor cores with x split
 *   into two f16 pieces (x to about 2^-22 relative; |x| must stay below 65504);
 *   otherwise in f32 FMAs.  f32 accumulation either way (order differs from a
 *   sequential sum; deterministic run to run).
 */
rz_status rz_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                       int64_t in_dim, rz_stream stream);

/*
 * rz_q4_0_gemv_bias -- rz_q4_0_gemv plus a bias added to every token's output:
 * y[t][r] = (W x_t)_r + bias[r] (the LM-head bias of preload_lm_head_bias,
 * realizar 0.8.5 src/cuda/executor/cached.rs).  bias f32 [out_dim], 4-byte
 * aligned; other arguments as rz_q4_0_gemv.
 */
rz_status rz_q4_0_gemv_bias(const void *w, const float *x, const float *bias, float *y, int64_t m, int64_t out_dim,
                            int64_t in_dim, rz_stream stream);

/*
 * rz_rmsnorm -- RMSNorm with optional fused Q8_1 quantisation (rms_norm_inplace in
 * using.rs; rmsnorm_gpu + q8_quantize_async in transformer_layer_gpu_true_dp4a):
 *   rms = sqrt(sum_{i<n} x_i^2 / n + eps);  y_i = x_i / rms * gamma_i (i < n),
 *   y_i = 0 for n <= i < n_pad (the zero padding of pad_and_upload_input).
 *   x      f32 [m][n_pad] (only the first n of each row are read)
 *   gamma  f32 [n]
 *   y      f32 [m][n_pad] output, or NULL
 *   q8     Q8_1 of m rows of n_pad (output), or NULL.  When given, it is exactly
 *          the Q8_1 quantisation of the f32 y this call computes.
 *   At least one of y, q8 non-NULL.  n >= 1, n_pad >= n, n_pad % 32 == 0 when q8.
 */
rz_status rz_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m, int64_t n,
                     int64_t n_pad, float eps, rz_stream stream);

/*
 * rz_residual_add -- out = a + b elementwise in f32 (residual_add_gpu, steps 7 and
 * 10 of transformer_layer_gpu_true_dp4a).  out may alias a or b.  Bit-exact.
 */
rz_status rz_residual_add(const float *a, const float *b, float *out, int64_t n, rz_stream stream);

/*
 * ---------------------------------------------------------------------------
 * Layer-level entry points.  They launch several kernels in stream order and
 * use a caller-provided device workspace (size from the *_workspace_bytes
 * function, base 16-byte aligned).  The workspace holds intermediates only; the
 * attention counters inside it must be zero before the first call (fill the
 * workspace with zeros once after allocating it); every completed call leaves
 * them zero again.  Calls that share a workspace must not overlap on the GPU.
 * ---------------------------------------------------------------------------
 */

/* One Q4_K decode layer (the weights of transformer_layer_gpu_true_dp4a).
 * Matrices (Q4_K, row-major [out][in]):
 *   wq [n_heads*head_dim][hidden_pad]   wk, wv [n_kv_heads*head_dim][hidden_pad]
 *   wo [hidden][q_pad]                  q_pad = n_heads*head_dim rounded up to 256
 *   wgate, wup [inter][hidden_pad]      wdown [hidden][inter]
 * attn_gamma, ffn_gamma: f32 [hidden].  hidden_pad % 256 == 0 (the zero padding of
 * pad_and_upload_input), inter % 256 == 0, head_dim % 32 == 0 and <= 256,
 * n_heads % n_kv_heads == 0 with at most 16 query heads per kv head.
 * rope_mode 0 rotates adjacent pairs (2i, 2i+1), 1 rotates (i, i + head_dim/2);
 * the angle of pair i at position p is p * rope_theta^(-2i/head_dim).
 * Fused Q|K|V layout (OwnedQKVWeights::Fused of realizar 0.8.4
 * clone_layer_weights.rs): wk = wv = NULL and wq holds the one matrix
 * [n_heads*head_dim + 2*n_kv_heads*head_dim][hidden_pad] (Q rows, then K, then V).
 * Biases (the Qwen2 QKV bias of preload_qkv_bias in realizar 0.8.5 cached.rs):
 * bq [n_heads*head_dim], bk, bv [n_kv_heads*head_dim] f32, each NULL for none,
 * added to the projections before RoPE; with the fused layout bq holds the fused
 * bias [q_dim + 2*kv_dim] and bk, bv must be NULL.  Biases need 4-byte alignment. */
typedef struct {
    const void *wq, *wk, *wv, *wo, *wgate, *wup, *wdown;
    const float *attn_gamma, *ffn_gamma;
    int32_t hidden, hidden_pad, n_heads, n_kv_heads, head_dim, inter;
    float eps, rope_theta;
    int32_t rope_mode;
    const float *bq, *bk, *bv;
} rz_layer_weights;

/* f32 KV cache of one layer.  Row p of sequence t (token t of a batch) is at
 * k + t*seq_stride + p*kv_dim (same for v), kv_dim = n_kv_heads*head_dim.
 * seq_stride is ignored when m == 1; otherwise >= max_seq*kv_dim and a multiple of 4
 * (every sequence starts 16-byte aligned).  1 <= max_seq <= 4096. */
typedef struct {
    float *k, *v;
    int64_t seq_stride;
    int32_t max_seq;
} rz_kv_cache;

/*
 * rz_swiglu_ffn -- out = x + W_down q8( silu(W_gate q8(n)) * (W_up q8(n)) ),
 * n = RMSNorm(x; gamma) (steps 8-10 of transformer_layer_gpu_true_dp4a;
 * fused_ffn_swiglu_gpu_true_dp4a; SiLU of the gate times up as in cuda_swiglu_ffn
 * of clone_layer_weights.rs).  x, out f32 [m][hidden_pad] (out may alias x;
 * out[.][hidden..hidden_pad) is written as 0).
 */
size_t rz_swiglu_ffn_workspace_bytes(int64_t m, int64_t hidden_pad, int64_t inter);
rz_status rz_swiglu_ffn(const float *x, const float *gamma, const void *w_gate, const void *w_up,
                        const void *w_down, float *out, int64_t m, int64_t hidden,
                        int64_t hidden_pad, int64_t inter, float eps, void *workspace,
                        size_t ws_bytes, rz_stream stream);

/*
 * rz_attention_decode -- RoPE on q and k at each token's position, append k and v
 * to the cache row `position`, then softmax(q k^T / sqrt(head_dim)) v over cache
 * rows 0..position with the GQA map kv_head = q_head / (n_heads / n_kv_heads)
 * (incremental_attention_async, step 4; first-token and GQA semantics of
 * forward_single_full_cuda_with_cache).
 *   q, k, v   f32 projections, token t at q + t*ld_qkv (same ld for k, v);
 *             q [n_heads*head_dim], k, v [n_kv_heads*head_dim] per token.
 *   positions device int32 [m] (each checked in the kernel against max_seq; a bad
 *             one records RZ_ERR_DEVICE, skips its cache write and yields zeros),
 *             or NULL to use `position` for every token (checked on the host).
 *   att       f32 [m][n_heads*head_dim] output, or NULL.
 *   att_q8    Q8_1 of m rows of q_pad (output, the O projection's input), or NULL.
 */
size_t rz_attention_workspace_bytes(int64_t m, int32_t n_heads, int32_t n_kv_heads,
                                    int32_t head_dim, int32_t max_seq);
rz_status rz_attention_decode(const float *q, const float *k, const float *v, int64_t ld_qkv,
                              const rz_kv_cache *kv, const int32_t *positions, int32_t position,
                              int64_t m, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                              float rope_theta, int32_t rope_mode, float *att, void *att_q8,
                              void *workspace, size_t ws_bytes, rz_stream stream);

/*
 * rz_decode_layer -- one decode step of one layer for m tokens (m sequences),
 * the step order of transformer_layer_gpu_true_dp4a.
 *   input, output f32 [m][hidden_pad] (zero padding kept; output may alias input)
 *   kv            this layer's cache, written at each token's position
 *   positions     device int32 [m] or NULL for the host `position`
 */
size_t rz_decode_layer_workspace_bytes(const rz_layer_weights *w, int64_t m, int32_t max_seq);
rz_status rz_decode_layer(const float *input, const rz_layer_weights *w, const rz_kv_cache *kv,
                          const int32_t *positions, int32_t position, int64_t m, float *output,
                          void *workspace, size_t ws_bytes, rz_stream stream);

/*
 * rz_decode_stack -- n_layers decode layers, then the output RMSNorm and the Q4_0
 * LM head (forward_all_layers_gpu_to_logits; GpuModelQ4::forward steps 4-5).
 *   layers, kvs   host arrays of n_layers descriptors (same hidden, hidden_pad,
 *                 eps and kv max_seq for every layer)
 *   out_gamma     f32 [hidden];  lm_head Q4_0 [vocab][hidden]
 *   lm_bias       f32 [vocab] added to the logits (preload_lm_head_bias in realizar
 *                 0.8.5 cached.rs), or NULL
 *   hidden_out    f32 [m][hidden_pad] final hidden state, or NULL
 *   logits        f32 [m][vocab]
 */
size_t rz_decode_stack_workspace_bytes(const rz_layer_weights *layers, int32_t n_layers, int64_t m,
                                       int32_t max_seq);
rz_status rz_decode_stack(const float *input, const rz_layer_weights *layers, const rz_kv_cache *kvs,
                          int32_t n_layers, const int32_t *positions, int32_t position, int64_t m,
                          const float *out_gamma, const void *lm_head, const float *lm_bias, int64_t vocab,
                          float *hidden_out, float *logits, void *workspace, size_t ws_bytes,
                          rz_stream stream);

/*
 * rz_decode_layers -- the n_layers decode layers of rz_decode_stack without the
 * output RMSNorm and the LM head (a pipeline stage, or a caller with its own
 * head).  output: f32 [m][hidden_pad], the final hidden state (padding zero).
 * Other arguments, checks and the workspace (rz_decode_stack_workspace_bytes)
 * as for rz_decode_stack.
 */
rz_status rz_decode_layers(const float *input, const rz_layer_weights *layers, const rz_kv_cache *kvs,
                           int32_t n_layers, const int32_t *positions, int32_t position, int64_t m, float *output,
                           void *workspace, size_t ws_bytes, rz_stream stream);

/*
 * The Q4_0 whole-model layer (GpuModelQ4::forward_layer of realizar 0.8.4
 * src/gpu/adapters/using.rs): every projection Q4_0 against f32 activations.
 *   wqkv   Q4_0 [n_heads*head_dim + 2*n_kv_heads*head_dim][hidden] (Q rows, then K, then V)
 *   wo     Q4_0 [hidden][n_heads*head_dim]
 *   wgate  Q4_0 [inter][hidden], or NULL for the GELU FFN
 *   wup    Q4_0 [inter][hidden]      wdown  Q4_0 [hidden][inter]
 *   attn_gamma, ffn_gamma f32 [hidden]
 * hidden and inter multiples of 32 (hidden <= 16384), head_dim a multiple of 32 in
 * [32, 256], rope as rz_layer_weights.
 * Step order: RMSNorm -> QKV GEMV -> RoPE q, k at the position, KV append,
 * attention over rows 0..position -> O GEMV -> + input -> RMSNorm -> FFN ->
 * + residual.  FFN: silu(gate) * up then down (ffn_swiglu_gpu) with a gate,
 * else GELU(up) then down (ffn_standard_gpu), GELU in its tanh form
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).  Intermediates are f32.
 */
typedef struct {
    const void *wqkv, *wo, *wgate, *wup, *wdown;
    const float *attn_gamma, *ffn_gamma;
    int32_t hidden, n_heads, n_kv_heads, head_dim, inter;
    float eps, rope_theta;
    int32_t rope_mode;
} rz_layer_weights_q4_0;

/*
 * rz_decode_layer_q4_0 -- one decode step of one Q4_0 layer for m tokens.
 *   input, output f32 [m][hidden] (output may alias input); kv, positions,
 *   position and the workspace (zero-filled once) as for rz_decode_layer.
 */
size_t rz_decode_layer_q4_0_workspace_bytes(const rz_layer_weights_q4_0 *w, int64_t m, int32_t max_seq);
rz_status rz_decode_layer_q4_0(const float *input, const rz_layer_weights_q4_0 *w, const rz_kv_cache *kv,
                               const int32_t *positions, int32_t position, int64_t m, float *output, void *workspace,
                               size_t ws_bytes, rz_stream stream);

/*
 * rz_decode_stack_launches -- the number of librz kernels one rz_decode_stack call
 * (with_head != 0, an LM head of `vocab` rows) or one rz_decode_layers call
 * (with_head == 0, vocab unused) launches for these layers, batch m and cache
 * length max_seq.  Memset nodes are not kernels and are not counted.
 * Returns 0 for arguments the calls would reject.
 */
int32_t rz_decode_stack_launches(const rz_layer_weights *layers, int32_t n_layers, int64_t m, int32_t max_seq,
                                 int32_t with_head, int64_t vocab);

/*
 * rz_swiglu_ffn_static -- the same computation as rz_swiglu_ffn, for callers that
 * cannot allocate device memory or pass a workspace (the paper has no
 * counterpart: this is a packaging variant of rz_swiglu_ffn).  Its intermediates
 * live in a fixed 512 KiB device array inside the library (every GPU that loads
 * the library holds one until the process exits); shapes whose scratch
 * (rz_swiglu_ffn_workspace_bytes) exceeds 512 KiB are rejected with
 * RZ_ERR_UNSUPPORTED.  It calls no allocator.  The first call on a device looks
 * up the array's device address (a runtime query), so make that first call before
 * any stream capture.  All calls share the array: calls that overlap on the GPU
 * race and must be ordered by the caller.  Arguments as for rz_swiglu_ffn.
 */
rz_status rz_swiglu_ffn_static(const float *x, const float *gamma, const void *w_gate, const void *w_up,
                               const void *w_down, float *out, int64_t m, int64_t hidden,
                               int64_t hidden_pad, int64_t inter, float eps, rz_stream stream);

/*
 * rz_check_device_error -- synchronise `stream`, read the device error word of the
 * current device and clear it.  *code_out (nullable) receives the raw code (0 = none).
 * Returns RZ_OK, RZ_ERR_TIMEOUT (a bounded wait ran out) or RZ_ERR_DEVICE (a
 * device-side range check failed and the access was skipped).
 */
rz_status rz_check_device_error(rz_stream stream, uint32_t *code_out);

/*
 * rz_set_pdl -- enable (default) or disable programmatic dependent launch between
 * consecutive librz kernels in a stream.  With it a GEMV starts streaming its
 * weights while the previous kernel finishes; results are identical either way.
 */
rz_status rz_set_pdl(int enable);

/*
 * rz_debug_stall_next_gemv -- test aid for the bounded-wait error path (off by
 * default).  The next Q4_K GEMV launch of this process leaves the first weight
 * stage of its CTA 0 unissued and bounds every wait of that CTA by wait_limit
 * polls (1024 <= wait_limit <= 2^22, else RZ_ERR_INVALID_ARG).  Its consumer warps
 * then run out of their wait, record code 0x101 in the device error word and
 * stop; the CTA still waits for every copy it did issue before it exits, so no
 * copy outlives the kernel.  rz_check_device_error then returns RZ_ERR_TIMEOUT,
 * and the output rows of CTA 0 of that launch are undefined.  One shot: the
 * setting clears itself at that launch.  The pages return errors instead of
 * panicking (GpuError in realizar 0.8.5 forward_utils.rs); this checks that a
 * wait that cannot complete ends in such an error and not in a hung GPU.
 */
rz_status rz_debug_stall_next_gemv(uint32_t wait_limit);


#ifdef __cplusplus
}
#endif
#endif /* RZ_H */
