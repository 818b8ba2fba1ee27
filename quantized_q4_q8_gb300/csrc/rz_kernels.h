// rz_kernels.h -- host-side launchers shared between the librz translation units.
// Arguments are already validated by the C-ABI layer (abi.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rz {

// A 2-D tiled tensor map (TMA descriptor) over a row-major array of `rows` rows
// whose rows are `row_stride` bytes apart and hold `inner` elements of
// `elem_bytes` bytes (1, 2 or 4), copied in boxes of box_inner x box_rows
// elements; out-of-range parts of a box read as zero.  Encoded through the
// driver's cuTensorMapEncodeTiled (looked up once through the runtime).
cudaError_t encode_tensor_map_2d(CUtensorMap *map, const void *base, int elem_bytes, uint64_t inner, uint64_t rows,
                                 uint64_t row_stride, uint32_t box_inner, uint32_t box_rows);
// The same for rank dimensions (dims[0] innermost; strides[i] = bytes between
// consecutive indices of dimension i + 1).
cudaError_t encode_tensor_map(CUtensorMap *map, const void *base, int elem_bytes, int rank, const uint64_t *dims,
                              const uint64_t *strides, const uint32_t *box);

// Device properties of the current device (cached per device).
struct DevInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
};
const DevInfo &dev_info();

// Device error word of the current device (a file-scope __device__ variable).
unsigned *dev_error_word();

// Test aid: non-zero makes the next Q4_K GEMV launch leave its first stage in
// CTA 0 unissued and bound that CTA's waits by this many polls (then reset to 0).
extern uint32_t g_stall_next_gemv;

// Launch with the programmatic-stream-serialization attribute (PDL) so that the
// kernel's weight prefetch overlaps the tail of the previous kernel in the stream.
extern bool g_use_pdl;

// ---------------------------------------------------------------- Q8_1
cudaError_t launch_q8_1_quantize(const float *x, void *q8, int64_t m, int64_t n, cudaStream_t s);

// ---------------------------------------------------------------- many-token Q4_K x Q8_1 (tensor cores)
// y[t][r] for m tokens (any m >= 1) with tcgen05.mma: a packing kernel turns the
// Q8_1 activations into tensor-core operands in `workspace`
// (q4k_gemm_tc_workspace_bytes), then one CTA per 128 tokens x 128 rows.
int64_t q4k_gemm_tc_workspace_bytes(int64_t m, int64_t in_dim);
int q4k_gemm_tc_launch_count();
cudaError_t launch_q4k_gemm_tc(const void *w, const void *q8, float *y, int64_t ldy, int64_t m, int64_t out_dim,
                               int64_t in_dim, void *workspace, cudaStream_t s);

// ---------------------------------------------------------------- norms / elementwise
cudaError_t launch_rmsnorm(const float *x, const float *gamma, float *y, void *q8, int64_t m,
                           int64_t n, int64_t n_pad, float eps, cudaStream_t s);
cudaError_t launch_residual_add(const float *a, const float *b, float *out, int64_t n,
                                cudaStream_t s);
// h = silu(g) * u (g != nullptr) or GELU(u), n values
cudaError_t launch_ffn_act(const float *g, const float *u, float *h, int64_t n, cudaStream_t s);

// ---------------------------------------------------------------- Q4_K x Q8_1 GEMV
enum Q4kEpilogue { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2 };

struct Q4kSegment {
    const void *w;     // Q4_K [rows][in_dim]
    float *y;          // [m][ldy], row r of token t at y[t * ldy + r]
    const float *res;  // [m][ldr] (EPI_RESID) or nullptr
    int64_t rows;
    int64_t ldy = 0;   // 0: rows
    int64_t ldr = 0;   // 0: rows
    const float *bias = nullptr;  // [rows] added to every token's output (EPI_STORE only)
    int64_t zero_to = 0;          // > rows: y[t][rows .. zero_to) is set to 0 (a padded hidden state)
};

// Up to three weight matrices with the same in_dim read against one Q8_1
// activation (the fused Q|K|V launch).  For EPI_SWIGLU seg[0] is the gate
// matrix, seg[1] the up matrix, and seg[0].y receives silu(gate) * up.
cudaError_t launch_q4k_gemv(const Q4kSegment *seg, int nseg, int epilogue, const void *q8,
                            int64_t m, int64_t in_dim, cudaStream_t s);

// The same GEMV with f32 activations quantised inside the kernel (every CTA
// quantises the whole input into its shared memory): with gamma != nullptr the
// input is first RMS-normalised over its first norm_n values (the fused
// RMSNorm -> Q8_1 of the decode layer), else quantised as it is (the Q8_1 of the
// FFN intermediate).  x: f32 [m][ldx].  Bit-identical to rz_rmsnorm / the Q8_1
// kernel followed by launch_q4k_gemv.
struct F32Input {
    const float *x;
    int64_t ldx;
    const float *gamma;  // nullptr: no norm
    int64_t norm_n;
    float eps;
};
bool q4k_gemv_f32_input_ok(int64_t m, int64_t in_dim);
// Whether a layer should let the GEMV quantise its f32 input (else a separate
// norm / quantise launch first).
bool q4k_gemv_f32_input_preferred(int64_t m, int64_t in_dim);
// launches one GEMV of m tokens takes (token groups when the activations exceed
// shared memory; Q8_1 input stages its codes in phases first)
int q4k_gemv_launch_count(int64_t m, int64_t in_dim, int epilogue, bool q8_input = true);

// From this many tokens on, the GEMV runs on the tensor cores (gemv_q4k_mma.cu).
constexpr int kMmaMinTokens = 4;
// Most tokens one tensor-core launch takes for this shape (0: none fit).
int q4k_gemv_mma_group(int64_t m, int64_t in_dim, int epilogue, bool q8_input);
cudaError_t launch_q4k_gemv_mma(const Q4kSegment *seg, int nseg, int epilogue, const int8_t *xq, const float *xd,
                                const float *xs, const F32Input *f32in, int64_t m, int64_t in_dim, cudaStream_t s);
cudaError_t launch_q4k_gemv_f32(const Q4kSegment *seg, int nseg, int epilogue, const F32Input &in,
                                int64_t m, int64_t in_dim, cudaStream_t s);

// Whether the stage ring of the GEMV fits in shared memory for this shape
// (two stages of one pack: rows up to about 47000 wide at m = 1).
bool q4k_gemv_supported(int64_t m, int64_t in_dim, int epilogue);

// Q4_K weights times f32 activations without Q8_1 (gemv_q4k_f32.cu): x [m][ldx],
// y [m][ldy], optional bias [out_dim]; tokens in groups that fit shared memory.
int q4k_f32_gemv_group(int64_t in_dim);
cudaError_t launch_q4k_f32_gemv(const void *w, const float *x, int64_t ldx, float *y, int64_t ldy, const float *bias,
                                int64_t m, int64_t out_dim, int64_t in_dim, cudaStream_t s);

cudaError_t launch_q4k_subblock_dots(const void *w, const void *q8, int32_t *I, int64_t out_dim,
                                     int64_t in_dim, cudaStream_t s);

// ---------------------------------------------------------------- attention
struct AttnArgs {
    CUtensorMap kmap, vmap;      // the caches as [m][max_seq][kv_dim] f32, boxes of one head x 64 rows
    const float *q, *k, *v;      // pre-RoPE projections of token t at + t * ld_qkv
    int64_t ld_qkv;
    double rope_f[128];          // rope_f[i] = (theta^(-2 / head_dim))^i: pair i turns by position * rope_f[i]
    float *kc, *vc;              // caches: token t at + t * seq_stride, row p at + p * kv_dim
    int64_t seq_stride;
    int max_seq;
    const int32_t *positions;    // device int32 [m], or nullptr to use `position`
    int position;
    int m, n_heads, n_kv_heads, head_dim, group, q_dim, q_pad, kv_dim;
    float rope_theta;
    int rope_mode;
    int chunk_len, n_chunks;     // n_chunks covers max_seq (workspace layout)
    int launch_chunks;           // chunks launched: enough for the host position, else n_chunks
    int att_bufs;                // set by launch_attention: 1 = K then V through one buffer, 2 = both
    int stream_slots;            // set by launch_attention for the streaming kernel: tiles in flight per warp,
    int stream_tab_tokens;       //   tokens whose RoPE angles a CTA tabulates,
    int stream_kmax;             //   record slots per (token, kv head)
    int stream_cluster;          //   CTAs per cluster of the cluster kernel
    float *part;                 // workspace of attention_part_bytes: the partial records
    int *counters;               // workspace: [m][n_kv_heads], zero before the first call
    float *att;                  // f32 [m][q_dim] output, or nullptr
    void *att_q8;                // Q8_1 of m rows of q_pad (output), or nullptr
    unsigned *err;
};

int attention_chunk_len(int max_seq, int n_kv_heads, int m);
// Bytes of the partial-record workspace (AttnArgs::part) for either attention kernel.
size_t attention_part_bytes(int64_t m, int n_kv_heads, int group, int head_dim, int max_seq);
size_t attention_smem_bytes(int group, int head_dim, int chunk_len);
// (table,) then split-sequence attention with RoPE, the KV append, the merge and
// the Q8_1 of the output.
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s);

// ---------------------------------------------------------------- Q4_0 GEMV
// bias (nullable) [out_dim] is added to every token's output row
// Kernels one launch_q4_0_gemv call starts for these shapes (the one-token ring
// kernel once per token, else one multi-token launch).
// The Q4_0 GEMV of one to eight tokens per launch on the tensor cores (the LM
// head; gemv_q4_0_mma.cu): rows with in_dim % 256 == 0, x
// 16-byte aligned, ldx % 4 == 0.  Tokens in equal groups of at most eight.
bool q4_0_head_mma_ok(int64_t m, int64_t out_dim, int64_t in_dim, const float *x, int64_t ldx);
int q4_0_head_mma_launches(int64_t m);
cudaError_t launch_q4_0_head_mma(const void *w, const float *x, int64_t ldx, float *y, int64_t m, int64_t out_dim,
                                 int64_t in_dim, const float *bias, cudaStream_t s);
int q4_0_gemv_launches(int64_t m, int64_t out_dim, int64_t in_dim);
cudaError_t launch_q4_0_gemv(const void *w, const float *x, float *y, int64_t m, int64_t out_dim,
                             int64_t in_dim, cudaStream_t s, const float *bias = nullptr);
// as above with activation row stride ldx (elements) between tokens
cudaError_t launch_q4_0_gemv_ld(const void *w, const float *x, int64_t ldx, float *y, int64_t m,
                                int64_t out_dim, int64_t in_dim, cudaStream_t s, const float *bias = nullptr);

// ---------------------------------------------------------------- layer / stack
// wk == wv == nullptr: wq is the fused [q_dim + 2 kv_dim][hidden_pad] matrix (and
// bq, when given, its fused bias).  Biases are optional.
struct LayerDesc {
    const void *wq, *wk, *wv, *wo, *wgate, *wup, *wdown;
    const float *attn_gamma, *ffn_gamma;
    int hidden, hidden_pad, n_heads, n_kv_heads, head_dim, inter;
    float eps, rope_theta;
    int rope_mode;
    const float *bq, *bk, *bv;
};

struct KvDesc {
    float *k, *v;
    int64_t seq_stride;
    int max_seq;
};

size_t ffn_workspace_bytes(int64_t m, int64_t hidden_pad, int64_t inter);
cudaError_t launch_swiglu_ffn(const float *x, const float *gamma, const void *w_gate, const void *w_up,
                              const void *w_down, float *out, int64_t m, int64_t hidden,
                              int64_t hidden_pad, int64_t inter, float eps, void *workspace,
                              cudaStream_t s);
size_t layer_workspace_bytes(const LayerDesc &L, int64_t m, int max_seq);
AttnArgs make_attn_args(const LayerDesc &L, int64_t m, const KvDesc &kv, const int32_t *positions,
                        int position, float *part, int *counters,
                        const float *q, const float *k, const float *v, int64_t ld_qkv, float *att,
                        void *att_q8);
cudaError_t launch_decode_layer(const float *input, const LayerDesc &L, const KvDesc &kv,
                                const int32_t *positions, int position, int64_t m, float *output,
                                void *workspace, cudaStream_t s);
size_t stack_workspace_bytes(const LayerDesc &L, int64_t m, int max_seq);

// The Q4_0 whole-model layer (every projection Q4_0 against f32 activations).
struct LayerQ40Desc {
    const void *wqkv, *wo, *wgate, *wup, *wdown;  // wgate nullptr: GELU FFN
    const float *attn_gamma, *ffn_gamma;
    int hidden, n_heads, n_kv_heads, head_dim, inter;
    float eps, rope_theta;
    int rope_mode;
};
size_t layer_q4_0_workspace_bytes(const LayerQ40Desc &L, int64_t m, int max_seq);
cudaError_t launch_decode_layer_q4_0(const float *input, const LayerQ40Desc &L, const KvDesc &kv,
                                     const int32_t *positions, int position, int64_t m, float *output,
                                     void *workspace, cudaStream_t s);
// logits == nullptr: the layers only, the final hidden state in hidden_out.
cudaError_t launch_decode_stack(const float *input, const LayerDesc *layers, int n_layers,
                                const KvDesc *kvs, const int32_t *positions, int position, int64_t m,
                                const float *out_gamma, const void *lm_head, const float *lm_bias, int64_t vocab,
                                float *hidden_out, float *logits, void *workspace, cudaStream_t s);
// kernels launched by one launch_decode_stack (with or without the head)
// vocab: rows of the LM head (with head only)
int stack_kernel_launches(const LayerDesc *layers, int n_layers, int64_t m, int max_seq, bool head,
                          int64_t vocab);

}  // namespace rz
