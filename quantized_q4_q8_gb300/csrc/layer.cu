// layer.cu -- the SwiGLU FFN, the decode layer and the decode stack as launch
// sequences on one stream (no host synchronisation, no allocation).
//
// Step order of transformer_layer_gpu_true_dp4a (realizar 0.8.5
// src/cuda/executor/cached.rs):
//   1 RMSNorm(attn) -> 2 Q8_1 once for Q, K and V -> 3 Q/K/V GEMVs ->
//   4 incremental attention -> 5 Q8_1 of the attention output -> 6 O GEMV ->
//   7 residual -> 8 RMSNorm(ffn) -> 9 SwiGLU FFN (gate, up, silu(gate) * up, Q8_1,
//   down) -> 10 residual.
// Fusions here: 1+2+3 are one launch: every CTA of the Q|K|V GEMV normalises
// and quantises the layer input into its shared memory, and the three matrices
// are one GEMV; 4+5 are one split-sequence attention kernel that also applies
// RoPE, appends k and v to the cache,
// and whose merging CTA quantises its heads; 6+7 are one GEMV with a residual
// epilogue; in 9 the norm + Q8_1 live in the gate/up GEMV, whose epilogue
// applies silu(gate) * up, and the Q8_1 of h lives in the down GEMV, whose
// epilogue adds the residual (10).  Five launches per layer.  When the batch is
// too large for the activations to sit in shared memory, the norm and the
// quantisation run as their own kernels instead.
// The stack (forward_all_layers_gpu_to_logits in realizar 0.8.5
// src/cuda/executor/layers/forward_utils.rs) chains the layers through two
// workspace buffers, then the output RMSNorm and the Q4_0 LM head.
#include <algorithm>

#include "rz_common.cuh"
#include "rz_kernels.h"

namespace rz {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static size_t q8_bytes(int64_t m, int64_t n) { return (size_t)(m * n + 8 * m * (n / 32)); }

size_t ffn_workspace_bytes(int64_t m, int64_t hidden_pad, int64_t inter)
{
    return align256(q8_bytes(m, hidden_pad)) + align256((size_t)m * inter * 4) +
           align256(q8_bytes(m, inter));
}

cudaError_t launch_swiglu_ffn(const float *x, const float *gamma, const void *w_gate, const void *w_up,
                              const void *w_down, float *out, int64_t m, int64_t hidden,
                              int64_t hidden_pad, int64_t inter, float eps, void *workspace,
                              cudaStream_t s)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *x8 = ws;
    ws += align256(q8_bytes(m, hidden_pad));
    float *h = reinterpret_cast<float *>(ws);
    ws += align256((size_t)m * inter * 4);
    void *h8 = ws;

    cudaError_t e;
    Q4kSegment gu[2] = {{w_gate, h, nullptr, inter, inter, 0}, {w_up, nullptr, nullptr, inter, 0, 0}};
    if (q4k_gemv_f32_input_preferred(m, hidden_pad)) {
        // RMSNorm -> Q8_1 inside the gate/up GEMV (every CTA normalises the input)
        e = launch_q4k_gemv_f32(gu, 2, EPI_SWIGLU, F32Input{x, hidden_pad, gamma, hidden, eps}, m, hidden_pad, s);
    } else {
        e = launch_rmsnorm(x, gamma, nullptr, x8, m, hidden, hidden_pad, eps, s);
        if (e != cudaSuccess) return e;
        e = launch_q4k_gemv(gu, 2, EPI_SWIGLU, x8, m, hidden_pad, s);
    }
    if (e != cudaSuccess) return e;
    // out's padding [hidden, hidden_pad) is zeroed by the down GEMV itself (a
    // memset node would end the programmatic-dependent-launch chain)
    Q4kSegment dn = {w_down, out, x, hidden, hidden_pad, hidden_pad, nullptr, hidden_pad};
    if (q4k_gemv_f32_input_preferred(m, inter)) {
        // Q8_1 of h inside the down GEMV
        e = launch_q4k_gemv_f32(&dn, 1, EPI_RESID, F32Input{h, inter, nullptr, 0, 0.0f}, m, inter, s);
    } else {
        e = launch_q8_1_quantize(h, h8, m, inter, s);
        if (e != cudaSuccess) return e;
        e = launch_q4k_gemv(&dn, 1, EPI_RESID, h8, m, inter, s);
    }
    return e;
}

// ---------------------------------------------------------------- decode layer
// Workspace of one layer: the attention merge counters first, then the
// intermediates of the step.
struct LayerWs {
    int *counters;
    void *x8;
    float *qkv, *part;
    void *a8;
    float *res1;
    void *ffn;
    float *h;  // the f32 FFN intermediate inside the FFN workspace
    size_t total;
};

static LayerWs layer_ws(const LayerDesc &L, int64_t m, int max_seq, uint8_t *base)
{
    LayerWs w{};
    const int q_dim = L.n_heads * L.head_dim, kv_dim = L.n_kv_heads * L.head_dim;
    const int q_pad = (q_dim + 255) / 256 * 256;
    const int group = L.n_heads / L.n_kv_heads;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    w.counters = reinterpret_cast<int *>(take((size_t)m * L.n_kv_heads * 4));
    w.x8 = take(q8_bytes(m, L.hidden_pad));
    w.qkv = reinterpret_cast<float *>(take((size_t)m * (q_dim + 2 * kv_dim) * 4));
    w.part = reinterpret_cast<float *>(take(attention_part_bytes(m, L.n_kv_heads, group, L.head_dim, max_seq)));
    w.a8 = take(q8_bytes(m, q_pad));
    w.res1 = reinterpret_cast<float *>(take((size_t)m * L.hidden_pad * 4));
    w.ffn = take(ffn_workspace_bytes(m, L.hidden_pad, L.inter));
    w.h = base ? reinterpret_cast<float *>(static_cast<uint8_t *>(w.ffn) + align256(q8_bytes(m, L.hidden_pad)))
               : nullptr;
    w.total = off;
    return w;
}

size_t layer_workspace_bytes(const LayerDesc &L, int64_t m, int max_seq)
{
    return layer_ws(L, m, max_seq, nullptr).total;
}

AttnArgs make_attn_args(const LayerDesc &L, int64_t m, const KvDesc &kv, const int32_t *positions,
                        int position, float *part, int *counters,
                        const float *q, const float *k, const float *v, int64_t ld_qkv, float *att,
                        void *att_q8)
{
    AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.ld_qkv = ld_qkv;
    // r^i by binary powering of r = theta^(-2 / head_dim), in double precision
    const double r = pow((double)L.rope_theta, -2.0 / (double)L.head_dim);
    for (int i = 0; i < L.head_dim / 2 && i < 128; ++i) {
        double f = 1.0, b = r;
        for (int e = i; e; e >>= 1) {
            if (e & 1) f *= b;
            b *= b;
        }
        a.rope_f[i] = f;
    }
    a.kc = kv.k;
    a.vc = kv.v;
    a.seq_stride = kv.seq_stride;
    a.max_seq = kv.max_seq;
    a.positions = positions;
    a.position = position;
    a.m = (int)m;
    a.n_heads = L.n_heads;
    a.n_kv_heads = L.n_kv_heads;
    a.head_dim = L.head_dim;
    a.group = L.n_heads / L.n_kv_heads;
    a.q_dim = L.n_heads * L.head_dim;
    a.q_pad = (a.q_dim + 255) / 256 * 256;
    a.kv_dim = L.n_kv_heads * L.head_dim;
    a.rope_theta = L.rope_theta;
    a.rope_mode = L.rope_mode;
    a.chunk_len = attention_chunk_len(kv.max_seq, L.n_kv_heads, (int)m);
    a.n_chunks = (kv.max_seq + a.chunk_len - 1) / a.chunk_len;
    a.launch_chunks = positions ? a.n_chunks : position / a.chunk_len + 1;
    a.part = part;
    a.counters = counters;
    a.att = att;
    a.att_q8 = att_q8;
    a.err = dev_error_word();
    return a;
}

cudaError_t launch_decode_layer(const float *input, const LayerDesc &L, const KvDesc &kv,
                                const int32_t *positions, int position, int64_t m, float *output,
                                void *workspace, cudaStream_t s)
{
    LayerWs w = layer_ws(L, m, kv.max_seq, static_cast<uint8_t *>(workspace));
    const int q_dim = L.n_heads * L.head_dim, kv_dim = L.n_kv_heads * L.head_dim;
    const int q_pad = (q_dim + 255) / 256 * 256;
    const int64_t ld_qkv = q_dim + 2 * kv_dim;

    cudaError_t e;
    Q4kSegment qkv[3] = {{L.wq, w.qkv, nullptr, q_dim, ld_qkv, 0, L.bq},
                         {L.wk, w.qkv + q_dim, nullptr, kv_dim, ld_qkv, 0, L.bk},
                         {L.wv, w.qkv + q_dim + kv_dim, nullptr, kv_dim, ld_qkv, 0, L.bv}};
    int nseg = 3;
    if (!L.wk) {
        // fused Q|K|V matrix: one segment of q_dim + 2 kv_dim rows
        qkv[0].rows = ld_qkv;
        nseg = 1;
    }
    if (q4k_gemv_f32_input_preferred(m, L.hidden_pad)) {
        // RMSNorm -> Q8_1 inside the Q|K|V GEMV
        e = launch_q4k_gemv_f32(qkv, nseg, EPI_STORE,
                                F32Input{input, L.hidden_pad, L.attn_gamma, L.hidden, L.eps}, m, L.hidden_pad, s);
    } else {
        e = launch_rmsnorm(input, L.attn_gamma, nullptr, w.x8, m, L.hidden, L.hidden_pad, L.eps, s);
        if (e != cudaSuccess) return e;
        e = launch_q4k_gemv(qkv, nseg, EPI_STORE, w.x8, m, L.hidden_pad, s);
    }
    if (e != cudaSuccess) return e;
    AttnArgs a = make_attn_args(L, m, kv, positions, position, w.part, w.counters,
                                w.qkv, w.qkv + q_dim, w.qkv + q_dim + kv_dim, ld_qkv, nullptr, w.a8);
    e = launch_attention(a, s);
    if (e != cudaSuccess) return e;
    Q4kSegment o = {L.wo, w.res1, input, L.hidden, L.hidden_pad, L.hidden_pad};
    e = launch_q4k_gemv(&o, 1, EPI_RESID, w.a8, m, q_pad, s);
    if (e != cudaSuccess) return e;
    return launch_swiglu_ffn(w.res1, L.ffn_gamma, L.wgate, L.wup, L.wdown, output, m, L.hidden,
                             L.hidden_pad, L.inter, L.eps, w.ffn, s);
}

// ---------------------------------------------------------------- stack
// Workspace: two layer-output buffers, the normalised final hidden state, then
// one layer workspace shared by every layer.
size_t stack_workspace_bytes(const LayerDesc &L, int64_t m, int max_seq)
{
    return 3 * align256((size_t)m * L.hidden_pad * 4) + layer_workspace_bytes(L, m, max_seq);
}

cudaError_t launch_decode_stack(const float *input, const LayerDesc *layers, int n_layers,
                                const KvDesc *kvs, const int32_t *positions, int position, int64_t m,
                                const float *out_gamma, const void *lm_head, const float *lm_bias, int64_t vocab,
                                float *hidden_out, float *logits, void *workspace, cudaStream_t s)
{
    const LayerDesc &L0 = layers[0];
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t hbytes = align256((size_t)m * L0.hidden_pad * 4);
    float *buf[2] = {reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + hbytes)};
    float *normed = reinterpret_cast<float *>(ws + 2 * hbytes);
    void *lws = ws + 3 * hbytes;
    const float *cur = input;
    cudaError_t e = cudaSuccess;
    for (int l = 0; l < n_layers; ++l) {
        float *out = (l == n_layers - 1 && hidden_out) ? hidden_out : buf[l & 1];
        e = launch_decode_layer(cur, layers[l], kvs[l], positions, position, m, out, lws, s);
        if (e != cudaSuccess) return e;
        cur = out;
    }
    if (!logits) return cudaSuccess;  // the layers only (rz_decode_layers)
    e = launch_rmsnorm(cur, out_gamma, normed, nullptr, m, L0.hidden, L0.hidden_pad, L0.eps, s);
    if (e != cudaSuccess) return e;
    return launch_q4_0_gemv_ld(lm_head, normed, L0.hidden_pad, logits, m, vocab, L0.hidden, s, lm_bias);
}

int stack_kernel_launches(const LayerDesc *layers, int n_layers, int64_t m, int max_seq, bool head,
                          int64_t vocab)
{
    (void)max_seq;
    const LayerDesc &L0 = layers[0];
    const int h = head ? 1 + q4_0_gemv_launches(m, vocab, L0.hidden) : 0;  // output RMSNorm, LM head
    const int q_pad = (L0.n_heads * L0.head_dim + 255) / 256 * 256;
    // a GEMV with its input normalised / quantised inside, or a separate kernel
    // for that and then the Q8_1-input GEMV
    auto gemv = [&](int64_t in_dim, int epi) {
        const int n = q4k_gemv_launch_count(m, in_dim, epi);
        return q4k_gemv_f32_input_preferred(m, in_dim) ? n : 1 + n;
    };
    int per_layer = 1 /* attention */ + q4k_gemv_launch_count(m, q_pad, EPI_RESID) /* O */;
    per_layer += gemv(L0.hidden_pad, EPI_STORE);   // RMSNorm -> Q|K|V
    per_layer += gemv(L0.hidden_pad, EPI_SWIGLU);  // RMSNorm -> gate/up
    per_layer += gemv(L0.inter, EPI_RESID);        // Q8_1 of h -> down
    return n_layers * per_layer + h;
}

// ---------------------------------------------------------------- Q4_0 layer
// GpuModelQ4::forward_layer (realizar 0.8.4 src/gpu/adapters/using.rs) for m
// tokens: RMSNorm -> fused QKV Q4_0 GEMV -> attention (RoPE, KV append, as in the
// Q4_K layer) -> O Q4_0 GEMV -> residual -> RMSNorm -> up (and gate) Q4_0 GEMVs
// -> silu(gate) * up or GELU(up) -> down Q4_0 GEMV -> residual.  Every
// intermediate is an f32 buffer, as on the page.
struct LayerQ40Ws {
    int *counters;
    float *normed, *qkv, *part, *att, *o, *res1, *n2, *u, *g, *h, *dn;
    size_t total;
};

static LayerQ40Ws layer_q4_0_ws(const LayerQ40Desc &L, int64_t m, int max_seq, uint8_t *base)
{
    LayerQ40Ws w{};
    const int q_dim = L.n_heads * L.head_dim, kv_dim = L.n_kv_heads * L.head_dim;
    const int group = L.n_heads / L.n_kv_heads;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += align256(bytes);
        return reinterpret_cast<float *>(p);
    };
    w.counters = reinterpret_cast<int *>(take((size_t)m * L.n_kv_heads * 4));
    w.normed = take((size_t)m * L.hidden * 4);
    w.qkv = take((size_t)m * (q_dim + 2 * kv_dim) * 4);
    w.part = take(attention_part_bytes(m, L.n_kv_heads, group, L.head_dim, max_seq));
    w.att = take((size_t)m * q_dim * 4);
    w.o = take((size_t)m * L.hidden * 4);
    w.res1 = take((size_t)m * L.hidden * 4);
    w.n2 = take((size_t)m * L.hidden * 4);
    w.u = take((size_t)m * L.inter * 4);
    w.g = take((size_t)m * L.inter * 4);
    w.h = take((size_t)m * L.inter * 4);
    w.dn = take((size_t)m * L.hidden * 4);
    w.total = off;
    return w;
}

size_t layer_q4_0_workspace_bytes(const LayerQ40Desc &L, int64_t m, int max_seq)
{
    return layer_q4_0_ws(L, m, max_seq, nullptr).total;
}

cudaError_t launch_decode_layer_q4_0(const float *input, const LayerQ40Desc &L, const KvDesc &kv,
                                     const int32_t *positions, int position, int64_t m, float *output,
                                     void *workspace, cudaStream_t s)
{
    LayerQ40Ws w = layer_q4_0_ws(L, m, kv.max_seq, static_cast<uint8_t *>(workspace));
    const int q_dim = L.n_heads * L.head_dim, kv_dim = L.n_kv_heads * L.head_dim;
    const int64_t ld_qkv = q_dim + 2 * kv_dim;
    cudaError_t e = launch_rmsnorm(input, L.attn_gamma, w.normed, nullptr, m, L.hidden, L.hidden, L.eps, s);
    if (e == cudaSuccess) e = launch_q4_0_gemv_ld(L.wqkv, w.normed, L.hidden, w.qkv, m, ld_qkv, L.hidden, s);
    if (e != cudaSuccess) return e;
    LayerDesc ld{};
    ld.n_heads = L.n_heads;
    ld.n_kv_heads = L.n_kv_heads;
    ld.head_dim = L.head_dim;
    ld.rope_theta = L.rope_theta;
    ld.rope_mode = L.rope_mode;
    AttnArgs a = make_attn_args(ld, m, kv, positions, position, w.part, w.counters, w.qkv,
                                w.qkv + q_dim, w.qkv + q_dim + kv_dim, ld_qkv, w.att, nullptr);
    e = launch_attention(a, s);
    if (e == cudaSuccess) e = launch_q4_0_gemv_ld(L.wo, w.att, q_dim, w.o, m, L.hidden, q_dim, s);
    if (e == cudaSuccess) e = launch_residual_add(input, w.o, w.res1, m * L.hidden, s);
    if (e == cudaSuccess) e = launch_rmsnorm(w.res1, L.ffn_gamma, w.n2, nullptr, m, L.hidden, L.hidden, L.eps, s);
    if (e == cudaSuccess) e = launch_q4_0_gemv_ld(L.wup, w.n2, L.hidden, w.u, m, L.inter, L.hidden, s);
    if (e == cudaSuccess && L.wgate) e = launch_q4_0_gemv_ld(L.wgate, w.n2, L.hidden, w.g, m, L.inter, L.hidden, s);
    if (e == cudaSuccess) e = launch_ffn_act(L.wgate ? w.g : nullptr, w.u, w.h, m * L.inter, s);
    if (e == cudaSuccess) e = launch_q4_0_gemv_ld(L.wdown, w.h, L.inter, w.dn, m, L.hidden, L.inter, s);
    if (e == cudaSuccess) e = launch_residual_add(w.res1, w.dn, output, m * L.hidden, s);
    return e;
}

}  // namespace rz
