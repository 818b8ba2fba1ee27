"""torch-facing helpers over the librz C ABI (marshalling and output allocation only)."""
from __future__ import annotations

import ctypes as C

from ._lib import call, load, status

__all__ = [
    "q8_1_size", "q4k_bytes", "q4_0_bytes",
    "rz_q8_1_quantize", "rz_q4k_q8_gemv", "rz_q4k_q8_subblock_dots", "rz_q4_0_gemv",
    "rz_q4k_q8_gemv_ex", "rz_rmsnorm_q4k_gemv", "q4k_q8_gemv_ex", "rmsnorm_q4k_gemv",
    "rz_q4k_q8_gemv_multi", "q4k_q8_gemv_multi",
    "rz_q4k_f32_gemv", "q4k_f32_gemv",
    "rz_q4k_q8_gemm", "q4k_q8_gemm_workspace_bytes", "q4k_q8_gemm",
    "rz_rmsnorm", "rz_residual_add", "rz_check_device_error", "rz_set_pdl", "rz_debug_stall_next_gemv",
    "q8_1_quantize", "q4k_q8_gemv", "q4k_q8_subblock_dots", "q4_0_gemv",
    "rmsnorm", "residual_add", "check_device_error", "set_pdl", "version",
    "DeviceLayer", "DeviceKV", "DeviceStack", "workspace", "swiglu_ffn_workspace_bytes",
    "swiglu_ffn", "rz_swiglu_ffn_static", "attention_workspace_bytes", "attention_decode",
    "decode_layer_workspace_bytes", "decode_layer", "rz_decode_stack", "decode_stack",
    "rz_decode_layers", "decode_layers", "DeviceLayerQ40", "decode_layer_q4_0",
]


def q8_1_size(m: int, n: int) -> int:
    """Bytes of a Q8_1 buffer of m rows of n values (int8 q | f32 d | f32 s)."""
    return m * n + 8 * m * (n // 32)


def q4k_bytes(out_dim: int, in_dim: int) -> int:
    return out_dim * (in_dim // 256) * 144


def q4_0_bytes(out_dim: int, in_dim: int) -> int:
    return out_dim * (in_dim // 32) * 18


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# ------------------------------------------------------------------ raw entry points
def rz_q8_1_quantize(x, q8, m, n, stream=None):
    return call("rz_q8_1_quantize", _ptr(x), _ptr(q8), m, n, _stream(stream))


def rz_q4k_q8_gemv(w, q8, y, m, out_dim, in_dim, stream=None):
    return call("rz_q4k_q8_gemv", _ptr(w), _ptr(q8), _ptr(y), m, out_dim, in_dim, _stream(stream))


def rz_q4k_q8_subblock_dots(w, q8, I, out_dim, in_dim, stream=None):
    return call("rz_q4k_q8_subblock_dots", _ptr(w), _ptr(q8), _ptr(I), out_dim, in_dim,
                _stream(stream))


def rz_q4k_q8_gemv_ex(w, q8, bias, residual, y, ld, m, out_dim, in_dim, stream=None):
    return call("rz_q4k_q8_gemv_ex", _ptr(w), _ptr(q8), _ptr(bias), _ptr(residual), _ptr(y), ld, m,
                out_dim, in_dim, _stream(stream))


def rz_rmsnorm_q4k_gemv(x, ldx, gamma, n, eps, ws, rows, biases, y, ldy, m, in_dim, stream=None):
    """ws, rows, biases: sequences of equal length (1..3); biases may be None."""
    k = len(ws)
    wp = (C.c_void_p * k)(*[_ptr(t) for t in ws])
    rp = (C.c_int64 * k)(*rows)
    bp = None if biases is None else (C.c_void_p * k)(*[_ptr(b) for b in biases])
    return call("rz_rmsnorm_q4k_gemv", _ptr(x), ldx, _ptr(gamma), n, eps, k, wp, rp, bp, _ptr(y), ldy,
                m, in_dim, _stream(stream))


def rz_q4k_q8_gemv_multi(q8, ws, rows, biases, y, ldy, m, in_dim, stream=None):
    """ws, rows, biases: sequences of equal length (1..3); biases may be None."""
    k = len(ws)
    wp = (C.c_void_p * k)(*[_ptr(t) for t in ws])
    rp = (C.c_int64 * k)(*rows)
    bp = None if biases is None else (C.c_void_p * k)(*[_ptr(b) for b in biases])
    return call("rz_q4k_q8_gemv_multi", _ptr(q8), k, wp, rp, bp, _ptr(y), ldy, m, in_dim, _stream(stream))


def q4k_q8_gemv_multi(q8, ws, rows, m, in_dim, biases=None, out=None, stream=None):
    """GEMVs of 1..3 matrices against one Q8_1 activation; returns f32 [m, sum(rows)]."""
    import torch
    if out is None:
        out = torch.empty((m, sum(rows)), dtype=torch.float32, device=q8.device)
    rz_q4k_q8_gemv_multi(q8, ws, rows, biases, out, out.shape[-1], m, in_dim, stream)
    return out


def rz_q4k_f32_gemv(w, x, bias, y, m, out_dim, in_dim, stream=None):
    return call("rz_q4k_f32_gemv", _ptr(w), _ptr(x), _ptr(bias), _ptr(y), m, out_dim, in_dim, _stream(stream))


def q4k_f32_gemv(w, x, out_dim, in_dim, bias=None, out=None, stream=None):
    """Q4_K weights times f32 activations x [m, in_dim] (no Q8_1) -> f32 [m, out_dim]."""
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, out_dim), dtype=torch.float32, device=w.device)
    rz_q4k_f32_gemv(w, x, bias, out, m, out_dim, in_dim, stream)
    return out


def rz_q4_0_gemv(w, x, y, m, out_dim, in_dim, stream=None):
    return call("rz_q4_0_gemv", _ptr(w), _ptr(x), _ptr(y), m, out_dim, in_dim, _stream(stream))


def rz_rmsnorm(x, gamma, y, q8, m, n, n_pad, eps, stream=None):
    return call("rz_rmsnorm", _ptr(x), _ptr(gamma), _ptr(y), _ptr(q8), m, n, n_pad, eps,
                _stream(stream))


def rz_residual_add(a, b, out, n, stream=None):
    return call("rz_residual_add", _ptr(a), _ptr(b), _ptr(out), n, _stream(stream))


def rz_check_device_error(stream=None):
    """Returns (status, code); status 0 when the device error word was clear."""
    code = C.c_uint32(0)
    st = status("rz_check_device_error", _stream(stream), C.byref(code))
    return st, code.value


def rz_set_pdl(enable: bool):
    return call("rz_set_pdl", 1 if enable else 0)


def rz_debug_stall_next_gemv(wait_limit: int):
    """Test aid: the next Q4_K GEMV launch runs out of a bounded wait (see rz.h)."""
    return call("rz_debug_stall_next_gemv", int(wait_limit))


# ------------------------------------------------------------------ tensor helpers
def _cuda_contig(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def q8_1_quantize(x, out=None, stream=None):
    """x: f32 CUDA [m, n] -> uint8 CUDA [q8_1_size(m, n)]."""
    import torch
    _cuda_contig(x, torch.float32, "x")
    m, n = (1, x.shape[0]) if x.dim() == 1 else x.shape
    if out is None:
        out = torch.empty(q8_1_size(m, n), dtype=torch.uint8, device=x.device)
    rz_q8_1_quantize(x, out, m, n, stream)
    return out


def q4k_q8_gemv(w, q8, m, out_dim, in_dim, out=None, stream=None):
    import torch
    _cuda_contig(w, torch.uint8, "w")
    _cuda_contig(q8, torch.uint8, "q8")
    if out is None:
        out = torch.empty((m, out_dim), dtype=torch.float32, device=w.device)
    rz_q4k_q8_gemv(w, q8, out, m, out_dim, in_dim, stream)
    return out


def rz_q4k_q8_gemm(w, q8, y, ldy, m, out_dim, in_dim, ws, ws_bytes, stream=None):
    return call("rz_q4k_q8_gemm", _ptr(w), _ptr(q8), _ptr(y), ldy, m, out_dim, in_dim, _ptr(ws), ws_bytes,
                _stream(stream))


def q4k_q8_gemm_workspace_bytes(m: int, in_dim: int) -> int:
    return int(load().rz_q4k_q8_gemm_workspace_bytes(m, in_dim))


def q4k_q8_gemm(w, q8, m, out_dim, in_dim, out=None, ws=None, stream=None):
    """y = W x_t for m tokens on the tensor cores (any m >= 1); y f32 [m, out_dim]."""
    import torch
    _cuda_contig(w, torch.uint8, "w")
    _cuda_contig(q8, torch.uint8, "q8")
    if out is None:
        out = torch.empty((m, out_dim), dtype=torch.float32, device=w.device)
    need = q4k_q8_gemm_workspace_bytes(m, in_dim)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=w.device)
    rz_q4k_q8_gemm(w, q8, out, out.shape[-1], m, out_dim, in_dim, ws, ws.numel(), stream)
    return out


def q4k_q8_gemv_ex(w, q8, m, out_dim, in_dim, bias=None, residual=None, out=None, ld=0,
                   stream=None):
    """y = W x (+ bias | + residual); y f32 [m, ld or out_dim]."""
    import torch
    if out is None:
        out = torch.empty((m, ld or out_dim), dtype=torch.float32, device=w.device)
    rz_q4k_q8_gemv_ex(w, q8, bias, residual, out, ld, m, out_dim, in_dim, stream)
    return out


def rmsnorm_q4k_gemv(x, gamma, n, eps, ws, rows, in_dim, biases=None, out=None, stream=None):
    """RMSNorm -> Q8_1 -> GEMVs of 1..3 matrices; returns f32 [m, sum(rows)]."""
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    ldx = x.shape[-1]
    if out is None:
        out = torch.empty((m, sum(rows)), dtype=torch.float32, device=x.device)
    rz_rmsnorm_q4k_gemv(x, ldx, gamma, n, eps, ws, rows, biases, out, out.shape[-1], m, in_dim, stream)
    return out


def q4k_q8_subblock_dots(w, q8, out_dim, in_dim, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((out_dim, in_dim // 32), dtype=torch.int32, device=w.device)
    rz_q4k_q8_subblock_dots(w, q8, out, out_dim, in_dim, stream)
    return out


def q4_0_gemv(w, x, out_dim, in_dim, out=None, bias=None, stream=None):
    import torch
    _cuda_contig(w, torch.uint8, "w")
    _cuda_contig(x, torch.float32, "x")
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, out_dim), dtype=torch.float32, device=w.device)
    if bias is None:
        rz_q4_0_gemv(w, x, out, m, out_dim, in_dim, stream)
    else:
        call("rz_q4_0_gemv_bias", _ptr(w), _ptr(x), _ptr(bias), _ptr(out), m, out_dim, in_dim, _stream(stream))
    return out


def rmsnorm(x, gamma, n, n_pad, eps, want_y=True, want_q8=True, stream=None):
    """x: f32 [m, n_pad] -> (y f32 [m, n_pad] or None, q8 uint8 or None)."""
    import torch
    _cuda_contig(x, torch.float32, "x")
    m = 1 if x.dim() == 1 else x.shape[0]
    y = torch.empty((m, n_pad), dtype=torch.float32, device=x.device) if want_y else None
    q8 = torch.empty(q8_1_size(m, n_pad), dtype=torch.uint8, device=x.device) if want_q8 else None
    rz_rmsnorm(x, gamma, y, q8, m, n, n_pad, eps, stream)
    return y, q8


def residual_add(a, b, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty_like(a)
    rz_residual_add(a, b, out, a.numel(), stream)
    return out


def check_device_error(stream=None):
    return rz_check_device_error(stream)


def set_pdl(enable: bool):
    rz_set_pdl(enable)


def version() -> str:
    return load().rz_version().decode()


# ------------------------------------------------------------------ layer-level helpers
class DeviceLayer:
    """One Q4_K decode layer resident on the GPU (torch tensors) and its C descriptor.

    weights: dict with uint8 CUDA tensors wq, wk, wv, wo, wgate, wup, wdown and f32
    CUDA tensors attn_gamma, ffn_gamma; optional f32 CUDA tensors bq, bk, bv (QKV
    bias).  The fused Q|K|V layout leaves wk and wv out (or None) and holds the one
    [q_dim + 2 kv_dim][hidden_pad] matrix in wq.  Shapes follow include/rz.h."""

    def __init__(self, weights: dict, hidden: int, hidden_pad: int, n_heads: int,
                 n_kv_heads: int, head_dim: int, inter: int, eps: float, rope_theta: float,
                 rope_mode: int):
        from ._lib import LayerWeightsStruct
        self.t = weights
        self.hidden, self.hidden_pad, self.n_heads = hidden, hidden_pad, n_heads
        self.n_kv_heads, self.head_dim, self.inter = n_kv_heads, head_dim, inter
        self.eps, self.rope_theta, self.rope_mode = eps, rope_theta, rope_mode

        def p(k):
            t = weights.get(k)
            return None if t is None else t.data_ptr()

        self.struct = LayerWeightsStruct(
            *[p(k) for k in ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown", "attn_gamma", "ffn_gamma")],
            hidden, hidden_pad, n_heads, n_kv_heads, head_dim, inter, eps, rope_theta, rope_mode,
            p("bq"), p("bk"), p("bv"))

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim


class DeviceKV:
    """f32 K and V caches [m][max_seq][kv_dim] of one layer and their C descriptor."""

    def __init__(self, k, v):
        from ._lib import KvCacheStruct
        import torch
        assert k.dtype == torch.float32 and k.is_cuda and k.is_contiguous() and k.dim() == 3
        self.k, self.v = k, v
        m, max_seq, kv_dim = k.shape
        self.max_seq = max_seq
        self.struct = KvCacheStruct(k.data_ptr(), v.data_ptr(), max_seq * kv_dim, max_seq)


def workspace(nbytes: int, device):
    """Zero-filled device workspace (the attention counters start at zero)."""
    import torch
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def swiglu_ffn_workspace_bytes(m, hidden_pad, inter):
    return load().rz_swiglu_ffn_workspace_bytes(m, hidden_pad, inter)


def swiglu_ffn(x, gamma, w_gate, w_up, w_down, hidden, hidden_pad, inter, eps, out=None,
               ws=None, stream=None):
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, hidden_pad), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(swiglu_ffn_workspace_bytes(m, hidden_pad, inter), x.device)
    call("rz_swiglu_ffn", _ptr(x), _ptr(gamma), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(out),
         m, hidden, hidden_pad, inter, eps, _ptr(ws), ws.numel(), _stream(stream))
    return out


def rz_swiglu_ffn_static(x, gamma, w_gate, w_up, w_down, out, m, hidden, hidden_pad, inter, eps,
                         stream=None):
    """The SwiGLU FFN with the library's static scratch (no workspace argument)."""
    return call("rz_swiglu_ffn_static", _ptr(x), _ptr(gamma), _ptr(w_gate), _ptr(w_up),
                _ptr(w_down), _ptr(out), m, hidden, hidden_pad, inter, eps, _stream(stream))


def attention_workspace_bytes(m, n_heads, n_kv_heads, head_dim, max_seq):
    return load().rz_attention_workspace_bytes(m, n_heads, n_kv_heads, head_dim, max_seq)


def attention_decode(q, k, v, ld_qkv, kv: "DeviceKV", n_heads, n_kv_heads, head_dim,
                     rope_theta, rope_mode, position=0, positions=None, want_att=True,
                     want_q8=True, ws=None, stream=None):
    import ctypes as C
    import torch
    m = kv.k.shape[0]
    q_dim = n_heads * head_dim
    q_pad = (q_dim + 255) // 256 * 256
    att = torch.empty((m, q_dim), dtype=torch.float32, device=q.device) if want_att else None
    a8 = torch.empty(q8_1_size(m, q_pad), dtype=torch.uint8, device=q.device) if want_q8 else None
    if ws is None:
        ws = workspace(attention_workspace_bytes(m, n_heads, n_kv_heads, head_dim, kv.max_seq),
                       q.device)
    call("rz_attention_decode", _ptr(q), _ptr(k), _ptr(v), ld_qkv, C.byref(kv.struct),
         _ptr(positions), position, m, n_heads, n_kv_heads, head_dim, rope_theta, rope_mode,
         _ptr(att), _ptr(a8), _ptr(ws), ws.numel(), _stream(stream))
    return att, a8


def decode_layer_workspace_bytes(layer: "DeviceLayer", m, max_seq):
    import ctypes as C
    return load().rz_decode_layer_workspace_bytes(C.byref(layer.struct), m, max_seq)


def decode_layer(x, layer: "DeviceLayer", kv: "DeviceKV", position=0, positions=None, out=None,
                 ws=None, stream=None):
    import ctypes as C
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, layer.hidden_pad), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(decode_layer_workspace_bytes(layer, m, kv.max_seq), x.device)
    call("rz_decode_layer", _ptr(x), C.byref(layer.struct), C.byref(kv.struct), _ptr(positions),
         position, m, _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    return out


class DeviceStack:
    """Layers + per-layer KV caches + output norm + Q4_0 LM head, with the host
    descriptor arrays the C ABI takes."""

    def __init__(self, layers, kvs, out_gamma, lm_head, vocab, lm_bias=None):
        from ._lib import KvCacheStruct, LayerWeightsStruct
        self.layers, self.kvs = layers, kvs
        self.out_gamma, self.lm_head, self.vocab, self.lm_bias = out_gamma, lm_head, vocab, lm_bias
        n = len(layers)
        self.lw = (LayerWeightsStruct * n)(*[l.struct for l in layers])
        self.kv = (KvCacheStruct * n)(*[k.struct for k in kvs])

    def workspace_bytes(self, m):
        return load().rz_decode_stack_workspace_bytes(self.lw, len(self.layers), m,
                                                      self.kvs[0].max_seq)

    def launches(self, m, with_head=True):
        """librz kernels one rz_decode_stack (or rz_decode_layers) call launches."""
        return load().rz_decode_stack_launches(self.lw, len(self.layers), m, self.kvs[0].max_seq,
                                               1 if with_head else 0, self.vocab)


def rz_decode_stack(x, stack: "DeviceStack", positions, position, m, hidden_out, logits, ws,
                    stream=None):
    return call("rz_decode_stack", _ptr(x), stack.lw, stack.kv, len(stack.layers),
                _ptr(positions), position, m, _ptr(stack.out_gamma), _ptr(stack.lm_head),
                _ptr(stack.lm_bias), stack.vocab, _ptr(hidden_out), _ptr(logits), _ptr(ws), ws.numel(),
                _stream(stream))


def rz_decode_layers(x, stack: "DeviceStack", positions, position, m, out, ws, stream=None):
    return call("rz_decode_layers", _ptr(x), stack.lw, stack.kv, len(stack.layers), _ptr(positions),
                position, m, _ptr(out), _ptr(ws), ws.numel(), _stream(stream))


def decode_layers(x, stack: "DeviceStack", position=0, positions=None, ws=None, stream=None):
    """The stack's layers without the output norm and LM head; returns the hidden state."""
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    out = torch.empty((m, stack.layers[0].hidden_pad), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(stack.workspace_bytes(m), x.device)
    rz_decode_layers(x, stack, positions, position, m, out, ws, stream)
    return out


def decode_stack(x, stack: "DeviceStack", position=0, positions=None, ws=None, stream=None,
                 want_hidden=True):
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    hp = stack.layers[0].hidden_pad
    hid = torch.empty((m, hp), dtype=torch.float32, device=x.device) if want_hidden else None
    logits = torch.empty((m, stack.vocab), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(stack.workspace_bytes(m), x.device)
    rz_decode_stack(x, stack, positions, position, m, hid, logits, ws, stream)
    return hid, logits


# ------------------------------------------------------------------ Q4_0 whole-model layer
class DeviceLayerQ40:
    """One Q4_0 layer on the GPU: uint8 CUDA tensors wqkv, wo, wup, wdown (and wgate
    for SwiGLU, absent for the GELU FFN), f32 attn_gamma, ffn_gamma."""

    def __init__(self, weights: dict, hidden: int, n_heads: int, n_kv_heads: int, head_dim: int, inter: int,
                 eps: float, rope_theta: float, rope_mode: int):
        from ._lib import LayerWeightsQ40Struct
        self.t = weights
        self.hidden, self.n_heads, self.n_kv_heads, self.head_dim, self.inter = hidden, n_heads, n_kv_heads, head_dim, inter

        def p(k):
            t = weights.get(k)
            return None if t is None else t.data_ptr()

        self.struct = LayerWeightsQ40Struct(
            *[p(k) for k in ("wqkv", "wo", "wgate", "wup", "wdown", "attn_gamma", "ffn_gamma")],
            hidden, n_heads, n_kv_heads, head_dim, inter, eps, rope_theta, rope_mode)


def decode_layer_q4_0(x, layer: DeviceLayerQ40, kv: "DeviceKV", position=0, positions=None, out=None, ws=None,
                      stream=None):
    import ctypes as C
    import torch
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, layer.hidden), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(load().rz_decode_layer_q4_0_workspace_bytes(C.byref(layer.struct), m, kv.max_seq), x.device)
    call("rz_decode_layer_q4_0", _ptr(x), C.byref(layer.struct), C.byref(kv.struct), _ptr(positions), position, m,
         _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    return out
