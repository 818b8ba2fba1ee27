"""numpy front end of the C oracle (test infrastructure only).

Array conventions (all C-contiguous):
  Q4_K weights  uint8 [out_dim, in_dim/256*144]
  Q4_0 weights  uint8 [out_dim, in_dim/32*18]
  Q8_1 buffer   uint8 [q8_1_size(m, n)]: int8 q[m][n] | f32 d[m][n/32] | f32 s[m][n/32]
  activations   float32 [m, n]
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import build as _build

__all__ = [
    "lib", "use_all_cores", "threads", "f32_to_f16", "f16_to_f64",
    "q4k_unpack", "q4k_pack", "q4k_dequantize",
    "q4_0_unpack", "q4_0_pack", "q4_0_dequantize",
    "q8_1_quantize", "q8_1_dequantize", "q8_1_fields", "q8_1_size",
    "q4k_q8_subblock_dots", "q4k_q8_gemv", "q4k_f32_gemv", "q4_0_gemv",
    "rmsnorm", "residual_add", "silu", "rope", "attention",
    "LayerWeights", "swiglu_ffn", "decode_layer", "decode_stack",
    "gelu", "LayerWeightsQ40", "decode_layer_q4_0",
    "Q4K_BYTES", "Q4_0_BYTES",
]

Q4K_BYTES = 144
Q4_0_BYTES = 18

_libs = {}
_use_omp = False


def lib():
    """The oracle library: single-threaded, unless use_all_cores(True) was called."""
    key = "omp" if _use_omp else "st"
    if key not in _libs:
        L = C.CDLL(_build.build(openmp=_use_omp))
        _declare(L)
        _libs[key] = L
    return _libs[key]


def use_all_cores(enable: bool) -> int:
    """Switch every following call to the all-core build (OpenMP over output rows
    and attention heads; identical results) or back; returns its thread count."""
    global _use_omp
    _use_omp = bool(enable)
    return threads()


def threads() -> int:
    return int(lib().orc_threads())


_u8p = C.POINTER(C.c_uint8)
_u16p = C.POINTER(C.c_uint16)
_i32p = C.POINTER(C.c_int32)
_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_i64 = C.c_int64


class _OrcLayer(C.Structure):
    _fields_ = [
        ("wq", _u8p), ("wk", _u8p), ("wv", _u8p), ("wo", _u8p),
        ("wgate", _u8p), ("wup", _u8p), ("wdown", _u8p),
        ("attn_gamma", _f32p), ("ffn_gamma", _f32p),
        ("hidden", _i64), ("hidden_pad", _i64), ("n_heads", _i64),
        ("n_kv_heads", _i64), ("head_dim", _i64), ("inter", _i64),
        ("eps", C.c_float), ("rope_theta", C.c_double), ("rope_mode", C.c_int),
        ("bq", _f32p), ("bk", _f32p), ("bv", _f32p),
    ]


class _OrcLayerQ40(C.Structure):
    _fields_ = [
        ("wqkv", _u8p), ("wo", _u8p), ("wgate", _u8p), ("wup", _u8p), ("wdown", _u8p),
        ("attn_gamma", _f32p), ("ffn_gamma", _f32p),
        ("hidden", _i64), ("n_heads", _i64), ("n_kv_heads", _i64), ("head_dim", _i64), ("inter", _i64),
        ("eps", C.c_float), ("rope_theta", C.c_double), ("rope_mode", C.c_int),
    ]


def _declare(L):
    sig = {
        "orc_threads": (C.c_int, []),
        "orc_f32_to_f16": (C.c_uint16, [C.c_float]),
        "orc_f16_to_f64": (C.c_double, [C.c_uint16]),
        "orc_f32_to_f16_array": (None, [_f32p, _u16p, _i64]),
        "orc_f16_to_f32_array": (None, [_u16p, _f32p, _i64]),
        "orc_q4k_unpack": (None, [_u8p, _u16p, _u16p, _u8p, _u8p, _u8p]),
        "orc_q4k_pack": (None, [C.c_uint16, C.c_uint16, _u8p, _u8p, _u8p, _u8p]),
        "orc_q4k_dequantize": (None, [_u8p, _i64, _f64p]),
        "orc_q4_0_unpack": (None, [_u8p, _u16p, _u8p]),
        "orc_q4_0_pack": (None, [C.c_uint16, _u8p, _u8p]),
        "orc_q4_0_dequantize": (None, [_u8p, _i64, _f64p]),
        "orc_q8_1_quantize": (None, [_f32p, _u8p, _i64, _i64]),
        "orc_q8_1_dequantize": (None, [_u8p, _f64p, _i64, _i64]),
        "orc_q4k_q8_subblock_dots": (None, [_u8p, _u8p, _i32p, _i64, _i64]),
        "orc_q4k_q8_gemv": (None, [_u8p, _u8p, _f32p, _i64, _i64, _i64]),
        "orc_q4_0_gemv": (None, [_u8p, _f32p, _f32p, _i64, _i64, _i64]),
        "orc_q4k_f32_gemv": (None, [_u8p, _f32p, _f32p, _i64, _i64, _i64]),
        "orc_rmsnorm": (None, [_f32p, _f32p, _f32p, _i64, _i64, _i64, C.c_float]),
        "orc_residual_add": (None, [_f32p, _f32p, _f32p, _i64]),
        "orc_silu": (C.c_double, [C.c_double]),
        "orc_rope": (None, [_f32p, _i64, _i64, _i64, C.c_double, C.c_int]),
        "orc_attention": (None, [_f32p, _f32p, _f32p, _i64, _i64, _i64, _i64, _f32p]),
        "orc_swiglu_ffn": (None, [_f32p, _f32p, _u8p, _u8p, _u8p, _f32p,
                                  _i64, _i64, _i64, C.c_float]),
        "orc_decode_layer": (None, [_f32p, C.POINTER(_OrcLayer), _f32p, _f32p, _i64, _f32p]),
        "orc_gelu": (C.c_double, [C.c_double]),
        "orc_decode_layer_q4_0": (None, [_f32p, C.POINTER(_OrcLayerQ40), _f32p, _f32p, _i64, _f32p]),
        "orc_decode_stack": (None, [_f32p, C.POINTER(_OrcLayer), _i64,
                                    C.POINTER(_f32p), C.POINTER(_f32p), _i64,
                                    _f32p, _u8p, _f32p, _i64, _i64, _i64, C.c_float,
                                    _f32p, _f32p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _p(a: np.ndarray, ct):
    assert a.flags.c_contiguous, "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ct))


def _u8(a):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ---------------------------------------------------------------- fp16
def f32_to_f16(x) -> np.ndarray:
    """float32 array -> uint16 binary16 bits (round to nearest even)."""
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16_array(_p(x, C.c_float), _p(out, C.c_uint16), x.size)
    return out


def f16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    L = lib()
    return np.array([L.orc_f16_to_f64(int(v)) for v in h.ravel()],
                    dtype=np.float64).reshape(h.shape)


# ---------------------------------------------------------------- Q4_K
def q4k_unpack(blk):
    """144-byte super-block -> (d_bits, dmin_bits, sc[8], m[8], q[256])."""
    blk = _u8(blk)
    assert blk.size == Q4K_BYTES
    d = C.c_uint16()
    dm = C.c_uint16()
    sc = np.zeros(8, np.uint8)
    mn = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    lib().orc_q4k_unpack(_p(blk, C.c_uint8), C.byref(d), C.byref(dm),
                         _p(sc, C.c_uint8), _p(mn, C.c_uint8), _p(q, C.c_uint8))
    return int(d.value), int(dm.value), sc, mn, q


def q4k_pack(d_bits, dmin_bits, sc, mn, q) -> np.ndarray:
    sc = _u8(sc)
    mn = _u8(mn)
    q = _u8(q)
    out = np.zeros(Q4K_BYTES, np.uint8)
    lib().orc_q4k_pack(int(d_bits), int(dmin_bits), _p(sc, C.c_uint8), _p(mn, C.c_uint8),
                       _p(q, C.c_uint8), _p(out, C.c_uint8))
    return out


def q4k_dequantize(w) -> np.ndarray:
    """Q4_K bytes [..., nsb*144] -> float64 [..., nsb*256]."""
    w = _u8(w)
    nblk = w.size // Q4K_BYTES
    out = np.empty(nblk * 256, np.float64)
    lib().orc_q4k_dequantize(_p(w, C.c_uint8), nblk, _p(out, C.c_double))
    return out.reshape(w.shape[:-1] + (w.shape[-1] // Q4K_BYTES * 256,))


# ---------------------------------------------------------------- Q4_0
def q4_0_unpack(blk):
    blk = _u8(blk)
    d = C.c_uint16()
    q = np.zeros(32, np.uint8)
    lib().orc_q4_0_unpack(_p(blk, C.c_uint8), C.byref(d), _p(q, C.c_uint8))
    return int(d.value), q


def q4_0_pack(d_bits, q) -> np.ndarray:
    q = _u8(q)
    out = np.zeros(Q4_0_BYTES, np.uint8)
    lib().orc_q4_0_pack(int(d_bits), _p(q, C.c_uint8), _p(out, C.c_uint8))
    return out


def q4_0_dequantize(w) -> np.ndarray:
    w = _u8(w)
    nblk = w.size // Q4_0_BYTES
    out = np.empty(nblk * 32, np.float64)
    lib().orc_q4_0_dequantize(_p(w, C.c_uint8), nblk, _p(out, C.c_double))
    return out.reshape(w.shape[:-1] + (w.shape[-1] // Q4_0_BYTES * 32,))


# ---------------------------------------------------------------- Q8_1
def q8_1_size(m: int, n: int) -> int:
    return m * n + 8 * m * (n // 32)


def q8_1_quantize(x) -> np.ndarray:
    """float32 [m, n] (n % 32 == 0) -> uint8 [q8_1_size(m, n)]."""
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    m, n = x.shape
    assert n % 32 == 0
    out = np.empty(q8_1_size(m, n), np.uint8)
    lib().orc_q8_1_quantize(_p(x, C.c_float), _p(out, C.c_uint8), m, n)
    return out


def q8_1_dequantize(q8, m, n) -> np.ndarray:
    q8 = _u8(q8)
    assert q8.size == q8_1_size(m, n)
    out = np.empty((m, n), np.float64)
    lib().orc_q8_1_dequantize(_p(q8, C.c_uint8), _p(out, C.c_double), m, n)
    return out


def q8_1_fields(q8, m, n):
    """Split a Q8_1 buffer into (d f32 [m, n/32], s f32 [m, n/32], q int8 [m, n/32, 32])."""
    q8 = _u8(q8).ravel()
    assert q8.size == q8_1_size(m, n)
    nb = n // 32
    q = q8[:m * n].view(np.int8).reshape(m, nb, 32)
    d = q8[m * n:m * n + 4 * m * nb].view(np.float32).reshape(m, nb)
    s = q8[m * n + 4 * m * nb:].view(np.float32).reshape(m, nb)
    return d, s, q


# ---------------------------------------------------------------- GEMVs
def q4k_q8_subblock_dots(w, x8, out_dim, in_dim) -> np.ndarray:
    w = _u8(w)
    x8 = _u8(x8)
    I = np.empty((out_dim, in_dim // 32), np.int32)
    lib().orc_q4k_q8_subblock_dots(_p(w, C.c_uint8), _p(x8, C.c_uint8), _p(I, C.c_int32),
                                   out_dim, in_dim)
    return I


def q4k_q8_gemv(w, x8, m, out_dim, in_dim) -> np.ndarray:
    w = _u8(w)
    x8 = _u8(x8)
    assert w.size == out_dim * (in_dim // 256) * Q4K_BYTES
    assert x8.size == q8_1_size(m, in_dim)
    y = np.empty((m, out_dim), np.float32)
    lib().orc_q4k_q8_gemv(_p(w, C.c_uint8), _p(x8, C.c_uint8), _p(y, C.c_float),
                          m, out_dim, in_dim)
    return y


def q4k_f32_gemv(w, x, out_dim, in_dim) -> np.ndarray:
    """Q4_K weights times f32 activations [m, in_dim] (no Q8_1) -> float32 [m, out_dim]."""
    w = _u8(w)
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    m = x.shape[0]
    assert x.shape[1] == in_dim and w.size == out_dim * (in_dim // 256) * Q4K_BYTES
    y = np.empty((m, out_dim), np.float32)
    lib().orc_q4k_f32_gemv(_p(w, C.c_uint8), _p(x, C.c_float), _p(y, C.c_float), m, out_dim, in_dim)
    return y


def q4_0_gemv(w, x, out_dim, in_dim) -> np.ndarray:
    w = _u8(w)
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    m = x.shape[0]
    assert x.shape[1] == in_dim
    assert w.size == out_dim * (in_dim // 32) * Q4_0_BYTES
    y = np.empty((m, out_dim), np.float32)
    lib().orc_q4_0_gemv(_p(w, C.c_uint8), _p(x, C.c_float), _p(y, C.c_float),
                        m, out_dim, in_dim)
    return y


# ---------------------------------------------------------------- elementwise
def rmsnorm(x, gamma, n, n_pad, eps) -> np.ndarray:
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    m = x.shape[0]
    assert x.shape[1] == n_pad
    g = _f32(gamma)
    y = np.empty((m, n_pad), np.float32)
    lib().orc_rmsnorm(_p(x, C.c_float), _p(g, C.c_float), _p(y, C.c_float), m, n, n_pad, eps)
    return y


def residual_add(a, b) -> np.ndarray:
    a = _f32(a)
    b = _f32(b)
    out = np.empty_like(a)
    lib().orc_residual_add(_p(a, C.c_float), _p(b, C.c_float), _p(out, C.c_float), a.size)
    return out


def silu(x: float) -> float:
    return lib().orc_silu(float(x))


def rope(v, n_heads, head_dim, pos, theta, mode) -> np.ndarray:
    v = _f32(v).copy()
    lib().orc_rope(_p(v, C.c_float), n_heads, head_dim, pos, theta, mode)
    return v


def attention(q, kc, vc, pos, n_heads, n_kv_heads, head_dim) -> np.ndarray:
    q = _f32(q)
    kc = _f32(kc)
    vc = _f32(vc)
    out = np.empty(n_heads * head_dim, np.float32)
    lib().orc_attention(_p(q, C.c_float), _p(kc, C.c_float), _p(vc, C.c_float), pos,
                        n_heads, n_kv_heads, head_dim, _p(out, C.c_float))
    return out


# ---------------------------------------------------------------- layer / stack
@dataclass
class LayerWeights:
    """Host copy of one layer (numpy).  Q4_K weights as uint8 row-major blocks."""
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    wgate: np.ndarray
    wup: np.ndarray
    wdown: np.ndarray
    attn_gamma: np.ndarray
    ffn_gamma: np.ndarray
    hidden: int
    hidden_pad: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int
    eps: float
    rope_theta: float
    rope_mode: int
    bq: np.ndarray = None
    bk: np.ndarray = None
    bv: np.ndarray = None

    def _struct(self):
        keep = {k: np.ascontiguousarray(getattr(self, k)) for k in
                ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")}
        keep["attn_gamma"] = _f32(self.attn_gamma)
        keep["ffn_gamma"] = _f32(self.ffn_gamma)
        for b in ("bq", "bk", "bv"):
            if getattr(self, b) is not None:
                keep[b] = _f32(getattr(self, b))
        s = _OrcLayer(
            wq=_p(keep["wq"], C.c_uint8), wk=_p(keep["wk"], C.c_uint8),
            wv=_p(keep["wv"], C.c_uint8), wo=_p(keep["wo"], C.c_uint8),
            wgate=_p(keep["wgate"], C.c_uint8), wup=_p(keep["wup"], C.c_uint8),
            wdown=_p(keep["wdown"], C.c_uint8),
            attn_gamma=_p(keep["attn_gamma"], C.c_float),
            ffn_gamma=_p(keep["ffn_gamma"], C.c_float),
            hidden=self.hidden, hidden_pad=self.hidden_pad, n_heads=self.n_heads,
            n_kv_heads=self.n_kv_heads, head_dim=self.head_dim, inter=self.inter,
            eps=self.eps, rope_theta=self.rope_theta, rope_mode=self.rope_mode,
            bq=_p(keep["bq"], C.c_float) if "bq" in keep else None,
            bk=_p(keep["bk"], C.c_float) if "bk" in keep else None,
            bv=_p(keep["bv"], C.c_float) if "bv" in keep else None)
        return s, keep


def swiglu_ffn(x, gamma, wgate, wup, wdown, hidden, hidden_pad, inter, eps) -> np.ndarray:
    x = _f32(x)
    g = _f32(gamma)
    out = np.empty(hidden_pad, np.float32)
    wg, wu, wd = _u8(wgate), _u8(wup), _u8(wdown)
    lib().orc_swiglu_ffn(_p(x, C.c_float), _p(g, C.c_float), _p(wg, C.c_uint8),
                         _p(wu, C.c_uint8), _p(wd, C.c_uint8), _p(out, C.c_float),
                         hidden, hidden_pad, inter, eps)
    return out


def decode_layer(x, lw: LayerWeights, kc: np.ndarray, vc: np.ndarray, pos: int) -> np.ndarray:
    """One token through one layer.  kc, vc (float32 [max_seq, kv_dim]) are
    updated in place at row pos."""
    assert kc.dtype == np.float32 and kc.flags.c_contiguous
    assert vc.dtype == np.float32 and vc.flags.c_contiguous
    x = _f32(x)
    s, keep = lw._struct()
    out = np.empty(lw.hidden_pad, np.float32)
    lib().orc_decode_layer(_p(x, C.c_float), C.byref(s), _p(kc, C.c_float),
                           _p(vc, C.c_float), pos, _p(out, C.c_float))
    del keep
    return out


def decode_stack(x, layers, kcs, vcs, pos, out_gamma, lm_head, vocab,
                 hidden=None, hidden_pad=None, eps=None, lm_bias=None):
    """Layers, output RMSNorm and the Q4_0 LM head; returns (hidden, logits)."""
    x = _f32(x)
    n = len(layers)
    hidden = layers[0].hidden if hidden is None else hidden
    hp = layers[0].hidden_pad if hidden_pad is None else hidden_pad
    eps = layers[0].eps if eps is None else eps
    structs = (_OrcLayer * max(n, 1))()
    keeps = []
    for i, lw in enumerate(layers):
        s, keep = lw._struct()
        structs[i] = s
        keeps.append(keep)
    kp = (_f32p * max(n, 1))(*[_p(k, C.c_float) for k in kcs])
    vp = (_f32p * max(n, 1))(*[_p(v, C.c_float) for v in vcs])
    og = _f32(out_gamma)
    lm = _u8(lm_head)
    hid = np.empty(hp, np.float32)
    logits = np.empty(vocab, np.float32)
    lb = None if lm_bias is None else _f32(lm_bias)
    lib().orc_decode_stack(_p(x, C.c_float), structs, n, kp, vp, pos, _p(og, C.c_float),
                           _p(lm, C.c_uint8), None if lb is None else _p(lb, C.c_float), vocab, hidden, hp, eps,
                           _p(hid, C.c_float), _p(logits, C.c_float))
    del keeps
    return hid, logits


# ---------------------------------------------------------------- Q4_0 whole-model layer
def gelu(x: float) -> float:
    return lib().orc_gelu(float(x))


@dataclass
class LayerWeightsQ40:
    """Host copy of one Q4_0 layer: fused QKV [q + 2 kv][hidden], O, optional gate,
    up, down (uint8 Q4_0 blocks); gammas f32 [hidden]."""
    wqkv: np.ndarray
    wo: np.ndarray
    wgate: np.ndarray   # or None: the GELU FFN
    wup: np.ndarray
    wdown: np.ndarray
    attn_gamma: np.ndarray
    ffn_gamma: np.ndarray
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int
    eps: float
    rope_theta: float
    rope_mode: int

    def _struct(self):
        keep = {k: _u8(getattr(self, k)) for k in ("wqkv", "wo", "wup", "wdown")}
        if self.wgate is not None:
            keep["wgate"] = _u8(self.wgate)
        keep["attn_gamma"] = _f32(self.attn_gamma)
        keep["ffn_gamma"] = _f32(self.ffn_gamma)
        s = _OrcLayerQ40(
            wqkv=_p(keep["wqkv"], C.c_uint8), wo=_p(keep["wo"], C.c_uint8),
            wgate=_p(keep["wgate"], C.c_uint8) if "wgate" in keep else None,
            wup=_p(keep["wup"], C.c_uint8), wdown=_p(keep["wdown"], C.c_uint8),
            attn_gamma=_p(keep["attn_gamma"], C.c_float), ffn_gamma=_p(keep["ffn_gamma"], C.c_float),
            hidden=self.hidden, n_heads=self.n_heads, n_kv_heads=self.n_kv_heads,
            head_dim=self.head_dim, inter=self.inter, eps=self.eps, rope_theta=self.rope_theta,
            rope_mode=self.rope_mode)
        return s, keep


def decode_layer_q4_0(x, lw: LayerWeightsQ40, kc: np.ndarray, vc: np.ndarray, pos: int) -> np.ndarray:
    """One token through one Q4_0 layer; kc, vc (float32 [max_seq, kv_dim]) updated at row pos."""
    assert kc.dtype == np.float32 and kc.flags.c_contiguous
    assert vc.dtype == np.float32 and vc.flags.c_contiguous
    x = _f32(x)
    s, keep = lw._struct()
    out = np.empty(lw.hidden, np.float32)
    lib().orc_decode_layer_q4_0(_p(x, C.c_float), C.byref(s), _p(kc, C.c_float), _p(vc, C.c_float), pos,
                                _p(out, C.c_float))
    del keep
    return out
