"""torch-facing helpers over the librz C ABI (marshalling and output allocation only)."""
from __future__ import annotations

import ctypes as C

from ._lib import call, load, status

__all__ = [
    "q8_1_size", "q4k_bytes", "q4_0_bytes",
    "rz_q8_1_quantize", "rz_q4k_q8_gemv", "rz_q4k_q8_subblock_dots", "rz_q4_0_gemv",
    "rz_rmsnorm", "rz_residual_add", "rz_check_device_error", "rz_set_pdl",
    "q8_1_quantize", "q4k_q8_gemv", "q4k_q8_subblock_dots", "q4_0_gemv",
    "rmsnorm", "residual_add", "check_device_error", "set_pdl", "version",
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


def q4k_q8_subblock_dots(w, q8, out_dim, in_dim, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((out_dim, in_dim // 32), dtype=torch.int32, device=w.device)
    rz_q4k_q8_subblock_dots(w, q8, out, out_dim, in_dim, stream)
    return out


def q4_0_gemv(w, x, out_dim, in_dim, out=None, stream=None):
    import torch
    _cuda_contig(w, torch.uint8, "w")
    _cuda_contig(x, torch.float32, "x")
    m = 1 if x.dim() == 1 else x.shape[0]
    if out is None:
        out = torch.empty((m, out_dim), dtype=torch.float32, device=w.device)
    rz_q4_0_gemv(w, x, out, m, out_dim, in_dim, stream)
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
