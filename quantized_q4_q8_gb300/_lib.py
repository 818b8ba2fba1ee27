"""ctypes binding of librz (argument marshalling only).

Every function here forwards to the C entry point of the same name in
include/rz.h.  Tensors are passed as raw device pointers (``tensor.data_ptr()``)
and the stream as ``torch.cuda.current_stream().cuda_stream`` unless given.
All computation happens in the CUDA kernels of librz; there is no fallback: if
the shared library is missing or fails to load, importing raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librz.so")

RZ_OK = 0
STATUS_NAMES = {
    0: "RZ_OK", 1: "RZ_ERR_INVALID_ARG", 2: "RZ_ERR_SHAPE", 3: "RZ_ERR_ALIGN",
    4: "RZ_ERR_CUDA", 5: "RZ_ERR_TIMEOUT", 6: "RZ_ERR_UNSUPPORTED", 7: "RZ_ERR_DEVICE",
}


class RzError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_vp = C.c_void_p
_i64 = C.c_int64
_i32 = C.c_int32
_f32 = C.c_float
_sz = C.c_size_t


class LayerWeightsStruct(C.Structure):
    """rz_layer_weights (device pointers and dims)."""
    _fields_ = [
        ("wq", _vp), ("wk", _vp), ("wv", _vp), ("wo", _vp),
        ("wgate", _vp), ("wup", _vp), ("wdown", _vp),
        ("attn_gamma", _vp), ("ffn_gamma", _vp),
        ("hidden", _i32), ("hidden_pad", _i32), ("n_heads", _i32), ("n_kv_heads", _i32),
        ("head_dim", _i32), ("inter", _i32),
        ("eps", _f32), ("rope_theta", _f32), ("rope_mode", _i32),
        ("bq", _vp), ("bk", _vp), ("bv", _vp),
    ]


class KvCacheStruct(C.Structure):
    """rz_kv_cache."""
    _fields_ = [("k", _vp), ("v", _vp), ("seq_stride", _i64), ("max_seq", _i32)]


class LayerWeightsQ40Struct(C.Structure):
    """rz_layer_weights_q4_0 (device pointers and dims)."""
    _fields_ = [
        ("wqkv", _vp), ("wo", _vp), ("wgate", _vp), ("wup", _vp), ("wdown", _vp),
        ("attn_gamma", _vp), ("ffn_gamma", _vp),
        ("hidden", _i32), ("n_heads", _i32), ("n_kv_heads", _i32), ("head_dim", _i32), ("inter", _i32),
        ("eps", _f32), ("rope_theta", _f32), ("rope_mode", _i32),
    ]


_LWP = C.POINTER(LayerWeightsStruct)
_LQP = C.POINTER(LayerWeightsQ40Struct)
_KVP = C.POINTER(KvCacheStruct)

# name -> argtypes (restype is rz_status = int unless listed in _RESTYPES)
SIGNATURES = {
    "rz_q8_1_quantize": [_vp, _vp, _i64, _i64, _vp],
    "rz_q4k_q8_gemv": [_vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "rz_q4k_q8_subblock_dots": [_vp, _vp, _vp, _i64, _i64, _vp],
    "rz_q4k_q8_gemv_ex": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp],
    "rz_q4k_q8_gemm_workspace_bytes": [_i64, _i64],
    "rz_q4k_q8_gemm": [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp],
    "rz_q4k_q8_gemv_multi": [_vp, _i32, C.POINTER(_vp), C.POINTER(_i64), C.POINTER(_vp), _vp, _i64, _i64,
                             _i64, _vp],
    "rz_rmsnorm_q4k_gemv": [_vp, _i64, _vp, _i64, _f32, _i32, C.POINTER(_vp), C.POINTER(_i64),
                            C.POINTER(_vp), _vp, _i64, _i64, _i64, _vp],
    "rz_q4_0_gemv": [_vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "rz_q4k_f32_gemv": [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "rz_rmsnorm": [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _vp],
    "rz_residual_add": [_vp, _vp, _vp, _i64, _vp],
    "rz_swiglu_ffn_workspace_bytes": [_i64, _i64, _i64],
    "rz_swiglu_ffn": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _vp, _sz, _vp],
    "rz_swiglu_ffn_static": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _vp],
    "rz_attention_workspace_bytes": [_i64, _i32, _i32, _i32, _i32],
    "rz_attention_decode": [_vp, _vp, _vp, _i64, _KVP, _vp, _i32, _i64, _i32, _i32, _i32, _f32,
                            _i32, _vp, _vp, _vp, _sz, _vp],
    "rz_decode_layer_workspace_bytes": [_LWP, _i64, _i32],
    "rz_decode_layer": [_vp, _LWP, _KVP, _vp, _i32, _i64, _vp, _vp, _sz, _vp],
    "rz_decode_stack_workspace_bytes": [_LWP, _i32, _i64, _i32],
    "rz_decode_stack": [_vp, _LWP, _KVP, _i32, _vp, _i32, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _vp,
                        _sz, _vp],
    "rz_q4_0_gemv_bias": [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "rz_decode_layer_q4_0_workspace_bytes": [_LQP, _i64, _i32],
    "rz_decode_layer_q4_0": [_vp, _LQP, _KVP, _vp, _i32, _i64, _vp, _vp, _sz, _vp],
    "rz_decode_layers": [_vp, _LWP, _KVP, _i32, _vp, _i32, _i64, _vp, _vp, _sz, _vp],
    "rz_decode_stack_launches": [_LWP, _i32, _i64, _i32, _i32, _i64],
    "rz_check_device_error": [_vp, C.POINTER(C.c_uint32)],
    "rz_set_pdl": [C.c_int],
    "rz_debug_stall_next_gemv": [C.c_uint32],
    "rz_last_error": [],
    "rz_version": [],
}
_RESTYPES = {"rz_last_error": C.c_char_p, "rz_version": C.c_char_p,
             "rz_swiglu_ffn_workspace_bytes": _sz, "rz_attention_workspace_bytes": _sz,
             "rz_decode_layer_workspace_bytes": _sz, "rz_decode_stack_workspace_bytes": _sz,
             "rz_decode_layer_q4_0_workspace_bytes": _sz, "rz_q4k_q8_gemm_workspace_bytes": _sz,
             "rz_decode_stack_launches": C.c_int32}

_lib = None


def load(path: str = LIB_PATH):
    """Load librz.so; raises if it is missing (build it with the package build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"librz is not built ({path} missing): run __graft_entry__.build() "
                          "or python quantized_q4_q8_gb300/build.py")
    lib = C.CDLL(path)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPES.get(name, C.c_int)
    _lib = lib
    return lib


def call(name: str, *args):
    """Call a status-returning entry point; raise RzError on failure."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != RZ_OK:
        raise RzError(name, st, lib.rz_last_error().decode())
    return st


def status(name: str, *args) -> int:
    """Call an entry point and return its raw status (no raise)."""
    return getattr(load(), name)(*args)


def last_error() -> str:
    return load().rz_last_error().decode()
