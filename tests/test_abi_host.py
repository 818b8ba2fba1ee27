"""Host-side checks of the C ABI (no GPU needed).

librz builds here (nvcc cross-compiles for sm_103a), loads without a GPU, and
exports every entry point include/rz.h declares.  Calls that need no launch
(argument validation, version) are exercised too: a rejected call must return
its error status before touching the device.
"""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(rz_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    import quantized_q4_q8_gb300 as rz
    path = rz.build()
    return C.CDLL(path), path


def test_header_declares_the_path(lib):
    names = _declared_symbols()
    for required in ("rz_q8_1_quantize", "rz_q4k_q8_gemv", "rz_q4_0_gemv", "rz_rmsnorm",
                     "rz_residual_add"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    L, path = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(rz_[a-z0-9_]+)$", out, flags=re.M))
    missing = _declared_symbols() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"
    for name in _declared_symbols():
        getattr(L, name)


def test_binding_signatures_cover_header(lib):
    from quantized_q4_q8_gb300 import _lib
    assert _declared_symbols() <= set(_lib.SIGNATURES), \
        sorted(_declared_symbols() - set(_lib.SIGNATURES))


def test_version_and_no_error(lib):
    from quantized_q4_q8_gb300 import _lib
    L = _lib.load()
    assert b"sm_103a" in L.rz_version()
    assert L.rz_last_error() == b""


@pytest.mark.parametrize("call,args,status", [
    ("rz_q8_1_quantize", (0, 16, 1, 32, None), 1),            # null x
    ("rz_q8_1_quantize", (16, 16, 1, 33, None), 2),           # n % 32
    ("rz_q8_1_quantize", (16, 17, 1, 32, None), 3),           # misaligned q8
    ("rz_q4k_q8_gemv", (16, 16, 16, 17, 4, 256, None), 2),    # m > 16
    ("rz_q4k_q8_gemv", (16, 16, 16, 1, 4, 300, None), 2),     # in_dim % 256
    ("rz_q4k_q8_gemv", (16, 16, 16, 0, 4, 256, None), 1),     # m = 0
    ("rz_q4k_q8_gemv", (24, 16, 16, 1, 4, 256, None), 3),     # misaligned w
    ("rz_q4_0_gemv", (16, 16, 16, 1, 4, 48, None), 2),        # in_dim % 32
    ("rz_rmsnorm", (16, 16, 0, 0, 1, 8, 8, 1e-6, None), 1),   # no output
    ("rz_rmsnorm", (16, 16, 16, 16, 1, 8, 40, 1e-6, None), 2),  # n_pad % 32 with q8
    ("rz_rmsnorm", (16, 16, 16, 0, 1, 9, 8, 1e-6, None), 1),  # n_pad < n
    ("rz_residual_add", (16, 16, 16, 0, None), 1),            # n = 0
])
def test_argument_checks_fail_before_launch(lib, call, args, status):
    """Rejected calls return their status and a message without any device work
    (these pointers are not device memory and there is no GPU here)."""
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    st = _lib.status(call, *args)
    assert st == status, (st, _lib.last_error())
    assert _lib.last_error()


@pytest.mark.parametrize("call,args,status", [
    ("rz_q4k_q8_subblock_dots", (16, 16, 16, 1, 300, None), 2),           # in_dim % 256
    ("rz_q4k_q8_subblock_dots", (16, 16, 0, 1, 256, None), 1),            # null output
    ("rz_q4k_q8_subblock_dots", (16, 16, 20, 1, 256, None), 3),           # misaligned output
    ("rz_q4k_q8_gemv_ex", (16, 16, 16, 16, 16, 0, 1, 4, 256, None), 6),   # bias and residual
    ("rz_q4k_q8_gemv_ex", (16, 16, None, None, 16, 3, 1, 4, 256, None), 2),   # ld < out_dim
    ("rz_q4k_q8_gemv_ex", (16, 16, 18, None, 16, 0, 1, 4, 256, None), 3),     # bias not 4-byte aligned
    ("rz_q4k_q8_gemv_ex", (16, 16, None, 24, 16, 0, 1, 4, 256, None), 3),     # residual misaligned
    ("rz_q4k_q8_gemm", (16, 16, 16, 0, 1, 4, 300, 16, 1 << 20, None), 2),     # in_dim % 256
    ("rz_q4k_q8_gemm", (16, 16, 16, 3, 1, 4, 256, 16, 1 << 20, None), 2),     # ldy < out_dim
    ("rz_q4k_q8_gemm", (16, 16, 16, 0, 1, 4, 256, None, 1 << 20, None), 1),   # no workspace
    ("rz_q4k_q8_gemm", (16, 16, 16, 0, 1, 4, 256, 16, 16, None), 1),          # workspace too small
    ("rz_q4k_q8_gemm", (16, 16, 18, 0, 1, 4, 256, 16, 1 << 20, None), 3),     # y not 4-byte aligned
    ("rz_q4k_f32_gemv", (16, 16, None, 16, 17, 4, 256, None), 2),         # m > 16
    ("rz_q4k_f32_gemv", (16, 16, None, 16, 1, 4, 300, None), 2),          # in_dim % 256
    ("rz_q4k_f32_gemv", (16, 20, None, 16, 1, 4, 256, None), 3),          # x misaligned
    ("rz_q4k_f32_gemv", (16, 16, 18, 16, 1, 4, 256, None), 3),            # bias not 4-byte aligned
    ("rz_q4_0_gemv_bias", (16, 16, None, 16, 1, 4, 32, None), 1),         # no bias
    ("rz_q4_0_gemv_bias", (16, 16, 16, 16, 1, 4, 48, None), 2),           # in_dim % 32
    ("rz_debug_stall_next_gemv", (100,), 1),                              # limit below 1024
    ("rz_debug_stall_next_gemv", ((1 << 22) + 1,), 1),                    # limit above 2^22
])
def test_more_argument_checks_fail_before_launch(lib, call, args, status):
    """The same for the other GEMV, GEMM and test-aid entry points."""
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    st = _lib.status(call, *args)
    assert st == status, (st, _lib.last_error())
    assert _lib.last_error()


def test_multi_matrix_argument_checks(lib):
    """rz_q4k_q8_gemv_multi and rz_rmsnorm_q4k_gemv take arrays of matrices: their
    count, rows, alignment and output stride are checked on the host."""
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    w = (C.c_void_p * 3)(16, 32, 48)
    rows = (C.c_int64 * 3)(4, 4, 4)
    bad_w = (C.c_void_p * 3)(16, 40, 48)       # second matrix misaligned
    bad_rows = (C.c_int64 * 3)(4, 0, 4)        # empty second matrix
    bias = (C.c_void_p * 3)(16, 18, 16)        # second bias not 4-byte aligned
    cases = [
        (("rz_q4k_q8_gemv_multi", 16, 4, w, rows, None, 16, 12, 1, 256, None), 1),       # n_mats > 3
        (("rz_q4k_q8_gemv_multi", 16, 3, w, rows, None, 16, 12, 17, 256, None), 2),     # m > 16
        (("rz_q4k_q8_gemv_multi", 16, 3, w, rows, None, 16, 12, 1, 300, None), 2),      # in_dim % 256
        (("rz_q4k_q8_gemv_multi", 16, 3, bad_w, rows, None, 16, 12, 1, 256, None), 3),
        (("rz_q4k_q8_gemv_multi", 16, 3, w, bad_rows, None, 16, 12, 1, 256, None), 1),
        (("rz_q4k_q8_gemv_multi", 16, 3, w, rows, bias, 16, 12, 1, 256, None), 3),
        (("rz_q4k_q8_gemv_multi", 16, 3, w, rows, None, 16, 11, 1, 256, None), 2),      # ldy < 12 rows
        (("rz_rmsnorm_q4k_gemv", 16, 256, 16, 256, 1e-6, 0, w, rows, None, 16, 12, 1, 256, None), 1),
        (("rz_rmsnorm_q4k_gemv", 16, 256, 16, 300, 1e-6, 3, w, rows, None, 16, 12, 1, 256, None), 2),  # n > in_dim
        (("rz_rmsnorm_q4k_gemv", 16, 128, 16, 256, 1e-6, 3, w, rows, None, 16, 12, 1, 256, None), 2),  # ldx < in_dim
        (("rz_rmsnorm_q4k_gemv", 16, 256, 16, 256, -1.0, 3, w, rows, None, 16, 12, 1, 256, None), 1),  # eps < 0
        (("rz_rmsnorm_q4k_gemv", 16, 256, 16, 256, 1e-6, 3, bad_w, rows, None, 16, 12, 1, 256, None), 3),
        (("rz_rmsnorm_q4k_gemv", 16, 256, 16, 256, 1e-6, 3, w, rows, None, 16, 8, 1, 256, None), 2),  # ldy
    ]
    for args, status in cases:
        st = _lib.status(*args)
        assert st == status, (args[0], st, _lib.last_error())
        assert _lib.last_error()


def _llama_like_layer(_lib, **over):
    f = dict(wq=16, wk=32, wv=48, wo=64, wgate=80, wup=96, wdown=112, attn_gamma=128, ffn_gamma=144,
             hidden=4096, hidden_pad=4096, n_heads=32, n_kv_heads=32, head_dim=128, inter=11008,
             eps=1e-6, rope_theta=1e4, rope_mode=0, bq=None, bk=None, bv=None)
    f.update(over)
    return _lib.LayerWeightsStruct(**f)


@pytest.mark.parametrize("over,status", [
    (dict(wo=72), 3),                          # a weight not 16-byte aligned
    (dict(wup=None), 1),                       # a weight missing
    (dict(wk=None, wv=None, bk=16), 1),        # fused Q|K|V with its K bias apart
    (dict(bq=18), 3),                          # bias not 4-byte aligned
    (dict(hidden_pad=4000), 2),                # hidden_pad not a multiple of 256
    (dict(hidden_pad=3840), 2),                # hidden_pad < hidden
    (dict(n_kv_heads=5), 2),                   # n_heads % n_kv_heads
    (dict(n_kv_heads=1), 6),                   # 32 query heads per kv head
    (dict(head_dim=48), 2),                    # head_dim not a multiple of 32
    (dict(head_dim=512), 2),                   # head_dim beyond 256
])
def test_layer_descriptor_checks_fail_before_the_device(lib, over, status):
    """rz_decode_layer validates the layer descriptor on the host before it
    queries the device (whose shared memory bounds the remaining checks)."""
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    L = _llama_like_layer(_lib, **over)
    st = _lib.status("rz_decode_layer", 16, C.byref(L), None, None, 0, 1, 16, None, 0, None)
    assert st == status, (st, _lib.last_error())
    assert _lib.last_error()
    # the batch size is checked with the descriptor
    st = _lib.status("rz_decode_layer", 16, C.byref(_llama_like_layer(_lib)), None, None, 0, 17, 16, None, 0, None)
    assert st == 2, (st, _lib.last_error())


def test_valid_layer_descriptor_reaches_the_device_check(lib):
    """A descriptor that passes the host checks is next refused for what is
    missing: here no sm_103a device (or, on a GPU machine, the missing KV cache)."""
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    st = _lib.status("rz_decode_layer", 16, C.byref(_llama_like_layer(_lib)), None, None, 0, 1, 16, None, 0, None)
    assert st != 0 and _lib.last_error()


@pytest.mark.parametrize("over,status", [
    (dict(wo=24), 3), (dict(wdown=None), 1), (dict(hidden=100), 2), (dict(inter=1000), 2),
    (dict(n_kv_heads=3), 2), (dict(head_dim=40), 2),
])
def test_q4_0_layer_descriptor_checks(lib, over, status):
    from quantized_q4_q8_gb300 import _lib
    _lib.load()
    f = dict(wqkv=16, wo=32, wgate=48, wup=64, wdown=80, attn_gamma=96, ffn_gamma=112, hidden=896,
             n_heads=14, n_kv_heads=2, head_dim=64, inter=4864, eps=1e-6, rope_theta=1e6, rope_mode=1)
    f.update(over)
    L = _lib.LayerWeightsQ40Struct(**f)
    st = _lib.status("rz_decode_layer_q4_0", 16, C.byref(L), None, None, 0, 1, 16, None, 0, None)
    assert st == status, (st, _lib.last_error())


def test_package_fails_loudly_without_library(tmp_path):
    from quantized_q4_q8_gb300 import _lib
    with pytest.raises(ImportError):
        _lib._lib_backup = _lib._lib
        try:
            _lib._lib = None
            _lib.load(str(tmp_path / "missing.so"))
        finally:
            _lib._lib = _lib._lib_backup
