"""Helpers for the GPU parity tests (imported by tests marked gpu only)."""
import numpy as np

import oracle


def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def row_norms_q4k(w):
    """L2 norm of every dequantised weight row (the ||row|| of the tolerance)."""
    return np.linalg.norm(oracle.q4k_dequantize(w), axis=-1)


def row_norms_q4_0(w):
    return np.linalg.norm(oracle.q4_0_dequantize(w), axis=-1)


def assert_gemv_close(y_gpu, y_ref, wnorm, what=""):
    """f32 outputs within 1e-5 relative plus 1e-6 * ||row|| absolute, per element."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    tol = 1e-5 * np.abs(y_ref) + 1e-6 * np.broadcast_to(wnorm, y_ref.shape)
    err = np.abs(y_gpu - y_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(tol, 1e-30)), err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
            f"gpu={y_gpu[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")
    return float((err / np.maximum(tol, 1e-30)).max())


def check_no_device_error():
    import quantized_q4_q8_gb300 as rz
    st, code = rz.check_device_error()
    assert st == 0 and code == 0, f"device error word 0x{code:x}"
