"""rz_swiglu_ffn_static: the SwiGLU FFN for callers that cannot allocate.

Some callers cannot give the library device memory -- a serving loop that must
never enter the CUDA allocator, or a plugin inside another runtime that owns all
device buffers -- so this entry point keeps its intermediates in a fixed array
inside the library.  This file checks, through the C ABI, that calls in a row --
after other shapes have left their intermediates in the array -- give results
bit-identical to rz_swiglu_ffn with a caller workspace (both run the same
kernels on the same inputs; only the scratch address differs, so a stale or
misplaced intermediate would show as a changed bit), that both agree with the
oracle within the FFN parity tolerance, and that shapes whose scratch would not
fit are refused.  It is collected last so that a failure here does not hide the
other tests.
"""
import numpy as np
import pytest

import rz_synth as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    return rz


def _rel_close(a, b, tol=1e-3):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert np.isfinite(a).all()
    assert np.abs(a - b).max() <= tol * np.abs(b).max()
    assert np.linalg.norm(a - b) <= tol * np.linalg.norm(b)


def _static_ffn(rz, x, gamma, t, shape, m):
    import torch
    out = torch.full((m, shape.hidden_pad), float("nan"), dtype=torch.float32, device=x.device)
    rz.rz_swiglu_ffn_static(x, gamma, t["wgate"], t["wup"], t["wdown"], out, m, shape.hidden,
                            shape.hidden_pad, shape.inter, shape.eps)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# order matters: later shapes find the intermediates of earlier ones in the array
@pytest.mark.parametrize("shape,m", [(S.QWEN2, 1), (S.QWEN2, 2), (S.LLAMA7B, 1)])
def test_static_scratch_ffn_matches_workspace_ffn_twice(rz, shape, m):
    import torch
    import oracle
    dev = torch.device("cuda:0")
    L = S.layer(shape, f"noalloc.{shape.hidden}")
    t = {k: torch.from_numpy(L.w[k]).to(dev) for k in ("wgate", "wup", "wdown")}
    gamma = torch.from_numpy(L.ffn_gamma).to(dev)
    xh = S.hidden_input(f"noalloc.x.{shape.hidden}.{m}", m, shape.hidden, shape.hidden_pad)
    x = torch.from_numpy(xh).to(dev)
    ref = rz.swiglu_ffn(x, gamma, t["wgate"], t["wup"], t["wdown"], shape.hidden,
                        shape.hidden_pad, shape.inter, shape.eps).cpu().numpy()
    for _ in range(2):
        got = _static_ffn(rz, x, gamma, t, shape, m)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        assert not got[:, shape.hidden:].any()
    if m == 2:
        # one more call at the same shape with one token, right after the two-token calls
        ref1 = rz.swiglu_ffn(x[:1].contiguous(), gamma, t["wgate"], t["wup"], t["wdown"], shape.hidden,
                             shape.hidden_pad, shape.inter, shape.eps).cpu().numpy()
        got1 = _static_ffn(rz, x[:1].contiguous(), gamma, t, shape, 1)
        assert np.array_equal(got1.view(np.uint32), ref1.view(np.uint32))
    # and the result is the FFN the oracle computes
    for tok in range(m):
        o = oracle.swiglu_ffn(xh[tok], L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"], shape.hidden,
                              shape.hidden_pad, shape.inter, shape.eps)
        _rel_close(ref[tok], o)
    st, code = rz.check_device_error()
    assert st == 0 and code == 0


def test_static_scratch_refuses_oversized_shapes(rz):
    import torch
    from quantized_q4_q8_gb300 import _lib
    dev = torch.device("cuda:0")
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    p = buf.data_ptr()
    # m = 16 tokens of the Llama-shaped FFN needs about 1 MiB of scratch
    st = _lib.status("rz_swiglu_ffn_static", p, p, p, p, p, p, 16, 4096, 4096, 11008, 1e-6,
                     torch.cuda.current_stream().cuda_stream)
    assert st == 6 and "512 KiB" in _lib.last_error()
