"""GPU error paths: a bounded wait that runs out ends in an error status, not a hang.

The pages propagate failures as errors (GpuError in realizar 0.8.5
forward_utils.rs) instead of panicking; on the GPU every wait of librz's kernels
is bounded for the same reason.  rz_debug_stall_next_gemv makes one GEMV launch
leave a weight stage of its CTA 0 unissued (a flag that nothing sets), with a
short bound on that CTA's waits: the consumers give up, the CTA waits for the
copies it did issue, and the host reads RZ_ERR_TIMEOUT / 0x101 from the device
error word.  The context stays usable: the next call is exact.
"""
import numpy as np
import pytest

import oracle
import rz_synth as S

from gpu_common import assert_gemv_close, check_no_device_error, row_norms_q4k, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    return rz


@pytest.mark.parametrize("out_dim,in_dim,m", [(4096, 4096, 1), (2048, 1024, 4)])
def test_stalled_gemv_reports_timeout_and_next_call_is_exact(rz, out_dim, in_dim, m):
    import torch
    w = S.q4k_weight(f"stall.{out_dim}.{in_dim}", out_dim, in_dim)
    x8 = oracle.q8_1_quantize(S.normal(f"stall.x.{in_dim}.{m}", (m, in_dim)))
    wd, xd = to_dev(w), to_dev(x8)
    check_no_device_error()
    good = rz.q4k_q8_gemv(wd, xd, m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()

    rz.rz_debug_stall_next_gemv(1 << 14)
    y = torch.full((m, out_dim), float("nan"), dtype=torch.float32, device=wd.device)
    rz.q4k_q8_gemv(wd, xd, m, out_dim, in_dim, out=y)      # the launch itself succeeds
    st, code = rz.check_device_error()                     # synchronises: the kernel ended
    assert st == 5 and code == 0x101, (st, hex(code))
    # CTAs other than CTA 0 ran normally: only a prefix of rows (CTA 0's range, a
    # few dozen at most) may differ
    yb = y.cpu().numpy()
    same = np.all(yb.view(np.uint32) == good.view(np.uint32), axis=0)
    first_ok = int(np.argmax(same))
    assert same[first_ok:].all() and first_ok <= 64, first_ok
    check_no_device_error()                                # the word was cleared

    again = rz.q4k_q8_gemv(wd, xd, m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    assert np.array_equal(again.view(np.uint32), good.view(np.uint32))
    y_ref = oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim)
    assert_gemv_close(again, y_ref, row_norms_q4k(w)[None, :], "after the stalled launch")


def test_stall_limit_is_checked_on_the_host(rz):
    from quantized_q4_q8_gb300 import _lib
    assert _lib.status("rz_debug_stall_next_gemv", 10) == 1
    assert _lib.status("rz_debug_stall_next_gemv", 1 << 30) == 1
