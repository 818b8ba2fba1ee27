"""GPU parity of the many-token Q4_K x Q8_1 product on the tensor cores
(rz_q4k_q8_gemm) against the CPU oracle's q4k_q8_gemv on the same seeded inputs.

Bars: f32 outputs within 1e-5 relative plus 1e-6 * ||row|| absolute per element
(the GEMV bar); bit-exact on integer-valued inputs, where every partial sum is an
integer below 2^24; bit-identical between two runs.
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


# (out_dim, in_dim, m): single tile; ragged rows and tokens over several tiles;
# one token; one row; rings that wrap many times (in_dim 4096 = 144 regions)
GEMM_CASES = [
    (128, 256, 128), (300, 1024, 200), (1, 256, 1), (129, 512, 129), (256, 4096, 17),
    (1000, 2048, 64), (77, 11008, 5), (513, 768, 300),
]


@pytest.mark.parametrize("out_dim,in_dim,m", GEMM_CASES)
def test_q4k_gemm_parity(rz, out_dim, in_dim, m):
    w = S.q4k_weight(f"ggemm.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"ggemm.x.{in_dim}.{m}", (m, in_dim))
    x8 = oracle.q8_1_quantize(x)
    y = rz.q4k_q8_gemm(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim)
    assert_gemv_close(y, y_ref, row_norms_q4k(w)[None, :], f"gemm {out_dim}x{in_dim} m={m}")


def test_q4k_gemm_integer_inputs_exact(rz):
    """Integer-valued inputs make the product exact in f32: d = dmin = 1, every
    6-bit scale and min and every 4-bit code drawn over its full range, and
    activations that are integers in [-7, 7] with a 127 in every block (d8 = 1,
    q8 = x, s = sum of the block's codes).  Then y = sum_j sc_j I_j - sum_j m_j s_j
    exactly (every partial sum an integer below 2^24): a wrong K order, nibble,
    scale, min, bf16 piece of s or token/row mapping cannot hide in rounding."""
    out_dim, in_dim, m = 300, 512, 150
    g = np.random.default_rng(7)
    nsb = in_dim // 256
    w = np.zeros((out_dim, nsb * 144), np.uint8)
    scs = g.integers(0, 64, (out_dim, nsb, 8))
    mns = g.integers(0, 64, (out_dim, nsb, 8))
    qs = g.integers(0, 16, (out_dim, nsb, 256))
    for r in range(out_dim):
        for b in range(nsb):
            w[r, b * 144:(b + 1) * 144] = oracle.q4k_pack(0x3C00, 0x3C00, scs[r, b].astype(np.uint8),
                                                          mns[r, b].astype(np.uint8), qs[r, b].astype(np.uint8))
    x = g.integers(-7, 8, (m, in_dim)).astype(np.float32)
    x[:, ::32] = 127.0
    x8 = oracle.q8_1_quantize(x)
    d8, s8, q8 = oracle.q8_1_fields(x8, m, in_dim)
    assert (d8 == 1.0).all() and np.array_equal(q8.reshape(m, in_dim), x.astype(np.int8))
    qi = x.astype(np.int64).reshape(m, nsb, 8, 32)
    # element e of super-block b: q[e] as stored in qs (the layout of q4k_pack)
    qv = qs.reshape(out_dim, nsb, 8, 32).astype(np.int64)
    I = np.einsum("tbjk,rbjk->trbj", qi, qv)                        # [m, out, nsb, 8]
    ssum = qi.sum(-1)                                               # [m, nsb, 8]
    expect = (I * scs[None]).sum((-1, -2)) - np.einsum("tbj,rbj->tr", ssum, mns)
    assert np.abs(expect).max() < 2 ** 24
    assert np.array_equal(oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim), expect.astype(np.float32))
    y = rz.q4k_q8_gemm(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    assert np.array_equal(y, expect.astype(np.float32))


def test_q4k_gemm_deterministic_and_strided(rz):
    import torch
    out_dim, in_dim, m = 384, 2048, 256
    w = to_dev(S.q4k_weight("gemmdet.w", out_dim, in_dim))
    x8 = to_dev(oracle.q8_1_quantize(S.normal("gemmdet.x", (m, in_dim))))
    a = rz.q4k_q8_gemm(w, x8, m, out_dim, in_dim).cpu().numpy()
    b = rz.q4k_q8_gemm(w, x8, m, out_dim, in_dim).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # a row stride beyond out_dim leaves the gap untouched
    big = torch.full((m, out_dim + 5), 7.0, dtype=torch.float32, device=w.device)
    rz.q4k_q8_gemm(w, x8, m, out_dim, in_dim, out=big)
    check_no_device_error()
    big = big.cpu().numpy()
    assert np.array_equal(big[:, :out_dim].view(np.uint32), a.view(np.uint32))
    assert (big[:, out_dim:] == 7.0).all()


@pytest.mark.parametrize("out_dim,in_dim", S.LLAMA_SWEEP)
def test_q4k_gemm_full_size(rz, out_dim, in_dim):
    """The Llama sweep with a 512-token prompt, the launch configuration the
    benchmark times; every row of sampled tokens (first and last of the tiles,
    the last token) against the oracle."""
    m = 512
    w = S.q4k_weight(f"sweep.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"gemmfull.x.{in_dim}", (m, in_dim))
    x8 = oracle.q8_1_quantize(x)
    y = rz.q4k_q8_gemm(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    pick = [0, 127, 128, 383, 511]
    xs8 = oracle.q8_1_quantize(x[pick])        # Q8_1 is per row: the same codes
    y_ref = oracle.q4k_q8_gemv(w, xs8, len(pick), out_dim, in_dim)
    assert_gemv_close(y[pick], y_ref, row_norms_q4k(w)[None, :], f"gemm sweep {out_dim}x{in_dim} m={m}")


def test_q4k_gemm_rejects_bad_arguments(rz):
    """Shape and workspace checks run on the host before any launch."""
    import torch
    from quantized_q4_q8_gb300._lib import RzError
    w = torch.zeros(144, dtype=torch.uint8, device="cuda")
    q8 = torch.zeros(rz.q8_1_size(1, 256), dtype=torch.uint8, device="cuda")
    y = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.zeros(rz.q4k_q8_gemm_workspace_bytes(1, 256), dtype=torch.uint8, device="cuda")
    for args, status in [((0, 1, 1, 255, ws, ws.numel()), 2),        # in_dim % 256: RZ_ERR_SHAPE
                         ((0, 1, 1, 256, ws, ws.numel() - 16), 1),   # workspace too small
                         ((0, 0, 1, 256, ws, ws.numel()), 1)]:       # m = 0
        with pytest.raises(RzError) as e:
            rz.rz_q4k_q8_gemm(w, q8, y, *args)
        assert e.value.status == status
    rz.rz_q4k_q8_gemm(w, q8, y, 0, 1, 1, 256, ws, ws.numel())
    check_no_device_error()
