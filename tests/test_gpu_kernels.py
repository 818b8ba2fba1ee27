"""GPU parity: each librz kernel against the CPU oracle on the same seeded inputs.

Bars: Q8_1 codes, d, s and the integer sub-block dots bit-exact; f32 GEMV
outputs within 1e-5 relative plus 1e-6 * ||row|| absolute; residual add
bit-exact; RMSNorm's fused Q8_1 bit-exact against the oracle's quantisation of
the GPU's own f32 output.
"""
import numpy as np
import pytest

import oracle
import rz_synth as S

from gpu_common import (assert_gemv_close, check_no_device_error, row_norms_q4_0,
                        row_norms_q4k, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    return rz


# ----------------------------------------------------------------------------- Q8_1
@pytest.mark.parametrize("m,n", [(1, 32), (1, 1024), (3, 896), (16, 4096), (1, 14336), (2, 4864)])
def test_q8_1_bit_exact(rz, m, n):
    x = S.normal(f"gq8.{m}.{n}", (m, n)) * np.float32(3.0)
    x[0, :32] = 0.0                       # an all-zero block
    if n >= 64:
        x[0, 32:64] = 0.0
        x[0, 40] = -7.25                  # one-hot block
    q8 = rz.q8_1_quantize(to_dev(x)).cpu().numpy()
    check_no_device_error()
    assert np.array_equal(q8, oracle.q8_1_quantize(x))


@pytest.mark.parametrize("lo,hi", [(-2.0, 2.0), (-44.0, -36.0), (-37.5, -30.0), (30.0, 37.0)])
def test_q8_1_boundary_quotients_bit_exact(rz, lo, hi):
    """Every element next to a rounding boundary of x / d ((k + 1/2) d, nudged by at
    most an ulp): the kernels decide these as the IEEE quotient does, as the
    format does, so the codes still match the oracle bit for bit.  Block maxima
    10^lo .. 10^hi: ordinary scales, subnormal maxima and scales (1/d beyond the
    f32 range), scales near the top of the range."""
    g = np.random.default_rng(11)
    nblk = 4096
    amax = (10.0 ** g.uniform(lo, hi, nblk)).astype(np.float32)
    amax = np.where(amax > 0, amax, np.float32(1e-45)).astype(np.float32)
    d = amax / np.float32(127)
    k = g.integers(-126, 126, (nblk, 31)).astype(np.float32)
    x = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    nudge = g.integers(-1, 2, x.shape)
    x = np.where(nudge > 0, np.nextafter(x, np.float32(np.inf)),
                 np.where(nudge < 0, np.nextafter(x, np.float32(-np.inf)), x))
    x = np.concatenate([amax[:, None], x], axis=1).astype(np.float32).reshape(4, -1)
    q8 = rz.q8_1_quantize(to_dev(x)).cpu().numpy()
    check_no_device_error()
    assert np.array_equal(q8, oracle.q8_1_quantize(x))


def test_q8_1_large_magnitudes_bit_exact(rz):
    x = S.normal("gq8.big", (2, 512)) * np.float32(4.0e4)
    q8 = rz.q8_1_quantize(to_dev(x)).cpu().numpy()
    assert np.array_equal(q8, oracle.q8_1_quantize(x))


# ----------------------------------------------------------------------------- Q4_K x Q8_1
@pytest.mark.parametrize("out_dim,in_dim", [(256, 1024), (7, 256), (33, 512), (129, 768),
                                            (64, 2048), (40, 1280), (17, 4864), (9, 11008),
                                            (5, 14336)])
def test_q4k_subblock_dots_bit_exact(rz, out_dim, in_dim):
    w = S.q4k_weight(f"gdots.{out_dim}.{in_dim}", out_dim, in_dim)
    x8 = oracle.q8_1_quantize(S.normal(f"gdots.x.{in_dim}", (1, in_dim)))
    I = rz.q4k_q8_subblock_dots(to_dev(w), to_dev(x8), out_dim, in_dim).cpu().numpy()
    assert np.array_equal(I, oracle.q4k_q8_subblock_dots(w, x8, out_dim, in_dim))


GEMV_CASES = [
    (256, 1024, 1),            # the small single-GEMV workload (4 super-blocks per row)
    (1, 256, 1), (3, 512, 1), (129, 768, 1), (37, 1280, 1), (61, 1792, 1),
    (300, 2048, 1), (1000, 4096, 1), (23, 4864, 1), (45, 11008, 1), (19, 14336, 1),
    (256, 1024, 2), (100, 1024, 3), (77, 4096, 4), (50, 2304, 5), (33, 4096, 8),
    (65, 1024, 16), (40, 4864, 16), (9, 14336, 16), (2000, 256, 7),
    # >= 64 rows per CTA on 152 SMs: the multi-token row-pair path (token groups
    # of 2, 3, 4 with a ragged last group; CTAs with an odd row count)
    (10001, 512, 2), (10001, 1024, 3), (9999, 512, 6), (9729, 2048, 16),
    # several laps of the stage ring per CTA (263 and 198 rows per CTA)
    (40000, 4096, 1), (30001, 2048, 3),
    # 16 units per CTA on 152 SMs (16 row pairs; 16 packs of two short rows): the
    # one-token launch takes its 16-warp instantiation
    (4864, 2048, 1), (4800, 1024, 1),
    # tensor-core GEMV whose int8 codes do not fit at once: staged in phases of K
    # (11008 and 14336 at 12 and 16 tokens; 22528: more phases)
    (300, 11008, 16), (100, 14336, 12), (64, 22528, 16),
]


@pytest.mark.parametrize("out_dim,in_dim,m", GEMV_CASES)
def test_q4k_gemv_parity(rz, out_dim, in_dim, m):
    w = S.q4k_weight(f"ggemv.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"ggemv.x.{in_dim}.{m}", (m, in_dim))
    x8 = oracle.q8_1_quantize(x)
    y = rz.q4k_q8_gemv(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim)
    assert_gemv_close(y, y_ref, row_norms_q4k(w)[None, :], f"{out_dim}x{in_dim} m={m}")


def test_q4k_gemv_deterministic(rz):
    out_dim, in_dim, m = 512, 4096, 4
    w = to_dev(S.q4k_weight("gdet.w", out_dim, in_dim))
    x8 = to_dev(oracle.q8_1_quantize(S.normal("gdet.x", (m, in_dim))))
    a = rz.q4k_q8_gemv(w, x8, m, out_dim, in_dim).cpu().numpy()
    b = rz.q4k_q8_gemv(w, x8, m, out_dim, in_dim).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("out_dim,in_dim", S.LLAMA_SWEEP)
@pytest.mark.parametrize("m", [1, 16])
def test_q4k_gemv_full_size(rz, out_dim, in_dim, m):
    """Full Llama-shaped sweep in the launch configuration the benchmark times;
    every output row of every token against the oracle."""
    w = S.q4k_weight(f"sweep.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"sweep.x.{in_dim}.{m}", (m, in_dim))
    x8 = oracle.q8_1_quantize(x)
    y = rz.q4k_q8_gemv(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim)
    assert_gemv_close(y, y_ref, row_norms_q4k(w)[None, :], f"sweep {out_dim}x{in_dim} m={m}")


def test_q4k_gemv_padding_invariance(rz):
    """896 -> 1024: zero-padded activations make the padded weight columns
    irrelevant on the GPU too (bit-identical outputs)."""
    out_dim = 896
    w = S.q4k_weight("gpad.w", out_dim, 1024)
    x = S.hidden_input("gpad.x", 1, 896, 1024)
    x8 = to_dev(oracle.q8_1_quantize(x))
    y_rand = rz.q4k_q8_gemv(to_dev(w), x8, 1, out_dim, 1024).cpu().numpy()
    w0 = w.copy()
    w0[:, 3 * 144 + 16 + 64:4 * 144] = 0   # chunks 2, 3 of super-block 3: elements 896..1023
    y_zero = rz.q4k_q8_gemv(to_dev(w0), x8, 1, out_dim, 1024).cpu().numpy()
    assert np.array_equal(y_rand.view(np.uint32), y_zero.view(np.uint32))


# ----------------------------------------------------------------------------- Q4_0
# in_dim a multiple of 256 runs on the tensor-core kernel (token groups of at
# most eight; 17 rows: one row per CTA; 5000 x 512: ragged last tile; 40000 x 256:
# 240 rows per CTA, 167 CTAs; 9 tokens: groups of 5 and 4).  Otherwise every token
# runs on the bulk-copy ring kernel (one launch per token) when a whole number of
# rows fills 16 bytes and the column warps divide 16 (896: two rows, column warps 1;
# 1408: two rows, column warps 2), else (in_dim 32, 992) on the multi-token
# register kernel
@pytest.mark.parametrize("out_dim,in_dim,m", [(100, 896, 1), (33, 4096, 1), (7, 32, 1), (40, 1408, 1),
                                              (50, 1000 // 32 * 32, 1), (64, 8192, 1),
                                              (102, 2048, 1), (30, 16384, 1), (998, 896, 1),
                                              (40, 896, 3), (17, 4096, 16), (300, 9216, 2),
                                              (1000, 4096, 8), (5000, 512, 5), (40000, 256, 4),
                                              (2048, 4096, 9), (64, 992, 4)])
def test_q4_0_gemv_parity(rz, out_dim, in_dim, m):
    w = S.q4_0_weight(f"gq40.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"gq40.x.{in_dim}.{m}", (m, in_dim))
    y = rz.q4_0_gemv(to_dev(w), to_dev(x), out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4_0_gemv(w, x, out_dim, in_dim)
    assert_gemv_close(y, y_ref, row_norms_q4_0(w)[None, :], f"q4_0 {out_dim}x{in_dim} m={m}")


def test_q4_0_gemv_tensor_core_bias_and_range(rz):
    """The tensor-core head with a bias, activations up to +-300 (the two f16
    pieces still carry x to about 2^-22) and exact zeros."""
    out_dim, in_dim, m = 3000, 1024, 6
    w = S.q4_0_weight("gq40b.w", out_dim, in_dim)
    x = (S.normal("gq40b.x", (m, in_dim)) * np.float32(100.0)).astype(np.float32)
    x[1, :300] = 0.0
    b = S.normal("gq40b.b", (out_dim,))
    y = rz.q4_0_gemv(to_dev(w), to_dev(x), out_dim, in_dim, bias=to_dev(b)).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4_0_gemv(w, x, out_dim, in_dim) + b[None, :].astype(np.float64)
    assert_gemv_close(y, y_ref, row_norms_q4_0(w)[None, :] * np.abs(x).max(), "q4_0 + bias")


@pytest.mark.parametrize("vocab,hidden,m", [(v, h, 1) for v, h in S.LM_HEADS] + [(32000, 4096, 16)])
def test_q4_0_lm_head_full_size(rz, vocab, hidden, m):
    """Both LM heads at full size (32000 x 4096 on the tensor-core kernel,
    151936 x 896 on the ring kernel), and the Llama head at 16 tokens (two groups
    of eight); every logit against the oracle."""
    w = S.q4_0_weight(f"lm.{vocab}.{hidden}", vocab, hidden)
    x = S.normal(f"lm.x.{hidden}.{m}" if m > 1 else f"lm.x.{hidden}", (m, hidden))
    y = rz.q4_0_gemv(to_dev(w), to_dev(x), vocab, hidden).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4_0_gemv(w, x, vocab, hidden)
    assert_gemv_close(y, y_ref, row_norms_q4_0(w)[None, :], f"lm head {vocab}")


# ----------------------------------------------------------------------------- RMSNorm / residual
@pytest.mark.parametrize("m,n,n_pad", [(1, 896, 1024), (1, 4096, 4096), (4, 896, 1024),
                                       (16, 4096, 4096), (1, 100, 128), (2, 5, 32)])
def test_rmsnorm_parity_and_fused_q8(rz, m, n, n_pad):
    x = S.hidden_input(f"gnorm.{m}.{n}", m, n, n_pad) * np.float32(5.0)
    g = S.uniform(f"gnorm.g.{n}", n, 0.5, 1.5)
    y, q8 = rz.rmsnorm(to_dev(x), to_dev(g), n, n_pad, 1e-6)
    y = y.cpu().numpy()
    q8 = q8.cpu().numpy()
    y_ref = oracle.rmsnorm(x, g, n, n_pad, 1e-6)
    assert np.allclose(y, y_ref, rtol=2e-6, atol=1e-6 * np.abs(y_ref).max())
    assert not y[:, n:].any()
    # the fused quantisation is exactly Q8_1 of the GPU's own f32 output
    assert np.array_equal(q8, oracle.q8_1_quantize(y))
    # against the fully-oracle path: codes differ by at most one step
    d1, s1, c1 = oracle.q8_1_fields(q8, m, n_pad)
    d2, s2, c2 = oracle.q8_1_fields(oracle.q8_1_quantize(y_ref), m, n_pad)
    assert np.abs(c1.astype(int) - c2.astype(int)).max() <= 1


def test_rmsnorm_y_only_and_q8_only(rz):
    x = S.hidden_input("gnorm2", 2, 896, 1024)
    g = S.uniform("gnorm2.g", 896, 0.5, 1.5)
    y, _ = rz.rmsnorm(to_dev(x), to_dev(g), 896, 1024, 1e-6, want_q8=False)
    _, q8 = rz.rmsnorm(to_dev(x), to_dev(g), 896, 1024, 1e-6, want_y=False)
    assert np.array_equal(q8.cpu().numpy(), oracle.q8_1_quantize(y.cpu().numpy()))


@pytest.mark.parametrize("n", [1, 3, 4, 896, 4097])
def test_residual_add_bit_exact(rz, n):
    a = S.normal(f"gres.a.{n}", n)
    b = S.normal(f"gres.b.{n}", n) * np.float32(1e3)
    out = rz.residual_add(to_dev(a), to_dev(b)).cpu().numpy()
    assert np.array_equal(out, oracle.residual_add(a, b))


def test_device_errors_none_after_suite(rz):
    check_no_device_error()


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_q4k_gemv_integer_inputs_exact(rz, m):
    """Integer-valued inputs make the GEMV exact in f32: d = 1, dmin = 0, scales and
    codes below 4 (so every partial sum stays below 2^24), and activations that
    are integers with a +-127 in every block (d8 = 1, q8 = x).  Then
    y = sum_j sc_j I_j exactly, and every kernel path -- the dp4a forms for one to
    three tokens and the tensor-core form from four on -- must return exactly
    that: a wrong sub-block dot, scale or column mapping cannot hide in rounding."""
    out_dim, in_dim = 1000, 512
    g = np.random.default_rng(100 + m)
    nsb = in_dim // 256
    w = np.zeros((out_dim, nsb * 144), np.uint8)
    blocks = []
    for r in range(out_dim):
        for b in range(nsb):
            sc = g.integers(0, 4, 8).astype(np.uint8)
            mn = g.integers(0, 64, 8).astype(np.uint8)
            q = g.integers(0, 4, 256).astype(np.uint8)
            w[r, b * 144:(b + 1) * 144] = oracle.q4k_pack(0x3C00, 0x0000, sc, mn, q)   # d = 1, dmin = 0
            blocks.append((sc, q))
    x = g.integers(-127, 128, (m, in_dim)).astype(np.float32)
    x[:, ::32] = 127.0                                   # every block's max is 127: d8 = 1
    x8 = oracle.q8_1_quantize(x)
    d8, s8, q8 = oracle.q8_1_fields(x8, m, in_dim)
    assert (d8 == 1.0).all() and np.array_equal(q8.reshape(m, in_dim), x.astype(np.int8))
    expect = np.zeros((m, out_dim), np.int64)
    qi = x.astype(np.int64).reshape(m, in_dim // 32, 32)
    for r in range(out_dim):
        for b in range(nsb):
            sc, q = blocks[r * nsb + b]
            I = (q.astype(np.int64).reshape(8, 32)[None] * qi[:, b * 8:(b + 1) * 8]).sum(-1)   # [m, 8]
            expect[:, r] += (I * sc.astype(np.int64)[None]).sum(-1)
    assert np.abs(expect).max() < 2 ** 24
    y = rz.q4k_q8_gemv(to_dev(w), to_dev(x8), m, out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    assert np.array_equal(y, expect.astype(np.float32))


# ----------------------------------------------------------------------------- Q4_K x f32
@pytest.mark.parametrize("out_dim,in_dim,m", [(256, 1024, 1), (7, 256, 1), (129, 768, 2), (1000, 4096, 1),
                                              (33, 4096, 3), (77, 11008, 5), (19, 14336, 1), (300, 2048, 16)])
def test_q4k_f32_gemv_parity(rz, out_dim, in_dim, m):
    w = S.q4k_weight(f"gf32.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"gf32.x.{in_dim}.{m}", (m, in_dim))
    y = rz.q4k_f32_gemv(to_dev(w), to_dev(x), out_dim, in_dim).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4k_f32_gemv(w, x, out_dim, in_dim)
    assert_gemv_close(y, y_ref, row_norms_q4k(w)[None, :], f"q4k x f32 {out_dim}x{in_dim} m={m}")


@pytest.mark.parametrize("out_dim,in_dim", S.LLAMA_SWEEP)
def test_q4k_f32_gemv_full_size(rz, out_dim, in_dim):
    """The Llama sweep at one token, every row, with a bias."""
    w = S.q4k_weight(f"sweep.{out_dim}.{in_dim}", out_dim, in_dim)
    x = S.normal(f"sweepf.x.{in_dim}", (1, in_dim))
    b = S.normal(f"sweepf.b.{out_dim}", out_dim)
    y = rz.q4k_f32_gemv(to_dev(w), to_dev(x), out_dim, in_dim, bias=to_dev(b)).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.residual_add(oracle.q4k_f32_gemv(w, x, out_dim, in_dim)[0], b)[None, :]
    assert_gemv_close(y, y_ref, row_norms_q4k(w)[None, :], f"q4k x f32 {out_dim}x{in_dim} + bias")
