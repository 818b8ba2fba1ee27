"""GPU parity of the variants beside the Q4_K x Q8_1 decode path: the bias and
residual epilogues, the fused RMSNorm -> Q8_1 -> Q|K|V launch, the fused Q|K|V
weight layout with QKV biases (Qwen2's preload_qkv_bias, OwnedQKVWeights::Fused),
the LM-head bias, and the Q4_0 whole-model layer with its SwiGLU and GELU FFNs
(GpuModelQ4::forward_layer, ffn_swiglu_gpu, ffn_standard_gpu).

Bars as in the other GPU tests: GEMV outputs within 1e-5 relative plus 1e-6 ||row||
per element; composite outputs within 1e-3 relative (max and L2).
"""
import numpy as np
import pytest

import oracle
import rz_synth as S

from gpu_common import assert_gemv_close, check_no_device_error, row_norms_q4_0, row_norms_q4k, to_dev
from test_gpu_layer import assert_rel, dev_layer, orc_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    return rz


# ----------------------------------------------------------------------------- epilogues
@pytest.mark.parametrize("m", [1, 2, 5, 16])
def test_gemv_bias_and_residual_epilogues(rz, m):
    out_dim, in_dim = 3000, 2048
    w = S.q4k_weight("gex.w", out_dim, in_dim)
    x8 = oracle.q8_1_quantize(S.normal(f"gex.x.{m}", (m, in_dim)))
    b = S.normal("gex.b", out_dim)
    res = S.normal(f"gex.r.{m}", (m, out_dim + 8))     # row stride ld = out_dim + 8
    y_ref = oracle.q4k_q8_gemv(w, x8, m, out_dim, in_dim)
    wn = row_norms_q4k(w)[None, :]
    yb = rz.q4k_q8_gemv_ex(to_dev(w), to_dev(x8), m, out_dim, in_dim, bias=to_dev(b)).cpu().numpy()
    assert_gemv_close(yb, np.stack([oracle.residual_add(y_ref[t], b) for t in range(m)]), wn, "bias")
    yr = rz.q4k_q8_gemv_ex(to_dev(w), to_dev(x8), m, out_dim, in_dim, residual=to_dev(res),
                           ld=out_dim + 8).cpu().numpy()
    assert_gemv_close(yr[:, :out_dim], np.stack([oracle.residual_add(y_ref[t], res[t, :out_dim]) for t in range(m)]),
                      wn, "residual")
    check_no_device_error()


@pytest.mark.parametrize("m", [1, 3, 8])
def test_rmsnorm_qkv_fused_launch(rz, m):
    """RMSNorm -> Q8_1 -> three GEMVs in one launch, with a bias on K only."""
    sh = S.QWEN2
    L = S.layer(sh, "gnq")
    x = S.hidden_input(f"gnq.x.{m}", m, sh.hidden, sh.hidden_pad)
    bk = S.normal("gnq.bk", sh.kv_dim)
    rows = [sh.q_dim, sh.kv_dim, sh.kv_dim]
    y = rz.rmsnorm_q4k_gemv(to_dev(x), to_dev(L.attn_gamma), sh.hidden, sh.eps,
                            [to_dev(L.w["wq"]), to_dev(L.w["wk"]), to_dev(L.w["wv"])], rows, sh.hidden_pad,
                            biases=[None, to_dev(bk), None]).cpu().numpy()
    check_no_device_error()
    x8 = oracle.q8_1_quantize(oracle.rmsnorm(x, L.attn_gamma, sh.hidden, sh.hidden_pad, sh.eps))
    off = 0
    for nm, r in zip(("wq", "wk", "wv"), rows):
        ref = oracle.q4k_q8_gemv(L.w[nm], x8, m, r, sh.hidden_pad)
        if nm == "wk":
            ref = np.stack([oracle.residual_add(ref[t], bk) for t in range(m)])
        # the normed input is quantised on the GPU from its own f32 norm: codes may
        # differ by one step from the oracle's, so the layer bar applies
        for t in range(m):
            assert_rel(y[t, off:off + r], ref[t], what=f"fused {nm} token {t}")
        off += r


@pytest.mark.parametrize("m", [1, 5, 16])
def test_q8_gemv_multi_matches_single_gemvs(rz, m):
    """Three matrices against one Q8_1 activation in one launch (how a layer runs
    Q|K|V from four tokens on), a bias on K only: each matrix's rows against the
    oracle's GEMV of the same Q8_1 codes, at the GEMV bar."""
    sh = S.QWEN2
    L = S.layer(sh, "gmq")
    x = S.normal(f"gmq.x.{m}", (m, sh.hidden_pad))
    x8 = oracle.q8_1_quantize(x)
    bk = S.normal("gmq.bk", sh.kv_dim)
    rows = [sh.q_dim, sh.kv_dim, sh.kv_dim]
    y = rz.q4k_q8_gemv_multi(to_dev(x8), [to_dev(L.w["wq"]), to_dev(L.w["wk"]), to_dev(L.w["wv"])], rows, m,
                             sh.hidden_pad, biases=[None, to_dev(bk), None]).cpu().numpy()
    check_no_device_error()
    off = 0
    for nm, r in zip(("wq", "wk", "wv"), rows):
        ref = oracle.q4k_q8_gemv(L.w[nm], x8, m, r, sh.hidden_pad)
        if nm == "wk":
            ref = np.stack([oracle.residual_add(ref[t], bk) for t in range(m)])
        assert_gemv_close(y[:, off:off + r], ref, row_norms_q4k(L.w[nm])[None, :], f"multi {nm} m={m}")
        off += r


# ----------------------------------------------------------------------------- QKV bias, fused layout
@pytest.mark.parametrize("fused", [False, True])
def test_decode_layer_qwen2_with_qkv_bias(rz, fused):
    """The Qwen2-shaped layer with QKV biases, the three matrices either separate or
    as one fused [q + 2 kv][hidden] matrix."""
    import torch
    sh = S.QWEN2
    L = S.layer(sh, "qb.l")
    bq, bk, bv = S.normal("qb.bq", sh.q_dim), S.normal("qb.bk", sh.kv_dim), S.normal("qb.bv", sh.kv_dim)
    pos, max_seq = 127, 160
    x = S.hidden_input("qb.x", 1, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, "qb.kv", max_seq, pos)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    w = {k: to_dev(v) for k, v in L.w.items()}
    w["attn_gamma"], w["ffn_gamma"] = to_dev(L.attn_gamma), to_dev(L.ffn_gamma)
    if fused:
        w["wq"] = to_dev(np.concatenate([L.w["wq"], L.w["wk"], L.w["wv"]], axis=0))
        w["wk"] = w["wv"] = None
        w["bq"] = to_dev(np.concatenate([bq, bk, bv]))
    else:
        w["bq"], w["bk"], w["bv"] = to_dev(bq), to_dev(bk), to_dev(bv)
    dl = rz.DeviceLayer(w, sh.hidden, sh.hidden_pad, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.inter, sh.eps,
                        sh.rope_theta, sh.rope_mode)
    out = rz.decode_layer(to_dev(x), dl, kv, position=pos).cpu().numpy()
    check_no_device_error()
    ol = orc_layer(L)
    ol.bq, ol.bk, ol.bv = bq, bk, bv
    kr, vr = kc[0].copy(), vc[0].copy()
    ref = oracle.decode_layer(x[0], ol, kr, vr, pos)
    assert_rel(out[0], ref, what=f"qwen2 layer with QKV bias (fused={fused})")
    # the cache rows carry the biased projections (v + bv, rope(k + bk))
    kn, vn = kc[0].copy(), vc[0].copy()
    oracle.decode_layer(x[0], orc_layer(L), kn, vn, pos)
    assert_rel(kv.v.cpu().numpy()[0, pos], vr[pos], what="v row")
    assert_rel(kv.k.cpu().numpy()[0, pos], kr[pos], what="k row")
    assert np.abs(vr[pos] - vn[pos] - bv).max() <= 1e-3 * np.abs(bv).max()


# ----------------------------------------------------------------------------- LM-head bias
def test_q4_0_gemv_bias_and_stack_lm_bias(rz):
    vocab, hidden = 32000, 4096
    w = S.q4_0_weight(f"lm.{vocab}.{hidden}", vocab, hidden)
    x = S.normal(f"lmb.x.{hidden}", (2, hidden))
    b = S.normal("lmb.b", vocab)
    y = rz.q4_0_gemv(to_dev(w), to_dev(x), vocab, hidden, bias=to_dev(b)).cpu().numpy()
    check_no_device_error()
    y_ref = oracle.q4_0_gemv(w, x, vocab, hidden)
    assert_gemv_close(y, np.stack([oracle.residual_add(y_ref[t], b) for t in range(2)]),
                      row_norms_q4_0(w)[None, :], "lm head + bias")
    # the stack with an LM-head bias (Qwen2 shape, one layer)
    sh = S.QWEN2
    L = S.layer(sh, "lmb.l0")
    og = S.uniform("lmb.og", sh.hidden, 0.5, 1.5)
    lm = S.q4_0_weight("lmb.lm", 1000, sh.hidden)
    lb = S.normal("lmb.lb", 1000)
    kc, vc = S.kv_prefill(sh, "lmb.kv", 64, 20)
    stack = rz.DeviceStack([dev_layer(rz, L)], [rz.DeviceKV(to_dev(kc), to_dev(vc))], to_dev(og), to_dev(lm), 1000,
                           lm_bias=to_dev(lb))
    xs = S.hidden_input("lmb.xs", 1, sh.hidden, sh.hidden_pad)
    _, logits = rz.decode_stack(to_dev(xs), stack, position=20)
    check_no_device_error()
    _, log_r = oracle.decode_stack(xs[0], [orc_layer(L)], [kc[0].copy()], [vc[0].copy()], 20, og, lm, 1000,
                                   lm_bias=lb)
    assert_rel(logits.cpu().numpy()[0], log_r, what="stack logits with LM-head bias")


# ----------------------------------------------------------------------------- Q4_0 whole-model layer
def _dev_q40(rz, sh, w):
    t = {k: (to_dev(v) if v is not None else None) for k, v in w.items()}
    return rz.DeviceLayerQ40(t, sh.hidden, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.inter, sh.eps,
                             sh.rope_theta, sh.rope_mode)


def _orc_q40(sh, w):
    return oracle.LayerWeightsQ40(wqkv=w["wqkv"], wo=w["wo"], wgate=w.get("wgate"), wup=w["wup"],
                                  wdown=w["wdown"], attn_gamma=w["attn_gamma"], ffn_gamma=w["ffn_gamma"],
                                  hidden=sh.hidden, n_heads=sh.n_heads, n_kv_heads=sh.n_kv_heads,
                                  head_dim=sh.head_dim, inter=sh.inter, eps=sh.eps, rope_theta=sh.rope_theta,
                                  rope_mode=sh.rope_mode)


@pytest.mark.parametrize("shape", [S.Q40_GELU, S.Q40_SWIGLU], ids=["gelu", "swiglu"])
@pytest.mark.parametrize("positions", [[300], [0], [17, 300, 5]])
def test_decode_layer_q4_0_parity(rz, shape, positions):
    sh = shape
    w = S.layer_q4_0(sh, f"q40.{sh.gated}")
    m = len(positions)
    max_seq = 320
    x = S.normal(f"q40.x.{sh.gated}.{m}", (m, sh.hidden))
    kc = np.zeros((m, max_seq, sh.kv_dim), np.float32)
    vc = np.zeros_like(kc)
    kc[:, :max(positions)] = S.normal(f"q40.k.{m}", (m, max(positions), sh.kv_dim)) if max(positions) else 0
    vc[:, :max(positions)] = S.normal(f"q40.v.{m}", (m, max(positions), sh.kv_dim)) if max(positions) else 0
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    pos_d = to_dev(np.array(positions, np.int32)) if m > 1 else None
    out = rz.decode_layer_q4_0(to_dev(x), _dev_q40(rz, sh, w), kv, position=positions[0],
                               positions=pos_d).cpu().numpy()
    check_no_device_error()
    kc_after = kv.k.cpu().numpy()
    ol = _orc_q40(sh, w)
    for t, p in enumerate(positions):
        kt, vt = kc[t].copy(), vc[t].copy()
        ref = oracle.decode_layer_q4_0(x[t], ol, kt, vt, p)
        assert_rel(out[t], ref, what=f"q4_0 layer ({'swiglu' if sh.gated else 'gelu'}) token {t} at {p}")
        assert_rel(kc_after[t, p], kt[p], tol=1e-4, what="k row")
