"""Pins of the oracle's arithmetic against what the mathematics and the pages fix.

  - integer sub-block dots: brute force over unpacked codes;
  - Q4_K x Q8_1 GEMV: the algebraic identity with dequantise-then-f64-dot (exact
    when the stored s equals d*sum(q), bounded by the s rounding otherwise);
  - zero padding 896 -> 1024 leaves the GEMV bit-identical (forward_utils.rs,
    pad_and_upload_input);
  - Q4_0 GEMV: exact integer sums with d = 1, linearity;
  - RMSNorm: closed form on constant input, unit RMS, padding zeros
    (using.rs, rms_norm_inplace);
  - SiLU, RoPE and attention invariants; the first-token case of the attention
    (clone_layer_weights.rs, forward_single_full_cuda_with_cache);
  - layer / stack: identities that hold with zero weights.
"""
import numpy as np
import pytest

import rz_synth as S


def _unpack_rows(orc, w, nsb):
    """-> d, dmin (f64 [R, nsb]), sc, m ([R, nsb, 8]), q ([R, nsb, 256])"""
    R = w.shape[0]
    d = np.zeros((R, nsb))
    dm = np.zeros((R, nsb))
    sc = np.zeros((R, nsb, 8), np.int64)
    mn = np.zeros((R, nsb, 8), np.int64)
    q = np.zeros((R, nsb, 256), np.int64)
    for r in range(R):
        for b in range(nsb):
            db, dmb, s_, m_, q_ = orc.q4k_unpack(w[r, b * 144:(b + 1) * 144])
            d[r, b], dm[r, b] = orc.f16_to_f64(np.array([db, dmb], np.uint16))
            sc[r, b], mn[r, b], q[r, b] = s_, m_, q_
    return d, dm, sc, mn, q


def test_subblock_dots_brute_force(orc):
    out_dim, in_dim = 5, 768
    w = S.q4k_weight("pin.dots.w", out_dim, in_dim)
    x8 = orc.q8_1_quantize(S.normal("pin.dots.x", (1, in_dim)))
    I = orc.q4k_q8_subblock_dots(w, x8, out_dim, in_dim)
    _, _, q8 = orc.q8_1_fields(x8, 1, in_dim)          # [1, in/32, 32]
    _, _, _, _, q = _unpack_rows(orc, w, in_dim // 256)
    q4 = q.reshape(out_dim, in_dim // 32, 32)
    brute = (q4 * q8[0].astype(np.int64)[None]).sum(axis=-1)
    assert np.array_equal(I, brute)


def test_gemv_identity_exact_case(orc):
    """When every stored s equals d8*sum(q8) exactly, the factored integer dot equals
    the dequantise-then-f64-dot up to f64 rounding."""
    g = np.random.default_rng(11)
    out_dim, in_dim, m = 6, 1024, 3
    w = S.q4k_weight("pin.exact.w", out_dim, in_dim)
    k = g.integers(-127, 128, (m, in_dim))
    k[:, ::32] = 127                     # amax 127 in every block -> d8 = 1/8 exactly
    k[:, 1::32] = -127                   # keeps |sum q| small so s = sum/8 is exact in fp16
    x = (k * 0.125).astype(np.float32)
    x8 = orc.q8_1_quantize(x)
    d8, s8, q8 = orc.q8_1_fields(x8, m, in_dim)
    assert np.all(d8 == 0.125)
    assert np.array_equal(s8.astype(np.float64), 0.125 * q8.astype(np.int64).sum(-1))
    y = orc.q4k_q8_gemv(w, x8, m, out_dim, in_dim).astype(np.float64)
    W = orc.q4k_dequantize(w)                # f64 [out, in]
    X = orc.q8_1_dequantize(x8, m, in_dim)   # f64 [m, in]
    ref = X @ W.T
    scale = np.abs(X) @ np.abs(W).T
    # the oracle returns f32: allow the f32 rounding of the result plus f64 noise
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2 ** -24 + 1e-12 * scale)


def test_gemv_identity_random_bounded_by_s_rounding(orc):
    out_dim, in_dim, m = 8, 1024, 2
    w = S.q4k_weight("pin.ident.w", out_dim, in_dim)
    x8 = orc.q8_1_quantize(S.normal("pin.ident.x", (m, in_dim)))
    y = orc.q4k_q8_gemv(w, x8, m, out_dim, in_dim).astype(np.float64)
    W = orc.q4k_dequantize(w)
    X = orc.q8_1_dequantize(x8, m, in_dim)
    ref = X @ W.T
    d8, s8, q8 = orc.q8_1_fields(x8, m, in_dim)
    s_true = d8.astype(np.float64) * q8.astype(np.int64).sum(-1)
    s_err = np.abs(s8.astype(np.float64) - s_true)               # [m, in/32]
    d, dm, sc, mn, q = _unpack_rows(orc, w, in_dim // 256)
    coef = (dm[..., None] * mn).reshape(out_dim, in_dim // 32)   # dmin_b * m_bj
    bound = s_err @ coef.T                                       # [m, out]
    scale = np.abs(X) @ np.abs(W).T
    diff = np.abs(y - ref)
    assert np.all(diff <= bound + np.abs(ref) * 2 ** -24 + 1e-12 * scale)
    assert bound.max() > 0     # the bound is live, not vacuous-zero


def test_gemv_catches_dropped_min_term(orc):
    """A variant without the -dmin*m*s term would be far outside the bound above."""
    out_dim, in_dim = 4, 512
    w = S.q4k_weight("pin.min.w", out_dim, in_dim)
    x8 = orc.q8_1_quantize(S.normal("pin.min.x", (1, in_dim)))
    y = orc.q4k_q8_gemv(w, x8, 1, out_dim, in_dim)[0].astype(np.float64)
    W = orc.q4k_dequantize(w)
    X = orc.q8_1_dequantize(x8, 1, in_dim)[0]
    d, dm, sc, mn, q = _unpack_rows(orc, w, in_dim // 256)
    no_min = ((d[..., None, None] * sc[..., None] *
               q.reshape(out_dim, -1, 8, 32)).reshape(out_dim, in_dim)) @ X
    assert np.max(np.abs(y - W @ X)) < 1e-3 * np.max(np.abs(y - no_min))


def test_padding_invariance_896_to_1024(orc):
    """Zero-padded activations make the padded weight columns irrelevant: random or
    zero weights there give bit-identical outputs."""
    out_dim = 64
    w = S.q4k_weight("pin.pad.w", out_dim, 1024)
    x = S.hidden_input("pin.pad.x", 2, 896, 1024)
    x8 = orc.q8_1_quantize(x)
    y_rand = orc.q4k_q8_gemv(w, x8, 2, out_dim, 1024)
    # zero the codes of elements 896..1023 (super-block 3, sub-blocks 4..7)
    w0 = w.copy()
    for r in range(out_dim):
        blk = w0[r, 3 * 144:4 * 144]
        d, dm, sc, mn, q = orc.q4k_unpack(blk)
        q[128:] = 0
        sc[4:] = 0
        mn[4:] = 0
        w0[r, 3 * 144:4 * 144] = orc.q4k_pack(d, dm, sc, mn, q)
    y_zero = orc.q4k_q8_gemv(w0, x8, 2, out_dim, 1024)
    assert np.array_equal(y_rand.view(np.uint32), y_zero.view(np.uint32))
    d8, s8, q8 = orc.q8_1_fields(x8, 2, 1024)
    assert not d8[:, 28:].any() and not s8[:, 28:].any() and not q8[:, 28:].any()


def test_q4_0_gemv_exact_integers(orc):
    g = np.random.default_rng(2)
    out_dim, in_dim = 7, 320
    w = S.q4_0_weight("pin.q40.w", out_dim, in_dim).reshape(out_dim, in_dim // 32, 18)
    w[:, :, 0], w[:, :, 1] = 0x00, 0x3C        # d = 1.0
    w = w.reshape(out_dim, -1)
    x = g.integers(-50, 51, (2, in_dim)).astype(np.float32)
    y = orc.q4_0_gemv(w, x, out_dim, in_dim)
    codes = np.zeros((out_dim, in_dim), np.int64)
    for r in range(out_dim):
        for b in range(in_dim // 32):
            _, q = orc.q4_0_unpack(w[r, b * 18:(b + 1) * 18])
            codes[r, b * 32:(b + 1) * 32] = q.astype(np.int64) - 8
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ codes.T)


def test_q4_0_gemv_linear(orc):
    out_dim, in_dim = 16, 256
    w = S.q4_0_weight("pin.q40lin.w", out_dim, in_dim)
    x = S.normal("pin.q40lin.x", (1, in_dim))
    z = S.normal("pin.q40lin.z", (1, in_dim))
    W = orc.q4_0_dequantize(w)
    y = lambda v: orc.q4_0_gemv(w, v, out_dim, in_dim).astype(np.float64)
    lhs = y((0.5 * x + 2.0 * z).astype(np.float32))      # exact in f32 (power-of-2 scales)
    rhs = 0.5 * y(x) + 2.0 * y(z)
    scale = np.abs(W) @ (np.abs(x) + np.abs(z)).T
    assert np.all(np.abs(lhs - rhs) <= 4 * 2 ** -24 * scale.T)


def test_rmsnorm_constant_closed_form(orc):
    for c, eps in [(0.01, 1e-6), (3.0, 1e-6), (-0.2, 1e-5)]:
        n, n_pad = 896, 1024
        x = np.zeros((1, n_pad), np.float32)
        x[0, :n] = c
        y = orc.rmsnorm(x, np.ones(n, np.float32), n, n_pad, eps)
        expect = np.float32(np.float32(c) / np.sqrt(np.float64(np.float32(c)) ** 2 + np.float32(eps)))
        assert np.allclose(y[0, :n], expect, rtol=2 ** -23, atol=0)
        assert not y[0, n:].any()


def test_rmsnorm_unit_rms_and_gamma(orc):
    x = S.hidden_input("pin.rms.x", 3, 896, 1024) * 7.0
    gam = S.uniform("pin.rms.g", 896, 0.5, 1.5)
    y = orc.rmsnorm(x, gam, 896, 1024, 0.0).astype(np.float64)
    rms = np.sqrt(np.mean((y[:, :896] / gam) ** 2, axis=1))
    assert np.allclose(rms, 1.0, rtol=1e-6)
    y2 = orc.rmsnorm(x * 0.25, gam, 896, 1024, 0.0)     # scale invariance at eps = 0
    assert np.allclose(y2, y, rtol=1e-6, atol=1e-7)


def test_silu_identities(orc):
    assert orc.silu(0.0) == 0.0
    for v in [0.1, 1.0, 3.3, 12.0]:
        assert abs((orc.silu(v) - orc.silu(-v)) - v) < 1e-14 * max(1, v)
    assert abs(orc.silu(40.0) - 40.0) < 1e-14 * 40
    assert abs(orc.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_invariants(orc, mode):
    hd, H = 64, 3
    v = S.normal(f"pin.rope.v{mode}", H * hd)
    assert np.array_equal(orc.rope(v, H, hd, 0, 1e4, mode), v)          # position 0
    r = orc.rope(v, H, hd, 37, 1e4, mode).astype(np.float64)
    assert np.allclose(np.linalg.norm(r.reshape(H, hd), axis=1),
                       np.linalg.norm(v.reshape(H, hd).astype(np.float64), axis=1), rtol=1e-6)
    # group property: rope(rope(v, 20), 17) = rope(v, 37)
    rr = orc.rope(orc.rope(v, H, hd, 20, 1e4, mode), H, hd, 17, 1e4, mode)
    assert np.allclose(rr, r, atol=1e-5)
    # relative position: <rope(q,p), rope(k,p')> depends on p - p' only
    q = S.normal(f"pin.rope.q{mode}", hd)
    k = S.normal(f"pin.rope.k{mode}", hd)
    a = np.dot(orc.rope(q, 1, hd, 50, 1e4, mode), orc.rope(k, 1, hd, 45, 1e4, mode))
    b = np.dot(orc.rope(q, 1, hd, 1005, 1e4, mode), orc.rope(k, 1, hd, 1000, 1e4, mode))
    assert abs(a - b) < 1e-4 * (1 + abs(a))


def test_rope_pairing_and_frequency_closed_form(orc):
    hd = 8
    p = 3
    theta = 1e4
    for mode, partner in [(0, {0: 1, 2: 3, 4: 5, 6: 7}), (1, {0: 4, 1: 5, 2: 6, 3: 7})]:
        for i, (a, b) in enumerate(partner.items()):
            v = np.zeros(hd, np.float32)
            v[a] = 1.0
            r = orc.rope(v, 1, hd, p, theta, mode)
            ang = p * theta ** (-2.0 * i / hd)
            assert abs(r[a] - np.cos(ang)) < 1e-6 and abs(r[b] - np.sin(ang)) < 1e-6
            others = [j for j in range(hd) if j not in (a, b)]
            assert not r[others].any()


def test_attention_first_token_is_v_expanded(orc):
    """Position 0 (empty cache before the token): the output is v, each q head taking
    its kv head q_head / (n_heads / n_kv_heads)."""
    H, Hkv, hd = 8, 2, 16
    q = S.normal("pin.att0.q", H * hd)
    kc = S.normal("pin.att0.k", (4, Hkv * hd))
    vc = S.normal("pin.att0.v", (4, Hkv * hd))
    out = orc.attention(q, kc, vc, 0, H, Hkv, hd)
    for h in range(H):
        kvh = h // (H // Hkv)
        assert np.array_equal(out[h * hd:(h + 1) * hd], vc[0, kvh * hd:(kvh + 1) * hd])


def test_attention_brute_force_and_uniform(orc):
    H, Hkv, hd, pos = 4, 2, 8, 9
    q = S.normal("pin.att.q", H * hd)
    kc = S.normal("pin.att.k", (12, Hkv * hd))
    vc = S.normal("pin.att.v", (12, Hkv * hd))
    out = orc.attention(q, kc, vc, pos, H, Hkv, hd)
    for h in range(H):
        kvh = h // 2
        K = kc[:pos + 1, kvh * hd:(kvh + 1) * hd].astype(np.float64)
        V = vc[:pos + 1, kvh * hd:(kvh + 1) * hd].astype(np.float64)
        s = K @ q[h * hd:(h + 1) * hd].astype(np.float64) / np.sqrt(hd)
        p = np.exp(s - s.max())
        p /= p.sum()
        assert np.allclose(out[h * hd:(h + 1) * hd], p @ V, rtol=1e-6, atol=1e-6)
    # identical keys -> uniform weights -> mean of the values
    kc_same = np.repeat(kc[:1], 12, axis=0)
    out = orc.attention(q, kc_same, vc, pos, H, Hkv, hd)
    for h in range(H):
        kvh = h // 2
        assert np.allclose(out[h * hd:(h + 1) * hd],
                           vc[:pos + 1, kvh * hd:(kvh + 1) * hd].mean(axis=0), atol=1e-6)


def _tiny_shape():
    return S.LayerShape(hidden=448, inter=512, n_heads=7, n_kv_heads=1, head_dim=64,
                        rope_theta=1e6, rope_mode=1)


def _orc_layer(orc, L):
    sh = L.shape
    return orc.LayerWeights(**L.w, attn_gamma=L.attn_gamma, ffn_gamma=L.ffn_gamma,
                            hidden=sh.hidden, hidden_pad=sh.hidden_pad, n_heads=sh.n_heads,
                            n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim, inter=sh.inter,
                            eps=sh.eps, rope_theta=sh.rope_theta, rope_mode=sh.rope_mode)


def test_layer_zero_weights_is_identity(orc):
    sh = _tiny_shape()
    L = S.layer(sh, "pin.zero")
    for k in L.w:
        L.w[k] = np.zeros_like(L.w[k])        # d = dmin = 0: every weight is 0
    lw = _orc_layer(orc, L)
    x = S.hidden_input("pin.zero.x", 1, sh.hidden, sh.hidden_pad)[0]
    kc, vc = S.kv_prefill(sh, "pin.zero", 16, 5)
    out = orc.decode_layer(x, lw, kc[0], vc[0], 5)
    assert np.array_equal(out, x)
    assert not kc[0, 5].any() and not vc[0, 5].any()   # k = v = 0 written at pos


def test_ffn_zero_down_or_gate_is_identity(orc):
    sh = _tiny_shape()
    L = S.layer(sh, "pin.ffn0")
    x = S.hidden_input("pin.ffn0.x", 1, sh.hidden, sh.hidden_pad)[0]
    for zero in ("wdown", "wgate"):
        w = dict(L.w)
        w[zero] = np.zeros_like(w[zero])
        out = orc.swiglu_ffn(x, L.ffn_gamma, w["wgate"], w["wup"], w["wdown"],
                             sh.hidden, sh.hidden_pad, sh.inter, sh.eps)
        assert np.array_equal(out, x)


def test_layer_first_token_composition(orc):
    """At position 0 the layer equals: x + O(q8(v expanded)) followed by the FFN, with
    v = V(q8(norm x)) -- the first-token case of forward_single_full_cuda_with_cache."""
    sh = _tiny_shape()
    L = S.layer(sh, "pin.first")
    lw = _orc_layer(orc, L)
    x = S.hidden_input("pin.first.x", 1, sh.hidden, sh.hidden_pad)[0]
    kc, vc = S.kv_prefill(sh, "pin.first", 8, 0)
    out = orc.decode_layer(x, lw, kc[0], vc[0], 0)
    n = orc.rmsnorm(x, L.attn_gamma, sh.hidden, sh.hidden_pad, sh.eps)
    x8 = orc.q8_1_quantize(n)
    v = orc.q4k_q8_gemv(L.w["wv"], x8, 1, sh.kv_dim, sh.hidden_pad)[0]
    att = np.zeros(sh.q_pad, np.float32)
    for h in range(sh.n_heads):
        kvh = h // (sh.n_heads // sh.n_kv_heads)
        att[h * sh.head_dim:(h + 1) * sh.head_dim] = v[kvh * sh.head_dim:(kvh + 1) * sh.head_dim]
    o = orc.q4k_q8_gemv(L.w["wo"], orc.q8_1_quantize(att), 1, sh.hidden, sh.q_pad)[0]
    r1 = np.zeros(sh.hidden_pad, np.float32)
    r1[:sh.hidden] = x[:sh.hidden] + o
    expect = orc.swiglu_ffn(r1, L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"],
                            sh.hidden, sh.hidden_pad, sh.inter, sh.eps)
    assert np.array_equal(out, expect)
    assert np.array_equal(vc[0, 0], v)


def test_stack_zero_layers_is_norm_then_head(orc):
    hidden, hp, vocab = 896, 1024, 100
    x = S.hidden_input("pin.stack0.x", 1, hidden, hp)[0]
    g = S.uniform("pin.stack0.g", hidden, 0.5, 1.5)
    lm = S.q4_0_weight("pin.stack0.lm", vocab, hidden)
    hid, logits = orc.decode_stack(x, [], [], [], 0, g, lm, vocab, hidden, hp, 1e-6)
    assert np.array_equal(hid, x)
    n = orc.rmsnorm(x, g, hidden, hp, 1e-6)[0, :hidden]
    assert np.array_equal(logits, orc.q4_0_gemv(lm, n, vocab, hidden)[0])


def test_ffn_gates_with_silu_of_gate_times_up(orc):
    """cuda_swiglu_ffn: SiLU is applied to the gate projection, then multiplied by up;
    both read the same quantised normed input; h is quantised again before down."""
    sh = _tiny_shape()
    L = S.layer(sh, "pin.ffnorder")
    x = S.hidden_input("pin.ffnorder.x", 1, sh.hidden, sh.hidden_pad)[0]
    out = orc.swiglu_ffn(x, L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"],
                         sh.hidden, sh.hidden_pad, sh.inter, sh.eps)
    x8 = orc.q8_1_quantize(orc.rmsnorm(x, L.ffn_gamma, sh.hidden, sh.hidden_pad, sh.eps))
    g = orc.q4k_q8_gemv(L.w["wgate"], x8, 1, sh.inter, sh.hidden_pad)[0].astype(np.float64)
    u = orc.q4k_q8_gemv(L.w["wup"], x8, 1, sh.inter, sh.hidden_pad)[0].astype(np.float64)
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    dn = orc.q4k_q8_gemv(L.w["wdown"], orc.q8_1_quantize(h), 1, sh.hidden, sh.inter)[0]
    assert np.allclose(out[:sh.hidden], x[:sh.hidden] + dn, rtol=0, atol=1e-6 * np.abs(dn).max())
    h_swapped = (u / (1.0 + np.exp(-u)) * g).astype(np.float32)
    dn_sw = orc.q4k_q8_gemv(L.w["wdown"], orc.q8_1_quantize(h_swapped), 1, sh.hidden, sh.inter)[0]
    assert np.abs(dn_sw - dn).max() > 1e-2 * np.abs(dn).max()


# ----------------------------------------------------------------------------- layer at position >= 1
def _k_of_layer(orc, L, x):
    """The new token's un-rotated key: K GEMV of the Q8_1 of the normed input."""
    sh = L.shape
    x8 = orc.q8_1_quantize(orc.rmsnorm(x, L.attn_gamma, sh.hidden, sh.hidden_pad, sh.eps))
    k = orc.q4k_q8_gemv(L.w["wk"], x8, 1, sh.kv_dim, sh.hidden_pad)[0]
    v = orc.q4k_q8_gemv(L.w["wv"], x8, 1, sh.kv_dim, sh.hidden_pad)[0]
    return k, v


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_writes_key_rotated_at_its_position(orc, mode):
    """forward_single_full_cuda_with_cache rotates the new token's k by RoPE at the
    token's position before it joins the cache: row pos of K holds rope(k, pos), row
    pos of V the plain v, and no other row changes."""
    sh = S.LayerShape(hidden=448, inter=512, n_heads=7, n_kv_heads=1, head_dim=64,
                      rope_theta=1e4, rope_mode=mode)
    L = S.layer(sh, f"pin.krow.{mode}")
    lw = _orc_layer(orc, L)
    x = S.hidden_input(f"pin.krow.x.{mode}", 1, sh.hidden, sh.hidden_pad)[0]
    pos = 9
    kc, vc = S.kv_prefill(sh, f"pin.krow.{mode}", 16, pos)
    k0, v0 = kc[0].copy(), vc[0].copy()
    orc.decode_layer(x, lw, kc[0], vc[0], pos)
    k, v = _k_of_layer(orc, L, x)
    assert np.array_equal(kc[0, pos], orc.rope(k, sh.n_kv_heads, sh.head_dim, pos, sh.rope_theta, mode))
    assert np.array_equal(vc[0, pos], v)
    others = np.arange(16) != pos
    assert np.array_equal(kc[0][others], k0[others]) and np.array_equal(vc[0][others], v0[others])
    # the rotation is not the identity here, nor the one of a neighbouring position
    for wrong in (k, orc.rope(k, sh.n_kv_heads, sh.head_dim, pos + 1, sh.rope_theta, mode),
                  orc.rope(k, sh.n_kv_heads, sh.head_dim, pos - 1, sh.rope_theta, mode)):
        assert np.abs(kc[0, pos] - wrong).max() > 1e-3 * np.abs(k).max()


def test_layer_uniform_attention_when_every_key_equals_the_new_one(orc):
    """Position 6 with every earlier K row equal to the new token's rotated key:
    all scores are the same number, the softmax is uniform and the attention output
    is the plain mean of V rows 0..6 (the new token's v included).  The layer then
    equals x + O(q8(mean v)) followed by the FFN, bit for bit."""
    sh = _tiny_shape()
    L = S.layer(sh, "pin.uni")
    lw = _orc_layer(orc, L)
    x = S.hidden_input("pin.uni.x", 1, sh.hidden, sh.hidden_pad)[0]
    pos = 6
    k, v = _k_of_layer(orc, L, x)
    kr = orc.rope(k, sh.n_kv_heads, sh.head_dim, pos, sh.rope_theta, sh.rope_mode)
    kc, vc = S.kv_prefill(sh, "pin.uni", 8, pos)
    kc[0, :pos] = kr
    out = orc.decode_layer(x, lw, kc[0], vc[0], pos)
    mean = [0.0] * sh.kv_dim
    for t in range(pos + 1):               # sequential f64 sum, rows in order
        row = vc[0, t]
        mean = [a + float(b) for a, b in zip(mean, row)]
    mean = np.array(mean) / (pos + 1)
    att = np.zeros(sh.q_pad, np.float32)
    for h in range(sh.n_heads):
        kvh = h // (sh.n_heads // sh.n_kv_heads)
        att[h * sh.head_dim:(h + 1) * sh.head_dim] = mean[kvh * sh.head_dim:(kvh + 1) * sh.head_dim]
    o = orc.q4k_q8_gemv(L.w["wo"], orc.q8_1_quantize(att), 1, sh.hidden, sh.q_pad)[0]
    r1 = np.zeros(sh.hidden_pad, np.float32)
    r1[:sh.hidden] = x[:sh.hidden] + o
    expect = orc.swiglu_ffn(r1, L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"],
                            sh.hidden, sh.hidden_pad, sh.inter, sh.eps)
    assert np.array_equal(out, expect)


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_query_rotated_at_its_position(orc, mode):
    """With W_q = W_k (so q = k before RoPE) and earlier K rows rope(k, j), the score
    of row j is k . R((j - pos) theta) k / sqrt(hd), which depends on |j - pos| only
    when the query is rotated at exactly `pos`.  Mirroring the rows about pos
    (rope(k, 2 pos - j) in place of rope(k, j)) must then leave the layer output
    unchanged up to f32 rounding, and mirroring about pos + 1 must not."""
    sh = S.LayerShape(hidden=512, inter=512, n_heads=4, n_kv_heads=4, head_dim=64,
                      rope_theta=1e4, rope_mode=mode)
    L = S.layer(sh, f"pin.qpos.{mode}")
    L.w["wq"] = L.w["wk"].copy()
    L.attn_gamma = np.full(sh.hidden, 0.01, np.float32)   # moderate scores: a soft softmax
    lw = _orc_layer(orc, L)
    x = S.hidden_input(f"pin.qpos.x.{mode}", 1, sh.hidden, sh.hidden_pad)[0]
    pos = 4
    k, _ = _k_of_layer(orc, L, x)
    rot = lambda p: orc.rope(k, sh.n_kv_heads, sh.head_dim, p, sh.rope_theta, mode)

    def run(center2):
        kc, vc = S.kv_prefill(sh, f"pin.qpos.{mode}", 8, pos)
        for j in range(pos):
            kc[0, j] = rot(center2 - j)
        return orc.decode_layer(x, lw, kc[0], vc[0], pos).astype(np.float64)

    kc, vc = S.kv_prefill(sh, f"pin.qpos.{mode}", 8, pos)
    for j in range(pos):
        kc[0, j] = rot(j)
    base = orc.decode_layer(x, lw, kc[0], vc[0], pos).astype(np.float64)
    mirrored = run(2 * pos)
    shifted = run(2 * (pos + 1))
    scale = np.abs(base).max()
    assert np.abs(mirrored - base).max() <= 1e-3 * scale
    assert np.abs(shifted - base).max() > 1e-2 * scale


# ----------------------------------------------------------------------------- projection biases
def test_zero_bias_is_no_bias(orc):
    sh = _tiny_shape()
    L = S.layer(sh, "pin.bias0")
    x = S.hidden_input("pin.bias0.x", 1, sh.hidden, sh.hidden_pad)[0]
    kc, vc = S.kv_prefill(sh, "pin.bias0", 8, 3)
    ref = orc.decode_layer(x, _orc_layer(orc, L), kc[0].copy(), vc[0].copy(), 3)
    lw = _orc_layer(orc, L)
    lw.bq = np.zeros(sh.q_dim, np.float32)
    lw.bk = np.zeros(sh.kv_dim, np.float32)
    lw.bv = np.zeros(sh.kv_dim, np.float32)
    assert np.array_equal(orc.decode_layer(x, lw, kc[0].copy(), vc[0].copy(), 3), ref)


def test_bias_on_zero_projections_is_the_bias(orc):
    """With W_q = W_k = W_v = 0 the projections are the biases themselves: the cache
    row at pos holds bv and rope(bk, pos), and the attention of a first token is bv
    expanded over the query heads."""
    sh = _tiny_shape()
    L = S.layer(sh, "pin.bias1")
    for k in ("wq", "wk", "wv"):
        L.w[k] = np.zeros_like(L.w[k])
    lw = _orc_layer(orc, L)
    lw.bq = S.normal("pin.bias1.bq", sh.q_dim)
    lw.bk = S.normal("pin.bias1.bk", sh.kv_dim)
    lw.bv = S.normal("pin.bias1.bv", sh.kv_dim)
    x = S.hidden_input("pin.bias1.x", 1, sh.hidden, sh.hidden_pad)[0]
    pos = 5
    kc, vc = S.kv_prefill(sh, "pin.bias1", 8, pos)
    orc.decode_layer(x, lw, kc[0], vc[0], pos)
    assert np.array_equal(vc[0, pos], lw.bv)
    assert np.array_equal(kc[0, pos], orc.rope(lw.bk, sh.n_kv_heads, sh.head_dim, pos, sh.rope_theta,
                                               sh.rope_mode))
    # first token: output = x + O(q8(bv expanded)) then the FFN
    kc0, vc0 = S.kv_prefill(sh, "pin.bias1b", 4, 0)
    out = orc.decode_layer(x, lw, kc0[0], vc0[0], 0)
    att = np.zeros(sh.q_pad, np.float32)
    for h in range(sh.n_heads):
        kvh = h // (sh.n_heads // sh.n_kv_heads)
        att[h * sh.head_dim:(h + 1) * sh.head_dim] = lw.bv[kvh * sh.head_dim:(kvh + 1) * sh.head_dim]
    o = orc.q4k_q8_gemv(L.w["wo"], orc.q8_1_quantize(att), 1, sh.hidden, sh.q_pad)[0]
    r1 = np.zeros(sh.hidden_pad, np.float32)
    r1[:sh.hidden] = x[:sh.hidden] + o
    expect = orc.swiglu_ffn(r1, L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"],
                            sh.hidden, sh.hidden_pad, sh.inter, sh.eps)
    assert np.array_equal(out, expect)


# ----------------------------------------------------------------------------- Q4_K x f32
def test_q4k_f32_gemv_exact_integers(orc):
    """d = 1, dmin = 0, integer activations: y = sum_j sc_j sum_k q_k x_k exactly."""
    g = np.random.default_rng(7)
    nsb, rows = 2, 5
    w = np.zeros((rows, nsb * 144), np.uint8)
    expect = np.zeros(rows, np.int64)
    x = g.integers(-50, 51, 256 * nsb).astype(np.float32)
    for r in range(rows):
        for b in range(nsb):
            sc = g.integers(0, 64, 8).astype(np.uint8)
            q = g.integers(0, 16, 256).astype(np.uint8)
            w[r, b * 144:(b + 1) * 144] = orc.q4k_pack(0x3C00, 0, sc, np.zeros(8, np.uint8), q)
            xi = x[b * 256:(b + 1) * 256].astype(np.int64).reshape(8, 32)
            expect[r] += int((sc.astype(np.int64) * (q.astype(np.int64).reshape(8, 32) * xi).sum(1)).sum())
    y = orc.q4k_f32_gemv(w, x, rows, 256 * nsb)[0]
    assert np.array_equal(y, expect.astype(np.float32))


def test_q4k_f32_gemv_min_term_alone(orc):
    """All codes zero: every weight is -dmin m_j, so y = -sum_b dmin_b sum_j m_j (sum of
    sub-block j of x), the min term and nothing else."""
    g = np.random.default_rng(8)
    rows, nsb = 4, 3
    w = np.zeros((rows, nsb * 144), np.uint8)
    x = g.standard_normal(256 * nsb).astype(np.float32)
    expect = np.zeros(rows)
    for r in range(rows):
        for b in range(nsb):
            mn = g.integers(0, 64, 8).astype(np.uint8)
            dmin = np.float16(g.uniform(1e-3, 1e-2))
            w[r, b * 144:(b + 1) * 144] = orc.q4k_pack(0x3C00, dmin.view(np.uint16), g.integers(0, 64, 8),
                                                     mn, np.zeros(256, np.uint8))
            xs = x[b * 256:(b + 1) * 256].astype(np.float64).reshape(8, 32).sum(1)
            expect[r] -= float(dmin) * (mn.astype(np.float64) * xs).sum()
    y = orc.q4k_f32_gemv(w, x, rows, 256 * nsb)[0]
    assert np.allclose(y, expect, rtol=1e-6, atol=1e-9)


def test_q4k_f32_gemv_close_to_q8_1_path(orc):
    """The Q8_1 path differs only by the activation rounding: |y_f32 - y_q8| <=
    sum_k |w_k| d8_k / 2 (each code is within half a step of x / d8), per row."""
    rows, in_dim = 64, 1024
    w = S.q4k_weight("pin.f32vq8", rows, in_dim)
    x = S.normal("pin.f32vq8.x", (1, in_dim))
    x8 = orc.q8_1_quantize(x)
    yf = orc.q4k_f32_gemv(w, x, rows, in_dim)[0].astype(np.float64)
    yq = orc.q4k_q8_gemv(w, x8, 1, rows, in_dim)[0].astype(np.float64)
    d8, _, _ = orc.q8_1_fields(x8, 1, in_dim)
    wd = orc.q4k_dequantize(w)
    bound = (np.abs(wd) * np.repeat(d8[0], 32)[None, :] / 2).sum(1) + 1e-5 * np.abs(yf)
    assert (np.abs(yf - yq) <= bound).all()
    assert np.abs(yf - yq).max() > 0   # the two paths are not the same computation


# ----------------------------------------------------------------------------- Q4_0 whole-model layer
def test_gelu_identities(orc):
    """GELU (tanh form): gelu(0) = 0; the odd part is x/2, so gelu(x) - gelu(-x) = x;
    gelu(x) -> x for large x and -> 0 for large negative x."""
    assert orc.gelu(0.0) == 0.0
    for x in (0.1, 0.5, 1.0, 2.5, 7.0):
        assert abs(orc.gelu(x) - orc.gelu(-x) - x) < 1e-14 * max(1.0, x)
    assert abs(orc.gelu(12.0) - 12.0) < 1e-12 and abs(orc.gelu(-12.0)) < 1e-12
    # between x * sigmoid(1.5 x) - 0.02 and x (a crude bracket that a wrong constant breaks)
    for x in (0.3, 1.0, 2.0):
        assert x / (1 + np.exp(-1.5 * x)) - 0.03 < orc.gelu(x) < x


def _q40_tiny(gated):
    return S.Q40Shape(hidden=256, inter=384, n_heads=4, n_kv_heads=2, head_dim=64, rope_theta=1e4,
                      rope_mode=0, gated=gated)


def _orc_q40(orc, sh, w):
    return orc.LayerWeightsQ40(wqkv=w["wqkv"], wo=w["wo"], wgate=w.get("wgate"), wup=w["wup"], wdown=w["wdown"],
                               attn_gamma=w["attn_gamma"], ffn_gamma=w["ffn_gamma"], hidden=sh.hidden,
                               n_heads=sh.n_heads, n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim,
                               inter=sh.inter, eps=sh.eps, rope_theta=sh.rope_theta, rope_mode=sh.rope_mode)


@pytest.mark.parametrize("gated", [False, True])
def test_q4_0_layer_zero_weights_is_identity(orc, gated):
    sh = _q40_tiny(gated)
    w = S.layer_q4_0(sh, f"pin.q40z.{gated}")
    for k in sh.weight_shapes():
        w[k] = np.zeros_like(w[k])
    x = S.normal(f"pin.q40z.x.{gated}", sh.hidden)
    kc = S.normal("pin.q40z.k", (8, sh.kv_dim))
    vc = S.normal("pin.q40z.v", (8, sh.kv_dim))
    out = orc.decode_layer_q4_0(x, _orc_q40(orc, sh, w), kc, vc, 5)
    assert np.array_equal(out, x)
    assert not kc[5].any() and not vc[5].any()


@pytest.mark.parametrize("gated", [False, True])
def test_q4_0_layer_first_token_composition(orc, gated):
    """Position 0: the layer is x + O(v expanded) followed by the FFN of the page:
    silu(gate) * up then down (ffn_swiglu_gpu) or GELU(up) then down
    (ffn_standard_gpu), every step an f32 buffer."""
    sh = _q40_tiny(gated)
    w = S.layer_q4_0(sh, f"pin.q40f.{gated}")
    x = S.normal(f"pin.q40f.x.{gated}", sh.hidden)
    kc = np.zeros((4, sh.kv_dim), np.float32)
    vc = np.zeros_like(kc)
    out = orc.decode_layer_q4_0(x, _orc_q40(orc, sh, w), kc, vc, 0)
    n = orc.rmsnorm(x, w["attn_gamma"], sh.hidden, sh.hidden, sh.eps)[0]
    qkv = orc.q4_0_gemv(w["wqkv"], n, sh.q_dim + 2 * sh.kv_dim, sh.hidden)[0]
    v = qkv[sh.q_dim + sh.kv_dim:]
    att = np.concatenate([v[(h // (sh.n_heads // sh.n_kv_heads)) * sh.head_dim:][:sh.head_dim]
                          for h in range(sh.n_heads)])
    r1 = orc.residual_add(x, orc.q4_0_gemv(w["wo"], att, sh.hidden, sh.q_dim)[0])
    n2 = orc.rmsnorm(r1, w["ffn_gamma"], sh.hidden, sh.hidden, sh.eps)[0]
    u = orc.q4_0_gemv(w["wup"], n2, sh.inter, sh.hidden)[0].astype(np.float64)
    if gated:
        g = orc.q4_0_gemv(w["wgate"], n2, sh.inter, sh.hidden)[0].astype(np.float64)
        h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    else:
        h = np.array([orc.gelu(t) for t in u], np.float32)
    expect = orc.residual_add(r1, orc.q4_0_gemv(w["wdown"], h, sh.hidden, sh.inter)[0])
    assert np.allclose(out, expect, rtol=0, atol=1e-6 * np.abs(expect).max())
    assert np.array_equal(vc[0], v)
