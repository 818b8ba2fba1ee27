"""GPU parity of the composite steps: attention, SwiGLU FFN, decode layer, stack.

Bars.  Attention (f32 in, f32 out): |gpu - oracle| <= 1e-5 |ref| + 1e-5 max|ref|;
the cache row written bit-exact for v and within 1e-6 relative for the rotated k;
the attention output's Q8_1 bit-exact against the oracle's quantisation of the
GPU's own f32 output.  Composite outputs that pass through Q8_1 re-quantisation
of values the GPU computes in f32 (FFN, layer, stack): within 1e-3 relative, as
max|gpu - ref| <= 1e-3 max|ref| and ||gpu - ref||_2 <= 1e-3 ||ref||_2.
"""
import numpy as np
import pytest

import oracle
import rz_synth as S

from conftest import ELEMENTWISE_REPORT
from gpu_common import check_no_device_error, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    return rz


def assert_rel(gpu, ref, tol=1e-3, what=""):
    """max|gpu - ref| <= tol max|ref| and ||gpu - ref||_2 <= tol ||ref||_2; the worst
    element-wise relative error over the elements with |ref| > 1e-2 max|ref| is
    recorded for the run's summary (a systematic bias on small outputs shows there)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    dmax = np.abs(gpu - ref).max()
    d2 = np.linalg.norm(gpu - ref)
    big = np.abs(ref) > 1e-2 * np.abs(ref).max()
    ew = float((np.abs(gpu - ref)[big] / np.abs(ref)[big]).max()) if big.any() else 0.0
    ELEMENTWISE_REPORT.append((what, ew, float(dmax / max(np.abs(ref).max(), 1e-30))))
    assert dmax <= tol * np.abs(ref).max(), f"{what}: max err {dmax:.3e} vs {tol} * {np.abs(ref).max():.3e}"
    assert d2 <= tol * np.linalg.norm(ref), f"{what}: l2 err {d2:.3e} vs {tol} * {np.linalg.norm(ref):.3e}"
    return dmax / np.abs(ref).max()


def dev_layer(rz, L):
    sh = L.shape
    w = {k: to_dev(v) for k, v in L.w.items()}
    w["attn_gamma"] = to_dev(L.attn_gamma)
    w["ffn_gamma"] = to_dev(L.ffn_gamma)
    return rz.DeviceLayer(w, sh.hidden, sh.hidden_pad, sh.n_heads, sh.n_kv_heads, sh.head_dim,
                          sh.inter, sh.eps, sh.rope_theta, sh.rope_mode)


def orc_layer(L):
    sh = L.shape
    return oracle.LayerWeights(**L.w, attn_gamma=L.attn_gamma, ffn_gamma=L.ffn_gamma,
                               hidden=sh.hidden, hidden_pad=sh.hidden_pad, n_heads=sh.n_heads,
                               n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim, inter=sh.inter,
                               eps=sh.eps, rope_theta=sh.rope_theta, rope_mode=sh.rope_mode)


# ----------------------------------------------------------------------------- attention
ATT_CASES = [
    # n_heads, n_kv_heads, head_dim, theta, mode, max_seq, positions
    (14, 2, 64, 1e6, 1, 160, [127]),
    (14, 2, 64, 1e6, 1, 160, [0]),
    (8, 8, 128, 1e4, 0, 300, [257]),
    (4, 1, 32, 1e4, 0, 50, [49]),
    (8, 2, 64, 1e4, 1, 2056, [2048]),
    (8, 4, 64, 1e4, 0, 100, [5, 0, 99]),
    # more (head, chunk) units than resident CTAs: two K/V buffers, several chunks
    # streamed per CTA
    (32, 32, 128, 1e4, 0, 2056, [2000]),
    # 63 chunk records per head exceed one buffer: two buffers
    (8, 8, 128, 1e4, 0, 4096, [4000]),
    # the Llama-7B head layout with several tokens at distinct positions
    (32, 32, 128, 1e4, 0, 1100, [1024, 3, 517, 0]),
    (32, 32, 128, 1e4, 0, 300, [5, 299, 64, 65, 0, 128, 200, 1, 7, 250, 33, 190, 2, 299, 100, 63]),
    # dispatch: more (token, kv head) segments than SMs (the flat tiled kernel);
    # two tokens in clusters of CTAs per segment; 16 query heads per kv head and
    # head_dim 256 (the chunk kernel)
    (32, 32, 128, 1e4, 0, 200, [5, 199, 64, 0, 100, 150]),
    (16, 16, 128, 1e4, 0, 700, [650, 11]),
    (32, 2, 64, 1e4, 1, 600, [555]),
    (4, 2, 256, 1e4, 0, 300, [200]),
]


@pytest.mark.parametrize("H,Hkv,hd,theta,mode,max_seq,positions", ATT_CASES)
def test_attention_decode_parity(rz, H, Hkv, hd, theta, mode, max_seq, positions):
    import torch
    m = len(positions)
    kv_dim, q_dim = Hkv * hd, H * hd
    sh = S.LayerShape(hidden=q_dim, inter=256, n_heads=H, n_kv_heads=Hkv, head_dim=hd,
                      rope_theta=theta, rope_mode=mode)
    kc, vc = S.kv_prefill(sh, f"gatt.{H}.{hd}.{m}", max_seq, max(positions), m)
    kc *= np.float32(0.5)
    q = S.normal(f"gatt.q.{H}.{hd}.{m}", (m, q_dim)) * np.float32(0.7)
    k = S.normal(f"gatt.k.{H}.{hd}.{m}", (m, kv_dim)) * np.float32(0.7)
    v = S.normal(f"gatt.v.{H}.{hd}.{m}", (m, kv_dim))
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    pos_d = to_dev(np.array(positions, np.int32)) if m > 1 else None
    qkv = to_dev(np.concatenate([q, k, v], axis=1))      # one row per token: q | k | v
    ld = q_dim + 2 * kv_dim
    att, a8 = rz.attention_decode(qkv, qkv[:, q_dim:], qkv[:, q_dim + kv_dim:], ld, kv, H, Hkv, hd,
                                  theta, mode, position=positions[0], positions=pos_d)
    att = att.cpu().numpy()
    a8 = a8.cpu().numpy()
    check_no_device_error()
    kc_after = kv.k.cpu().numpy()
    vc_after = kv.v.cpu().numpy()
    q_pad = (q_dim + 255) // 256 * 256
    for t, p in enumerate(positions):
        qr = oracle.rope(q[t], H, hd, p, theta, mode)
        kr = oracle.rope(k[t], Hkv, hd, p, theta, mode)
        assert np.array_equal(vc_after[t, p], v[t])
        assert np.allclose(kc_after[t, p], kr, rtol=1e-6, atol=1e-6 * np.abs(kr).max())
        kct = kc[t].copy()
        vct = vc[t].copy()
        kct[p] = kr
        vct[p] = v[t]
        ref = oracle.attention(qr, kct, vct, p, H, Hkv, hd).astype(np.float64)
        err = np.abs(att[t] - ref)
        assert np.all(err <= 1e-5 * np.abs(ref) + 1e-5 * np.abs(ref).max()), (t, err.max())
    # the fused Q8_1 of the output is exactly the format applied to the f32 output
    padded = np.zeros((m, q_pad), np.float32)
    padded[:, :q_dim] = att
    assert np.array_equal(a8, oracle.q8_1_quantize(padded))
    # the other cache rows are untouched
    for t, p in enumerate(positions):
        mask = np.ones(max_seq, bool)
        mask[p] = False
        assert np.array_equal(kc_after[t][mask], kc[t][mask])


def test_results_identical_without_pdl(rz):
    """Programmatic dependent launch changes only when kernels may start: a Qwen2
    layer (the cluster attention kernel) and 6-token attention over 32 kv heads
    (192 segments: the flat kernel) give the same bits with it switched off."""
    sh = S.QWEN2
    L = S.layer(sh, "pdl.l")
    dl = dev_layer(rz, L)
    x = to_dev(S.hidden_input("pdl.x", 1, sh.hidden, sh.hidden_pad))
    kc, vc = S.kv_prefill(sh, "pdl.kv", 160, 77)
    H, Hkv, hd, max_seq = 32, 32, 128, 200
    positions = [5, 199, 64, 0, 100, 150]
    ash = S.LayerShape(hidden=H * hd, inter=256, n_heads=H, n_kv_heads=Hkv, head_dim=hd, rope_theta=1e4,
                       rope_mode=0)
    akc, avc = S.kv_prefill(ash, "pdl.att", max_seq, max(positions), len(positions))
    qkv = to_dev(S.normal("pdl.qkv", (len(positions), (H + 2 * Hkv) * hd)))
    pos_d = to_dev(np.array(positions, np.int32))
    runs = []
    try:
        for pdl in (True, False):
            rz.set_pdl(pdl)
            kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
            out = rz.decode_layer(x, dl, kv, position=77).cpu().numpy()
            akv = rz.DeviceKV(to_dev(akc), to_dev(avc))
            att, a8 = rz.attention_decode(qkv, qkv[:, H * hd:], qkv[:, (H + Hkv) * hd:], (H + 2 * Hkv) * hd, akv,
                                          H, Hkv, hd, 1e4, 0, positions=pos_d)
            check_no_device_error()
            runs.append((out, kv.k.cpu().numpy(), att.cpu().numpy(), a8.cpu().numpy(), akv.k.cpu().numpy()))
    finally:
        rz.set_pdl(True)
    for a, b in zip(*runs):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_attention_first_token_is_v(rz):
    """Position 0: every query head returns the value of its kv head (the first-token
    case of forward_single_full_cuda_with_cache), to f32 rounding of the weights."""
    H, Hkv, hd = 14, 2, 64
    kc = np.zeros((1, 8, Hkv * hd), np.float32)
    vc = np.zeros_like(kc)
    q = S.normal("gfirst.q", (1, H * hd))
    k = S.normal("gfirst.k", (1, Hkv * hd))
    v = S.normal("gfirst.v", (1, Hkv * hd))
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    att, _ = rz.attention_decode(to_dev(q), to_dev(k), to_dev(v), H * hd, kv, H, Hkv, hd, 1e6, 1,
                                 position=0)
    att = att.cpu().numpy()[0]
    for h in range(H):
        kvh = h // (H // Hkv)
        assert np.array_equal(att[h * hd:(h + 1) * hd], v[0, kvh * hd:(kvh + 1) * hd])


def test_attention_bad_device_position_is_reported(rz):
    """A device-resident position outside the cache is caught in the kernel: the
    error word reports it, the cache is not written, the output is zeros."""
    H, Hkv, hd, max_seq = 4, 2, 32, 16
    kc = S.normal("gbad.k", (2, max_seq, Hkv * hd))
    vc = S.normal("gbad.v", (2, max_seq, Hkv * hd))
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    qkv = to_dev(S.normal("gbad.qkv", (2, H * hd + 2 * Hkv * hd)))
    ld = H * hd + 2 * Hkv * hd
    pos = to_dev(np.array([3, max_seq + 5], np.int32))
    att, _ = rz.attention_decode(qkv, qkv[:, H * hd:], qkv[:, H * hd + Hkv * hd:], ld, kv, H, Hkv, hd,
                                 1e4, 0, positions=pos)
    st, code = rz.check_device_error()
    assert st == 7 and code == 0x201
    assert np.array_equal(kv.k.cpu().numpy()[1], kc[1])
    assert not att.cpu().numpy()[1].any()
    check_no_device_error()   # the word was cleared


# ----------------------------------------------------------------------------- SwiGLU FFN
# wide gate/up (9984 rows) and wide down (9984 rows): the multi-token row-pair
# path with the SwiGLU and the residual epilogues
WIDE_INTER = S.LayerShape(hidden=512, inter=9984, n_heads=8, n_kv_heads=8, head_dim=64,
                          rope_theta=1e4, rope_mode=0)
WIDE_HIDDEN = S.LayerShape(hidden=9984, inter=512, n_heads=8, n_kv_heads=8, head_dim=64,
                           rope_theta=1e4, rope_mode=0)


# (LLAMA7B, 16): the activations of down (16 x 11008) exceed shared memory, so
# down runs as token groups, each with its slice of the residual
@pytest.mark.parametrize("shape,m", [(S.QWEN2, 1), (S.QWEN2, 3), (S.LLAMA7B, 1), (S.LLAMA7B, 2),
                                     (S.LLAMA7B, 16), (WIDE_INTER, 5), (WIDE_HIDDEN, 3)])
def test_swiglu_ffn_parity(rz, shape, m):
    L = S.layer(shape, f"gffn.{shape.hidden}")
    x = S.hidden_input(f"gffn.x.{shape.hidden}.{m}", m, shape.hidden, shape.hidden_pad)
    out = rz.swiglu_ffn(to_dev(x), to_dev(L.ffn_gamma), to_dev(L.w["wgate"]), to_dev(L.w["wup"]),
                        to_dev(L.w["wdown"]), shape.hidden, shape.hidden_pad, shape.inter,
                        shape.eps).cpu().numpy()
    check_no_device_error()
    for t in range(m):
        ref = oracle.swiglu_ffn(x[t], L.ffn_gamma, L.w["wgate"], L.w["wup"], L.w["wdown"],
                                shape.hidden, shape.hidden_pad, shape.inter, shape.eps)
        assert_rel(out[t], ref, what=f"ffn token {t}")
        assert not out[t, shape.hidden:].any()


# ----------------------------------------------------------------------------- decode layer
@pytest.mark.parametrize("pos", [127, 0])
def test_decode_layer_qwen2_parity(rz, pos):
    """The Qwen2-0.5B-shaped layer at position 127 (and the first token)."""
    sh = S.QWEN2
    L = S.layer(sh, "qwen2.l0")
    max_seq = 160
    x = S.hidden_input("qwen2.x", 1, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, "qwen2.kv", max_seq, pos)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    out = rz.decode_layer(to_dev(x), dev_layer(rz, L), kv, position=pos).cpu().numpy()
    check_no_device_error()
    kc_r, vc_r = kc[0].copy(), vc[0].copy()
    ref = oracle.decode_layer(x[0], orc_layer(L), kc_r, vc_r, pos)
    assert_rel(out[0], ref, what="qwen2 layer")
    assert not out[0, sh.hidden:].any()
    assert_rel(kv.k.cpu().numpy()[0, pos], kc_r[pos], tol=1e-4, what="k row")
    assert_rel(kv.v.cpu().numpy()[0, pos], vc_r[pos], tol=1e-4, what="v row")


def test_decode_layer_batched_positions(rz):
    """m = 4 sequences at different positions through one launch sequence; each
    matches the oracle run alone."""
    import torch
    sh = S.QWEN2
    L = S.layer(sh, "qwen2.b")
    positions = [5, 127, 0, 63]
    m, max_seq = len(positions), 128
    x = S.hidden_input("qwen2.bx", m, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, "qwen2.bkv", max_seq, max(positions), m)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    out = rz.decode_layer(to_dev(x), dev_layer(rz, L), kv,
                          positions=to_dev(np.array(positions, np.int32))).cpu().numpy()
    check_no_device_error()
    ol = orc_layer(L)
    for t, p in enumerate(positions):
        kt, vt = kc[t].copy(), vc[t].copy()
        ref = oracle.decode_layer(x[t], ol, kt, vt, p)
        assert_rel(out[t], ref, what=f"token {t} at {p}")


def test_decode_layer_llama_parity(rz):
    sh = S.LLAMA7B
    L = S.layer(sh, "llama.l0")
    pos, max_seq = 128, 256
    x = S.hidden_input("llama.x", 1, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, "llama.kv", max_seq, pos)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    out = rz.decode_layer(to_dev(x), dev_layer(rz, L), kv, position=pos).cpu().numpy()
    check_no_device_error()
    ref = oracle.decode_layer(x[0], orc_layer(L), kc[0].copy(), vc[0].copy(), pos)
    assert_rel(out[0], ref, what="llama layer")


def test_decode_layer_in_place(rz):
    import torch
    sh = S.QWEN2
    L = S.layer(sh, "qwen2.ip")
    x = S.hidden_input("qwen2.ipx", 1, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, "qwen2.ipkv", 64, 10)
    dl = dev_layer(rz, L)
    a = rz.decode_layer(to_dev(x), dl, rz.DeviceKV(to_dev(kc), to_dev(vc)), position=10).cpu().numpy()
    xd = to_dev(x)
    rz.decode_layer(xd, dl, rz.DeviceKV(to_dev(kc), to_dev(vc)), position=10, out=xd)
    assert np.array_equal(xd.cpu().numpy(), a)


# ----------------------------------------------------------------------------- stack
def test_decode_stack_qwen2_two_layers_and_lm_head(rz):
    """Two Qwen2-shaped layers, output norm and the 151936 x 896 Q4_0 LM head."""
    sh = S.QWEN2
    vocab = 151936
    layers = [S.layer(sh, f"qs.l{i}") for i in range(2)]
    out_gamma = S.uniform("qs.og", sh.hidden, 0.5, 1.5)
    lm = S.q4_0_weight("qs.lm", vocab, sh.hidden)
    pos, max_seq = 127, 128
    x = S.hidden_input("qs.x", 1, sh.hidden, sh.hidden_pad)
    kvs_h = [S.kv_prefill(sh, f"qs.kv{i}", max_seq, pos) for i in range(2)]
    kvs = [rz.DeviceKV(to_dev(k), to_dev(v)) for k, v in kvs_h]
    stack = rz.DeviceStack([dev_layer(rz, L) for L in layers], kvs, to_dev(out_gamma), to_dev(lm), vocab)
    hid, logits = rz.decode_stack(to_dev(x), stack, position=pos)
    hid = hid.cpu().numpy()
    logits = logits.cpu().numpy()
    check_no_device_error()
    hid_r, log_r = oracle.decode_stack(x[0], [orc_layer(L) for L in layers],
                                       [k[0].copy() for k, _ in kvs_h], [v[0].copy() for _, v in kvs_h],
                                       pos, out_gamma, lm, vocab)
    assert_rel(hid[0], hid_r, what="stack hidden")
    assert_rel(logits[0], log_r, what="stack logits")


def test_stack_as_first_call_in_a_fresh_process(rz, tmp_path):
    """A process whose first librz call is the layer-level entry point (no earlier
    kernel call) gets through the host-side shape checks."""
    import subprocess
    import sys
    code = r"""
import sys, numpy as np, torch
sys.path.insert(0, %r)
import quantized_q4_q8_gb300 as rz, rz_synth as S
sh = S.QWEN2
dev = torch.device("cuda:0")
w = S.layer_device(sh, "fresh", dev)
L = rz.DeviceLayer(w, sh.hidden, sh.hidden_pad, sh.n_heads, sh.n_kv_heads, sh.head_dim, sh.inter,
                   sh.eps, sh.rope_theta, sh.rope_mode)
kv = rz.DeviceKV(*S.kv_prefill_device(sh, "fresh.kv", 16, 3, 1, dev))
stack = rz.DeviceStack([L], [kv], torch.ones(sh.hidden, device=dev), S.q4_0_weight_device("fresh.lm", 64, sh.hidden, dev), 64)
x = torch.zeros((1, sh.hidden_pad), device=dev); x[:, :sh.hidden] = 1.0
hid, logits = rz.decode_stack(x, stack, position=3)
torch.cuda.synchronize()
assert torch.isfinite(logits).all()
print("fresh ok")
""" % (str(__import__("os").path.dirname(__import__("os").path.dirname(__file__))),)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stderr[-3000:]


# ----------------------------------------------------------------------------- Llama-shaped, several tokens
LLAMA_POSITIONS = {
    4: [1024, 3, 517, 0],
    16: [599, 0, 1, 63, 64, 65, 127, 128, 300, 511, 512, 513, 200, 17, 450, 598],
}


@pytest.mark.parametrize("m", [4, 16])
def test_decode_layer_llama_batched_parity(rz, m):
    """The Llama-7B-shaped layer (32/32 heads of 128, hidden 4096, inter 11008) for m
    sequences at distinct positions (the batched-decode configuration); each token
    matches the oracle run alone on its own cache."""
    sh = S.LLAMA7B
    L = S.layer(sh, "llama.bl")
    positions = LLAMA_POSITIONS[m]
    max_seq = max(positions) + 1
    x = S.hidden_input(f"llama.bx.{m}", m, sh.hidden, sh.hidden_pad)
    kc, vc = S.kv_prefill(sh, f"llama.bkv.{m}", max_seq, max(positions), m)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    out = rz.decode_layer(to_dev(x), dev_layer(rz, L), kv,
                          positions=to_dev(np.array(positions, np.int32))).cpu().numpy()
    check_no_device_error()
    kc_after = kv.k.cpu().numpy()
    ol = orc_layer(L)
    for t, p in enumerate(positions):
        kt, vt = kc[t].copy(), vc[t].copy()
        ref = oracle.decode_layer(x[t], ol, kt, vt, p)
        assert_rel(out[t], ref, what=f"llama layer m={m} token {t} at {p}")
        assert_rel(kc_after[t, p], kt[p], tol=1e-4, what=f"k row token {t}")


def _llama_stack(rz, tag, n_layers, max_seq, filled, m, vocab=S.LLAMA_VOCAB):
    sh = S.LLAMA7B
    layers = [S.layer(sh, f"{tag}.l{i}") for i in range(n_layers)]
    out_gamma = S.uniform(f"{tag}.og", sh.hidden, 0.5, 1.5)
    lm = S.q4_0_weight(f"{tag}.lm", vocab, sh.hidden)
    kvs_h = [S.kv_prefill(sh, f"{tag}.kv{i}", max_seq, filled, m) for i in range(n_layers)]
    kvs = [rz.DeviceKV(to_dev(k), to_dev(v)) for k, v in kvs_h]
    stack = rz.DeviceStack([dev_layer(rz, L) for L in layers], kvs, to_dev(out_gamma), to_dev(lm), vocab)
    return layers, out_gamma, lm, kvs_h, stack


def test_decode_stack_llama_two_layers_and_lm_head(rz):
    """The benchmarked step shape through the launch sequence: two Llama-7B-shaped
    layers at position 1024, the output norm and the 32000 x 4096 Q4_0 LM head."""
    sh = S.LLAMA7B
    pos, max_seq = 1024, 1025
    layers, og, lm, kvs_h, stack = _llama_stack(rz, "ls", 2, max_seq, pos, 1)
    x = S.hidden_input("ls.x", 1, sh.hidden, sh.hidden_pad)
    hid, logits = rz.decode_stack(to_dev(x), stack, position=pos)
    hid = hid.cpu().numpy()
    logits = logits.cpu().numpy()
    check_no_device_error()
    hid_r, log_r = oracle.decode_stack(x[0], [orc_layer(L) for L in layers],
                                       [k[0].copy() for k, _ in kvs_h], [v[0].copy() for _, v in kvs_h],
                                       pos, og, lm, S.LLAMA_VOCAB)
    assert_rel(hid[0], hid_r, what="llama stack hidden")
    assert_rel(logits[0], log_r, what="llama stack logits")


@pytest.mark.parametrize("m", [4, 16])
def test_decode_stack_llama_batched(rz, m):
    """Two Llama-7B-shaped layers and the 32000 x 4096 head for m sequences at
    distinct positions (device-resident positions)."""
    sh = S.LLAMA7B
    positions = LLAMA_POSITIONS[m]
    max_seq = max(positions) + 1
    layers, og, lm, kvs_h, stack = _llama_stack(rz, f"lsb{m}", 2, max_seq, max(positions), m)
    x = S.hidden_input(f"lsb.x.{m}", m, sh.hidden, sh.hidden_pad)
    hid, logits = rz.decode_stack(to_dev(x), stack, positions=to_dev(np.array(positions, np.int32)))
    hid = hid.cpu().numpy()
    logits = logits.cpu().numpy()
    check_no_device_error()
    ols = [orc_layer(L) for L in layers]
    for t, p in enumerate(positions):
        hid_r, log_r = oracle.decode_stack(x[t], ols, [k[t].copy() for k, _ in kvs_h],
                                           [v[t].copy() for _, v in kvs_h], p, og, lm, S.LLAMA_VOCAB)
        assert_rel(hid[t], hid_r, what=f"llama stack m={m} token {t} hidden")
        assert_rel(logits[t], log_r, what=f"llama stack m={m} token {t} logits")


@pytest.mark.parametrize("m", [1, 4])
def test_decode_stack_graph_replay(rz, m):
    """rz_decode_stack captured once into a CUDA graph (positions in device memory)
    and replayed for two consecutive decode steps: each replay matches the oracle
    run on the same caches, the second step seeing the rows the first one wrote."""
    import torch
    sh = S.LLAMA7B
    p0 = [200, 5, 77, 0][:m]
    max_seq = 256
    layers, og, lm, kvs_h, stack = _llama_stack(rz, f"lg{m}", 2, max_seq, max(p0), m)
    dev = torch.device("cuda:0")
    xs = [S.hidden_input(f"lg.x{s}.{m}", m, sh.hidden, sh.hidden_pad) for s in range(2)]
    x_d = to_dev(xs[0])
    pos_d = to_dev(np.array(p0, np.int32))
    ws = rz.workspace(stack.workspace_bytes(m), dev)
    hid = torch.empty((m, sh.hidden_pad), dtype=torch.float32, device=dev)
    logits = torch.empty((m, S.LLAMA_VOCAB), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream()
    # warm-up call outside the graph sets the kernels' attributes; it writes the
    # cache rows at p0 that the first replay then overwrites with the same values
    rz.rz_decode_stack(x_d, stack, pos_d, 0, m, hid, logits, ws, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        rz.rz_decode_stack(x_d, stack, pos_d, 0, m, hid, logits, ws, stream=stream)
    torch.cuda.synchronize()
    ols = [orc_layer(L) for L in layers]
    kcs = [[k[t].copy() for k, _ in kvs_h] for t in range(m)]
    vcs = [[v[t].copy() for _, v in kvs_h] for t in range(m)]
    for step in range(2):
        x_d.copy_(torch.from_numpy(xs[step]))
        pos = [p + step for p in p0]
        pos_d.copy_(torch.from_numpy(np.array(pos, np.int32)))
        g.replay()
        torch.cuda.synchronize()
        check_no_device_error()
        h_g, l_g = hid.cpu().numpy(), logits.cpu().numpy()
        for t in range(m):
            hid_r, log_r = oracle.decode_stack(xs[step][t], ols, kcs[t], vcs[t], pos[t], og, lm,
                                               S.LLAMA_VOCAB)
            assert_rel(h_g[t], hid_r, what=f"graph m={m} step {step} token {t} hidden")
            assert_rel(l_g[t], log_r, what=f"graph m={m} step {step} token {t} logits")
