"""GPU parity of the persistent decode kernel (one cooperative launch per step of
up to 32 layers) beyond the shared layer/stack cases in test_gpu_layer.py:
the Llama-7B-shaped step at the benchmark position, consecutive steps through
the cache the kernel appends to, stacks longer than one launch, a bad device
position, and run-to-run determinism.

Bar (values re-quantised to Q8_1 inside the layer): within 1e-3 relative, as
max|gpu - ref| <= 1e-3 max|ref| and ||gpu - ref||_2 <= 1e-3 ||ref||_2.
"""
import numpy as np
import pytest

import oracle
import rz_synth as S

from gpu_common import check_no_device_error, to_dev
from test_gpu_layer import assert_rel, dev_layer, orc_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rz():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q4_q8_gb300 as rz
    rz.load()
    rz.set_persistent(True)
    return rz


def _stack(rz, sh, tag, n_layers, max_seq, filled, vocab):
    layers = [S.layer(sh, f"{tag}.l{i}") for i in range(n_layers)]
    out_gamma = S.uniform(f"{tag}.og", sh.hidden, 0.5, 1.5)
    lm = S.q4_0_weight(f"{tag}.lm", vocab, sh.hidden)
    kvs_h = [S.kv_prefill(sh, f"{tag}.kv{i}", max_seq, filled) for i in range(n_layers)]
    kvs = [rz.DeviceKV(to_dev(k), to_dev(v)) for k, v in kvs_h]
    stack = rz.DeviceStack([dev_layer(rz, L) for L in layers], kvs, to_dev(out_gamma), to_dev(lm), vocab)
    ref_kc = [k[0].copy() for k, _ in kvs_h]
    ref_vc = [v[0].copy() for _, v in kvs_h]
    return layers, out_gamma, lm, stack, kvs, ref_kc, ref_vc


def test_llama_step_at_benchmark_position(rz):
    """Two Llama-7B-shaped layers at position 1024 of a 2056-row cache, the
    output norm and the 32000 x 4096 Q4_0 LM head (the benchmark's step, cut to
    two layers so that the oracle stays quick)."""
    sh = S.LLAMA7B
    pos, max_seq, vocab = 1024, S.LLAMA_MAX_SEQ, S.LLAMA_VOCAB
    layers, og, lm, stack, kvs, kc, vc = _stack(rz, sh, "pl", 2, max_seq, pos, vocab)
    x = S.hidden_input("pl.x", 1, sh.hidden, sh.hidden_pad)
    hid, logits = rz.decode_stack(to_dev(x), stack, position=pos)
    hid, logits = hid.cpu().numpy(), logits.cpu().numpy()
    check_no_device_error()
    hid_r, log_r = oracle.decode_stack(x[0], [orc_layer(L) for L in layers], kc, vc, pos, og, lm, vocab)
    assert_rel(hid[0], hid_r, what="hidden")
    assert_rel(logits[0], log_r, what="logits")
    for i in range(2):
        assert_rel(kvs[i].k.cpu().numpy()[0, pos], kc[i][pos], tol=1e-4, what=f"k row layer {i}")
        assert np.array_equal(kvs[i].k.cpu().numpy()[0, :pos], kc[i][:pos]), "earlier cache rows changed"


def test_consecutive_steps_share_the_cache(rz):
    """Three steps in a row (positions 62, 63, 64: the last crosses a chunk
    boundary), each reading the rows the previous ones appended."""
    sh = S.QWEN2
    max_seq, vocab = 96, 512
    layers, og, lm, stack, kvs, kc, vc = _stack(rz, sh, "pc", 2, max_seq, 62, vocab)
    ol = [orc_layer(L) for L in layers]
    for step, pos in enumerate([62, 63, 64]):
        x = S.hidden_input(f"pc.x{step}", 1, sh.hidden, sh.hidden_pad)
        hid, logits = rz.decode_stack(to_dev(x), stack, position=pos)
        check_no_device_error()
        hid_r, log_r = oracle.decode_stack(x[0], ol, kc, vc, pos, og, lm, vocab)
        assert_rel(hid.cpu().numpy()[0], hid_r, what=f"hidden step {step}")
        assert_rel(logits.cpu().numpy()[0], log_r, what=f"logits step {step}")


def test_stack_longer_than_one_launch(rz):
    """34 layers: two persistent launches chained through the workspace."""
    sh = S.QWEN2
    n, max_seq, pos, vocab = 34, 40, 33, 256
    layers, og, lm, stack, kvs, kc, vc = _stack(rz, sh, "plong", n, max_seq, pos, vocab)
    x = S.hidden_input("plong.x", 1, sh.hidden, sh.hidden_pad)
    hid, logits = rz.decode_stack(to_dev(x), stack, position=pos)
    check_no_device_error()
    hid_r, log_r = oracle.decode_stack(x[0], [orc_layer(L) for L in layers], kc, vc, pos, og, lm, vocab)
    assert_rel(hid.cpu().numpy()[0], hid_r, what="hidden")
    assert_rel(logits.cpu().numpy()[0], log_r, what="logits")


def test_identical_calls_give_identical_bits(rz):
    """Fixed-order reductions everywhere: the atomic counters only choose which
    warp merges, never the order of a sum."""
    sh = S.LLAMA7B
    L = S.layer(sh, "pdet")
    pos, max_seq = 300, 320
    x = to_dev(S.hidden_input("pdet.x", 1, sh.hidden, sh.hidden_pad))
    kc, vc = S.kv_prefill(sh, "pdet.kv", max_seq, pos)
    dl = dev_layer(rz, L)
    outs = []
    for _ in range(2):
        kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
        outs.append(rz.decode_layer(x, dl, kv, position=pos).cpu().numpy())
    check_no_device_error()
    assert np.array_equal(outs[0], outs[1])


def test_bad_device_position_is_reported(rz):
    """A device-resident position outside the cache: the kernel records 0x201,
    writes no cache row, and the step still ends (finite output)."""
    sh = S.QWEN2
    L = S.layer(sh, "pbad")
    max_seq = 32
    x = to_dev(S.hidden_input("pbad.x", 1, sh.hidden, sh.hidden_pad))
    kc, vc = S.kv_prefill(sh, "pbad.kv", max_seq, 8)
    kv = rz.DeviceKV(to_dev(kc), to_dev(vc))
    out = rz.decode_layer(x, dev_layer(rz, L), kv, positions=to_dev(np.array([max_seq + 7], np.int32)))
    st, code = rz.check_device_error()
    assert st == 7 and code == 0x201
    assert np.isfinite(out.cpu().numpy()).all()
    assert np.array_equal(kv.k.cpu().numpy(), kc)
    check_no_device_error()
