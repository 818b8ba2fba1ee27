"""The all-core oracle build (OpenMP over independent output rows and attention
heads) that the benchmark's CPU baseline uses gives bit-identical results to the
single-threaded build the parity tests use: each row is summed in the same order."""
import numpy as np
import pytest

import rz_synth as S


@pytest.fixture
def both():
    import oracle
    try:
        oracle.use_all_cores(True)
    except Exception as e:   # no OpenMP toolchain
        oracle.use_all_cores(False)
        pytest.skip(f"no all-core build: {e}")
    yield oracle
    oracle.use_all_cores(False)


def test_all_core_build_matches_single_thread(both):
    orc = both
    assert orc.threads() >= 1
    w = S.q4k_weight("omp.w", 300, 1024)
    x8 = None
    sh = S.LayerShape(hidden=448, inter=512, n_heads=7, n_kv_heads=1, head_dim=64,
                      rope_theta=1e6, rope_mode=1)
    L = S.layer(sh, "omp.l")
    x = S.hidden_input("omp.x", 1, sh.hidden, sh.hidden_pad)[0]
    kc, vc = S.kv_prefill(sh, "omp.kv", 16, 9)
    lm = S.q4_0_weight("omp.lm", 200, sh.hidden)

    def run():
        nonlocal x8
        x8 = orc.q8_1_quantize(S.normal("omp.x8", (3, 1024)))
        y = orc.q4k_q8_gemv(w, x8, 3, 300, 1024)
        lw = orc.LayerWeights(**L.w, attn_gamma=L.attn_gamma, ffn_gamma=L.ffn_gamma,
                              hidden=sh.hidden, hidden_pad=sh.hidden_pad, n_heads=sh.n_heads,
                              n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim, inter=sh.inter,
                              eps=sh.eps, rope_theta=sh.rope_theta, rope_mode=sh.rope_mode)
        out = orc.decode_layer(x, lw, kc[0].copy(), vc[0].copy(), 9)
        logits = orc.q4_0_gemv(lm, x[:sh.hidden], 200, sh.hidden)
        return y, out, logits

    a = run()
    orc.use_all_cores(False)
    b = run()
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))
