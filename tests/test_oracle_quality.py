"""Pins of the 4-bit quality proxy and the quality-aware format ranking (the
PagedWeight feedback loop; the scoring m[e] * q[e] is a reading).

Independent references: a hand-worked ranking, brute force (a stable sort of
the scores), the plain importance ranking as the q = 1 special case; for the
error proxy, the same page on both sides (error 0), and the proxy's invariance
to the order of the sampled tokens and additivity over them. The library's
host ranking is compared with the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import synth


def test_rank_quality_hand(orc):
    m = np.array([0.5, 0.9, 0.2, 0.9, 0.1])
    q = np.array([0.4, 0.1, 2.0, 0.1, 0.0])
    # scores 0.2, 0.09, 0.4, 0.09, 0.0 -> top 2: experts 2, 0; top 3 adds expert 1 (tie with 3: lower id)
    assert orc.rank_formats_quality(m, q, 2).tolist() == [0, 1, 0, 1, 1]
    assert orc.rank_formats_quality(m, q, 3).tolist() == [0, 0, 0, 1, 1]


@pytest.mark.parametrize("E,n_hi", [(16, 4), (256, 64), (7, 0), (5, 9)])
def test_rank_quality_brute_force(orc, E, n_hi):
    g = np.random.default_rng(E + n_hi)
    m = g.random(E)
    q = np.round(g.random(E), 1)  # coarse values: ties occur
    score = m * q
    order = sorted(range(E), key=lambda e: (-score[e], e))
    want = np.ones(E, np.uint8)
    want[order[:n_hi]] = 0
    assert np.array_equal(orc.rank_formats_quality(m, q, n_hi), want)
    # q = 1 everywhere: the plain importance ranking
    assert np.array_equal(orc.rank_formats_quality(m, np.ones(E), n_hi), orc.rank_formats(m, n_hi))


def test_library_ranking_matches_oracle(orc):
    import paged_quantized_expert_gb300 as pqe
    pqe.load()
    for seed in range(8):
        g = np.random.default_rng(seed)
        E = int(g.integers(1, 300))
        n_hi = int(g.integers(0, E + 2))
        m = np.round(g.random(E), 2)
        q = np.round(g.random(E), 2)
        fmt = torch.zeros(E, dtype=torch.uint8)
        pqe.pqe_rank_formats_quality(torch.from_numpy(m), torch.from_numpy(q), n_hi, fmt)
        assert np.array_equal(fmt.numpy(), orc.rank_formats_quality(m, q, n_hi)), seed


def _expert(orc, cfg, e):
    w13, w2 = synth.expert_weights(cfg, e)
    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    w8 = (q13, s13, q2, s2)
    w4 = orc.quant_mxfp4_rows(q13, s13) + orc.quant_mxfp4_rows(q2, s2)
    return w8, w4


def test_quant_error_zero_for_one_page(orc):
    # the same page on both sides: the difference vanishes exactly, whatever the format
    cfg = synth.small_config(E=2, H=256, I=128, k=1, T=6, cid=95)
    w8, w4 = _expert(orc, cfg, 0)
    x = synth.activations(cfg, 6)
    for w, f in ((w8, 0), (w4, 1)):
        d2, r2 = orc.quant_error_sums(x, w, w, 128, fmt8=f, fmt4=f)
        assert r2 > 0 and d2 == 0.0


def test_quant_error_positive_and_order_free(orc):
    cfg = synth.small_config(E=2, H=256, I=128, k=1, T=12, cid=94)
    w8, w4 = _expert(orc, cfg, 1)
    x = synth.activations(cfg, 12)
    d2, r2 = orc.quant_error_sums(x, w8, w4, 128)
    assert r2 > 0 and 0 < d2 < r2  # 4 bits lose something, far less than the signal
    perm = np.random.default_rng(0).permutation(12)
    d2p, r2p = orc.quant_error_sums(x[perm], w8, w4, 128)
    assert d2p == pytest.approx(d2, rel=1e-12) and r2p == pytest.approx(r2, rel=1e-12)
    # sums over tokens: two halves add up to the whole
    a2, b2 = orc.quant_error_sums(x[:5], w8, w4, 128), orc.quant_error_sums(x[5:], w8, w4, 128)
    assert a2[0] + b2[0] == pytest.approx(d2, rel=1e-12) and a2[1] + b2[1] == pytest.approx(r2, rel=1e-12)
