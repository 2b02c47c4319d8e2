"""Pins of the oracle's per-expert bit-width assignment (importance EMA + rank).

Independent references: numpy's lexsort for the ranking, numpy's bincount for
the gate mass, and the closed form of an EMA under a constant input.
"""
import numpy as np


def test_rank_matches_lexsort_with_ties(orc):
    g = np.random.default_rng(0)
    for _ in range(20):
        E = int(g.integers(4, 300))
        n_hi = int(g.integers(0, E + 1))
        m = g.integers(0, 5, E).astype(np.float64)  # many exact ties
        fmt = orc.rank_formats(m, n_hi)
        order = np.lexsort((np.arange(E), -m))       # m desc, then id asc
        ref = np.ones(E, np.uint8)
        ref[order[:n_hi]] = 0
        assert np.array_equal(fmt, ref)


def test_alpha_zero_is_gate_mass(orc):
    g = np.random.default_rng(1)
    T, k, E = 50, 4, 16
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    gates = g.random((T, k)).astype(np.float32)
    m = g.random(E)
    fmt = np.zeros(E, np.uint8)
    orc.importance_step(m, ids, gates, E, step=0, fmt=fmt, alpha=0.0, every=64, n_hi=4)
    ref = np.bincount(ids.reshape(-1), weights=gates.reshape(-1).astype(np.float64), minlength=E) / T
    assert np.allclose(m, ref, rtol=1e-15, atol=0)


def test_ema_constant_input_closed_form_and_rerank_steps(orc):
    T, k, E = 8, 2, 8
    ids = np.tile(np.array([[3, 5]], np.int32), (T, 1))
    gates = np.tile(np.array([[0.75, 0.25]], np.float32), (T, 1))
    m = np.zeros(E)
    fmt = np.ones(E, np.uint8)
    reranks = []
    for step in range(200):
        if orc.importance_step(m, ids, gates, E, step, fmt, alpha=0.9, every=64, n_hi=1):
            reranks.append(step)
    # m_n = (1 - 0.9^n) * mass for a constant mass
    assert np.allclose(m[3], (1 - 0.9 ** 200) * 0.75, rtol=1e-12)
    assert np.allclose(m[5], (1 - 0.9 ** 200) * 0.25, rtol=1e-12)
    assert reranks == [63, 127, 191]
    assert fmt.tolist() == [1, 1, 1, 0, 1, 1, 1, 1]
