"""Pins of the oracle's router (logits, top-k, gates) and permutation.

Independent references: fp64 dot products with the recursive-summation error
bound, exact sums of powers of two, numpy's stable sort, scipy's softmax and
bincount, and invariants of a permutation.
"""
import numpy as np
import pytest
import scipy.special

import synth


def _bf16(a):
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def test_logits_exact_on_powers_of_two(orc):
    # every product and partial sum is exactly representable -> result is the exact dot
    g = np.random.default_rng(3)
    T, H, E = 5, 96, 7
    x = (2.0 ** g.integers(-4, 4, (T, H))) * g.choice([-1, 1], (T, H))
    w = (2.0 ** g.integers(-4, 4, (E, H))) * g.choice([-1, 1], (E, H))
    lg = orc.router_logits(_bf16(x), w.astype(np.float32))
    assert np.array_equal(lg.astype(np.float64), x @ w.T)


def test_logits_within_summation_bound(orc):
    cfg = synth.WORKLOADS["tiny"]
    x = synth.activations(cfg, 64)
    w = synth.router_weights(cfg)
    lg = orc.router_logits(x, w).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    exact = xf @ w.astype(np.float64).T
    mag = np.abs(xf) @ np.abs(w.astype(np.float64)).T
    n = cfg.H // 32 + 5  # longest chain: H/32 fused adds, then 5 tree levels
    u = 2.0 ** -24
    assert np.all(np.abs(lg - exact) <= n * u / (1 - n * u) * mag)
    # a dropped or doubled term would be far outside: the bound is tight enough to see one
    one_term = np.abs(xf[:, :1] * w[:, 0].astype(np.float64)[None, :])
    assert np.median(one_term) > 50 * np.median(n * u * mag)


def _stable_topk(logits, k):
    # numpy stable sort of -logit keeps ascending id among equal logits
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


@pytest.mark.parametrize("E,k", [(8, 2), (16, 1), (64, 8), (256, 8), (5, 5)])
def test_topk_matches_stable_sort_with_ties(orc, E, k):
    g = np.random.default_rng(E * 10 + k)
    T = 200
    # small integer logits: many exact ties
    logits = g.integers(-3, 3, (T, E)).astype(np.float32)
    ids, gates = orc.topk_gates(logits, k)
    assert np.array_equal(ids, _stable_topk(logits, k))


def test_topk_on_trace_ties(orc):
    cfg = synth.WORKLOADS["decode"]
    logits = synth.routing_logits(cfg, 64, 0)
    ids, _ = orc.topk_gates(logits, cfg.k)
    assert np.array_equal(ids, _stable_topk(logits, cfg.k))
    # the trace holds at least one exact tie across the k boundary
    srt = -np.sort(-logits, axis=1)
    assert np.any(srt[:, cfg.k - 1] == srt[:, cfg.k])


def test_gates_are_renormalised_softmax(orc):
    g = np.random.default_rng(5)
    logits = (g.standard_normal((100, 32)) * 3).astype(np.float32)
    ids, gates = orc.topk_gates(logits, 4)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    picked = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    ref = picked / picked.sum(axis=1, keepdims=True)
    assert np.allclose(gates, ref, rtol=1e-12, atol=0)
    assert np.allclose(gates.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(gates, axis=1) <= 0)  # ordered by logit


def test_gates_k1_is_one(orc):
    logits = np.random.default_rng(6).standard_normal((10, 9)).astype(np.float32)
    ids, gates = orc.topk_gates(logits, 1)
    assert np.all(gates == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(logits, axis=1))


@pytest.mark.parametrize("T,k,E", [(64, 2, 8), (1, 8, 256), (0, 8, 16), (333, 3, 17), (4096, 8, 512)])
def test_permute_matches_stable_sort(orc, T, k, E):
    g = np.random.default_rng(T + k + E)
    ids = np.stack([g.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    counts, offsets, perm_src, inv = orc.permute(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert counts.sum() == T * k
    assert np.array_equal(perm_src, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv[perm_src], np.arange(T * k))        # bijection
    for e in range(E):
        seg = perm_src[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
