"""Host parts of the product (no CUDA calls) against the oracle, bit for bit:
the LRU page table and the importance-ranked bit-width assignment.
"""
import numpy as np
import pytest
import torch

import synth
from tests.test_oracle_lru import HAND_TRACE


def _pqe():
    import paged_quantized_expert_gb300 as pqe
    pqe.load()
    return pqe


def _counts(E, used):
    c = np.zeros(E, np.int32)
    c[list(used)] = 1
    return c


def test_lru_hand_trace_matches(orc):
    pqe = _pqe()
    lru = pqe.LRU(6, 3)
    for step, (used, table, misses, wb, slots, last) in enumerate(HAND_TRACE):
        pt, me, md, got_wb = lru.page_table_update(torch.from_numpy(_counts(6, used)))
        assert list(zip(me.tolist(), md.tolist())) == misses and got_wb == wb
        se, lu, st = lru.state()
        assert se.tolist() == slots and lu.tolist() == last and st == step + 1


@pytest.mark.parametrize("E,S,maxk,steps", [(256, 32, 64, 400), (512, 46, 40, 300), (8, 8, 8, 50), (16, 0, 3, 30)])
def test_lru_random_traces_match_oracle(orc, E, S, maxk, steps):
    pqe = _pqe()
    a = pqe.LRU(E, S)
    b = orc.LRU(E, S)
    g = np.random.default_rng(E * 7 + S)
    for step in range(steps):
        n = int(g.integers(0, maxk + 1))
        used = g.choice(E, n, replace=False)
        counts = _counts(E, used) * g.integers(1, 5, E).astype(np.int32)
        pt, me, md, wb = a.page_table_update(torch.from_numpy(counts))
        pt2, me2, md2, wb2 = b.step(counts)
        assert np.array_equal(pt.numpy(), pt2) and wb == wb2
        assert np.array_equal(me.numpy(), me2) and np.array_equal(md.numpy(), md2)
        se, lu, st = a.state()
        se2, lu2, st2 = b.state()
        assert np.array_equal(se.numpy(), se2) and np.array_equal(lu.numpy(), lu2) and st == st2


def test_lru_trace_of_config_2(orc):
    # the decode layer's trace at T=8 through both pools
    pqe = _pqe()
    cfg = synth.WORKLOADS["decode"]
    tr = synth.RoutingTrace(cfg, 8)
    a, b = pqe.LRU(cfg.E, cfg.S), orc.LRU(cfg.E, cfg.S)
    for s in range(64):
        ids, _ = orc.topk_gates(tr.step(s), cfg.k)
        counts = np.bincount(ids.reshape(-1), minlength=cfg.E).astype(np.int32)
        r1 = a.page_table_update(torch.from_numpy(counts))
        r2 = b.step(counts)
        assert np.array_equal(r1[0].numpy(), r2[0]) and np.array_equal(r1[1].numpy(), r2[1])


def test_lru_invalidate(orc):
    pqe = _pqe()
    a = pqe.LRU(8, 4)
    a.page_table_update(torch.from_numpy(_counts(8, [1, 2, 3])))
    a.invalidate(2)
    se, _, _ = a.state()
    assert se.tolist() == [1, -1, 3, -1]
    pt, me, md, _ = a.page_table_update(torch.from_numpy(_counts(8, [2])))
    assert me.tolist() == [2] and md.tolist() == [1]   # lowest empty slot


def test_importance_matches_oracle(orc):
    pqe = _pqe()
    cfg = synth.WORKLOADS["mixed"]
    T, k, E = 256, cfg.k, cfg.E
    m_a = synth.importance_init(cfg)
    m_b = m_a.copy()
    f_a = np.zeros(E, np.uint8)
    f_b = np.zeros(E, np.uint8)
    pqe.pqe_rank_formats(torch.from_numpy(m_a), 64, torch.from_numpy(f_a))
    f_b[:] = orc.rank_formats(m_b, 64)
    assert np.array_equal(f_a, f_b) and int((f_a == 0).sum()) == 64
    tr = synth.RoutingTrace(cfg, T)
    for s in range(130):
        ids, g64 = orc.topk_gates(tr.step(s), k)
        g = g64.astype(np.float32)
        r1 = pqe.pqe_importance_step(torch.from_numpy(m_a), torch.from_numpy(ids), torch.from_numpy(g), T, k, E,
                                     0.9, s, 64, 64, torch.from_numpy(f_a))
        r2 = orc.importance_step(m_b, ids, g, E, s, f_b, alpha=0.9, every=64, n_hi=64)
        assert r1 == r2
        assert np.array_equal(m_a, m_b) and np.array_equal(f_a, f_b)
