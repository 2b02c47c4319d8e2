"""A bounded device wait that runs out: the failure path of the weight-stream
FFN kernel, made to happen without any GPU fault. A test hook raises the
phase-1 completion count that phase 2 of every expert waits for, so those
waits can never be satisfied; with a short wait limit they expire, the kernel
ORs PQE_STATUS_TIMEOUT into the status word and runs to its end, the call
returns, and the same context then computes a correct layer again."""
import time

import numpy as np
import pytest
import torch

import synth
from tests.test_gpu_ffn import Pages, check_tokens, run_layer

pytestmark = pytest.mark.gpu


def test_phase2_wait_expires_sets_timeout_and_returns(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    T = 16  # 32 assignments over 8 experts: every batch <= 8 rows, the weight stream alone
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)))
    x = synth.activations(cfg, T)
    logits = np.random.default_rng(5).standard_normal((T, cfg.E)).astype(np.float32)
    ids, g = orc.topk_gates(logits, cfg.k)
    assert np.bincount(ids.reshape(-1), minlength=cfg.E).max() <= 8
    pqe.pqe_set_wait_limit(2000)
    pqe.pqe_test_set_phase2_bias(1)
    try:
        t0 = time.perf_counter()
        res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
        elapsed = time.perf_counter() - t0
    finally:
        pqe.pqe_test_set_phase2_bias(0)
        pqe.pqe_set_wait_limit(0)
    assert res["status"] & pqe.PQE_STATUS_TIMEOUT
    assert elapsed < 30.0
    # the context is still usable: the same layer again, correct and clean
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    assert res["status"] == 0 and np.array_equal(res["ids"], ids)
    check_tokens(orc, pages, cfg, x, ids, g, res, np.arange(T, dtype=np.int32))
