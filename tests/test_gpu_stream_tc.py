"""GPU parity of the tensor-core weight stream (tcgen05 MMAs with the weight
rows as the 128-row operand and each token's activations as two E4M3 terms)
against the oracle, through moe_paged_ffn with every page FP8 (expert_fmt
NULL). The kernel is forced with the stream-kernel test hook, so small layers
take it too; each case is held to the same bounds as the CUDA-core stream
(max |y - ref| / ||ref_t|| <= 2e-2, and a relative L2 error of 5e-3 for tokens
whose experts all take a weight stream)."""
import numpy as np
import pytest
import torch

import synth
from tests import helpers
from tests.test_gpu_ffn import DEV, Pages, check_tokens, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture
def tc_stream(cuda_lib):
    cuda_lib.pqe_test_set_stream_kernel(2)
    try:
        yield cuda_lib
    finally:
        cuda_lib.pqe_test_set_stream_kernel(0)


def _layer(pqe, orc, cfg, T, logits, x=None, needed=None, page_table=None, pool=None, pages=None):
    ids, gates = orc.topk_gates(logits, cfg.k)
    if pages is None:
        pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)) if needed is None else needed)
    if x is None:
        x = synth.activations(cfg, T)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, page_table=page_table, fmt_dev=None,
                    pool=pages.pool if pool is None else pool)
    assert np.array_equal(res["ids"], ids)
    return pages, x, ids, gates, res


@pytest.mark.parametrize("E,H,I,k,T", [
    (8, 256, 128, 2, 16),     # a few items, most CTAs idle
    (9, 256, 128, 2, 25),     # ragged per-expert batches of 3..8 rows
    (40, 512, 256, 4, 36),    # batches of 0..8 rows, an expert's items over several CTAs
    (64, 1024, 384, 8, 24),   # K = 1024 in 8 stages; I = 384: six phase-1 items per expert
    (3, 256, 640, 1, 7),      # I > H: the h tile is the longer one
    # steps of at most 8 tokens: x and perm_src staged in shared memory
    (9, 256, 128, 2, 8),      # batches of 1..8 rows from a staged x
    (40, 512, 256, 4, 5),     # an expert's items over several CTAs, staged x
    (64, 1024, 384, 8, 1),    # one token, eight experts
])
def test_tc_stream_small_layers(tc_stream, orc, E, H, I, k, T):
    pqe = tc_stream
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=94)
    logits = np.random.default_rng(T + E).standard_normal((T, E)).astype(np.float32)
    ids, _ = orc.topk_gates(logits, k)
    assert np.bincount(ids.reshape(-1), minlength=E).max() <= 8  # every batch on the weight stream
    pages, x, ids, gates, res = _layer(pqe, orc, cfg, T, logits)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


@pytest.mark.parametrize("shift", [18, -18])
def test_tc_stream_activation_magnitude_extremes(tc_stream, orc, shift):
    # |x| (and so |h|) far from 1: each token's E4M3 terms are taken relative
    # to its own amax, so the relative bound holds at any scale
    pqe = tc_stream
    cfg = synth.WORKLOADS["tiny"]
    T = 6
    x = synth.activations(cfg, T)
    xf = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** shift)
    xs = (xf.view(np.uint32) >> 16).astype(np.uint16)
    logits = np.random.default_rng(7).standard_normal((T, cfg.E)).astype(np.float32)
    pages, _, ids, gates, res = _layer(pqe, orc, cfg, T, logits, x=xs)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, xs, ids, gates, res, np.arange(T, dtype=np.int32))


@pytest.mark.parametrize("T,n_check", [(1, 1), (8, 4), (64, 4)])
def test_tc_stream_decode_layer_shapes(tc_stream, orc, T, n_check):
    # the decode-shaped layer (E=256, H=2048, I=512, top-8); at T=64 batches of
    # 9 rows and more take the tensor-core GEMM chain on a side stream beside it
    pqe = tc_stream
    cfg = synth.WORKLOADS["decode"]
    logits = synth.routing_logits(cfg, T, 2)
    ids, _ = orc.topk_gates(logits, cfg.k)
    tokens = helpers.sample_tokens(T, n_check, seed=T)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    # checked tokens include one whose experts all take the weight stream
    stream_only = [t for t in range(T) if counts[ids[t]].max() < helpers.TC_MIN_ROWS]
    if stream_only:
        tokens = np.unique(np.append(tokens, stream_only[0])).astype(np.int32)
    needed = set(ids[tokens].reshape(-1).tolist())
    pages = Pages(pqe, orc, cfg, needed=needed, seed=T)
    x = synth.activations(cfg, T, 2)
    _, _, ids, gates, res = _layer(pqe, orc, cfg, T, logits, x=x, pages=pages)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, tokens)


@pytest.mark.parametrize("T", [3, 16])
def test_tc_stream_bad_page_staged_and_unstaged(tc_stream, orc, T):
    # a routed expert whose page-table entry points outside the pool, with x
    # staged in shared memory (T <= 8) and without: flagged, its rows of
    # out_perm are zero, the other experts' rows match the oracle
    pqe = tc_stream
    E, H, I, k = 6, 256, 128, 2
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=89)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)))
    logits = np.random.default_rng(23 + T).standard_normal((T, E)).astype(np.float32)
    ids, gates = orc.topk_gates(logits, k)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    bad_e = int(np.argmax(counts))
    pt = np.arange(E, dtype=np.int32)
    pt[bad_e] = E + 3
    x = synth.activations(cfg, T)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, page_table=torch.from_numpy(pt).to(DEV), fmt_dev=None,
                    pool=pages.pool)
    assert res["status"] & pqe.PQE_STATUS_BAD_PAGE
    op = res["out_perm"].float().cpu().numpy()
    _, offsets, _, _ = orc.permute(ids, E)
    assert np.all(op[np.arange(offsets[bad_e], offsets[bad_e + 1])] == 0)
    ok_tokens = np.array([t for t in range(T) if bad_e not in ids[t]], dtype=np.int32)
    if len(ok_tokens):
        check_tokens(orc, pages, cfg, x, ids, gates, res, ok_tokens)


def test_tc_stream_slot_indirection_and_bad_page(tc_stream, orc):
    # experts in permuted slots of a larger pool; then one routed expert points
    # outside the pool: flagged, its rows of out_perm are zero, the others exact
    pqe = tc_stream
    E, H, I, k, T = 6, 256, 128, 2, 16
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=95)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)))
    stride = pqe.slot_stride(H, I)
    perm = np.array([4, 0, 5, 2, 1, 3])
    pool2 = torch.zeros(8 * stride, dtype=torch.uint8, device=DEV)
    for e in range(E):
        pool2[perm[e] * stride:(perm[e] + 1) * stride].copy_(pages.pool_mem[e * stride:(e + 1) * stride])
    p2 = pqe.make_pool(pool2, 8, H, I)
    logits = np.random.default_rng(3).standard_normal((T, E)).astype(np.float32)
    pt = torch.from_numpy(perm.astype(np.int32)).to(DEV)
    _, x, ids, gates, res = _layer(pqe, orc, cfg, T, logits, page_table=pt, pool=p2, pages=pages)
    assert np.bincount(ids.reshape(-1), minlength=E).max() <= 8
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))
    bad = perm.copy()
    bad[3] = 9
    res = run_layer(pqe, cfg, T, x, logits_np=logits, page_table=torch.from_numpy(bad.astype(np.int32)).to(DEV),
                    fmt_dev=None, pool=p2)
    assert res["status"] & pqe.PQE_STATUS_BAD_PAGE
    op = res["out_perm"].float().cpu().numpy()
    _, offsets, _, _ = orc.permute(ids, E)
    assert np.all(op[np.arange(offsets[3], offsets[4])] == 0)
    assert np.any(op[np.arange(offsets[0], offsets[1])] != 0)


@pytest.mark.parametrize("T", [6, 36])
def test_tc_stream_graph_replay_bit_identical(tc_stream, orc, T):
    # the FFN call eager and replayed from a CUDA graph: the same out_perm bit
    # for bit (no atomics in the arithmetic, a fixed MMA order); T=6 stages x
    pqe = tc_stream
    E, H, I, k = 40, 512, 256, 4
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=96)
    logits = np.random.default_rng(13).standard_normal((T, E)).astype(np.float32)
    ids, _ = orc.topk_gates(logits, k)
    pages = Pages(pqe, orc, cfg, needed=set())
    A = T * k
    xd = torch.from_numpy(synth.activations(cfg, T).view(np.int16)).to(DEV)
    idsd = torch.from_numpy(ids.astype(np.int32)).to(DEV)
    counts = torch.zeros(E, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    perm_src = torch.zeros(A, dtype=torch.int32, device=DEV)
    inv = torch.zeros(A, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pws = torch.zeros(pqe.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    pqe.moe_permute(idsd, T, k, E, counts, offsets, perm_src, inv, pws, status)
    pt = torch.arange(E, dtype=torch.int32, device=DEV)
    fws = torch.zeros(pqe.moe_paged_ffn_workspace_size(T, k, E, H, I), dtype=torch.uint8, device=DEV)
    eager = torch.zeros((A, H), dtype=torch.bfloat16, device=DEV)
    pqe.moe_paged_ffn(xd, perm_src, offsets, pt, None, pages.pool, T, k, E, eager, fws, status)
    torch.cuda.synchronize()
    replay = torch.zeros((A, H), dtype=torch.bfloat16, device=DEV)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            pqe.moe_paged_ffn(xd, perm_src, offsets, pt, None, pages.pool, T, k, E, replay, fws, status, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        replay.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))
    assert status.item() == 0


def test_tc_stream_phase2_wait_expires(tc_stream, orc):
    # the phase-2 count wait of the tensor-core stream runs out (test bias):
    # PQE_STATUS_TIMEOUT, the call returns, and the context computes the layer
    # correctly afterwards
    import time
    pqe = tc_stream
    E, H, I, k, T = 40, 512, 256, 4, 36
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=97)
    logits = np.random.default_rng(13).standard_normal((T, E)).astype(np.float32)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)))
    x = synth.activations(cfg, T)
    pqe.pqe_set_wait_limit(2000)
    pqe.pqe_test_set_phase2_bias(1)
    try:
        t0 = time.perf_counter()
        res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=None, pool=pages.pool)
        elapsed = time.perf_counter() - t0
    finally:
        pqe.pqe_test_set_phase2_bias(0)
        pqe.pqe_set_wait_limit(0)
    assert res["status"] & pqe.PQE_STATUS_TIMEOUT
    assert elapsed < 30.0
    _, _, ids, gates, res = _layer(pqe, orc, cfg, T, logits, x=x, pages=pages)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


def test_stream_kernel_hook_rejects_unknown_kind(cuda_lib):
    with pytest.raises(cuda_lib.PqeError):
        cuda_lib.pqe_test_set_stream_kernel(3)
    cuda_lib.pqe_test_set_stream_kernel(0)
