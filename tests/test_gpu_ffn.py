"""GPU parity of the expert FFN + combine over the slot pool, called through the
C-ABI one step at a time (moe_route -> moe_permute -> moe_paged_ffn ->
moe_combine), against the oracle.

Tolerance per token t: max_i |y - ref| / ||ref_t||_2 <= 2e-2 (stated bound);
the CUDA-core path is also held to a relative L2 error of 5e-3.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import synth
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Pages:
    """Expert pages on the device, in slots 0..E-1 of one pool (identity table),
    plus the oracle's copy of the experts the checked tokens use."""

    def __init__(self, pqe, orc, cfg, needed, fp4=(), seed=0):
        self.pqe, self.cfg = pqe, cfg
        E, H, I = cfg.E, cfg.H, cfg.I
        self.pool_mem, self.pool = pqe.alloc_pool(E, H, I)
        stride = pqe.slot_stride(H, I)
        self.fmt = torch.zeros(E, dtype=torch.uint8)
        self.experts = orc.ExpertSet(E)
        gen = torch.Generator(device=DEV)
        gen.manual_seed(1000 + seed)
        lay8 = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
        def oracle_expert(e):
            # the workload's weights and the oracle's quantisation of them (the
            # C oracle releases the GIL, so experts run on all host cores)
            w13, w2 = synth.expert_weights(cfg, e)
            q13, s13 = orc.quant_e4m3_rows(w13)
            q2, s2 = orc.quant_e4m3_rows(w2)
            if e in fp4:
                return w13, w2, (1, *orc.quant_mxfp4_rows(q13, s13), *orc.quant_mxfp4_rows(q2, s2))
            return w13, w2, (0, q13, s13, q2, s2)

        order = list(range(E))
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as pool:
            for b0 in range(0, E, 32):  # bounded batches: the fp32 weights of a batch at a time
                batch = [e for e in order[b0:b0 + 32] if e in needed]
                done = dict(zip(batch, pool.map(oracle_expert, batch)))
                for e in order[b0:b0 + 32]:
                    if e in needed:
                        w13, w2, rec = done.pop(e)
                        w13d, w2d = torch.from_numpy(w13).to(DEV), torch.from_numpy(w2).to(DEV)
                        self.experts.set(e, *rec)
                    else:
                        w13d = torch.randn(2 * I, H, device=DEV, generator=gen) * 0.02
                        w2d = torch.randn(H, I, device=DEV, generator=gen) * 0.02
                    slot = self.pool_mem[e * stride:(e + 1) * stride]
                    pqe.pqe_pack_fp8_page(w13d, w2d, H, I, slot)
                    if e in fp4:
                        tmp = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I), dtype=torch.uint8, device=DEV)
                        pqe.pqe_pack_mxfp4_page(slot, H, I, tmp)
                        slot.zero_()
                        slot[:tmp.numel()].copy_(tmp)
                        self.fmt[e] = pqe.PQE_FMT_MXFP4
        torch.cuda.synchronize()
        # the library's pages of the needed experts are the oracle's bytes
        for e in sorted(needed)[:2]:
            if e in fp4:
                continue
            got = self.pool_mem[e * stride:e * stride + lay8["bytes"]].cpu().numpy()
            q13, s13, q2, s2 = helpers.split_fp8_page(got, lay8, H, I)
            w13, w2 = synth.expert_weights(cfg, e)
            assert np.array_equal(q13, orc.quant_e4m3_rows(w13)[0])
        self.fmt_dev = self.fmt.to(DEV)


def run_layer(pqe, cfg, T, x_np, logits_np=None, w_r_np=None, page_table=None, fmt_dev=None, pool=None):
    E, H, k = cfg.E, cfg.H, cfg.k
    A = T * k
    x = torch.from_numpy(x_np.view(np.int16)).to(DEV)
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    gw = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    if w_r_np is not None:
        lg = torch.zeros((T, E), dtype=torch.float32, device=DEV)
        pqe.moe_route(x, torch.from_numpy(w_r_np).to(DEV), lg, T, H, E, k, ids, gw)
    else:
        pqe.moe_route(None, None, torch.from_numpy(logits_np).to(DEV), T, H, E, k, ids, gw)
    counts = torch.zeros(E, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    perm_src = torch.zeros(A, dtype=torch.int32, device=DEV)
    inv = torch.zeros(A, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(pqe.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    pqe.moe_permute(ids, T, k, E, counts, offsets, perm_src, inv, ws, status)
    pt = page_table if page_table is not None else torch.arange(E, dtype=torch.int32, device=DEV)
    out_perm = torch.zeros((A, H), dtype=torch.bfloat16, device=DEV)
    fws = torch.zeros(pqe.moe_paged_ffn_workspace_size(T, k, E, H, cfg.I), dtype=torch.uint8, device=DEV)
    pqe.moe_paged_ffn(x, perm_src, offsets, pt, fmt_dev, pool, T, k, E, out_perm, fws, status)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    pqe.moe_combine(out_perm, inv, gw, T, k, H, y)
    torch.cuda.synchronize()
    return {"y": y, "ids": ids.cpu().numpy(), "gates": gw.cpu().numpy(), "status": int(status.item()),
            "out_perm": out_perm}


def check_tokens(orc, pages, cfg, x_np, ids, gates_ref, res, tokens, l2_bound=None):
    ref = orc.moe_ffn(x_np, ids, gates_ref, pages.experts, cfg.I, tokens=tokens)
    y = helpers.bf16_to_f64(res["y"])[tokens]
    st = helpers.error_stats(y, ref)
    fp4 = set(np.nonzero(pages.fmt.numpy() == 1)[0].tolist())
    bound = helpers.l2_bounds(ids, tokens, cfg.E, fp4, cfg.H, cfg.I) if l2_bound is None else l2_bound
    assert st["max_over_l2"] <= helpers.TOL_MAX_OVER_L2, st
    assert np.all(st["l2_per_token"] <= bound), (st, bound)
    return st


def test_tiny_layer_end_to_end(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)))
    x = synth.activations(cfg, 64)
    w_r = synth.router_weights(cfg)
    res = run_layer(pqe, cfg, 64, x, w_r_np=w_r, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, g = orc.topk_gates(orc.router_logits(x, w_r), cfg.k)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, g, res, np.arange(64, dtype=np.int32))


@pytest.mark.parametrize("shift,fp4", [(18, ()), (-18, ()), (18, (3,)), (-18, (3,))])
def test_activation_magnitude_extremes(cuda_lib, orc, shift, fp4):
    # |x| (and so |h|) far from 1: the weight stream brings its f16 activations
    # into range with a power-of-two factor per token and K slice; the bound is
    # relative, so the same tolerance holds at any scale
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    T = 6
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)), fp4=set(fp4))
    x = synth.activations(cfg, T)
    xf = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** shift)
    xs = (xf.view(np.uint32) >> 16).astype(np.uint16)
    logits = np.random.default_rng(7).standard_normal((T, cfg.E)).astype(np.float32)
    logits[:, 3] += 2.0  # the 4-bit expert is routed
    res = run_layer(pqe, cfg, T, xs, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, g = orc.topk_gates(logits, cfg.k)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, xs, ids, g, res, np.arange(T, dtype=np.int32))


@pytest.mark.parametrize("E,H,I,k,T,fp4", [
    (5, 192, 64, 3, 37, ()),
    (5, 192, 64, 3, 37, (1, 3)),
    (9, 256, 128, 2, 129, (0, 1, 2, 3, 4, 5, 6, 7, 8)),
    (3, 64, 192, 1, 11, (2,)),
])
def test_small_ragged_layers(cuda_lib, orc, E, H, I, k, T, fp4):
    pqe = cuda_lib
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=92)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)), fp4=set(fp4))
    x = synth.activations(cfg, T)
    g = np.random.default_rng(T)
    logits = g.standard_normal((T, E)).astype(np.float32)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, gates = orc.topk_gates(logits, k)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


@pytest.mark.parametrize("T,n_check", [(1, 1), (8, 4), (64, 3)])
def test_decode_layer_shapes(cuda_lib, orc, T, n_check):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["decode"]
    logits = synth.routing_logits(cfg, T, 2)
    ids, gates = orc.topk_gates(logits, cfg.k)
    tokens = helpers.sample_tokens(T, n_check, seed=T)
    needed = set(ids[tokens].reshape(-1).tolist())
    pages = Pages(pqe, orc, cfg, needed=needed, seed=T)
    x = synth.activations(cfg, T, 2)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, tokens)


def test_slot_indirection_and_bad_page(cuda_lib, orc):
    # experts live in permuted slots; one routed expert points outside the pool
    pqe = cuda_lib
    cfg = synth.small_config(E=6, H=128, I=64, k=2, T=40, cid=93)
    pages = Pages(pqe, orc, cfg, needed=set(range(6)))
    stride = pqe.slot_stride(cfg.H, cfg.I)
    perm = np.array([4, 0, 5, 2, 1, 3])
    pool2 = torch.zeros(8 * stride, dtype=torch.uint8, device=DEV)
    for e in range(6):
        pool2[perm[e] * stride:(perm[e] + 1) * stride].copy_(pages.pool_mem[e * stride:(e + 1) * stride])
    p2 = pqe.make_pool(pool2, 8, cfg.H, cfg.I)
    x = synth.activations(cfg, 40)
    logits = np.random.default_rng(1).standard_normal((40, 6)).astype(np.float32)
    pt = torch.from_numpy(perm.astype(np.int32)).to(DEV)
    res = run_layer(pqe, cfg, 40, x, logits_np=logits, page_table=pt, fmt_dev=pages.fmt_dev, pool=p2)
    ids, gates = orc.topk_gates(logits, 2)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(40, dtype=np.int32))
    # expert 3 -> slot 9 (outside the 8-slot pool): flagged, its rows are zero
    bad = perm.copy()
    bad[3] = 9
    res = run_layer(pqe, cfg, 40, x, logits_np=logits, page_table=torch.from_numpy(bad.astype(np.int32)).to(DEV),
                    fmt_dev=pages.fmt_dev, pool=p2)
    assert res["status"] & pqe.PQE_STATUS_BAD_PAGE
    op = res["out_perm"].float().cpu().numpy()
    flat = ids.reshape(-1)
    _, offsets, perm_src, _ = orc.permute(ids, 6)
    rows3 = np.arange(offsets[3], offsets[4])
    assert np.all(op[rows3] == 0) and np.any(op[np.arange(offsets[0], offsets[1])] != 0)


# ---- tensor-core path (batches of >= TC_MIN_ROWS rows on FP8 or MXFP4 pages) --------------
# the per-token L2 bound follows the path (helpers.l2_bounds)


@pytest.mark.parametrize("E,H,I,k,T", [(4, 256, 128, 1, 300), (3, 512, 256, 2, 700), (6, 256, 384, 3, 1000)])
def test_tensor_core_path_small(cuda_lib, orc, E, H, I, k, T):
    pqe = cuda_lib
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=97)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)))
    x = synth.activations(cfg, T)
    g = np.random.default_rng(T + H)
    logits = g.standard_normal((T, E)).astype(np.float32)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, gates = orc.topk_gates(logits, k)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert counts.max() >= helpers.TC_MIN_ROWS  # at least one expert on the tensor-core path
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


def test_mixed_paths_one_call(cuda_lib, orc):
    # some experts with large batches (tensor cores), some small (CUDA cores), one 4-bit
    pqe = cuda_lib
    E, H, I, k, T = 8, 256, 128, 2, 200
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=98)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)), fp4={5})
    x = synth.activations(cfg, T)
    g = np.random.default_rng(5)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[:, 0] += 3.0   # expert 0 in almost every token
    logits[:, 5] += 3.0   # the 4-bit expert too: its MXFP4 page on the block-scaled tensor-core path
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, gates = orc.topk_gates(logits, k)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert counts[0] >= helpers.TC_MIN_ROWS and counts[5] >= helpers.TC_MIN_ROWS
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


@pytest.mark.parametrize("H,I", [(512, 256), (2048, 512)])
def test_tensor_core_path_4bit_pages(cuda_lib, orc, H, I):
    # most experts hold MXFP4 pages and batches of ~75 rows: their E2M1 weights
    # and E8M0 block scales go straight into the block-scaled MMA; one FP8
    # expert and one small 4-bit batch (weight stream) ride along
    pqe = cuda_lib
    E, k, T = 8, 2, 300
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=96)
    fp4 = {0, 1, 2, 3, 4, 6, 7}
    pages = Pages(pqe, orc, cfg, needed=set(range(E)), fp4=fp4)
    x = synth.activations(cfg, T)
    g = np.random.default_rng(H)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[:, 7] -= 4.0  # expert 7: a handful of rows (weight-stream path)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, gates = orc.topk_gates(logits, k)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert min(counts[e] for e in fp4 if e != 7) >= helpers.TC_MIN_ROWS and counts[7] < helpers.TC_MIN_ROWS
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


def tile_cover_tokens(orc, ids, E, k, tile=128):
    """Tokens whose rows are the first and the last row of every `tile`-row
    tile of every expert's batch (batch order of the permutation), so every
    tensor-core tile, and every weight-stream batch, has a checked row."""
    _, offsets, perm_src, _ = orc.permute(ids, E)
    rows = []
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        for t0 in range(a, b, tile):
            rows += [t0, min(t0 + tile, b) - 1]
    return np.unique(perm_src[np.array(rows, np.int64)] // k).astype(np.int32)


@pytest.mark.parametrize("wl,T", [("batched", 16384), ("large", 4096), ("mixed", 4096)])
def test_full_size_batched(cuda_lib, orc, wl, T):
    # the full module-batched, large-layer and mixed-precision steps (mixed: the
    # 192 experts outside the top quarter by the seeded importance hold MXFP4
    # pages, multiplied by the block-scaled MMA); checked: every token whose row
    # opens or closes a 128-row tile of some expert's batch
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    logits = synth.routing_logits(cfg, T, 0)
    ids, gates = orc.topk_gates(logits, cfg.k)
    tokens = tile_cover_tokens(orc, ids, cfg.E, cfg.k)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    assert len(tokens) >= int(np.sum(np.ceil(counts / 128.0)))  # at least one token per tile
    needed = set(ids[tokens].reshape(-1).tolist())
    fp4 = set()
    if wl == "mixed":
        m = synth.importance_init(cfg)
        order = np.lexsort((np.arange(cfg.E), -m))  # importance descending, ties to the lower id
        fp4 = set(order[cfg.E // 4:].tolist())
        assert sum(counts[e] >= helpers.TC_MIN_ROWS for e in fp4) > 100
    pages = Pages(pqe, orc, cfg, needed=needed, fp4=fp4, seed=cfg.cid)
    x = synth.activations(cfg, T, 0)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, tokens)


def test_wide_hidden_fallback_path(cuda_lib, orc):
    # H = 8192: 8 gate/up row pairs (128 KiB) do not fit two stages of the
    # streaming kernel's ring, so the grid-stride CUDA-core kernels run
    pqe = cuda_lib
    E, H, I, k, T = 2, 8192, 64, 2, 5
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=99)
    pages = Pages(pqe, orc, cfg, needed=set(range(E)), fp4={1})
    x = synth.activations(cfg, T)
    logits = np.random.default_rng(3).standard_normal((T, E)).astype(np.float32)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    ids, gates = orc.topk_gates(logits, k)
    assert res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))


def test_decode_step_tensor_core_batches_beside_stream(cuda_lib, orc):
    # a decode-sized step (at most 4 rows per routed expert on average) in which
    # two experts have 14 rows: their batches take the tensor-core path on the
    # side stream while the weight stream takes the rest. Every token is checked
    # against the oracle, and a CUDA-graph replay of the same FFN call (fork and
    # join captured) gives the eager out_perm bit for bit.
    pqe = cuda_lib
    E, H, I, k, T = 64, 256, 128, 4, 32
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, cid=89)
    g = np.random.default_rng(5)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[:14, 0] += 8.0
    logits[14:28, 1] += 8.0
    ids, gates = orc.topk_gates(logits, k)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert counts[0] >= helpers.TC_MIN_ROWS and counts[1] >= helpers.TC_MIN_ROWS
    assert helpers.TC_MIN_ROWS <= T * k <= 4 * E
    pages = Pages(pqe, orc, cfg, needed=set(range(E)))
    x = synth.activations(cfg, T)
    res = run_layer(pqe, cfg, T, x, logits_np=logits, fmt_dev=pages.fmt_dev, pool=pages.pool)
    assert np.array_equal(res["ids"], ids) and res["status"] == 0
    check_tokens(orc, pages, cfg, x, ids, gates, res, np.arange(T, dtype=np.int32))

    # the FFN call alone, eager and then replayed from a graph
    A = T * k
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    idsd = torch.from_numpy(ids.astype(np.int32)).to(DEV)
    counts_d = torch.zeros(E, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    perm_src = torch.zeros(A, dtype=torch.int32, device=DEV)
    inv = torch.zeros(A, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pws = torch.zeros(pqe.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    pqe.moe_permute(idsd, T, k, E, counts_d, offsets, perm_src, inv, pws, status)
    pt = torch.arange(E, dtype=torch.int32, device=DEV)
    fws = torch.zeros(pqe.moe_paged_ffn_workspace_size(T, k, E, H, I), dtype=torch.uint8, device=DEV)
    eager = torch.zeros((A, H), dtype=torch.bfloat16, device=DEV)
    pqe.moe_paged_ffn(xd, perm_src, offsets, pt, pages.fmt_dev, pages.pool, T, k, E, eager, fws, status)
    torch.cuda.synchronize()
    replay = torch.zeros((A, H), dtype=torch.bfloat16, device=DEV)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            pqe.moe_paged_ffn(xd, perm_src, offsets, pt, pages.fmt_dev, pages.pool, T, k, E, replay, fws, status,
                              stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        replay.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))
    assert status.item() == 0
