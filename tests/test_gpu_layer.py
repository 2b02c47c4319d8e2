"""GPU parity of the layer runtime (pqe_layer_step): a routing trace through the
per-layer LRU slot pool with side-stream refills from pinned host pages.

Per step: the LRU state and misses equal the oracle's pool driven by the
oracle's routing (bit for bit), and sampled tokens of y match the oracle FFN
within the tolerance."""
import numpy as np
import pytest
import torch

import synth
from tests import helpers
from tests.test_gpu_ffn import Pages

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host_tier(pqe, pages: Pages):
    cfg = pages.cfg
    stride = pqe.slot_stride(cfg.H, cfg.I)
    host = pages.pool_mem.view(cfg.E, stride).cpu().pin_memory()
    nbytes = [pqe.page_bytes(int(pages.fmt[e]), cfg.H, cfg.I) for e in range(cfg.E)]
    return host, nbytes


def _run_trace(pqe, orc, cfg, T, steps, S, W, check_every, n_check, side=True, host_api=False):
    # experts the checked tokens of the checked steps use get oracle weights
    tr = synth.RoutingTrace(cfg, T)
    logits_all = [tr.step(s) for s in range(steps)]
    checks = {}
    needed = set()
    for s in range(0, steps, check_every):
        ids, g = orc.topk_gates(logits_all[s], cfg.k)
        tok = helpers.sample_tokens(T, n_check, seed=s)
        checks[s] = (ids, g, tok)
        needed |= set(ids[tok].reshape(-1).tolist())
    pages = Pages(pqe, orc, cfg, needed=needed, seed=7)
    host, nbytes = _host_tier(pqe, pages)
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, S, W, T, host, nbytes, expert_fmt=pages.fmt_dev)
    ref_lru = orc.LRU(cfg.E, S)
    stream = torch.cuda.current_stream()
    side_stream = torch.cuda.Stream() if side else None
    y = torch.zeros((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    if host_api:
        y_host = torch.zeros((T, cfg.H), dtype=torch.bfloat16).pin_memory()
    worst = {"max_over_l2": 0.0, "l2": 0.0}
    n_wb = 0
    for s in range(steps):
        x_np = synth.activations(cfg, T, s)
        if host_api:
            x_host = torch.from_numpy(x_np.view(np.int16)).pin_memory()
            lg_host = torch.from_numpy(logits_all[s]).pin_memory()
            info = layer.step_host(x_host, y_host, T, logits_host=lg_host, stream=stream, side_stream=side_stream)
            y.copy_(y_host.view(torch.bfloat16))
        else:
            x = torch.from_numpy(x_np.view(np.int16)).to(DEV)
            lg = torch.from_numpy(logits_all[s]).to(DEV)
            info = layer.step(x, y, T, logits=lg, stream=stream, side_stream=side_stream)
        ids_ref, _ = orc.topk_gates(logits_all[s], cfg.k)
        counts = np.bincount(ids_ref.reshape(-1), minlength=cfg.E).astype(np.int32)
        pt, me, md, wb = ref_lru.step(counts)
        se, lu, st = layer.lru_state()
        se2, lu2, st2 = ref_lru.state()
        assert np.array_equal(se.numpy(), se2) and np.array_equal(lu.numpy(), lu2) and st == st2
        assert info.n_miss == len(me) and info.working_buffer == int(wb)
        n_wb += int(wb)
        torch.cuda.synchronize()
        if s in checks:
            ids, g, tok = checks[s]
            got_ids = layer.device_view("topk_ids", torch.int32, (T, cfg.k)).cpu().numpy()
            assert np.array_equal(got_ids, ids)
            ref = orc.moe_ffn(x_np, ids, g, pages.experts, cfg.I, tokens=tok)
            st_ = helpers.error_stats(helpers.bf16_to_f64(y)[tok], ref)
            bound = helpers.l2_bounds(ids, tok, cfg.E, (), cfg.H, cfg.I)
            assert st_["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st_["l2_per_token"] <= bound), (s, st_)
            worst = {k: max(worst[k], st_[k]) for k in worst}
    status = layer.device_view("status", torch.int32, (1,)).item()
    assert status == 0
    layer.close()
    return worst, n_wb


def test_layer_trace_config2_T1(cuda_lib, orc):
    cfg = synth.CONFIGS[2]
    _run_trace(cuda_lib, orc, cfg, T=1, steps=40, S=cfg.S, W=cfg.k, check_every=13, n_check=1)


def test_layer_trace_config2_T8_same_stream(cuda_lib, orc):
    cfg = synth.CONFIGS[2]
    _run_trace(cuda_lib, orc, cfg, T=8, steps=24, S=cfg.S, W=64, check_every=11, n_check=2, side=False)


def test_layer_trace_config2_T64_working_buffer(cuda_lib, orc):
    cfg = synth.CONFIGS[2]
    worst, n_wb = _run_trace(cuda_lib, orc, cfg, T=64, steps=6, S=cfg.S, W=cfg.E, check_every=5, n_check=2)
    assert n_wb == 6   # |U| > 32 at T=64 every step


def test_layer_step_host_buffers(cuda_lib, orc):
    cfg = synth.small_config(E=12, H=256, I=128, k=3, T=20, S=5, cid=94, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=12)
    _run_trace(cuda_lib, orc, cfg, T=20, steps=12, S=5, W=12, check_every=4, n_check=20, host_api=True)


def test_layer_compressed_host_tier(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.small_config(E=10, H=256, I=128, k=2, T=6, S=3, cid=95, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=10)
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)), seed=3)
    stride = pqe.slot_stride(cfg.H, cfg.I)
    fp8 = pages.pool_mem.view(cfg.E, stride).cpu()
    bound = pqe.pqe_huff_page_bound(cfg.H, cfg.I)
    comp = torch.zeros((cfg.E, bound), dtype=torch.uint8)
    luts = torch.zeros((cfg.E, 2 * 4096), dtype=torch.uint8)
    sizes = []
    for e in range(cfg.E):
        n = pqe.pqe_huff_encode_page(fp8[e].contiguous(), cfg.H, cfg.I, comp[e], luts[e, :4096], luts[e, 4096:])
        sizes.append(n)
    host = comp.pin_memory()
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, cfg.E, cfg.T[0], host, sizes, compressed=True,
                              luts=luts.to(DEV), expert_fmt=pages.fmt_dev)
    tr = synth.RoutingTrace(cfg, 6)
    ref_lru = orc.LRU(cfg.E, cfg.S)
    y = torch.zeros((6, cfg.H), dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    total_miss = 0
    for s in range(10):
        logits = tr.step(s)
        x_np = synth.activations(cfg, 6, s)
        info = layer.step(torch.from_numpy(x_np.view(np.int16)).to(DEV), y, 6,
                          logits=torch.from_numpy(logits).to(DEV), side_stream=side)
        total_miss += info.n_miss
        ids, g = orc.topk_gates(logits, cfg.k)
        ref_lru.step(np.bincount(ids.reshape(-1), minlength=cfg.E).astype(np.int32))
        torch.cuda.synchronize()
        ref = orc.moe_ffn(x_np, ids, g, pages.experts, cfg.I)
        st = helpers.error_stats(helpers.bf16_to_f64(y), ref)
        bound = helpers.l2_bounds(ids, np.arange(6), cfg.E, (), cfg.H, cfg.I)
        assert st["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st["l2_per_token"] <= bound), (s, st)
    assert total_miss > 0
    assert layer.device_view("status", torch.int32, (1,)).item() == 0
    # the resident slots hold the decoded FP8 pages byte for byte
    se, _, _ = layer.lru_state()
    lay = pqe.page_layout(pqe.PQE_FMT_FP8, cfg.H, cfg.I)
    for slot, e in enumerate(se.tolist()):
        if e >= 0:
            got = layer.pool_mem[slot * stride:slot * stride + lay["bytes"]].cpu()
            assert torch.equal(got, fp8[e, :lay["bytes"]])
    layer.close()


def test_layer_capacity_error(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.small_config(E=8, H=64, I=64, k=4, T=4, S=2, cid=96)
    pages = Pages(pqe, orc, cfg, needed=set(), seed=1)
    host, nbytes = _host_tier(pqe, pages)
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, 2, 1, 4, host, nbytes)
    logits = np.tile(np.arange(8, dtype=np.float32), (4, 1))  # 4 experts > 2 slots, 2 misses > W=1
    x = torch.zeros((4, cfg.H), dtype=torch.int16, device=DEV)
    y = torch.zeros((4, cfg.H), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pqe.PqeError) as ei:
        layer.step(x, y, 4, logits=torch.from_numpy(logits).to(DEV))
    assert ei.value.code == pqe.PQE_ERR_CAPACITY
    torch.cuda.synchronize()
    layer.close()
