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


def _ram_tier(pqe, host, nbytes, S_ram, W_ram, path, n_threads=4):
    """A RAM tier of S_ram slots (+ W_ram working entries) over a paging file
    holding the host tier's pages; RAM is pinned (the GPU pulls from it)."""
    E = len(nbytes)
    offs = pqe.pqe_paging_file_write(path, [host[e] for e in range(E)], nbytes)
    slot = -(-max(nbytes) // 4096) * 4096
    buf = torch.zeros((S_ram + W_ram) * slot + 4096, dtype=torch.uint8).pin_memory()
    a = (-buf.data_ptr()) % 4096
    ram = buf[a:a + (S_ram + W_ram) * slot]
    tier = pqe.RamTier(path, offs, nbytes, S_ram, W_ram, ram, slot, n_threads=n_threads)
    tier._buf = buf
    return tier


def _run_trace(pqe, orc, cfg, T, steps, S, W, check_every, n_check, side=True, host_api=False, device_pager=False,
               ram_slots=None, ram_wb=0, tmp_path=None, overlap_groups=0):
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
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, S, W, T, host, nbytes, expert_fmt=pages.fmt_dev,
                              device_pager=device_pager, overlap_groups=overlap_groups)
    ref_lru = orc.LRU(cfg.E, S)
    tier = ref_ram = None
    if ram_slots is not None:
        tier = _ram_tier(pqe, host, nbytes, ram_slots, ram_wb, str(tmp_path / "experts.pqe"))
        layer.attach_ram_tier(tier)
        ref_ram = orc.LRU(cfg.E, ram_slots)
        n_file = 0
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
        if not device_pager:
            assert info.n_miss == len(me) and info.working_buffer == int(wb)
        if tier is not None:  # the RAM tier: the oracle's LRU with ram_slots, driven by the VRAM misses
            need = np.zeros(cfg.E, np.int32)
            need[me] = 1
            _, r_miss, _, _ = ref_ram.step(need)
            rse, rlu, rst, _ = tier.state()
            se3, lu3, st3 = ref_ram.state()
            assert rse == se3.tolist() and rlu == lu3.tolist() and rst == st3
            assert info.n_file_read == len(r_miss)
            n_file += len(r_miss)
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
    if tier is not None:
        assert n_file > 0
        tier.close()
    return worst, n_wb


def test_layer_trace_decode_T1(cuda_lib, orc):
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=1, steps=40, S=cfg.S, W=cfg.k, check_every=13, n_check=1)


def test_layer_trace_decode_T8_same_stream(cuda_lib, orc):
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=8, steps=24, S=cfg.S, W=64, check_every=11, n_check=2, side=False)


def test_layer_trace_decode_T64_working_buffer(cuda_lib, orc):
    cfg = synth.WORKLOADS["decode"]
    worst, n_wb = _run_trace(cuda_lib, orc, cfg, T=64, steps=6, S=cfg.S, W=cfg.E, check_every=5, n_check=2)
    assert n_wb == 6   # |U| > 32 at T=64 every step


def test_layer_ram_tier_decode_T8(cuda_lib, orc, tmp_path):
    """Pages come from a paging file through 40 RAM slots (of 256 experts) and
    32 VRAM slots: RAM misses are read from the file, then pulled to VRAM."""
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=8, steps=24, S=cfg.S, W=64, check_every=7, n_check=2, ram_slots=40,
               ram_wb=64, tmp_path=tmp_path)


def test_layer_ram_tier_working_entries_T64(cuda_lib, orc, tmp_path):
    """T=64: ~140 VRAM misses per step against 128 RAM slots, so the RAM tier
    takes working-entry steps too."""
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=64, steps=5, S=cfg.S, W=cfg.E, check_every=4, n_check=2, ram_slots=128,
               ram_wb=cfg.E, tmp_path=tmp_path)


def test_layer_step_host_buffers(cuda_lib, orc):
    cfg = synth.small_config(E=12, H=256, I=128, k=3, T=20, S=5, cid=94, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=12)
    _run_trace(cuda_lib, orc, cfg, T=20, steps=12, S=5, W=12, check_every=4, n_check=20, host_api=True)


@pytest.mark.parametrize("mode", ["host", "ram", "device", "device_overlap"])
def test_layer_compressed_host_tier(cuda_lib, orc, tmp_path, mode):
    """Compressed pages pulled and decoded into the slots; with "ram", they
    come from a paging file through a RAM tier of 4 slots (compressed pages in
    RAM and in the file, as the article's compressed configurations hold);
    with "device", the LRU runs on the GPU and a decode kernel reads the step's
    miss list there (in two overlapped refill groups with "device_overlap")."""
    ram = mode == "ram"
    device = mode.startswith("device")
    pqe = cuda_lib
    cfg = synth.small_config(E=10, H=256, I=128, k=2, T=6, S=3, cid=95, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=10)
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)), seed=3)
    stride = pqe.slot_stride(cfg.H, cfg.I)
    fp8 = pages.pool_mem.view(cfg.E, stride).cpu()
    bound = pqe.pqe_huff_page_bound(cfg.H, cfg.I)
    comp = torch.zeros((cfg.E, bound), dtype=torch.uint8)
    luts = torch.zeros((cfg.E, 2 * pqe.PQE_HUFF_LUT_BYTES), dtype=torch.uint8)
    sizes = []
    for e in range(cfg.E):
        n = pqe.pqe_huff_encode_page(fp8[e].contiguous(), cfg.H, cfg.I, comp[e], luts[e, :pqe.PQE_HUFF_LUT_BYTES], luts[e, pqe.PQE_HUFF_LUT_BYTES:])
        sizes.append(n)
    host = comp.pin_memory()
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, cfg.E, cfg.T[0], host, sizes, compressed=True,
                              luts=luts.to(DEV), expert_fmt=pages.fmt_dev, device_pager=device,
                              overlap_groups=2 if mode == "device_overlap" else 0)
    tier = None
    if ram:
        tier = _ram_tier(pqe, host, sizes, 4, cfg.E, str(tmp_path / "comp.pqe"), n_threads=2)
        layer.attach_ram_tier(tier)
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
        if device:  # the GPU-resident LRU against the oracle's, every step
            se_, lu_, st_ = layer.lru_state()
            se2, lu2, st2 = ref_lru.state()
            assert np.array_equal(se_.numpy(), se2) and np.array_equal(lu_.numpy(), lu2) and st_ == st2, s
        ref = orc.moe_ffn(x_np, ids, g, pages.experts, cfg.I)
        st = helpers.error_stats(helpers.bf16_to_f64(y), ref)
        bound = helpers.l2_bounds(ids, np.arange(6), cfg.E, (), cfg.H, cfg.I)
        assert st["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st["l2_per_token"] <= bound), (s, st)
    if device:
        total_miss = int(layer.device_stats()["misses"])
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
    if tier is not None:
        assert tier.state()[3]["reads"] > 0
        tier.close()


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


def test_layer_device_pager_trace(cuda_lib, orc):
    # LRU state, misses and refills on the GPU: same slot states as the oracle
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=8, steps=30, S=cfg.S, W=cfg.E, check_every=7, n_check=3, device_pager=True)


def test_layer_device_pager_working_buffer(cuda_lib, orc):
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=64, steps=5, S=cfg.S, W=cfg.E, check_every=4, n_check=2, device_pager=True)


@pytest.mark.parametrize("groups", [1, 3])
def test_layer_device_pager_overlapped_refills(cuda_lib, orc, groups):
    # misses refilled in groups on the side stream while the FFN runs in passes
    # (resident experts first, then each group's): same LRU states as the oracle
    # and every token of the checked steps within the bounds
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=8, steps=30, S=cfg.S, W=cfg.E, check_every=5, n_check=8, device_pager=True,
               overlap_groups=groups)


@pytest.mark.parametrize("T,groups", [(8, 3), (64, 5)])
def test_layer_overlapped_steps_bit_identical(cuda_lib, orc, T, groups):
    # the passes compute every expert with the same kernels and summation order
    # as one FFN call: y, the page table and the LRU state equal a plain layer's
    # bit for bit, step after step
    pqe = cuda_lib
    cfg = synth.WORKLOADS["decode"]
    pages = Pages(pqe, orc, cfg, needed=set(), seed=3)
    host, nbytes = _host_tier(pqe, pages)
    tr = synth.RoutingTrace(cfg, T)
    mk = lambda g: pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, cfg.E, T, host, nbytes,
                                     expert_fmt=pages.fmt_dev, device_pager=True, overlap_groups=g)
    plain, ovl = mk(0), mk(groups)
    side = torch.cuda.Stream()
    y0 = torch.zeros((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    y1 = torch.zeros_like(y0)
    for s in range(6):
        x = torch.from_numpy(synth.activations(cfg, T, s).view(np.int16)).to(DEV)
        lg = torch.from_numpy(tr.step(s)).to(DEV)
        plain.step(x, y0, T, logits=lg, side_stream=side)
        ovl.step(x, y1, T, logits=lg, side_stream=side)
        torch.cuda.synchronize()
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), s
        pt0 = plain.device_view("page_table", torch.int32, (cfg.E,)).clone()
        pt1 = ovl.device_view("page_table", torch.int32, (cfg.E,)).clone()
        assert torch.equal(pt0, pt1), s
        a, b = plain.lru_state(), ovl.lru_state()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and a[2] == b[2], s
    for l in (plain, ovl):
        assert l.device_view("status", torch.int32, (1,)).item() == 0
        l.close()


def test_layer_device_pager_overlapped_working_buffer(cuda_lib, orc):
    # every routed expert a miss: the resident pass is empty, four refill groups
    cfg = synth.WORKLOADS["decode"]
    _run_trace(cuda_lib, orc, cfg, T=64, steps=5, S=cfg.S, W=cfg.E, check_every=2, n_check=8, device_pager=True,
               overlap_groups=4)


@pytest.mark.parametrize("groups", [0, 2])
def test_layer_device_pager_graph_replay(cuda_lib, orc, groups):
    # with the device pager a whole step has no host synchronisation: capture it
    # once in a CUDA graph and replay it on new inputs copied into its buffers
    # (groups > 0: the refill groups on a side stream inside the graph)
    pqe = cuda_lib
    cfg = synth.small_config(E=16, H=256, I=128, k=2, T=8, S=4, cid=80, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=8)
    T = 8
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)), seed=11)
    host, nbytes = _host_tier(pqe, pages)
    layer = pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, cfg.E, T, host, nbytes, expert_fmt=pages.fmt_dev,
                              device_pager=True, overlap_groups=groups)
    side = torch.cuda.Stream() if groups else None
    tr = synth.RoutingTrace(cfg, T)
    logits_all = [tr.step(s) for s in range(8)]
    x_buf = torch.zeros((T, cfg.H), dtype=torch.int16, device=DEV)
    lg_buf = torch.zeros((T, cfg.E), dtype=torch.float32, device=DEV)
    y = torch.zeros((T, cfg.H), dtype=torch.bfloat16, device=DEV)
    # step 0 eagerly (also warms up the launch paths), then capture step 1
    x_buf.copy_(torch.from_numpy(synth.activations(cfg, T, 0).view(np.int16)))
    lg_buf.copy_(torch.from_numpy(logits_all[0]))
    layer.step(x_buf, y, T, logits=lg_buf, side_stream=side)
    torch.cuda.synchronize()
    ref_lru = orc.LRU(cfg.E, cfg.S)
    ref_lru.step(np.bincount(orc.topk_gates(logits_all[0], cfg.k)[0].reshape(-1), minlength=cfg.E).astype(np.int32))
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            layer.step(x_buf, y, T, logits=lg_buf, stream=stream, side_stream=side)
    torch.cuda.synchronize()
    # capture did not run the step: the LRU state is still after step 0
    assert layer.lru_state()[2] == 1
    for s in range(1, 8):
        x_np = synth.activations(cfg, T, s)
        x_buf.copy_(torch.from_numpy(x_np.view(np.int16)))
        lg_buf.copy_(torch.from_numpy(logits_all[s]))
        g.replay()
        torch.cuda.synchronize()
        ids, gates = orc.topk_gates(logits_all[s], cfg.k)
        ref_lru.step(np.bincount(ids.reshape(-1), minlength=cfg.E).astype(np.int32))
        se, lu, st = layer.lru_state()
        se2, lu2, st2 = ref_lru.state()
        assert np.array_equal(se.numpy(), se2) and np.array_equal(lu.numpy(), lu2) and st == st2, s
        ref = orc.moe_ffn(x_np, ids, gates, pages.experts, cfg.I)
        st_ = helpers.error_stats(helpers.bf16_to_f64(y), ref)
        bound = helpers.l2_bounds(ids, np.arange(T), cfg.E, (), cfg.H, cfg.I)
        assert st_["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st_["l2_per_token"] <= bound), (s, st_)
    assert layer.device_view("status", torch.int32, (1,)).item() == 0
    layer.close()


@pytest.mark.parametrize("groups", [0, 3])
def test_layer_step_host_graph_replays(cuda_lib, orc, groups):
    # pqe_layer_step_host on a device-pager layer replays each step shape from a
    # graph after its second call: y, the page table and the LRU state equal
    # those of the same layer stepping eagerly, bit for bit, across step sizes,
    # a changed wait limit (the graph is captured again) and the oracle's LRU;
    # replayed calls count no launch of their own
    pqe = cuda_lib
    cfg = synth.small_config(E=16, H=256, I=128, k=2, T=8, S=4, cid=81, reuse_p=0.5, zipf_s=1.1,
                             router_gemm=False, steps=14)
    pages = Pages(pqe, orc, cfg, needed=set(range(cfg.E)), seed=12)
    host, nbytes = _host_tier(pqe, pages)
    mk = lambda: pqe.PagedMoELayer(cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, cfg.E, 8, host, nbytes,
                                   expert_fmt=pages.fmt_dev, device_pager=True, overlap_groups=groups)
    graphed, eager = mk(), mk()
    eager.set_step_graphs(False)
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    Ts = [8, 8, 8, 5, 8, 5, 5, 8, 8, 3, 5, 8, 8, 8]
    ref_lru = orc.LRU(cfg.E, cfg.S)
    y_g = torch.zeros((8, cfg.H), dtype=torch.int16).pin_memory()
    y_e = torch.zeros_like(y_g).pin_memory()
    calls = {}  # calls of each step size since the settings last changed
    try:
        for s, T in enumerate(Ts):
            if s == 9:
                pqe.pqe_set_wait_limit(1 << 23)  # a new setting: shapes are captured again
                calls = {}
            tr = synth.RoutingTrace(cfg, T)
            lg = tr.step(s)
            x_np = synth.activations(cfg, T, s)
            x_h = torch.from_numpy(x_np.view(np.int16)).pin_memory()
            lg_h = torch.from_numpy(lg).pin_memory()
            n0 = pqe.kernel_launches()
            graphed.step_host(x_h, y_g, T, logits_host=lg_h, stream=stream, side_stream=side)
            n_graphed = pqe.kernel_launches() - n0
            eager.step_host(x_h, y_e, T, logits_host=lg_h, stream=stream, side_stream=side)
            c = calls.get(T, 0)  # 0: eager, 1: captured and launched, then replays
            assert (n_graphed == 0) == (c >= 2), (s, T, c, n_graphed)
            calls[T] = c + 1
            assert torch.equal(y_g[:T], y_e[:T]), s
            pt0 = graphed.device_view("page_table", torch.int32, (cfg.E,)).clone()
            pt1 = eager.device_view("page_table", torch.int32, (cfg.E,)).clone()
            assert torch.equal(pt0, pt1), s
            ids, gates = orc.topk_gates(lg, cfg.k)
            ref_lru.step(np.bincount(ids.reshape(-1), minlength=cfg.E).astype(np.int32))
            se, lu, st = graphed.lru_state()
            se2, lu2, st2 = ref_lru.state()
            assert np.array_equal(se.numpy(), se2) and np.array_equal(lu.numpy(), lu2) and st == st2, s
            ref = orc.moe_ffn(x_np, ids, gates, pages.experts, cfg.I)
            y = y_g[:T].view(torch.bfloat16)
            st_ = helpers.error_stats(helpers.bf16_to_f64(y), ref)
            bound = helpers.l2_bounds(ids, np.arange(T), cfg.E, (), cfg.H, cfg.I)
            assert st_["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st_["l2_per_token"] <= bound), (s, st_)
    finally:
        pqe.pqe_set_wait_limit(0)
    for l in (graphed, eager):
        assert l.device_view("status", torch.int32, (1,)).item() == 0
        l.close()


def test_layer_mixed_precision_reranking(cuda_lib, orc):
    # config-5 behaviour at a small size: every `every` steps the experts are
    # re-ranked by the EMA of their gate mass; the top quarter keep FP8 pages,
    # the rest get 4-bit pages; a changed expert's page is swapped on the host
    # and its resident copy forgotten, so its next use refills the new page
    pqe = cuda_lib
    E, H, I, k, T, every, n_hi = 32, 256, 128, 4, 48, 6, 8
    cfg = synth.small_config(E=E, H=H, I=I, k=k, T=T, S=E, cid=81, reuse_p=0.7, zipf_s=1.1, router_gemm=False,
                             steps=24)
    stride = pqe.slot_stride(H, I)
    lay8 = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
    n8, n4 = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I), pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I)
    fp8_pages = torch.zeros((E, stride), dtype=torch.uint8)
    fp4_pages = torch.zeros((E, stride), dtype=torch.uint8)
    ex8, ex4 = {}, {}
    dev_page = torch.zeros(stride, dtype=torch.uint8, device=DEV)
    dev_p4 = torch.zeros(n4, dtype=torch.uint8, device=DEV)
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e)
        pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(DEV), torch.from_numpy(w2).to(DEV), H, I, dev_page)
        pqe.pqe_pack_mxfp4_page(dev_page, H, I, dev_p4)
        fp8_pages[e] = dev_page.cpu()
        fp4_pages[e, :n4] = dev_p4.cpu()
        q13, s13 = orc.quant_e4m3_rows(w13)
        q2, s2 = orc.quant_e4m3_rows(w2)
        ex8[e] = (q13, s13, q2, s2)
        ex4[e] = orc.quant_mxfp4_rows(q13, s13) + orc.quant_mxfp4_rows(q2, s2)
    fp8_pages, fp4_pages = fp8_pages.pin_memory(), fp4_pages.pin_memory()
    m_lib = synth.importance_init(cfg)
    m_orc = m_lib.copy()
    fmt = np.zeros(E, np.uint8)
    pqe.pqe_rank_formats(torch.from_numpy(m_lib), n_hi, torch.from_numpy(fmt))
    fmt_orc = orc.rank_formats(m_orc, n_hi)
    assert np.array_equal(fmt, fmt_orc)
    host = [fp8_pages[e] if fmt[e] == 0 else fp4_pages[e] for e in range(E)]
    sizes = [n8 if fmt[e] == 0 else n4 for e in range(E)]
    fmt_dev = torch.from_numpy(fmt.copy()).to(DEV)
    layer = pqe.PagedMoELayer(E, H, I, k, E, 0, T, host, sizes, expert_fmt=fmt_dev)
    ref_lru = orc.LRU(E, E)
    tr = synth.RoutingTrace(cfg, T)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    n_changes = 0
    for s in range(24):
        logits = tr.step(s)
        x_np = synth.activations(cfg, T, s)
        layer.step(torch.from_numpy(x_np.view(np.int16)).to(DEV), y, T, logits=torch.from_numpy(logits).to(DEV))
        torch.cuda.synchronize()
        ids = layer.device_view("topk_ids", torch.int32, (T, k)).cpu().numpy()
        gates32 = layer.device_view("topk_w", torch.float32, (T, k)).cpu().numpy()
        ids_ref, gates_ref = orc.topk_gates(logits, k)
        assert np.array_equal(ids, ids_ref)
        ref_lru.step(np.bincount(ids.reshape(-1), minlength=E).astype(np.int32))
        assert np.array_equal(layer.lru_state()[0].numpy(), ref_lru.state()[0])
        experts = orc.ExpertSet(E)
        for e in range(E):
            experts.set(e, int(fmt[e]), *(ex8[e] if fmt[e] == 0 else ex4[e]))
        ref = orc.moe_ffn(x_np, ids_ref, gates_ref, experts, I)
        st = helpers.error_stats(helpers.bf16_to_f64(y), ref)
        bound = helpers.l2_bounds(ids_ref, np.arange(T), E, set(np.nonzero(fmt == 1)[0].tolist()), H, I)
        assert st["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and np.all(st["l2_per_token"] <= bound), (s, st)
        # importance and re-ranking: library (host) and oracle bit for bit
        old = fmt.copy()
        r1 = pqe.pqe_importance_step(torch.from_numpy(m_lib), torch.from_numpy(ids), torch.from_numpy(gates32),
                                     T, k, E, 0.9, s, every, n_hi, torch.from_numpy(fmt))
        r2 = orc.importance_step(m_orc, ids, gates32, E, s, fmt_orc, alpha=0.9, every=every, n_hi=n_hi)
        assert r1 == r2 and np.array_equal(m_lib, m_orc) and np.array_equal(fmt, fmt_orc)
        for e in np.nonzero(fmt != old)[0]:
            page = fp8_pages[e] if fmt[e] == 0 else fp4_pages[e]
            layer.set_host_page(int(e), page, n8 if fmt[e] == 0 else n4)
            ref_lru.invalidate(int(e))
            n_changes += 1
        if (fmt != old).any():
            fmt_dev.copy_(torch.from_numpy(fmt))
    assert n_changes > 0
    assert int((fmt == 0).sum()) == n_hi
    assert layer.device_view("status", torch.int32, (1,)).item() == 0
    layer.close()


def test_layer_large_shapes_compressed(cuda_lib, orc):
    # E=512, H=2560, I=640, 46 slots, Huffman-compressed host tier decoded on the
    # GPU after every refill. 16 distinct pages, expert e uses page e % 16.
    pqe = cuda_lib
    cfg = synth.WORKLOADS["large"]
    E, H, I, k, S, T = cfg.E, cfg.H, cfg.I, cfg.k, cfg.S, 1
    n_src = 16
    stride = pqe.slot_stride(H, I)
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    bound = pqe.pqe_huff_page_bound(H, I)
    comp = torch.zeros((n_src, bound), dtype=torch.uint8)
    luts_src = torch.zeros((n_src, 2 * pqe.PQE_HUFF_LUT_BYTES), dtype=torch.uint8)
    sizes_src, src_w = [], []
    dev_page = torch.zeros(stride, dtype=torch.uint8, device=DEV)
    for j in range(n_src):
        w13, w2 = synth.expert_weights(cfg, j)
        pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(DEV), torch.from_numpy(w2).to(DEV), H, I, dev_page)
        page = dev_page[:nb].cpu().contiguous()
        sizes_src.append(pqe.pqe_huff_encode_page(page, H, I, comp[j], luts_src[j, :pqe.PQE_HUFF_LUT_BYTES], luts_src[j, pqe.PQE_HUFF_LUT_BYTES:]))
        q13, s13 = orc.quant_e4m3_rows(w13)
        q2, s2 = orc.quant_e4m3_rows(w2)
        src_w.append((q13, s13, q2, s2))
        assert sizes_src[-1] < 0.9 * nb
    comp = comp.pin_memory()
    host = [comp[e % n_src] for e in range(E)]
    sizes = [sizes_src[e % n_src] for e in range(E)]
    luts = luts_src[torch.arange(E) % n_src].contiguous().to(DEV)
    experts = orc.ExpertSet(E)
    for e in range(E):
        experts.set(e, 0, *src_w[e % n_src])
    layer = pqe.PagedMoELayer(E, H, I, k, S, E, T, host, sizes, compressed=True, luts=luts)
    ref_lru = orc.LRU(E, S)
    tr = synth.RoutingTrace(cfg, T)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    misses = 0
    for s in range(12):
        logits = tr.step(s)
        x_np = synth.activations(cfg, T, s)
        info = layer.step(torch.from_numpy(x_np.view(np.int16)).to(DEV), y, T,
                          logits=torch.from_numpy(logits).to(DEV), side_stream=side)
        misses += info.n_miss
        ids, g = orc.topk_gates(logits, k)
        _, me, _, _ = ref_lru.step(np.bincount(ids.reshape(-1), minlength=E).astype(np.int32))
        assert info.n_miss == len(me)
        torch.cuda.synchronize()
        assert np.array_equal(layer.lru_state()[0].numpy(), ref_lru.state()[0])
        ref = orc.moe_ffn(x_np, ids, g, experts, I)
        st = helpers.error_stats(helpers.bf16_to_f64(y), ref)
        assert st["max_over_l2"] <= helpers.TOL_MAX_OVER_L2 and st["l2"] <= helpers.TOL_L2_GEMV, (s, st)
    assert misses >= 8
    assert layer.device_view("status", torch.int32, (1,)).item() == 0
    layer.close()
