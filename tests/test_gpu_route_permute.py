"""GPU parity: page quantisers, router and permutation against the oracle.

Bit-exact for codes, ids, permutation and counts; gates within 1e-6 relative
(fp32 exp against the oracle's fp64).
"""
import numpy as np
import pytest
import torch

import synth
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sync():
    torch.cuda.synchronize()


# ---- quantisers ---------------------------------------------------------------

@pytest.mark.parametrize("wl,e", [("tiny", 0), ("tiny", 7), ("decode", 11), ("large", 300)])
def test_fp8_page_pack_bit_exact(cuda_lib, orc, wl, e):
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    H, I = cfg.H, cfg.I
    w13, w2 = synth.expert_weights(cfg, e)
    page = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_FP8, H, I), dtype=torch.uint8, device=DEV)
    pqe.pqe_pack_fp8_page(torch.from_numpy(w13).to(DEV), torch.from_numpy(w2).to(DEV), H, I, page)
    _sync()
    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    ref = helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, H, I), H, I, q13, s13, q2, s2)
    assert np.array_equal(page.cpu().numpy(), ref)


def test_fp8_quant_ties_subnormals_zeros(cuda_lib, orc):
    pqe = cuda_lib
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2                 # exact ties once s == 1
    g = np.random.default_rng(0)
    rows = []
    for chunk in np.array_split(np.concatenate([mids, vals]), 4):
        r = np.zeros(64, np.float32)
        r[: len(chunk)] = chunk[:64]
        r[-1] = 448.0                                  # amax 448 -> s = 1 exactly
        rows.append(r * g.choice([-1, 1], 64).astype(np.float32))
    rows.append(np.zeros(64, np.float32))             # all zero -> s = 1
    neg = np.zeros(64, np.float32)
    neg[:] = -0.0
    neg[0] = 1.0
    neg[1:8] = -1e-12                                  # tiny negatives round to -0
    rows.append(neg)
    rows.append((g.standard_normal(64) * 1e-30).astype(np.float32))  # tiny rows: scale itself tiny
    w = np.stack(rows).astype(np.float32)
    q = torch.zeros(w.shape, dtype=torch.uint8, device=DEV)
    s = torch.zeros(w.shape[0], dtype=torch.float32, device=DEV)
    pqe.pqe_quantize_fp8_rows(torch.from_numpy(w).to(DEV), q, s)
    _sync()
    qr, sr = orc.quant_e4m3_rows(w)
    assert np.array_equal(s.cpu().numpy(), sr)
    assert np.array_equal(q.cpu().numpy(), qr)


@pytest.mark.parametrize("wl,e", [("tiny", 2), ("mixed", 40)])
def test_mxfp4_page_pack_bit_exact(cuda_lib, orc, wl, e):
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    H, I = cfg.H, cfg.I
    w13, w2 = synth.expert_weights(cfg, e)
    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    fp8 = helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, H, I), H, I, q13, s13, q2, s2)
    fp4 = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I), dtype=torch.uint8, device=DEV)
    pqe.pqe_pack_mxfp4_page(torch.from_numpy(fp8).to(DEV), H, I, fp4)
    _sync()
    lay = pqe.page_layout(pqe.PQE_FMT_MXFP4, H, I)
    a13, x13, a2, x2 = helpers.split_mxfp4_page(fp4.cpu().numpy(), lay, H, I)
    r13, y13 = orc.quant_mxfp4_rows(q13, s13)
    r2, y2 = orc.quant_mxfp4_rows(q2, s2)
    assert np.array_equal(x13, y13) and np.array_equal(x2, y2)
    assert np.array_equal(a13, r13) and np.array_equal(a2, r2)


def test_mxfp4_quant_hand_groups(cuda_lib, orc):
    pqe = cuda_lib
    g0 = [3.0, 1.0, -0.5, 0.25] + [0.0] * 28
    g1 = [1.0, 0.375, -0.0625] + [0.0] * 29
    g2 = [0.0] * 32
    g3 = [448.0, -448.0, 0.001953125, 5.5] + [0.0] * 28   # saturating block, e4m3 subnormal
    row = g0 + g1 + g2 + g3
    q8 = np.array([[orc.e4m3_encode(v) for v in row]], np.uint8)
    s8 = np.array([1.0], np.float32)
    q4 = torch.zeros((1, 64), dtype=torch.uint8, device=DEV)
    x8 = torch.zeros((1, 4), dtype=torch.uint8, device=DEV)
    pqe.pqe_quantize_mxfp4_rows(torch.from_numpy(q8).to(DEV), torch.from_numpy(s8).to(DEV), q4, x8)
    _sync()
    r4, rx = orc.quant_mxfp4_rows(q8, s8)
    assert np.array_equal(x8.cpu().numpy(), rx) and np.array_equal(q4.cpu().numpy(), r4)


# ---- router -------------------------------------------------------------------

def _route(pqe, T, H, E, k, x=None, w_r=None, logits=None):
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    gw = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    lg = logits if logits is not None else torch.zeros((T, E), dtype=torch.float32, device=DEV)
    pqe.moe_route(x, w_r, lg, T, H, E, k, ids, gw)
    _sync()
    return ids.cpu().numpy(), gw.cpu().numpy(), lg.cpu().numpy()


def test_route_router_gemm_tiny_bit_exact(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    x = synth.activations(cfg, 64)
    w_r = synth.router_weights(cfg)
    ids, gw, lg = _route(pqe, 64, cfg.H, cfg.E, cfg.k, torch.from_numpy(x.view(np.int16)).to(DEV),
                         torch.from_numpy(w_r).to(DEV))
    ref_lg = orc.router_logits(x, w_r)
    assert np.array_equal(lg.view(np.uint32), ref_lg.view(np.uint32))
    ref_ids, ref_g = orc.topk_gates(ref_lg, cfg.k)
    assert np.array_equal(ids, ref_ids)
    assert np.allclose(gw, ref_g, rtol=1e-6, atol=0)


@pytest.mark.parametrize("H,E,k,T", [(96, 5, 3, 33), (2048, 256, 8, 7), (4096, 64, 4, 130)])
def test_route_router_gemm_other_shapes(cuda_lib, orc, H, E, k, T):
    pqe = cuda_lib
    cfg = synth.small_config(E=E, H=H, I=64, k=k, T=T, cid=91)
    x = synth.activations(cfg, T)
    w_r = synth.router_weights(cfg)
    ids, gw, lg = _route(pqe, T, H, E, k, torch.from_numpy(x.view(np.int16)).to(DEV), torch.from_numpy(w_r).to(DEV))
    ref_lg = orc.router_logits(x, w_r)
    assert np.array_equal(lg.view(np.uint32), ref_lg.view(np.uint32))
    assert np.array_equal(ids, orc.topk_gates(ref_lg, k)[0])


@pytest.mark.parametrize("wl,T,step", [("decode", 64, 0), ("decode", 64, 5), ("decode", 1, 3), ("batched", 16384, 0), ("large", 4096, 0)])
def test_route_trace_logits(cuda_lib, orc, wl, T, step):
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    logits = synth.routing_logits(cfg, T, step)
    ids, gw, _ = _route(pqe, T, cfg.H, cfg.E, cfg.k, logits=torch.from_numpy(logits).to(DEV))
    ref_ids, ref_g = orc.topk_gates(logits, cfg.k)
    assert np.array_equal(ids, ref_ids)
    assert np.allclose(gw, ref_g, rtol=1e-6, atol=0)
    assert np.allclose(gw.sum(1), 1.0, atol=2e-6)


@pytest.mark.parametrize("E,k", [(1024, 32), (1024, 1), (33, 32), (32, 32), (1, 1), (40, 7)])
def test_route_extremes_with_ties(cuda_lib, orc, E, k):
    pqe = cuda_lib
    g = np.random.default_rng(E + k)
    T = 50
    logits = g.integers(-2, 3, (T, E)).astype(np.float32)   # many exact ties
    logits[0, :] = 0.0
    logits[1, ::2] = -0.0                                     # signed zeros tie too
    ids, gw, _ = _route(pqe, T, 64, E, k, logits=torch.from_numpy(logits).to(DEV))
    ref_ids, ref_g = orc.topk_gates(logits, k)
    assert np.array_equal(ids, ref_ids)
    assert np.allclose(gw, ref_g, rtol=1e-6, atol=0)


def test_route_empty(cuda_lib):
    pqe = cuda_lib
    pqe.moe_route(None, None, None, 0, 64, 8, 2, None, None)  # T == 0: no-op


# ---- permutation ----------------------------------------------------------------

def _permute(pqe, ids_np, E):
    T, k = ids_np.shape
    A = T * k
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).to(DEV)
    counts = torch.zeros(E, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    perm_src = torch.full((max(A, 1),), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((max(A, 1),), -7, dtype=torch.int32, device=DEV)
    ws = torch.zeros(max(pqe.moe_permute_workspace_size(T, k, E), 256), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pqe.moe_permute(ids, T, k, E, counts, offsets, perm_src, inv, ws, status)
    _sync()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm_src.cpu().numpy()[:A], inv.cpu().numpy()[:A], \
        int(status.item())


@pytest.mark.parametrize("wl,T", [("tiny", 64), ("decode", 1), ("decode", 64), ("batched", 16384), ("large", 4096)])
def test_permute_bit_exact_on_traces(cuda_lib, orc, wl, T):
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    if cfg.router_gemm:
        ids, _ = orc.topk_gates(orc.router_logits(synth.activations(cfg, T), synth.router_weights(cfg)), cfg.k)
    else:
        ids, _ = orc.topk_gates(synth.routing_logits(cfg, T, 0), cfg.k)
    got = _permute(pqe, ids, cfg.E)
    ref = orc.permute(ids, cfg.E)
    for a, b in zip(got[:4], ref):
        assert np.array_equal(a, b)
    assert got[4] == 0


# one chunk (a single kernel) up to 2048 assignments: the boundary, E = 1024 (four
# experts per thread in its scan), one token; then several chunks
@pytest.mark.parametrize("T,k,E", [(256, 8, 256), (64, 32, 1024), (1, 1, 1024), (2048, 1, 7),
                                   (2049, 1, 3), (5000, 3, 1024), (257, 32, 1000), (3, 2, 2)])
def test_permute_bit_exact_random(cuda_lib, orc, T, k, E):
    pqe = cuda_lib
    g = np.random.default_rng(T + E)
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    got = _permute(pqe, ids, E)
    for a, b in zip(got[:4], orc.permute(ids, E)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("E,T", [(16, 300), (1024, 300), (16, 700)])
def test_permute_bad_ids_flagged(cuda_lib, orc, E, T):
    # one chunk (T*4 <= 2048) and several (T = 700)
    pqe = cuda_lib
    g = np.random.default_rng(9)
    ids = g.integers(0, E, (T, 4)).astype(np.int32)
    ids[5, 1] = -1
    ids[77, 3] = E
    counts, offsets, perm_src, inv, status = _permute(pqe, ids, E)
    assert status & pqe.PQE_STATUS_BAD_EXPERT_ID
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < E)
    assert np.array_equal(counts, np.bincount(flat[ok], minlength=E))
    assert inv[5 * 4 + 1] == -1 and inv[77 * 4 + 3] == -1
    n = int(ok.sum())
    assert np.array_equal(perm_src[:n], np.nonzero(ok)[0][np.argsort(flat[ok], kind="stable")])
    assert np.all(perm_src[n:] == -1)


def test_permute_empty(cuda_lib):
    pqe = cuda_lib
    counts = torch.full((8,), 5, dtype=torch.int32, device=DEV)
    offsets = torch.full((9,), 5, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pqe.moe_permute(None, 0, 2, 8, counts, offsets, None, None, None, status)
    _sync()
    assert counts.sum().item() == 0 and offsets.sum().item() == 0
