"""Pins of the oracle's expert FFN and combine.

Independent references: a closed form on constructed weights (identity /
permutation matrices), and PyTorch's own linear + SiLU composition (a library
routine) on weights dequantised by PyTorch's float8 view and by the OCP MX
value tables.
"""
import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import synth

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _torch_deq_fp8(q, s):
    v = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64)
    return v * torch.from_numpy(s.astype(np.float64))[:, None]


def _torch_deq_fp4(q4, e8):
    nib = np.empty((q4.shape[0], q4.shape[1] * 2), np.uint8)
    nib[:, 0::2] = q4 & 15
    nib[:, 1::2] = q4 >> 4
    sc = np.ldexp(1.0, e8.astype(np.int64) - 127)
    return torch.from_numpy(E2M1[nib] * np.repeat(sc, 32, axis=1))


def _swiglu_ffn(x, w13, w2, I):
    u = F.linear(x, w13)
    return F.linear(F.silu(u[..., :I]) * u[..., I:], w2)


def test_closed_form_identity_experts(orc):
    # I = H. Expert e: gate rows = c_e * Id, up rows = Id, w2 = d_e * P_e (P_e a
    # permutation). Then o = d_e * P_e (SiLU(c_e x) * x) and y = sum_j g_j o_j.
    # Distinct c_e / d_e / P_e expose a swapped gate/up half, a transposed w2,
    # a wrong expert index or a wrong gate.
    H = I = 64
    E, k, T = 4, 2, 16
    g = np.random.default_rng(0)
    c = [0.5, 1.0, 2.0, 4.0]
    d = [1.0, -2.0, 0.25, 3.0]
    perms = [g.permutation(H) for _ in range(E)]
    ex = orc.ExpertSet(E)
    for e in range(E):
        w13 = np.zeros((2 * I, H), np.uint8)
        w13[np.arange(I), np.arange(I)] = 0x38          # 1.0
        w13[I + np.arange(I), np.arange(I)] = 0x38
        s13 = np.array([c[e]] * I + [1.0] * I, np.float32)
        w2 = np.zeros((H, I), np.uint8)
        w2[np.arange(H), perms[e]] = 0x38
        s2 = np.full(H, d[e], np.float32)
        ex.set(e, 0, w13, s13, w2, s2)
    x = synth.to_bf16_bits(g.standard_normal((T, H)).astype(np.float32))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    logits = g.standard_normal((T, E)).astype(np.float32)
    ids, gates = orc.topk_gates(logits, k)
    y = orc.moe_ffn(x, ids, gates, ex, I)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            h = scipy.special.expit(c[e] * xf[t]) * c[e] * xf[t] * xf[t]
            ref[t] += gates[t, j] * d[e] * h[perms[e]]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def _fp8_experts(orc, cfg, E):
    ex = orc.ExpertSet(E)
    deq = []
    for e in range(E):
        w13, w2 = synth.expert_weights(cfg, e)
        q13, s13 = orc.quant_e4m3_rows(w13)
        q2, s2 = orc.quant_e4m3_rows(w2)
        ex.set(e, 0, q13, s13, q2, s2)
        deq.append((_torch_deq_fp8(q13, s13), _torch_deq_fp8(q2, s2)))
    return ex, deq


def test_single_expert_matches_torch(orc):
    cfg = synth.small_config(E=3, H=128, I=64, k=1, T=24)
    ex, deq = _fp8_experts(orc, cfg, cfg.E)
    x = synth.activations(cfg, 24)
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    ids = np.full((24, 1), 2, np.int32)
    gates = np.ones((24, 1))
    y = orc.moe_ffn(x, ids, gates, ex, cfg.I)
    ref = _swiglu_ffn(xt, deq[2][0], deq[2][1], cfg.I).numpy()
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_all_experts_is_dense_mixture(orc):
    # k = E: every expert is picked and the gates are the full softmax
    cfg = synth.WORKLOADS["tiny"]
    ex, deq = _fp8_experts(orc, cfg, cfg.E)
    x = synth.activations(cfg, 64)
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    logits = synth.router_weights(cfg)[:, :1].T.repeat(64, 0) + \
        np.random.default_rng(2).standard_normal((64, cfg.E)).astype(np.float32)
    ids, gates = orc.topk_gates(logits, cfg.E)
    y = orc.moe_ffn(x, ids, gates, ex, cfg.I)
    soft = scipy.special.softmax(logits.astype(np.float64), axis=1)
    ref = sum(soft[:, e:e + 1] * _swiglu_ffn(xt, deq[e][0], deq[e][1], cfg.I).numpy() for e in range(cfg.E))
    assert np.allclose(y, ref, rtol=1e-9, atol=1e-12)


def test_fp4_experts_match_torch(orc):
    cfg = synth.small_config(E=2, H=128, I=64, k=2, T=10)
    ex = orc.ExpertSet(2)
    deq = []
    for e in range(2):
        w13, w2 = synth.expert_weights(cfg, e)
        q13, s13 = orc.quant_e4m3_rows(w13)
        q2, s2 = orc.quant_e4m3_rows(w2)
        a13, b13 = orc.quant_mxfp4_rows(q13, s13)
        a2, b2 = orc.quant_mxfp4_rows(q2, s2)
        ex.set(e, 1, a13, b13, a2, b2)
        deq.append((_torch_deq_fp4(a13, b13), _torch_deq_fp4(a2, b2)))
    x = synth.activations(cfg, 10)
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    ids = np.tile(np.array([[1, 0]], np.int32), (10, 1))
    gates = np.tile(np.array([[0.75, 0.25]]), (10, 1))
    y = orc.moe_ffn(x, ids, gates, ex, cfg.I)
    ref = 0.75 * _swiglu_ffn(xt, *deq[1], cfg.I) + 0.25 * _swiglu_ffn(xt, *deq[0], cfg.I)
    assert np.allclose(y, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_token_subset_equals_full(orc):
    cfg = synth.WORKLOADS["tiny"]
    ex, _ = _fp8_experts(orc, cfg, cfg.E)
    x = synth.activations(cfg, 64)
    lg = orc.router_logits(x, synth.router_weights(cfg))
    ids, gates = orc.topk_gates(lg, cfg.k)
    full = orc.moe_ffn(x, ids, gates, ex, cfg.I)
    sub = orc.moe_ffn(x, ids, gates, ex, cfg.I, tokens=[63, 0, 17])
    assert np.array_equal(sub, full[[63, 0, 17]])
