"""Shared test helpers: page assembly, tolerance measures, expert sets.

Pages for the CUDA path are packed by the library (pqe_pack_fp8_page /
pqe_pack_mxfp4_page); the oracle quantises the same fp32 weights itself and
the two byte images are compared. Nothing here computes the layer.
"""
from __future__ import annotations

import numpy as np

import synth

# Tolerance of the layer output (bf16) against the oracle (fp64), per token t:
#   max_i |y[t,i] - ref[t,i]| / ||ref[t]||_2 <= 2e-2   (the stated bound)
TOL_MAX_OVER_L2 = 2e-2
# The weight-streaming path multiplies exact weights by x (bf16, exact in its
# scaled f16 form) with fp32 sums, rounds h to 11 bits and out_perm and y to
# bf16 (relative 2^-9 each), so its relative L2 error per token is far
# smaller; this bound catches a wrong term that the stated bound would let
# through.
TOL_L2_GEMV = 5e-3
# The tensor-core path (per-expert batches of >= TC_MIN_ROWS rows; MXFP4
# pages multiplied exactly with their block scales) rounds x and h per row to
# E4M3 (about 2-3% RMS each); its relative L2 error per token stays below 0.1,
# which a dropped expert term (~1/k) breaks.
TOL_L2_TC = 0.1
TC_MIN_ROWS = 9


def l2_bounds(ids: np.ndarray, tokens, E: int, fp4=(), H: int = 0, I: int = 0) -> np.ndarray:
    """Per checked token: the L2 bound of the path its experts take."""
    counts = np.bincount(ids.reshape(-1), minlength=E)
    tc_shape = (H % 256 == 0 and I % 128 == 0 and H >= 256 and I >= 128) if H else True
    # FP8 and 4-bit experts alike (the block-scaled MMA multiplies MXFP4 pages as they are)
    tc_exp = (counts >= TC_MIN_ROWS) & tc_shape & (ids.size >= TC_MIN_ROWS)
    out = np.full(len(tokens), TOL_L2_GEMV)
    for i, t in enumerate(tokens):
        if tc_exp[ids[t]].any():
            out[i] = TOL_L2_TC
    return out


def bf16_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to("cpu").view(torch.int16).numpy().astype(np.uint16).astype(np.uint32).__lshift__(16) \
        .view(np.float32).astype(np.float64)


def error_stats(y: np.ndarray, ref: np.ndarray) -> dict:
    nrm = np.linalg.norm(ref, axis=1)
    nrm = np.where(nrm == 0, 1.0, nrm)
    max_over_l2 = np.max(np.abs(y - ref), axis=1) / nrm
    l2 = np.linalg.norm(y - ref, axis=1) / nrm
    return {"max_over_l2": float(max_over_l2.max()), "l2": float(l2.max()), "l2_per_token": l2}


def fp8_page_host(layout: dict, H: int, I: int, q13, s13, q2, s2) -> np.ndarray:
    page = np.zeros(layout["bytes"], np.uint8)
    page[layout["w13"]:layout["w13"] + 2 * I * H] = q13.reshape(-1)
    page[layout["w2"]:layout["w2"] + H * I] = q2.reshape(-1)
    page[layout["s13"]:layout["s13"] + 8 * I] = s13.astype(np.float32).view(np.uint8)
    page[layout["s2"]:layout["s2"] + 4 * H] = s2.astype(np.float32).view(np.uint8)
    return page


def split_fp8_page(page: np.ndarray, layout: dict, H: int, I: int):
    q13 = page[layout["w13"]:layout["w13"] + 2 * I * H].reshape(2 * I, H)
    q2 = page[layout["w2"]:layout["w2"] + H * I].reshape(H, I)
    s13 = page[layout["s13"]:layout["s13"] + 8 * I].view(np.float32)
    s2 = page[layout["s2"]:layout["s2"] + 4 * H].view(np.float32)
    return q13, s13, q2, s2


def split_mxfp4_page(page: np.ndarray, layout: dict, H: int, I: int):
    q13 = page[layout["w13"]:layout["w13"] + I * H].reshape(2 * I, H // 2)
    q2 = page[layout["w2"]:layout["w2"] + H * I // 2].reshape(H, I // 2)
    x13 = page[layout["s13"]:layout["s13"] + 2 * I * H // 32].reshape(2 * I, H // 32)
    x2 = page[layout["s2"]:layout["s2"] + H * I // 32].reshape(H, I // 32)
    return q13, x13, q2, x2


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if T <= n:
        return np.arange(T, dtype=np.int32)
    g = np.random.default_rng(seed)
    s = np.sort(g.choice(T, n, replace=False)).astype(np.int32)
    s[0], s[-1] = 0, T - 1  # keep both ends: the first and the ragged last tile
    return np.unique(s)
