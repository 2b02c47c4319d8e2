"""Seeded synthetic inputs for the paged, quantized MoE expert layer.

This module is shared by the oracle-side tests and the CUDA path. It draws
random numbers and shapes them into the workloads' structure; it holds none of
the layer's arithmetic (no quantisation, routing, permutation or FFN math).

Shapes follow the model sizes the pages quote:
  * 40 MoE layers x 256 experts ~= 30 GiB of FP8 expert weights
    (vllm-expert-pager article, "はじめに") -> 3 MiB per expert = 3*H*I bytes
    with H=2048, I=512;
  * 48 layers x 512 experts = 112.5 GiB (same article, Table 3 prose)
    -> 4.6875 MiB per expert = 3*H*I with H=2560, I=640.
Routing skew follows the pages' observation that recently chosen experts are
chosen again (same article, "エキスパート重みの階層ページング"): a token slot
keeps its previous expert set with probability 0.7, else draws k distinct
experts from a Zipf(s=1.1) law over a seeded permutation of the ids.

All draws use numpy's PCG64 seeded from ``SEED_BASE + 1000*config + step``
plus a per-tensor tag, so any tensor can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Iterator

import numpy as np

SEED_BASE = 20260720

# per-tensor tags mixed into the seed sequence
_TAG_X = 1
_TAG_WR = 2
_TAG_W13 = 3
_TAG_W2 = 4
_TAG_TRACE = 5
_TAG_IMPORTANCE = 6
_TAG_PERM = 7


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """One MoE layer workload."""
    cid: int            # config number (1..5)
    name: str
    E: int              # experts
    H: int              # hidden size
    I: int              # expert intermediate size
    k: int              # experts per token
    T: tuple            # token counts per step that the workload uses
    S: int              # cache slots (VRAM tier) per layer
    steps: int          # steps in the routing trace
    reuse_p: float      # probability a token slot keeps its previous set
    zipf_s: float       # Zipf exponent of expert popularity
    router_gemm: bool   # logits = x . W_r^T (True) or given fp32 logits
    compressed: bool    # host tier holds Huffman-coded pages
    mixed: bool         # per-expert FP8 / 4-bit pages
    tie_frac: float = 0.01  # fraction of tokens with an exact tie at rank k/k+1

    @property
    def page_bytes_fp8(self) -> int:
        """FP8 weight bytes of one expert: w13 [2I,H] + w2 [H,I]."""
        return 3 * self.H * self.I


# The layer workloads, by what they are. The first field of each is its seed
# namespace (inputs drawn for a workload depend on it, not on the name).
WORKLOADS = {
    "tiny": LayerConfig(1, "tiny layer, all experts resident", E=8, H=256, I=128, k=2,
                   T=(64,), S=8, steps=1, reuse_p=0.0, zipf_s=0.0,
                   router_gemm=True, compressed=False, mixed=False, tie_frac=0.0),
    "decode": LayerConfig(2, "decode-shaped paged layer", E=256, H=2048, I=512, k=8,
                   T=(1, 8, 64), S=32, steps=256, reuse_p=0.7, zipf_s=1.1,
                   router_gemm=False, compressed=False, mixed=False),
    "batched": LayerConfig(3, "module-batched prefill layer", E=256, H=2048, I=512, k=8,
                   T=(16384,), S=32, steps=1, reuse_p=0.0, zipf_s=1.1,
                   router_gemm=False, compressed=False, mixed=False),
    "large": LayerConfig(4, "large paged layer, compressed host tier", E=512, H=2560, I=640, k=8,
                   T=(1, 4096), S=46, steps=256, reuse_p=0.7, zipf_s=1.1,
                   router_gemm=False, compressed=True, mixed=False),
    "mixed": LayerConfig(5, "mixed per-expert precision layer", E=256, H=2048, I=512, k=8,
                   T=(4096,), S=256, steps=256, reuse_p=0.7, zipf_s=1.1,
                   router_gemm=False, compressed=False, mixed=True),
}


def small_config(E=4, H=64, I=32, k=2, T=16, S=None, cid=90, **kw) -> LayerConfig:
    """A small layer of arbitrary shape, for tests that sweep sizes."""
    return LayerConfig(cid, "small", E=E, H=H, I=I, k=k, T=(T,), S=E if S is None else S,
                       steps=kw.pop("steps", 1), reuse_p=kw.pop("reuse_p", 0.0),
                       zipf_s=kw.pop("zipf_s", 0.0), router_gemm=kw.pop("router_gemm", True),
                       compressed=kw.pop("compressed", False), mixed=kw.pop("mixed", False),
                       tie_frac=kw.pop("tie_frac", 0.0))


def _rng(cfg: LayerConfig, step: int, tag: int, sub: int = 0) -> np.random.Generator:
    seed = SEED_BASE + 1000 * cfg.cid + step
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, sub])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def activations(cfg: LayerConfig, T: int, step: int = 0) -> np.ndarray:
    """x: bf16 bit patterns [T, H], values N(0, 1)."""
    g = _rng(cfg, step, _TAG_X, T)
    return to_bf16_bits(g.standard_normal((T, cfg.H), dtype=np.float32))


def router_weights(cfg: LayerConfig) -> np.ndarray:
    """W_r: fp32 [E, H], N(0, 0.02)."""
    g = _rng(cfg, 0, _TAG_WR)
    return (g.standard_normal((cfg.E, cfg.H), dtype=np.float32) * np.float32(0.02)).astype(np.float32)


def expert_weights(cfg: LayerConfig, e: int) -> tuple[np.ndarray, np.ndarray]:
    """Unquantised fp32 weights of expert e: w13 [2I, H] (gate rows then up rows), w2 [H, I].

    Drawn N(0, 0.02); each expert has its own stream so any subset can be made alone.
    """
    g13 = _rng(cfg, 0, _TAG_W13, e)
    g2 = _rng(cfg, 0, _TAG_W2, e)
    w13 = g13.standard_normal((2 * cfg.I, cfg.H), dtype=np.float32) * np.float32(0.02)
    w2 = g2.standard_normal((cfg.H, cfg.I), dtype=np.float32) * np.float32(0.02)
    return w13.astype(np.float32), w2.astype(np.float32)


def importance_init(cfg: LayerConfig) -> np.ndarray:
    """Seeded initial importance score per expert, U(0, 1), float64 [E]."""
    return _rng(cfg, 0, _TAG_IMPORTANCE).random(cfg.E)


def _zipf_probs(E: int, s: float) -> np.ndarray:
    w = 1.0 / np.power(np.arange(1, E + 1, dtype=np.float64), s)
    return w / w.sum()


class RoutingTrace:
    """Router logits for a sequence of steps, fp32 [T, E] each.

    A token slot keeps its previous step's expert set with probability
    ``reuse_p``; otherwise it draws k distinct experts from Zipf(s) over a
    seeded permutation of the expert ids (sampling without replacement).
    Logits are N(0,1) noise, plus 6.0 on the chosen experts, minus 0.25 times
    the draw rank. A fraction ``tie_frac`` of tokens get an exact tie between
    their k-th and (k+1)-th largest logits, to exercise the lower-id rule.
    """

    def __init__(self, cfg: LayerConfig, T: int, layer: int = 0, vectorized: bool = False):
        """vectorized: draw the fresh sets of a step all at once (Gumbel top-k:
        the k largest of log p + Gumbel noise, in descending order, which is
        the same distribution as k sequential draws without replacement);
        another random stream than the token-by-token draws, for long traces."""
        self.cfg, self.T, self.layer, self.vectorized = cfg, T, layer, vectorized
        self._perm = _rng(cfg, 0, _TAG_PERM, layer).permutation(cfg.E)
        self._p = _zipf_probs(cfg.E, cfg.zipf_s) if cfg.zipf_s > 0 else np.full(cfg.E, 1.0 / cfg.E)
        self._prev = None

    def _sets_vectorized(self, g: np.random.Generator) -> np.ndarray:
        cfg, T = self.cfg, self.T
        fresh = np.ones(T, bool) if self._prev is None else g.random(T) >= cfg.reuse_p
        sets = np.empty((T, cfg.k), dtype=np.int64) if self._prev is None else self._prev.copy()
        n = int(fresh.sum())
        if n:
            key = np.log(self._p)[None, :] + g.gumbel(size=(n, cfg.E))
            top = np.argpartition(-key, cfg.k - 1, axis=1)[:, :cfg.k]
            order = np.argsort(-np.take_along_axis(key, top, axis=1), axis=1, kind="stable")
            sets[fresh] = self._perm[np.take_along_axis(top, order, axis=1)]
        return sets

    def _fresh(self, g: np.random.Generator) -> np.ndarray:
        ranks = g.choice(self.cfg.E, size=self.cfg.k, replace=False, p=self._p)
        return self._perm[ranks]

    def step(self, s: int) -> np.ndarray:
        cfg, T = self.cfg, self.T
        g = _rng(cfg, s, _TAG_TRACE, T + (self.layer << 20))
        if self.vectorized:
            sets = self._sets_vectorized(g)
        else:
            sets = np.empty((T, cfg.k), dtype=np.int64)
            for t in range(T):
                if self._prev is not None and g.random() < cfg.reuse_p:
                    sets[t] = self._prev[t]
                else:
                    sets[t] = self._fresh(g)
        self._prev = sets
        logits = g.standard_normal((T, cfg.E), dtype=np.float32)
        bump = np.float32(6.0) - np.float32(0.25) * np.arange(cfg.k, dtype=np.float32)
        rows = np.repeat(np.arange(T), cfg.k)
        logits[rows, sets.reshape(-1)] += np.tile(bump, T)
        n_tie = int(round(cfg.tie_frac * T))
        if n_tie == 0 and cfg.tie_frac > 0 and T >= 8:
            n_tie = 1
        if n_tie:
            for t in g.choice(T, size=n_tie, replace=False):
                order = np.argsort(-logits[t], kind="stable")
                logits[t, order[cfg.k]] = logits[t, order[cfg.k - 1]]
        return logits.astype(np.float32)

    def __iter__(self) -> Iterator[np.ndarray]:
        for s in range(self.cfg.steps):
            yield self.step(s)


def routing_logits(cfg: LayerConfig, T: int, step: int = 0) -> np.ndarray:
    """Logits of one step (replays the trace up to ``step``)."""
    tr = RoutingTrace(cfg, T)
    out = None
    for s in range(step + 1):
        out = tr.step(s)
    return out
