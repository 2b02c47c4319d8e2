"""Python access to the CPU oracle (pqe_oracle.c).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package. It never imports the product
package, and the product never imports it.

``build()`` compiles pqe_oracle.c with gcc into ``oracle/_build/``; the
wrappers below only marshal numpy arrays into the C functions.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pqe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

HUF_G = 64        # symbols per chunk in the compressed-row format
HUF_LMAX = 12     # longest code


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, OpenMP over tokens in the FFN only)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


P = C.c_void_p


def _declare(L):
    sig = {
        "orc_e4m3_value": (C.c_double, [C.c_uint8]),
        "orc_e4m3_encode": (C.c_uint8, [C.c_float]),
        "orc_e2m1_value": (C.c_double, [C.c_uint8]),
        "orc_e2m1_encode": (C.c_uint8, [C.c_float]),
        "orc_e8m0_value": (C.c_double, [C.c_uint8]),
        "orc_quant_e4m3_rows": (None, [P, C.c_int, C.c_int, P, P]),
        "orc_quant_mxfp4_rows": (None, [P, P, C.c_int, C.c_int, P, P]),
        "orc_router_logits": (None, [P, P, C.c_int, C.c_int, C.c_int, P]),
        "orc_topk_gates": (None, [P, C.c_int, C.c_int, C.c_int, P, P]),
        "orc_permute": (None, [P, C.c_int, C.c_int, C.c_int, P, P, P, P]),
        "orc_lru_create": (P, [C.c_int, C.c_int]),
        "orc_lru_destroy": (None, [P]),
        "orc_lru_state": (None, [P, P, P, P]),
        "orc_lru_step": (C.c_int, [P, P, P, P, P, P]),
        "orc_lru_invalidate": (None, [P, C.c_int]),
        "orc_moe_ffn": (None, [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P, P, C.c_int, P]),
        "orc_num_threads": (C.c_int, []),
        "orc_set_num_threads": (None, [C.c_int]),
        "orc_huff_lengths": (C.c_int, [P, C.c_int, P]),
        "orc_huff_codes": (None, [P, P]),
        "orc_huff_encode": (C.c_int64, [P, C.c_int, C.c_int, C.c_int, P, P, P, P, P]),
        "orc_huff_decode": (C.c_int, [P, P, P, P, P, C.c_int, C.c_int, P]),
        "orc_rank_formats": (None, [P, C.c_int, C.c_int, P]),
        "orc_rank_formats_quality": (None, [P, P, C.c_int, C.c_int, P]),
        "orc_importance_step": (C.c_int, [P, P, P, C.c_int, C.c_int, C.c_int, C.c_double,
                                          C.c_int64, C.c_int, C.c_int, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- number formats --------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(v)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(v)


def e8m0_value(code: int) -> float:
    return lib().orc_e8m0_value(code)


def quant_e4m3_rows(w: np.ndarray):
    """fp32 [R, C] -> (codes uint8 [R, C], scales fp32 [R])."""
    w = _c(w, np.float32)
    R, Cc = w.shape
    q = np.empty((R, Cc), np.uint8)
    s = np.empty(R, np.float32)
    lib().orc_quant_e4m3_rows(_p(w), R, Cc, _p(q), _p(s))
    return q, s


def quant_mxfp4_rows(q8: np.ndarray, s8: np.ndarray):
    """FP8 codes + row scales [R, C] -> (nibble pairs uint8 [R, C/2], e8m0 uint8 [R, C/32])."""
    q8 = _c(q8, np.uint8)
    s8 = _c(s8, np.float32)
    R, Cc = q8.shape
    q4 = np.empty((R, Cc // 2), np.uint8)
    e8 = np.empty((R, Cc // 32), np.uint8)
    lib().orc_quant_mxfp4_rows(_p(q8), _p(s8), R, Cc, _p(q4), _p(e8))
    return q4, e8


def dequant_e4m3_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_value(b) for b in range(256)])
    return table[q] * s.astype(np.float64)[:, None]


def dequant_mxfp4_rows(q4: np.ndarray, e8: np.ndarray) -> np.ndarray:
    R = q4.shape[0]
    nib = np.empty((R, q4.shape[1] * 2), np.uint8)
    nib[:, 0::2] = q4 & 15
    nib[:, 1::2] = q4 >> 4
    vals = np.array([e2m1_value(b) for b in range(16)])[nib]
    sc = np.array([e8m0_value(b) for b in range(256)])[e8]
    return vals * np.repeat(sc, 32, axis=1)


# ---- router and permutation ------------------------------------------------

def router_logits(x_bf16: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    w = _c(w_r, np.float32)
    T, H = x.shape
    E = w.shape[0]
    out = np.empty((T, E), np.float32)
    lib().orc_router_logits(_p(x), _p(w), T, H, E, _p(out))
    return out


def topk_gates(logits: np.ndarray, k: int):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    g = np.empty((T, k), np.float64)
    lib().orc_topk_gates(_p(lg), T, E, k, _p(ids), _p(g))
    return ids, g


def permute(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    A = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_src = np.empty(A, np.int32)
    inv = np.empty(A, np.int32)
    lib().orc_permute(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm_src), _p(inv))
    return counts, offsets, perm_src, inv


# ---- LRU slot pool ----------------------------------------------------------

class LRU:
    """Per-layer VRAM slot pool state (see orc_lru_step for the rules)."""

    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self._h = lib().orc_lru_create(E, S)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_lru_destroy(self._h)
            self._h = None

    def step(self, counts: np.ndarray):
        counts = _c(counts, np.int32)
        table = np.empty(self.E, np.int32)
        me = np.empty(self.E, np.int32)
        md = np.empty(self.E, np.int32)
        n = np.zeros(1, np.int32)
        wb = lib().orc_lru_step(self._h, _p(counts), _p(table), _p(me), _p(md), _p(n))
        return table, me[: n[0]].copy(), md[: n[0]].copy(), bool(wb)

    def invalidate(self, e: int):
        lib().orc_lru_invalidate(self._h, int(e))

    def state(self):
        se = np.empty(self.S, np.int32)
        lu = np.empty(self.S, np.int64)
        st = np.zeros(1, np.int64)
        lib().orc_lru_state(self._h, _p(se), _p(lu), _p(st))
        return se, lu, int(st[0])


# ---- expert FFN -------------------------------------------------------------

class _Expert(C.Structure):
    _fields_ = [("fmt", C.c_int32), ("pad", C.c_int32), ("w13", C.c_void_p), ("s13", C.c_void_p),
                ("w2", C.c_void_p), ("s2", C.c_void_p)]


class ExpertSet:
    """Quantised weights of E experts, by format.

    fmt 0: (w13 codes [2I,H], s13 fp32 [2I], w2 codes [H,I], s2 fp32 [H]);
    fmt 1: (w13 nibbles [2I,H/2], e8m0 [2I,H/32], w2 nibbles [H,I/2], e8m0 [H,I/32]).
    Experts not present stay NULL and must not be routed to.
    """

    def __init__(self, E: int):
        self.E = E
        self._arr = (_Expert * E)()
        self._keep = {}

    def set(self, e: int, fmt: int, w13, s13, w2, s2):
        arrs = [np.ascontiguousarray(a) for a in (w13, s13, w2, s2)]
        self._keep[e] = arrs
        self._arr[e] = _Expert(fmt, 0, *[a.ctypes.data for a in arrs])

    def has(self, e: int) -> bool:
        return e in self._keep

    def ptr(self):
        return C.cast(self._arr, C.c_void_p)


def moe_ffn(x_bf16: np.ndarray, ids: np.ndarray, gates: np.ndarray, experts: ExpertSet, I: int,
            tokens=None) -> np.ndarray:
    """y [n, H] fp64 for the listed tokens (all tokens if ``tokens`` is None)."""
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    g = _c(gates, np.float64)
    T, H = x.shape
    k = ids.shape[1]
    needed = np.unique(ids if tokens is None else ids[np.asarray(tokens)])
    for e in needed:
        if not experts.has(int(e)):
            raise ValueError(f"expert {e} has no weights in the ExpertSet")
    if tokens is None:
        y = np.empty((T, H), np.float64)
        lib().orc_moe_ffn(_p(x), T, H, I, k, _p(ids), _p(g), experts.ptr(), None, 0, _p(y))
    else:
        tl = _c(tokens, np.int32)
        y = np.empty((len(tl), H), np.float64)
        lib().orc_moe_ffn(_p(x), T, H, I, k, _p(ids), _p(g), experts.ptr(), _p(tl), len(tl), _p(y))
    return y


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(n)


# ---- Huffman codec ----------------------------------------------------------

def huff_lengths(freq, lmax: int = HUF_LMAX) -> np.ndarray:
    f = _c(freq, np.uint64)
    assert f.shape == (16,)
    ln = np.zeros(16, np.uint8)
    rc = lib().orc_huff_lengths(_p(f), lmax, _p(ln))
    if rc != 0:
        raise ValueError("alphabet does not fit the length limit")
    return ln


def huff_codes(lengths) -> np.ndarray:
    ln = _c(lengths, np.uint8)
    code = np.zeros(16, np.uint32)
    lib().orc_huff_codes(_p(ln), _p(code))
    return code


def huff_encode(q: np.ndarray, lmax: int = HUF_LMAX) -> dict:
    """Compress an FP8 matrix [R, C] (C % 64 == 0) into the row/chunk format."""
    q = _c(q, np.uint8)
    R, Cc = q.shape
    assert Cc % HUF_G == 0
    ln = np.zeros(16, np.uint8)
    rw = np.zeros(R + 1, np.uint32)
    cb = np.zeros(R * (Cc // HUF_G), np.uint16)
    nib = np.zeros(R * Cc // 2, np.uint8)
    nw = lib().orc_huff_encode(_p(q), R, Cc, lmax, _p(ln), _p(rw), _p(cb), _p(nib), None)
    if nw < 0:
        raise ValueError("code construction failed")
    words = np.zeros(max(int(nw), 1), np.uint32)
    lib().orc_huff_encode(_p(q), R, Cc, lmax, _p(ln), _p(rw), _p(cb), _p(nib), _p(words))
    return {"lengths": ln, "row_word": rw, "chunk_bit": cb, "nibbles": nib,
            "words": words[: int(nw)], "rows": R, "cols": Cc}


def huff_decode(enc: dict) -> tuple[np.ndarray, int]:
    """-> (FP8 bytes [R, C], status: 0 ok, -2 corrupt)."""
    R, Cc = enc["rows"], enc["cols"]
    q = np.zeros((R, Cc), np.uint8)
    words = _c(enc["words"], np.uint32)
    if words.size == 0:
        words = np.zeros(1, np.uint32)
    rc = lib().orc_huff_decode(_p(_c(enc["lengths"], np.uint8)), _p(_c(enc["row_word"], np.uint32)),
                               _p(_c(enc["chunk_bit"], np.uint16)), _p(_c(enc["nibbles"], np.uint8)),
                               _p(words), R, Cc, _p(q))
    return q, rc


# ---- bit-width assignment ----------------------------------------------------

def rank_formats(m: np.ndarray, n_hi: int) -> np.ndarray:
    m = _c(m, np.float64)
    fmt = np.empty(m.shape[0], np.uint8)
    lib().orc_rank_formats(_p(m), m.shape[0], n_hi, _p(fmt))
    return fmt


def rank_formats_quality(m: np.ndarray, q: np.ndarray, n_hi: int) -> np.ndarray:
    """Top n_hi of m[e] * q[e] keep FP8 (0), the rest MXFP4 (1); ties to the lower id."""
    m = _c(m, np.float64)
    q = _c(q, np.float64)
    fmt = np.empty(m.shape[0], np.uint8)
    lib().orc_rank_formats_quality(_p(m), _p(q), m.shape[0], n_hi, _p(fmt))
    return fmt


def quant_error_sums(x_bf16: np.ndarray, w8: tuple, w4: tuple, I: int, fmt8: int = 0, fmt4: int = 1) -> tuple:
    """The 4-bit quality proxy of one expert on tokens x: (sum ||y4 - y8||^2,
    sum ||y8||^2) in fp64, y8 / y4 the expert's SwiGLU FFN from its FP8 page
    (q13, s13, q2, s2) and its MXFP4 page (a13, x13, a2, x2). fmt8 / fmt4 name
    the formats of the two pages (FP8 0, MXFP4 1)."""
    n = x_bf16.shape[0]
    ex = ExpertSet(2)
    ex.set(0, fmt8, *w8)
    ex.set(1, fmt4, *w4)
    ones = np.ones((n, 1), np.float32)
    y8 = moe_ffn(x_bf16, np.zeros((n, 1), np.int32), ones, ex, I)
    y4 = moe_ffn(x_bf16, np.ones((n, 1), np.int32), ones, ex, I)
    return float(np.sum((y4 - y8) ** 2)), float(np.sum(y8 ** 2))


def importance_step(m: np.ndarray, ids: np.ndarray, gates_f32: np.ndarray, E: int, step: int,
                    fmt: np.ndarray, alpha: float = 0.9, every: int = 64, n_hi: int = 64) -> bool:
    """Updates m and fmt in place; returns True when the formats were re-ranked."""
    assert m.dtype == np.float64 and fmt.dtype == np.uint8
    ids = _c(ids, np.int32)
    g = _c(gates_f32, np.float32)
    T, k = ids.shape
    return bool(lib().orc_importance_step(_p(m), _p(ids), _p(g), T, k, E, alpha, step, every,
                                          n_hi, _p(fmt)))
