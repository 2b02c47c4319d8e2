"""Pins of the oracle's lossless FP8 page codec (per-row exponent Huffman) and
of the page sizes the pages print.

Independent references: exact round trip, the Kraft equality, a textbook
Huffman construction (heapq) for the optimal cost, brute force over length
vectors when the length limit binds, prefix-freeness, and the sizes and
compression band printed in the vllm-expert-pager article.
"""
import heapq
import itertools
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _textbook_huffman_cost(freq):
    f = [int(x) for x in freq if x > 0]
    if len(f) <= 1:
        return sum(f)
    heap = list(f)
    heapq.heapify(heap)
    cost = 0
    while len(heap) > 1:
        a = heapq.heappop(heap)
        b = heapq.heappop(heap)
        cost += a + b
        heapq.heappush(heap, a + b)
    return cost


def _textbook_max_len(freq):
    # depth of the textbook tree (ties broken arbitrarily: only used as a guard)
    items = [(int(w), i, 0) for i, w in enumerate(freq) if w > 0]
    heapq.heapify(items)
    cnt = len(freq)
    while len(items) > 1:
        a = heapq.heappop(items)
        b = heapq.heappop(items)
        heapq.heappush(items, (a[0] + b[0], cnt, max(a[2], b[2]) + 1))
        cnt += 1
    return items[0][2]


def _cost(freq, lens):
    return int(sum(int(f) * int(l) for f, l in zip(freq, lens)))


@pytest.mark.parametrize("seed", range(20))
def test_lengths_optimal_and_complete(orc, seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(2, 17))
    freq = np.zeros(16, np.uint64)
    freq[g.choice(16, n, replace=False)] = g.integers(1, 10 ** g.integers(1, 7), n)
    lens = orc.huff_lengths(freq)
    used = freq > 0
    assert np.all(lens[~used] == 0) and np.all(lens[used] >= 1) and lens.max() <= 12
    assert sum(2.0 ** -int(l) for l in lens[used]) == 1.0          # Kraft equality
    if _textbook_max_len(freq) <= 12:
        assert _cost(freq, lens) == _textbook_huffman_cost(freq)


def test_length_limit_binding_brute_force(orc):
    # Fibonacci-like weights force long codes; brute-force the best length vector
    g = np.random.default_rng(7)
    for trial in range(30):
        n = int(g.integers(3, 7))
        lmax = int(g.integers(int(np.ceil(np.log2(n))), 5))
        w = np.sort(g.integers(1, 200, n))[::-1] ** 2
        freq = np.zeros(16, np.uint64)
        syms = g.choice(16, n, replace=False)
        freq[syms] = w
        lens = orc.huff_lengths(freq, lmax)
        assert lens.max() <= lmax
        best = min(sum(int(wi) * li for wi, li in zip(w, L))
                   for L in itertools.product(range(1, lmax + 1), repeat=n)
                   if sum(2.0 ** -l for l in L) <= 1.0)
        assert _cost(freq, lens) == best


def test_single_symbol_and_canonical_codes(orc):
    freq = np.zeros(16, np.uint64)
    freq[9] = 100
    lens = orc.huff_lengths(freq)
    assert lens[9] == 1 and lens.sum() == 1
    freq = np.array([5, 0, 9, 1, 1, 0, 3, 0, 0, 0, 0, 0, 0, 0, 0, 30], np.uint64)
    lens = orc.huff_lengths(freq)
    codes = orc.huff_codes(lens)
    used = [s for s in range(16) if lens[s]]
    strs = {s: format(int(codes[s]), f"0{lens[s]}b") for s in used}
    for a, b in itertools.permutations(used, 2):
        assert not strs[b].startswith(strs[a])                     # prefix-free
    order = sorted(used, key=lambda s: (lens[s], s))
    vals = [int(codes[s]) << (16 - int(lens[s])) for s in order]
    assert vals == sorted(vals) and len(set(vals)) == len(vals)   # canonical order


def _synthetic_fp8(orc, cfg, e):
    w13, w2 = synth.expert_weights(cfg, e)
    return orc.quant_e4m3_rows(w13)[0], orc.quant_e4m3_rows(w2)[0]


def test_roundtrip_synthetic_pages(orc):
    for wl in ("tiny", "decode"):
        cfg = synth.WORKLOADS[wl]
        for q in _synthetic_fp8(orc, cfg, 3):
            enc = orc.huff_encode(q)
            dec, rc = orc.huff_decode(enc)
            assert rc == 0 and np.array_equal(dec, q)


@pytest.mark.parametrize("kind", ["zero", "single", "uniform16", "skewed", "random_bytes", "negzero"])
def test_roundtrip_adversarial(orc, kind):
    g = np.random.default_rng(hash(kind) % 1000)
    R, Cc = 5, 256
    if kind == "zero":
        q = np.zeros((R, Cc), np.uint8)
    elif kind == "single":
        q = np.full((R, Cc), 0x41, np.uint8)
    elif kind == "uniform16":
        q = (np.arange(R * Cc) % 256).astype(np.uint8).reshape(R, Cc)
    elif kind == "skewed":
        # Fibonacci symbol counts: the unlimited Huffman tree is 15 deep, so
        # the 12-bit limit binds
        fib = [1, 1]
        while len(fib) < 16:
            fib.append(fib[-1] + fib[-2])
        R = 11
        sym = np.concatenate([np.full(c, s) for s, c in enumerate(fib)])
        sym = np.concatenate([sym, np.full(R * Cc - sym.size, 15)])
        g.shuffle(sym)
        sym = sym.reshape(R, Cc)
        q = ((sym << 3) | g.integers(0, 8, (R, Cc)) | (g.integers(0, 2, (R, Cc)) << 7)).astype(np.uint8)
        q[q == 0x7F] = 0x7E
        q[q == 0xFF] = 0xFE
    elif kind == "negzero":
        q = np.full((R, Cc), 0x80, np.uint8)
    else:
        q = g.integers(0, 256, (R, Cc)).astype(np.uint8)
    enc = orc.huff_encode(q)
    dec, rc = orc.huff_decode(enc)
    assert rc == 0 and np.array_equal(dec, q)
    if kind == "skewed":
        assert enc["lengths"].max() == 12


def test_corrupt_streams_are_reported(orc):
    cfg = synth.WORKLOADS["tiny"]
    q = _synthetic_fp8(orc, cfg, 0)[1]
    enc = orc.huff_encode(q)
    short = dict(enc)
    rw = enc["row_word"].copy()
    rw[1] -= 1                                    # row 0 loses its last word
    short["row_word"] = rw
    _, rc = orc.huff_decode(short)
    assert rc == -2
    # single-symbol code: any 1 bit is not a code word
    q1 = np.full((2, 64), 0x41, np.uint8)
    enc1 = orc.huff_encode(q1)
    enc1["words"] = enc1["words"].copy()
    enc1["words"][0] |= np.uint32(1 << 31)
    _, rc = orc.huff_decode(enc1)
    assert rc == -2


def _compressed_bytes(enc):
    return (enc["words"].size * 4 + enc["chunk_bit"].size * 2 + enc["row_word"].size * 4
            + enc["nibbles"].size)


def test_page_sizes_match_pages(orc):
    with open(os.path.join(GOLDEN, "page_sizes.txt")) as f:
        rows = [l.split()[:5] for l in f if l.strip() and not l.startswith("#")]
    for layers, experts, H, I, gib in rows:
        cfg = synth.LayerConfig(0, "", int(experts), int(H), int(I), 8, (1,), 0, 0, 0, 0, False, False, False)
        assert cfg.page_bytes_fp8 * int(experts) * int(layers) == float(gib) * 2 ** 30
    assert synth.WORKLOADS["decode"].page_bytes_fp8 == 3 * 2 ** 20
    assert synth.WORKLOADS["large"].page_bytes_fp8 == int(4.6875 * 2 ** 20)


def test_compression_ratio_plausible(orc):
    # Plausibility only (not parity): the pages report a bit over 10% saving on
    # real weights; N(0, 0.02) rows scaled to 448 have a lower exponent entropy,
    # so the synthetic saving is larger. Both must lie in (0, 50%].
    with open(os.path.join(GOLDEN, "compression_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    page_ratios = [float(c) / float(u) for _, _, u, c in rows]
    assert all(0.85 <= r <= 0.9 for r in page_ratios)
    cfg = synth.WORKLOADS["decode"]
    tot = comp = 0
    for q in _synthetic_fp8(orc, cfg, 5):
        enc = orc.huff_encode(q)
        tot += q.size
        comp += _compressed_bytes(enc)
    ratio = comp / tot
    assert 0.5 < ratio < min(page_ratios)
