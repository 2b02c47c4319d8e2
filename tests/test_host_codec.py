"""The product's host-side page encoder against the oracle's encoder: every
section of a compressed page is bit-identical, and the product's code table
agrees with the oracle's canonical codes. CPU only.
"""
import numpy as np
import pytest
import torch

import synth
from tests import helpers


def _pqe():
    import paged_quantized_expert_gb300 as pqe
    pqe.load()
    return pqe


HDR = 256


def _sections(comp: np.ndarray, H: int, I: int):
    hdr = comp[:HDR]
    u64 = hdr[48:48 + 8 * 12].view(np.uint64)
    off_scales = int(u64[0])
    m13 = [int(v) for v in u64[1:6]]
    m2 = [int(v) for v in u64[6:11]]
    out = {"len13": hdr[16:32].copy(), "len2": hdr[32:48].copy(),
           "scales": comp[off_scales:off_scales + 4 * (2 * I + H)].copy()}
    for name, m, rows, cols in (("13", m13, 2 * I, H), ("2", m2, H, I)):
        rw, cb, nb, wd, nw = m
        out["row_word" + name] = comp[rw:rw + 4 * (rows + 1)].view(np.uint32)
        out["chunk_bit" + name] = comp[cb:cb + 2 * rows * (cols // 64)].view(np.uint16)
        out["nibbles" + name] = comp[nb:nb + rows * cols // 2]
        out["words" + name] = comp[wd:wd + 4 * nw].view(np.uint32)
    return out


def _encode_page(pqe, page: np.ndarray, H: int, I: int):
    out = torch.zeros(pqe.pqe_huff_page_bound(H, I), dtype=torch.uint8)
    l13 = torch.zeros(pqe.PQE_HUFF_LUT_BYTES, dtype=torch.uint8)
    l2 = torch.zeros(pqe.PQE_HUFF_LUT_BYTES, dtype=torch.uint8)
    n = pqe.pqe_huff_encode_page(torch.from_numpy(page), H, I, out, l13, l2)
    return out[:n].numpy(), l13.numpy(), l2.numpy()


def _prefix_symbol(bits: int, nbits: int, lengths, codes):
    """The symbol whose code word is a prefix of the nbits-bit value `bits`
    (MSB first), with its length; (None, 0) if none fits."""
    for s in range(16):
        L = int(lengths[s])
        if L and L <= nbits and (bits >> (nbits - L)) == int(codes[s]):
            return s, L
    return None, 0


def _check_code_table(lut: np.ndarray, lengths, codes):
    """Every entry holds the whole code words at the front of its 12-bit
    window (at most 5): their total length in bits 0-3, their number in bits
    4-6, the first one's length in bits 7-10, the symbols from bit 12 (first
    lowest, unused slots zero); decoding stops where no whole code word fits
    the rest. A window that no code word prefixes reads n = 1, length 0 and
    bit 11 set."""
    assert lut.size == 4096
    for w in range(4096):
        ent = int(lut[w])
        tot, n, l0, inv, syms = ent & 15, (ent >> 4) & 7, (ent >> 7) & 15, (ent >> 11) & 1, ent >> 12
        rest, left, got = w, 12, []
        while len(got) < 5:
            s, L = _prefix_symbol(rest, left, lengths, codes)
            if s is None:
                break
            got.append((s, L))
            left -= L
            rest &= (1 << left) - 1
        if not got:
            assert (tot, n, l0, inv, syms) == (0, 1, 0, 1, 0), (w, ent)
            continue
        assert inv == 0 and n == len(got), (w, ent, got)
        assert tot == sum(L for _, L in got)
        assert l0 == got[0][1]
        assert syms == sum(s << (4 * i) for i, (s, _) in enumerate(got))


def _check_page(orc, pqe, page, H, I):
    lay = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
    comp, l13, l2 = _encode_page(pqe, page, H, I)
    sec = _sections(comp, H, I)
    q13, s13, q2, s2 = helpers.split_fp8_page(page, lay, H, I)
    for name, q, lut in (("13", q13, l13), ("2", q2, l2)):
        ref = orc.huff_encode(q)
        assert np.array_equal(sec["len" + name], ref["lengths"])
        assert np.array_equal(sec["row_word" + name], ref["row_word"])
        assert np.array_equal(sec["chunk_bit" + name], ref["chunk_bit"])
        assert np.array_equal(sec["nibbles" + name], ref["nibbles"])
        assert np.array_equal(sec["words" + name], ref["words"])
        # code table: checked entry by entry against the oracle's canonical codes
        _check_code_table(lut.view(np.uint32), ref["lengths"], orc.huff_codes(ref["lengths"]))
    assert np.array_equal(sec["scales"], page[lay["s13"]:lay["s13"] + 4 * (2 * I + H)])
    return comp


@pytest.mark.parametrize("wl,e", [("tiny", 0), ("tiny", 5), ("decode", 17)])
def test_encoder_matches_oracle_on_synthetic_pages(orc, wl, e):
    pqe = _pqe()
    cfg = synth.WORKLOADS[wl]
    w13, w2 = synth.expert_weights(cfg, e)
    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    page = helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, cfg.H, cfg.I), cfg.H, cfg.I, q13, s13, q2, s2)
    comp = _check_page(orc, pqe, page, cfg.H, cfg.I)
    assert comp.size < 0.9 * page.size


@pytest.mark.parametrize("kind", ["zero", "single", "random", "fib"])
def test_encoder_matches_oracle_adversarial(orc, kind):
    pqe = _pqe()
    H, I = 128, 64
    g = np.random.default_rng(len(kind))
    if kind == "zero":
        q13, q2 = np.zeros((2 * I, H), np.uint8), np.zeros((H, I), np.uint8)
    elif kind == "single":
        q13, q2 = np.full((2 * I, H), 0x3A, np.uint8), np.full((H, I), 0xC1, np.uint8)
    elif kind == "random":
        q13, q2 = g.integers(0, 256, (2 * I, H)).astype(np.uint8), g.integers(0, 256, (H, I)).astype(np.uint8)
    else:
        fib = [1, 1]
        while len(fib) < 16:
            fib.append(fib[-1] + fib[-2])
        sym = np.concatenate([np.full(c, s) for s, c in enumerate(fib)])
        sym = np.concatenate([sym, np.full(2 * I * H - sym.size, 15)])
        g.shuffle(sym)
        q13 = ((sym.reshape(2 * I, H) << 3) | g.integers(0, 7, (2 * I, H))).astype(np.uint8)
        q2 = g.integers(0, 0x7E, (H, I)).astype(np.uint8)
    s13 = np.ones(2 * I, np.float32)
    s2 = np.full(H, 0.5, np.float32)
    page = helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, H, I), H, I, q13, s13, q2, s2)
    _check_page(orc, pqe, page, H, I)


def test_encoder_refuses_rows_beyond_16_bit_chunk_offsets():
    """Chunk offsets are 16-bit: a row whose chunks would start past bit 65535
    (here 16384 symbols of ~10-bit codes) is refused, not wrapped."""
    pqe = _pqe()
    H, I = 16384, 64
    g = np.random.default_rng(5)
    q13 = np.where(g.random((2 * I, H)) < 0.9, 0x38, 0x40).astype(np.uint8)
    q13[3] = g.permutation(np.repeat(np.arange(8, 16, dtype=np.uint8), H // 8)) << 3
    q2 = np.full((H, I), 0x38, np.uint8)
    page = helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, H, I), H, I, q13, np.ones(2 * I, np.float32), q2,
                                 np.ones(H, np.float32))
    with pytest.raises(pqe.PqeError) as ei:
        _encode_page(pqe, page, H, I)
    assert ei.value.code == pqe.PQE_ERR_CAPACITY
