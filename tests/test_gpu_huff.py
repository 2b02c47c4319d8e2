"""GPU decode of compressed FP8 pages: bit-exact reconstruction of the FP8
bytes and scales, corrupt pages flagged in the status word (no fault), and the
copy-then-decode slot refill."""
import numpy as np
import pytest
import torch

import synth
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fp8_page(pqe, orc, cfg, e):
    w13, w2 = synth.expert_weights(cfg, e)
    q13, s13 = orc.quant_e4m3_rows(w13)
    q2, s2 = orc.quant_e4m3_rows(w2)
    return helpers.fp8_page_host(pqe.page_layout(pqe.PQE_FMT_FP8, cfg.H, cfg.I), cfg.H, cfg.I, q13, s13, q2, s2)


def _encode(pqe, page, H, I):
    out = torch.zeros(pqe.pqe_huff_page_bound(H, I), dtype=torch.uint8)
    l13 = torch.zeros(pqe.PQE_HUFF_LUT_BYTES, dtype=torch.uint8)
    l2 = torch.zeros(pqe.PQE_HUFF_LUT_BYTES, dtype=torch.uint8)
    n = pqe.pqe_huff_encode_page(torch.from_numpy(page), H, I, out, l13, l2)
    return out[:n].clone(), torch.cat([l13, l2])


def _decode(pqe, comp, luts, H, I, comp_bytes=None):
    dev = torch.zeros(comp.numel() + 256, dtype=torch.uint8, device=DEV)
    dev[:comp.numel()].copy_(comp)
    lut = luts.to(DEV)
    out = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_FP8, H, I), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pqe.fp8_exp_huff_decode(dev, comp.numel() if comp_bytes is None else comp_bytes, lut[:pqe.PQE_HUFF_LUT_BYTES], lut[pqe.PQE_HUFF_LUT_BYTES:], H, I,
                            out, status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("wl,e", [("tiny", 1), ("decode", 0), ("decode", 200), ("large", 511)])
def test_decode_bit_exact(cuda_lib, orc, wl, e):
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    page = _fp8_page(pqe, orc, cfg, e)
    comp, luts = _encode(pqe, page, cfg.H, cfg.I)
    assert comp.numel() < page.size
    out, status = _decode(pqe, comp, luts, cfg.H, cfg.I)
    assert status == 0
    assert np.array_equal(out, page)


@pytest.mark.parametrize("kind", ["zero", "single", "random", "negzero"])
def test_decode_adversarial(cuda_lib, kind):
    pqe = cuda_lib
    H, I = 128, 64
    g = np.random.default_rng(3)
    lay = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
    if kind == "zero":
        q13, q2 = np.zeros((2 * I, H), np.uint8), np.zeros((H, I), np.uint8)
    elif kind == "single":
        q13, q2 = np.full((2 * I, H), 0x45, np.uint8), np.full((H, I), 0xB8, np.uint8)
    elif kind == "negzero":
        q13, q2 = np.full((2 * I, H), 0x80, np.uint8), np.full((H, I), 0x80, np.uint8)
    else:
        q13, q2 = g.integers(0, 256, (2 * I, H)).astype(np.uint8), g.integers(0, 256, (H, I)).astype(np.uint8)
    page = helpers.fp8_page_host(lay, H, I, q13, np.ones(2 * I, np.float32), q2, np.ones(H, np.float32))
    comp, luts = _encode(pqe, page, H, I)
    out, status = _decode(pqe, comp, luts, H, I)
    assert status == 0 and np.array_equal(out, page)


def test_corrupt_pages_flagged(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    page = _fp8_page(pqe, orc, cfg, 2)
    comp, luts = _encode(pqe, page, cfg.H, cfg.I)
    # truncated page: the header's sections no longer fit
    _, status = _decode(pqe, comp, luts, cfg.H, cfg.I, comp_bytes=comp.numel() // 2)
    assert status & pqe.PQE_STATUS_CORRUPT_STREAM
    # bad magic
    bad = comp.clone()
    bad[0] ^= 0xFF
    _, status = _decode(pqe, bad, luts, cfg.H, cfg.I)
    assert status & pqe.PQE_STATUS_CORRUPT_STREAM
    # a single-symbol matrix: a set bit is no code word
    H, I = 64, 64
    lay = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
    p1 = helpers.fp8_page_host(lay, H, I, np.full((2 * I, H), 0x40, np.uint8), np.ones(2 * I, np.float32),
                               np.full((H, I), 0x40, np.uint8), np.ones(H, np.float32))
    c1, l1 = _encode(pqe, p1, H, I)
    hdr = c1[:256].numpy()
    off_words13 = int(hdr[48:48 + 96].view(np.uint64)[4])
    c1 = c1.clone()
    c1[off_words13 + 3] |= 0x80          # first word, MSB (little-endian byte 3)
    _, status = _decode(pqe, c1, l1, H, I)
    assert status & pqe.PQE_STATUS_CORRUPT_STREAM
    # row offsets that run past the stream
    c2, l2 = _encode(pqe, p1, H, I)
    hdr = c2[:256].numpy()
    off_rw13 = int(hdr[48:48 + 96].view(np.uint64)[1])
    c2 = c2.clone()
    c2[off_rw13 + 4 * 5:off_rw13 + 4 * 6] = torch.tensor([0xFF, 0xFF, 0xFF, 0x7F], dtype=torch.uint8)
    _, status = _decode(pqe, c2, l2, H, I)
    assert status & pqe.PQE_STATUS_CORRUPT_STREAM


def test_slot_fill_compressed(cuda_lib, orc):
    pqe = cuda_lib
    cfg = synth.WORKLOADS["tiny"]
    page = _fp8_page(pqe, orc, cfg, 4)
    comp, luts = _encode(pqe, page, cfg.H, cfg.I)
    pinned = comp.pin_memory()
    pool_mem, pool = pqe.alloc_pool(3, cfg.H, cfg.I)
    staging = torch.zeros(pqe.pqe_huff_page_bound(cfg.H, cfg.I), dtype=torch.uint8, device=DEV)
    lut = luts.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record(side)  # creates the CUDA event (torch makes it lazily); the library records it again
    pqe.slot_fill_compressed(pool, 2, pinned, comp.numel(), staging, lut[:pqe.PQE_HUFF_LUT_BYTES], lut[pqe.PQE_HUFF_LUT_BYTES:], status, stream=side,
                             done_event=ev)
    ev.synchronize()
    stride = pqe.slot_stride(cfg.H, cfg.I)
    got = pool_mem[2 * stride:2 * stride + page.size].cpu().numpy()
    assert int(status.item()) == 0 and np.array_equal(got, page)
    assert int(torch.count_nonzero(pool_mem[:2 * stride]).item()) == 0


def _page_from_codes(pqe, H, I, q13, q2):
    lay = pqe.page_layout(pqe.PQE_FMT_FP8, H, I)
    g = np.random.default_rng(H + I)
    return helpers.fp8_page_host(lay, H, I, q13, g.random(2 * I).astype(np.float32), q2,
                                 g.random(H).astype(np.float32))


def test_decode_batch_one_launch_with_a_corrupt_page(cuda_lib, orc):
    """Several pages of one shape in one launch (device-resident sources); a
    corrupt page in the middle is flagged and the others stay bit-exact."""
    pqe = cuda_lib
    cfg = synth.WORKLOADS["decode"]
    H, I = cfg.H, cfg.I
    pages, comps, luts = [], [], []
    for e in (3, 77, 150, 255):
        p = _fp8_page(pqe, orc, cfg, e)
        c, l = _encode(pqe, p, H, I)
        pages.append(p)
        comps.append(c)
        luts.append(l)
    bad = comps[1].clone()
    bad[0] ^= 0xFF  # bad magic
    srcs = [c.to(DEV) for c in (comps[0], bad, comps[2], comps[3])]
    lut = [l.to(DEV) for l in luts]
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    out = torch.zeros((4, nb), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    LB = pqe.PQE_HUFF_LUT_BYTES
    n0 = pqe.kernel_launches()
    pqe.fp8_exp_huff_decode_batch(srcs, [c.numel() for c in comps], [l[:LB] for l in lut], [l[LB:] for l in lut], H,
                                  I, [out[i] for i in range(4)], status)
    torch.cuda.synchronize()
    assert pqe.kernel_launches() - n0 == 1
    assert int(status.item()) & pqe.PQE_STATUS_CORRUPT_STREAM
    got = out.cpu().numpy()
    for i in (0, 2, 3):
        assert np.array_equal(got[i], pages[i])


@pytest.mark.parametrize("wl", ["tiny", "large"])
def test_slot_fill_compressed_batch_from_pinned_host(cuda_lib, orc, wl):
    """Compressed pages pulled from pinned host memory and decoded in one pass
    into pool entries (cache slots and working buffer), bit-exact; untouched
    entries stay zero."""
    pqe = cuda_lib
    cfg = synth.WORKLOADS[wl]
    H, I = cfg.H, cfg.I
    experts = (0, 5, 2) if wl == "tiny" else (511, 7, 300)
    pages, comps, luts = [], [], []
    for e in experts:
        p = _fp8_page(pqe, orc, cfg, e)
        c, l = _encode(pqe, p, H, I)
        pages.append(p)
        comps.append(c.pin_memory())
        luts.append(l.to(DEV))
    stride = pqe.slot_stride(H, I)
    pool_mem = torch.zeros(4 * stride, dtype=torch.uint8, device=DEV)
    wb = torch.zeros(2 * stride, dtype=torch.uint8, device=DEV)
    pool = pqe.make_pool(pool_mem, 4, H, I, wb, 2)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    LB = pqe.PQE_HUFF_LUT_BYTES
    dests = [3, 0, 5]  # two cache slots and working-buffer entry 1
    side = torch.cuda.Stream()
    pqe.slot_fill_compressed_batch(pool, dests, comps, [c.numel() for c in comps], [l[:LB] for l in luts],
                                   [l[LB:] for l in luts], status, stream=side)
    side.synchronize()
    assert int(status.item()) == 0
    nb = pages[0].size
    mem = {3: pool_mem[3 * stride:3 * stride + nb], 0: pool_mem[:nb], 5: wb[stride:stride + nb]}
    for d, p in zip(dests, pages):
        assert np.array_equal(mem[d].cpu().numpy(), p)
    assert int(torch.count_nonzero(pool_mem[stride:3 * stride]).item()) == 0
    assert int(torch.count_nonzero(wb[:stride]).item()) == 0


def test_long_rows_at_the_format_limit(cuda_lib):
    """H=16384 rows of uniformly random bytes: 16 equally frequent exponents,
    4-bit codes, the last chunk of a row starting at bit 65280 (16-bit chunk
    offsets): 2048 code words per row, decoded bit-exact. A row whose chunks
    would start past bit 65535 cannot be represented; the encoder refuses it."""
    pqe = cuda_lib
    H, I = 16384, 64
    g = np.random.default_rng(11)
    q13 = g.integers(0, 256, (2 * I, H)).astype(np.uint8)
    q2 = g.integers(0, 256, (H, I)).astype(np.uint8)
    page = _page_from_codes(pqe, H, I, q13, q2)
    comp, luts = _encode(pqe, page, H, I)
    l13, _ = pqe.pqe_huff_page_lengths(comp)
    assert int(l13.min()) == 4 and int(l13.max()) == 4
    out, status = _decode(pqe, comp, luts, H, I)
    assert status == 0
    assert np.array_equal(out, page)
    # one row of rare exponents (8..15, 2048 each: ~10-bit codes) overflows its chunk offsets
    q13 = np.where(g.random((2 * I, H)) < 0.9, 0x38, 0x40).astype(np.uint8)
    q13[37] = g.permutation(np.repeat(np.arange(8, 16, dtype=np.uint8), H // 8)) << 3
    bad = _page_from_codes(pqe, H, I, q13, q2)
    with pytest.raises(pqe.PqeError) as ei:
        _encode(pqe, bad, H, I)
    assert ei.value.code == pqe.PQE_ERR_CAPACITY
