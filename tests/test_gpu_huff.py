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
    l13 = torch.zeros(4096, dtype=torch.uint8)
    l2 = torch.zeros(4096, dtype=torch.uint8)
    n = pqe.pqe_huff_encode_page(torch.from_numpy(page), H, I, out, l13, l2)
    return out[:n].clone(), torch.cat([l13, l2])


def _decode(pqe, comp, luts, H, I, comp_bytes=None):
    dev = torch.zeros(comp.numel() + 256, dtype=torch.uint8, device=DEV)
    dev[:comp.numel()].copy_(comp)
    lut = luts.to(DEV)
    out = torch.zeros(pqe.page_bytes(pqe.PQE_FMT_FP8, H, I), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pqe.fp8_exp_huff_decode(dev, comp.numel() if comp_bytes is None else comp_bytes, lut[:4096], lut[4096:], H, I,
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
    pqe.slot_fill_compressed(pool, 2, pinned, comp.numel(), staging, lut[:4096], lut[4096:], status, stream=side,
                             done_event=ev)
    ev.synchronize()
    stride = pqe.slot_stride(cfg.H, cfg.I)
    got = pool_mem[2 * stride:2 * stride + page.size].cpu().numpy()
    assert int(status.item()) == 0 and np.array_equal(got, page)
    assert int(torch.count_nonzero(pool_mem[:2 * stride]).item()) == 0
