"""GPU: refills from the pinned host tier, one page at a time (slot_fill) and
all misses of a step in one kernel (slot_fill_batch); the destination bytes
equal the host pages and nothing else in the pool changes."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_slot_fill_batch_cache_and_working_buffer(cuda_lib):
    pqe = cuda_lib
    H, I = 256, 128
    stride = pqe.slot_stride(H, I)
    n_slots, n_wb = 5, 4
    pool_mem = torch.zeros(n_slots * stride, dtype=torch.uint8, device=DEV)
    wb_mem = torch.zeros(n_wb * stride, dtype=torch.uint8, device=DEV)
    pool = pqe.make_pool(pool_mem, n_slots, H, I, wb_mem, n_wb)
    g = torch.Generator().manual_seed(0)
    host = torch.randint(0, 256, (6, stride), dtype=torch.uint8, generator=g).pin_memory()
    fp8 = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    fp4 = pqe.page_bytes(pqe.PQE_FMT_MXFP4, H, I)
    dests = [3, 0, 6, 8, 1]
    srcs = [host[0], host[2], host[5], host[1], host[4]]
    sizes = [fp8, fp4, fp8, fp4, fp8]
    pqe.slot_fill_batch(pool, dests, srcs, sizes)
    torch.cuda.synchronize()
    exp_pool = torch.zeros_like(pool_mem).cpu()
    exp_wb = torch.zeros_like(wb_mem).cpu()
    for d, s, n in zip(dests, srcs, sizes):
        tgt, off = (exp_pool, d * stride) if d < n_slots else (exp_wb, (d - n_slots) * stride)
        tgt[off:off + n] = s[:n]
    assert torch.equal(pool_mem.cpu(), exp_pool)
    assert torch.equal(wb_mem.cpu(), exp_wb)


def test_slot_fill_batch_many_pages(cuda_lib):
    # more pages than one launch carries (128): the call splits them
    pqe = cuda_lib
    H, I = 64, 64
    stride = pqe.slot_stride(H, I)
    n = 300
    pool_mem = torch.zeros(n * stride, dtype=torch.uint8, device=DEV)
    pool = pqe.make_pool(pool_mem, n, H, I)
    host = torch.randint(0, 256, (n, stride), dtype=torch.uint8).pin_memory()
    nb = pqe.page_bytes(pqe.PQE_FMT_FP8, H, I)
    perm = np.random.default_rng(1).permutation(n)
    pqe.slot_fill_batch(pool, perm.tolist(), [host[i] for i in range(n)], [nb] * n)
    torch.cuda.synchronize()
    got = pool_mem.view(n, stride).cpu()
    for i in range(n):
        assert torch.equal(got[perm[i], :nb], host[i, :nb])


def test_slot_fill_batch_rejects_bad_entries(cuda_lib):
    pqe = cuda_lib
    H, I = 64, 64
    pool_mem, pool = pqe.alloc_pool(2, H, I)
    host = torch.zeros((1, pqe.slot_stride(H, I)), dtype=torch.uint8).pin_memory()
    with pytest.raises(pqe.PqeError):
        pqe.slot_fill_batch(pool, [2], [host[0]], [16])          # outside the pool
    with pytest.raises(pqe.PqeError):
        pqe.slot_fill_batch(pool, [0], [host[0]], [24])          # not a multiple of 16
    with pytest.raises(pqe.PqeError):
        pqe.slot_fill_batch(pool, [0], [host[0]], [pqe.slot_stride(H, I) + 16])
