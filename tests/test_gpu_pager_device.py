"""GPU-resident pager: the device LRU step equals the oracle's LRU bit for bit
(page table, misses in order, destinations, slot state, step counter), and the
device-driven refill copies exactly the missed pages."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _counts(E, used, g):
    c = np.zeros(E, np.int32)
    c[list(used)] = g.integers(1, 6, len(used))
    return c


@pytest.mark.parametrize("E,S,maxk,steps", [(256, 32, 70, 120), (1024, 1024, 200, 40), (16, 4, 8, 80),
                                             (8, 0, 3, 10), (512, 46, 60, 60)])
def test_device_lru_matches_oracle(cuda_lib, orc, E, S, maxk, steps):
    pqe = cuda_lib
    state = torch.zeros(pqe.pqe_lru_device_bytes(E, S), dtype=torch.uint8, device=DEV)
    pqe.pqe_lru_device_init(state, E, S)
    ref = orc.LRU(E, S)
    page_bytes = torch.full((E,), 4096, dtype=torch.int64, device=DEV)
    pt = torch.zeros(E, dtype=torch.int32, device=DEV)
    miss = torch.zeros(3 * E + 3, dtype=torch.int32, device=DEV)
    g = np.random.default_rng(E + S)
    for step in range(steps):
        used = g.choice(E, int(g.integers(0, maxk + 1)), replace=False)
        c = _counts(E, used, g)
        if step % 17 == 5 and S > 0:                  # forget one resident expert now and then
            se_now = ref.state()[0]
            res = se_now[se_now >= 0]
            if res.size:
                e = int(res[0])
                ref.invalidate(e)
                pqe.pqe_lru_device_invalidate(state, E, S, e)
        pqe.page_table_update_device(state, E, S, torch.from_numpy(c).to(DEV), page_bytes, pt, miss)
        table, me, md, wb = ref.step(c)
        m = miss.cpu().numpy()
        n = int(m[0])
        assert np.array_equal(pt.cpu().numpy(), table), step
        assert n == len(me) and bool(m[1]) == wb, step
        assert np.array_equal(m[2:2 + n], me) and np.array_equal(m[2 + E:2 + E + n], md), step
        assert np.array_equal(m[2 + 2 * E:2 + 2 * E + n + 1], np.arange(n + 1)), step  # 1 segment per 4 KiB page
        se, lu, st, stats = pqe.pqe_lru_device_state(state, E, S)
        se2, lu2, st2 = ref.state()
        assert np.array_equal(se.numpy(), se2) and np.array_equal(lu.numpy(), lu2) and st == st2, step


def test_device_fill_copies_missed_pages(cuda_lib, orc):
    pqe = cuda_lib
    E, S, H, I = 12, 4, 128, 64
    stride = pqe.slot_stride(H, I)
    pool_mem = torch.zeros(S * stride, dtype=torch.uint8, device=DEV)
    wb_mem = torch.zeros(E * stride, dtype=torch.uint8, device=DEV)
    pool = pqe.make_pool(pool_mem, S, H, I, wb_mem, E)
    host = torch.randint(0, 256, (E, stride), dtype=torch.uint8).pin_memory()
    sizes = [pqe.page_bytes(pqe.PQE_FMT_FP8 if e % 3 else pqe.PQE_FMT_MXFP4, H, I) for e in range(E)]
    ptrs = torch.tensor([host[e].data_ptr() for e in range(E)], dtype=torch.int64, device=DEV)
    nbytes = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    state = torch.zeros(pqe.pqe_lru_device_bytes(E, S), dtype=torch.uint8, device=DEV)
    pqe.pqe_lru_device_init(state, E, S)
    pt = torch.zeros(E, dtype=torch.int32, device=DEV)
    miss = torch.zeros(3 * E + 3, dtype=torch.int32, device=DEV)
    for used in ([1, 4, 7], [0, 1, 2, 3, 4, 5, 6, 8], [2, 9]):
        c = np.zeros(E, np.int32)
        c[used] = 1
        pqe.page_table_update_device(state, E, S, torch.from_numpy(c).to(DEV), nbytes, pt, miss)
        pqe.slot_fill_device(pool, miss, E, ptrs, nbytes)
        torch.cuda.synchronize()
        table = pt.cpu().numpy()
        for e in used:
            d = int(table[e])
            buf = pool_mem if d < S else wb_mem
            off = (d if d < S else d - S) * stride
            assert torch.equal(buf[off:off + sizes[e]].cpu(), host[e, :sizes[e]]), (used, e)
