"""The host-RAM tier over a paging file (expert-pager article, エキスパート重みの
階層ページング and SSD階層), host only: the paging file holds every page at a
4096-byte offset; the RAM tier's LRU state equals the oracle's LRU driven, step
by step, by the VRAM tier's misses with RAM_SLOTS slots; every page it hands
out is the page's bytes, read from the file on a RAM miss. No GPU needed.
"""
import os

import numpy as np
import pytest
import torch


def _pqe():
    import paged_quantized_expert_gb300 as pqe
    pqe.load()
    return pqe


def _aligned(nbytes, align=4096):
    buf = np.zeros(nbytes + align, np.uint8)
    off = (-buf.ctypes.data) % align
    return buf[off:off + nbytes]


def _pages(E, g, sizes=None):
    sizes = sizes or [int(g.integers(1, 9)) * 1000 + int(g.integers(0, 64)) * 16 for _ in range(E)]
    return [g.integers(0, 256, n).astype(np.uint8) for n in sizes]


def test_paging_file_layout(tmp_path):
    pqe = _pqe()
    g = np.random.default_rng(1)
    pages = _pages(5, g, [4096, 5000, 1, 8192, 12345])
    path = str(tmp_path / "experts.pqe")
    offs = pqe.pqe_paging_file_write(path, pages, [p.size for p in pages])
    exp, at = [], 0
    for p in pages:
        exp.append(at)
        at += -(-p.size // 4096) * 4096
    assert offs == exp and os.path.getsize(path) == at
    raw = np.fromfile(path, np.uint8)
    for o, p in zip(offs, pages):
        assert np.array_equal(raw[o:o + p.size], p)
        pad_end = o + -(-p.size // 4096) * 4096
        assert not raw[o + p.size:pad_end].any()


def _counts(E, used):
    c = np.zeros(E, np.int32)
    c[list(used)] = 1
    return c


@pytest.mark.parametrize("E,S_vram,S_ram,maxk,steps", [(64, 8, 20, 12, 120), (32, 4, 32, 6, 60), (48, 0, 6, 16, 50)])
def test_ram_tier_matches_oracle_lru_on_vram_misses(tmp_path, orc, E, S_vram, S_ram, maxk, steps):
    pqe = _pqe()
    g = np.random.default_rng(E + S_ram)
    pages = _pages(E, g)
    path = str(tmp_path / "experts.pqe")
    offs = pqe.pqe_paging_file_write(path, pages, [p.size for p in pages])
    slot = 16384
    W_ram = E
    ram = _aligned((S_ram + W_ram) * slot)
    tier = pqe.RamTier(path, offs, [p.size for p in pages], S_ram, W_ram, ram, slot, n_threads=3)
    vram = pqe.LRU(E, S_vram)
    ref_vram, ref_ram = orc.LRU(E, S_vram), orc.LRU(E, S_ram)
    zipf = 1.0 / np.arange(1, E + 1) ** 1.1
    zipf /= zipf.sum()
    for step in range(steps):
        k = int(g.integers(1, maxk + 1))
        used = g.choice(E, k, replace=False, p=zipf)
        counts = _counts(E, used)
        _, me, _, _ = vram.page_table_update(torch.from_numpy(counts))
        _, rme, _, _ = ref_vram.step(counts)
        assert sorted(me.tolist()) == sorted(rme.tolist())
        need = np.zeros(E, np.int32)
        need[me.numpy()] = 1
        addr, queued, n_read, working = tier.request(need)
        tier.wait()
        table, r_miss, _, r_wb = ref_ram.step(need)
        assert n_read == len(r_miss) and working == r_wb
        assert sorted(e for e in range(E) if queued[e]) == sorted(r_miss.tolist())
        se, lu, st, _ = tier.state()
        rse, rlu, rst = ref_ram.state()
        assert se == rse.tolist() and lu == rlu.tolist() and st == rst
        for e in range(E):
            if not need[e]:
                assert addr[e] is None
                continue
            assert addr[e] == tier.ram_addr + int(table[e]) * slot  # the oracle's slot or working entry
            got = np.ctypeslib.as_array((np.ctypeslib.ctypes.c_uint8 * pages[e].size).from_address(addr[e]))
            assert np.array_equal(got, pages[e])
    stats = tier.state()[3]
    assert stats["reads"] > 0 and isinstance(stats["direct_io"], bool)
    tier.close()


def test_ram_tier_capacity_and_io_errors(tmp_path):
    pqe = _pqe()
    g = np.random.default_rng(7)
    E = 10
    pages = _pages(E, g)
    path = str(tmp_path / "experts.pqe")
    offs = pqe.pqe_paging_file_write(path, pages, [p.size for p in pages])
    slot = 16384
    ram = _aligned((2 + 3) * slot)
    tier = pqe.RamTier(path, offs, [p.size for p in pages], 2, 3, ram, slot, n_threads=2)
    with pytest.raises(pqe.PqeError) as ei:  # 5 pages needed: 2 slots + 3 entries hold only 3 of a working step
        tier.request([1, 1, 1, 1, 1, 0, 0, 0, 0, 0])
    assert ei.value.code == pqe.PQE_ERR_CAPACITY
    tier.close()
    # a paging file cut short: the read fails and the wait reports it
    with open(path, "r+b") as f:
        f.truncate(offs[E - 1])
    tier = pqe.RamTier(path, offs, [p.size for p in pages], 2, 3, ram, slot, n_threads=2, direct_io=False)
    need = [0] * E
    need[E - 1] = 1
    tier.request(need)
    with pytest.raises(pqe.PqeError) as ei:
        tier.wait()
    assert ei.value.code == pqe.PQE_ERR_IO
    tier.close()
    # bad configurations are refused
    with pytest.raises(pqe.PqeError):
        pqe.RamTier(path, offs, [p.size for p in pages], 2, 3, ram[1:], slot)   # RAM not 4096-aligned
    with pytest.raises(pqe.PqeError):
        pqe.RamTier(path, offs, [p.size for p in pages], 2, 3, ram, 4096)       # a page larger than a slot
