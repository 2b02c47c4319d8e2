"""The C-ABI library loads and exports every entry point include/pqe.h declares.

CPU only: no compute call needs a GPU here.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "pqe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^PQE_API [^(]*?\b([a-z_0-9]+)\(", text, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("moe_route", "moe_permute", "moe_paged_ffn", "moe_combine", "page_table_update", "slot_fill",
              "fp8_exp_huff_decode"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import ctypes
    import paged_quantized_expert_gb300 as pqe
    lib = pqe.load()
    for n in _declared():
        assert hasattr(lib, n), n
    # and the binding declares a signature for each of them, under the same name
    assert sorted(pqe.ABI_SYMBOLS) == _declared()
    raw = ctypes.CDLL(pqe.LIB_PATH)
    for n in _declared():
        getattr(raw, n)


def test_host_only_calls_without_gpu():
    import paged_quantized_expert_gb300 as pqe
    pqe.load()
    assert pqe.lib().pqe_abi_version() == 1
    assert pqe.page_bytes(pqe.PQE_FMT_FP8, 2048, 512) == 3 * 2 ** 20 + 4 * (2 * 512 + 2048)
    assert pqe.page_bytes(pqe.PQE_FMT_MXFP4, 2048, 512) == 1572864 + 98304
    assert pqe.slot_stride(2560, 640) % 4096 == 0
    assert pqe.page_bytes(pqe.PQE_FMT_FP8, 100, 512) == 0   # H not a multiple of 64
    assert pqe.lib().pqe_strerror(-4) == b"corrupt compressed page"


def test_invalid_arguments_are_rejected_before_any_launch():
    import paged_quantized_expert_gb300 as pqe
    lib = pqe.load()
    # k > E, E too large, null outputs: all refused on the host
    assert lib.moe_route(None, None, None, 4, 64, 4, 8, None, None, None) == pqe.PQE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, None, 4, 64, 2000, 8, None, None, None) == pqe.PQE_ERR_INVALID_ARG
    assert lib.moe_permute(None, 4, 2, 8, None, None, None, None, None, 0, None, None) == pqe.PQE_ERR_INVALID_ARG
    assert lib.moe_combine(None, None, None, 4, 2, 100, None, None) == pqe.PQE_ERR_INVALID_ARG
    assert lib.pqe_lru_create(0, 4) is None
