"""Python binding of libpqe: the MoE expert layer over paged, quantized expert
weights on one GB300 (sm_103a).

Each function below has the name of a C entry point in include/pqe.h and only
marshals arguments: tensors become device (or host) pointers, streams become
cudaStream_t handles, non-zero return codes become PqeError. All compute
happens in the CUDA library; there is no other implementation, and loading
fails loudly when the library cannot be built or loaded.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from . import build as _build

PQE_OK = 0
PQE_ERR_INVALID_ARG = -1
PQE_ERR_CUDA = -2
PQE_ERR_CAPACITY = -3
PQE_ERR_CORRUPT = -4
PQE_ERR_TIMEOUT = -5
PQE_ERR_UNSUPPORTED = -6
PQE_ERR_IO = -7

PQE_STATUS_BAD_EXPERT_ID = 0x1
PQE_STATUS_CORRUPT_STREAM = 0x2
PQE_STATUS_BAD_PAGE = 0x4
PQE_STATUS_TIMEOUT = 0x8

PQE_FMT_FP8 = 0
PQE_FMT_MXFP4 = 1
PQE_HUFF_LUT_BYTES = 16384

LIB_PATH = _build.LIB


class PqeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.pqe_strerror(code).decode() if _lib else str(code)
        extra = ""
        if code == PQE_ERR_CUDA and _lib:
            extra = f" (cudaError {_lib.pqe_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{code}]{extra}")
        self.code = code


class pqe_layer_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("E", "H", "I", "k", "S", "W", "max_T", "compressed", "device_pager",
                                         "overlap_groups")]


class pqe_step_info(C.Structure):
    _fields_ = [("n_routed", C.c_int32), ("n_miss", C.c_int32), ("working_buffer", C.c_int32),
                ("n_file_read", C.c_int32), ("h2d_bytes", C.c_int64)]


class pqe_ram_tier_config(C.Structure):
    _fields_ = [("E", C.c_int32), ("S", C.c_int32), ("W", C.c_int32), ("n_threads", C.c_int32),
                ("direct_io", C.c_int32), ("pad", C.c_int32), ("slot_bytes", C.c_uint64)]


class pqe_layer_buffers_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("status", "topk_ids", "topk_w", "counts", "offsets", "perm_src", "inv",
                                          "page_table", "out_perm", "x_in", "logits_in", "y_out")]


class pqe_pool(C.Structure):
    _fields_ = [("base", C.c_void_p), ("wb_base", C.c_void_p), ("slot_stride", C.c_size_t),
                ("n_slots", C.c_int32), ("n_wb", C.c_int32), ("H", C.c_int32), ("I", C.c_int32)]


_lib: Optional[C.CDLL] = None
P = C.c_void_p
I32 = C.c_int
SZ = C.c_size_t

_SIGS = {
    "pqe_strerror": (C.c_char_p, [I32]),
    "pqe_abi_version": (I32, []),
    "pqe_last_cuda_error": (I32, []),
    "pqe_kernel_launches": (C.c_uint64, []),
    "pqe_set_wait_limit": (I32, [C.c_uint32]),
    "pqe_test_set_phase2_bias": (I32, [C.c_uint32]),
    "pqe_test_set_stream_kernel": (I32, [C.c_int]),
    "pqe_layer_set_ffn_events": (I32, [P, P, P]),
    "pqe_layer_set_step_graphs": (I32, [P, I32]),
    "pqe_page_bytes": (SZ, [I32, I32, I32]),
    "pqe_slot_stride": (SZ, [I32, I32]),
    "pqe_quantize_fp8_rows": (I32, [P, I32, I32, P, P, P]),
    "pqe_quantize_mxfp4_rows": (I32, [P, P, I32, I32, P, P, P]),
    "moe_route": (I32, [P, P, P, I32, I32, I32, I32, P, P, P]),
    "moe_permute_workspace_size": (SZ, [I32, I32, I32]),
    "moe_permute": (I32, [P, I32, I32, I32, P, P, P, P, P, SZ, P, P]),
    "moe_permute_static_max_words": (SZ, []),
    "moe_permute_static": (I32, [P, I32, I32, I32, P, P, P, P, P, P]),
    "moe_paged_ffn_workspace_size": (SZ, [I32, I32, I32, I32, I32]),
    "moe_paged_ffn": (I32, [P, P, P, P, P, C.POINTER(pqe_pool), I32, I32, I32, P, P, SZ, P, P]),
    "moe_combine": (I32, [P, P, P, I32, I32, I32, P, P]),
    "pqe_lru_create": (P, [I32, I32]),
    "pqe_lru_destroy": (None, [P]),
    "pqe_lru_state": (I32, [P, P, P, P]),
    "pqe_lru_invalidate": (I32, [P, I32]),
    "page_table_update": (I32, [P, P, P, P, P, P, P]),
    "slot_fill": (I32, [C.POINTER(pqe_pool), I32, P, SZ, P, P]),
    "slot_fill_batch": (I32, [C.POINTER(pqe_pool), I32, P, P, P, P, P]),
    "pqe_huff_page_bound": (SZ, [I32, I32]),
    "pqe_huff_encode_page": (I32, [P, I32, I32, P, SZ, C.POINTER(C.c_size_t), P, P]),
    "pqe_huff_page_lengths": (I32, [P, P, P]),
    "pqe_huff_build_lut": (I32, [P, P]),
    "fp8_exp_huff_decode": (I32, [P, SZ, P, P, I32, I32, P, P, P]),
    "slot_fill_compressed": (I32, [C.POINTER(pqe_pool), I32, P, SZ, P, SZ, P, P, P, P, P]),
    "fp8_exp_huff_decode_batch": (I32, [I32, P, P, P, P, I32, I32, P, P, P]),
    "slot_fill_compressed_batch": (I32, [C.POINTER(pqe_pool), I32, P, P, P, P, P, P, P, P]),
    "pqe_importance_step": (I32, [P, P, P, I32, I32, I32, C.c_double, C.c_int64, I32, I32, P, P]),
    "pqe_rank_formats": (I32, [P, I32, I32, P]),
    "pqe_module_batch_size": (C.c_int64, [I32, I32, I32, I32, C.c_double, C.c_double, I32]),
    "pqe_rank_formats_quality": (I32, [P, P, I32, I32, P]),
    "pqe_quality_workspace_size": (SZ, [I32, I32, I32]),
    "pqe_expert_quant_error": (I32, [P, I32, P, P, I32, I32, P, P, SZ, P, P]),
    "pqe_pool_slot_addr": (P, [C.POINTER(pqe_pool), I32]),
    "pqe_lru_device_bytes": (SZ, [I32, I32]),
    "pqe_lru_device_init": (I32, [P, I32, I32, P]),
    "pqe_lru_device_invalidate": (I32, [P, I32, I32, I32, P]),
    "pqe_lru_device_state": (I32, [P, I32, I32, P, P, P, P, P]),
    "page_table_update_device": (I32, [P, I32, I32, P, P, P, P, P]),
    "slot_fill_device": (I32, [C.POINTER(pqe_pool), P, I32, P, P, P]),
    "pqe_layer_device_stats": (I32, [P, P, P, P, P, P]),
    "pqe_pack_fp8_page": (I32, [P, P, I32, I32, P, P]),
    "pqe_pack_mxfp4_page": (I32, [P, I32, I32, P, P]),
    "pqe_layer_scratch_bytes": (SZ, [P]),
    "pqe_layer_create": (P, [P, C.POINTER(pqe_pool), P, P, P, P, P, SZ]),
    "pqe_layer_destroy": (None, [P]),
    "pqe_layer_set_host_page": (I32, [P, I32, P, SZ]),
    "pqe_layer_buffers": (I32, [P, P]),
    "pqe_layer_lru_state": (I32, [P, P, P, P]),
    "pqe_layer_step": (I32, [P, P, P, P, I32, P, P, P, P]),
    "pqe_layer_step_host": (I32, [P, P, P, P, I32, P, P, P, P]),
    "pqe_layer_attach_ram_tier": (I32, [P, P]),
    "pqe_paging_file_write": (I32, [C.c_char_p, I32, P, P, P]),
    "pqe_ram_tier_create": (P, [C.POINTER(pqe_ram_tier_config), C.c_char_p, P, P, P]),
    "pqe_ram_tier_destroy": (None, [P]),
    "pqe_ram_tier_request": (I32, [P, P, P, P, P, P]),
    "pqe_ram_tier_wait": (I32, [P]),
    "pqe_ram_tier_state": (I32, [P, P, P, P, P]),
    "pqe_ram_tier_page_bytes": (SZ, [P, I32]),
}

# every entry point of include/pqe.h
ABI_SYMBOLS = tuple(_SIGS)


def load(build_if_needed: bool = True) -> C.CDLL:
    """Load libpqe.so (building it first when its sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_needed:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpqe.so is missing at {LIB_PATH}; build it with paged_quantized_expert_gb300.build")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def lib() -> C.CDLL:
    return _lib if _lib is not None else load()


def _check(fn: str, rc: int):
    if rc != PQE_OK:
        raise PqeError(fn, rc)


def _nbytes(t) -> int:
    """Byte size of a buffer tensor (any dtype)."""
    return t.numel() * t.element_size()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors passed to libpqe must be contiguous")
        return t.data_ptr()
    raise TypeError(f"cannot pass {type(t)} as a pointer")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _event(ev) -> Optional[int]:
    if ev is None:
        return None
    if isinstance(ev, torch.cuda.Event):
        return ev.cuda_event
    return int(ev)


# ---- page layout ---------------------------------------------------------------

def page_bytes(fmt: int, H: int, I: int) -> int:
    return lib().pqe_page_bytes(fmt, H, I)


def slot_stride(H: int, I: int) -> int:
    return lib().pqe_slot_stride(H, I)


def page_layout(fmt: int, H: int, I: int) -> dict:
    """Byte offsets of the page sections (pqe.h, "Expert pages and the slot pool")."""
    ih = H * I
    if fmt == PQE_FMT_FP8:
        return {"w13": 0, "w2": 2 * ih, "s13": 3 * ih, "s2": 3 * ih + 8 * I, "bytes": page_bytes(fmt, H, I)}
    return {"w13": 0, "w2": ih, "s13": 3 * ih // 2, "s2": 3 * ih // 2 + ih // 16, "bytes": page_bytes(fmt, H, I)}


def make_pool(base: Optional[torch.Tensor], n_slots: int, H: int, I: int, wb: Optional[torch.Tensor] = None,
              n_wb: int = 0) -> pqe_pool:
    """Describe cache slots (``base``) and working-buffer entries (``wb``) for the library."""
    stride = slot_stride(H, I)
    if n_slots and (base is None or base.numel() * base.element_size() < n_slots * stride):
        raise ValueError("pool tensor too small")
    if n_wb and (wb is None or wb.numel() * wb.element_size() < n_wb * stride):
        raise ValueError("working-buffer tensor too small")
    return pqe_pool(base.data_ptr() if n_slots else None, wb.data_ptr() if n_wb else None, stride, n_slots, n_wb,
                    H, I)


def alloc_pool(n_slots: int, H: int, I: int, device="cuda") -> tuple[torch.Tensor, pqe_pool]:
    """A pool of n_slots cache slots and no working buffer."""
    t = torch.zeros(max(n_slots, 1) * slot_stride(H, I), dtype=torch.uint8, device=device)
    return t, make_pool(t, n_slots, H, I)


def alloc_working_buffer(n_wb: int, H: int, I: int, device="cuda") -> torch.Tensor:
    return torch.zeros(max(n_wb, 1) * slot_stride(H, I), dtype=torch.uint8, device=device)


def pqe_pool_slot_addr(pool: pqe_pool, dest: int) -> Optional[int]:
    return lib().pqe_pool_slot_addr(C.byref(pool), dest)


# ---- quantisers ----------------------------------------------------------------

def pqe_quantize_fp8_rows(w, q, scale, stream=None):
    rows, cols = w.shape
    _check("pqe_quantize_fp8_rows", lib().pqe_quantize_fp8_rows(_ptr(w), rows, cols, _ptr(q), _ptr(scale),
                                                                _stream(stream)))


def pqe_quantize_mxfp4_rows(q8, s8, q4, x8, stream=None):
    rows, cols = q8.shape
    _check("pqe_quantize_mxfp4_rows", lib().pqe_quantize_mxfp4_rows(_ptr(q8), _ptr(s8), rows, cols, _ptr(q4),
                                                                    _ptr(x8), _stream(stream)))


# ---- hot path ------------------------------------------------------------------

def moe_route(x, w_router, logits, T, H, E, k, topk_ids, topk_w, stream=None):
    _check("moe_route", lib().moe_route(_ptr(x), _ptr(w_router), _ptr(logits), T, H, E, k, _ptr(topk_ids),
                                        _ptr(topk_w), _stream(stream)))


def moe_permute_workspace_size(T, k, E) -> int:
    return lib().moe_permute_workspace_size(T, k, E)


def moe_permute(topk_ids, T, k, E, counts, offsets, perm_src, inv, ws, status, stream=None):
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("moe_permute", lib().moe_permute(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm_src),
                                            _ptr(inv), _ptr(ws), nbytes, _ptr(status), _stream(stream)))


def moe_permute_static(topk_ids, T, k, E, counts, offsets, perm_src, inv, status, stream=None):
    """moe_permute with the library's own fixed device scratch (no workspace argument)."""
    _check("moe_permute_static", lib().moe_permute_static(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets),
                                                          _ptr(perm_src), _ptr(inv), _ptr(status), _stream(stream)))


def moe_paged_ffn_workspace_size(T, k, E, H, I) -> int:
    return lib().moe_paged_ffn_workspace_size(T, k, E, H, I)


def moe_paged_ffn(x, perm_src, offsets, page_table, expert_fmt, pool: pqe_pool, T, k, E, out_perm, ws, status,
                  stream=None):
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("moe_paged_ffn", lib().moe_paged_ffn(_ptr(x), _ptr(perm_src), _ptr(offsets), _ptr(page_table),
                                                _ptr(expert_fmt), C.byref(pool), T, k, E, _ptr(out_perm),
                                                _ptr(ws), nbytes, _ptr(status), _stream(stream)))


def moe_combine(out_perm, inv, topk_w, T, k, H, y, stream=None):
    _check("moe_combine", lib().moe_combine(_ptr(out_perm), _ptr(inv), _ptr(topk_w), T, k, H, _ptr(y),
                                            _stream(stream)))


# ---- pager ---------------------------------------------------------------------

class LRU:
    """Host LRU state of one layer's slot pool (pqe_lru)."""

    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self._h = lib().pqe_lru_create(E, S)
        if not self._h:
            raise PqeError("pqe_lru_create", PQE_ERR_INVALID_ARG)
        self._pt = torch.empty(E, dtype=torch.int32)
        self._me = torch.empty(E, dtype=torch.int32)
        self._md = torch.empty(E, dtype=torch.int32)
        self._n = torch.zeros(2, dtype=torch.int32)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.pqe_lru_destroy(h)
            self._h = None

    def page_table_update(self, counts_host: torch.Tensor, page_table_host: torch.Tensor = None):
        """-> (page_table [E], miss_expert [n], miss_dest [n], working_buffer_mode)"""
        pt = self._pt if page_table_host is None else page_table_host
        nm = self._n[0:1]
        wb = self._n[1:2]
        _check("page_table_update", lib().page_table_update(self._h, _ptr(counts_host), _ptr(pt), _ptr(self._me),
                                                            _ptr(self._md), _ptr(nm), _ptr(wb)))
        n = int(nm.item())
        return pt, self._me[:n], self._md[:n], bool(wb.item())

    def state(self):
        se = torch.empty(self.S, dtype=torch.int32)
        lu = torch.empty(self.S, dtype=torch.int64)
        st = torch.zeros(1, dtype=torch.int64)
        _check("pqe_lru_state", lib().pqe_lru_state(self._h, _ptr(se), _ptr(lu), _ptr(st)))
        return se, lu, int(st.item())

    def invalidate(self, expert: int):
        _check("pqe_lru_invalidate", lib().pqe_lru_invalidate(self._h, expert))


def page_table_update(lru: LRU, counts_host, page_table_host=None):
    return lru.page_table_update(counts_host, page_table_host)


def slot_fill_batch(pool: pqe_pool, dests, pinned_srcs, nbytes, stream=None, done_event=None):
    """dests: entries; pinned_srcs: pinned tensors (or addresses); nbytes: bytes per page."""
    n = len(dests)
    d = (C.c_int32 * n)(*[int(x) for x in dests])
    s = (C.c_void_p * n)(*[_ptr(x) for x in pinned_srcs])
    b = (C.c_size_t * n)(*[int(x) for x in nbytes])
    _check("slot_fill_batch", lib().slot_fill_batch(C.byref(pool), n, C.cast(d, C.c_void_p), C.cast(s, C.c_void_p),
                                                    C.cast(b, C.c_void_p), _stream(stream), _event(done_event)))


def slot_fill(pool: pqe_pool, dest: int, pinned_src, nbytes: int, stream=None, done_event=None):
    _check("slot_fill", lib().slot_fill(C.byref(pool), dest, _ptr(pinned_src), nbytes, _stream(stream),
                                        _event(done_event)))


# ---- compressed host tier ---------------------------------------------------------

def pqe_huff_page_bound(H: int, I: int) -> int:
    return lib().pqe_huff_page_bound(H, I)


def pqe_huff_encode_page(fp8_page: torch.Tensor, H: int, I: int, out: torch.Tensor, lut13: torch.Tensor,
                         lut2: torch.Tensor) -> int:
    """Host tensors. Returns the compressed size in bytes."""
    n = C.c_size_t(0)
    _check("pqe_huff_encode_page", lib().pqe_huff_encode_page(_ptr(fp8_page), H, I, _ptr(out), _nbytes(out),
                                                              C.byref(n), _ptr(lut13), _ptr(lut2)))
    return n.value


def pqe_huff_page_lengths(comp_page: torch.Tensor):
    l13 = torch.zeros(16, dtype=torch.uint8)
    l2 = torch.zeros(16, dtype=torch.uint8)
    _check("pqe_huff_page_lengths", lib().pqe_huff_page_lengths(_ptr(comp_page), _ptr(l13), _ptr(l2)))
    return l13, l2


def pqe_huff_build_lut(lengths: torch.Tensor, lut: torch.Tensor):
    _check("pqe_huff_build_lut", lib().pqe_huff_build_lut(_ptr(lengths), _ptr(lut)))


def fp8_exp_huff_decode(comp_page, comp_bytes, lut13, lut2, H, I, fp8_page, status, stream=None):
    _check("fp8_exp_huff_decode", lib().fp8_exp_huff_decode(_ptr(comp_page), comp_bytes, _ptr(lut13), _ptr(lut2),
                                                            H, I, _ptr(fp8_page), _ptr(status), _stream(stream)))


def _ptr_array(xs):
    return (C.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def fp8_exp_huff_decode_batch(comp_pages, comp_bytes, lut13, lut2, H, I, fp8_pages, status, stream=None):
    """Lists of n tensors (or addresses): compressed pages (device or pinned host), their sizes, code tables,
    destinations; one launch per 128 pages."""
    n = len(comp_pages)
    cb = (C.c_size_t * n)(*[int(b) for b in comp_bytes])
    arrs = [_ptr_array(x) for x in (comp_pages, lut13, lut2, fp8_pages)]
    _check("fp8_exp_huff_decode_batch", lib().fp8_exp_huff_decode_batch(
        n, C.cast(arrs[0], C.c_void_p), C.cast(cb, C.c_void_p), C.cast(arrs[1], C.c_void_p),
        C.cast(arrs[2], C.c_void_p), H, I, C.cast(arrs[3], C.c_void_p), _ptr(status), _stream(stream)))


def slot_fill_compressed_batch(pool: pqe_pool, dests, pinned_comp, comp_bytes, lut13, lut2, status, stream=None,
                               done_event=None):
    n = len(dests)
    d = (C.c_int32 * n)(*[int(x) for x in dests])
    cb = (C.c_size_t * n)(*[int(b) for b in comp_bytes])
    arrs = [_ptr_array(x) for x in (pinned_comp, lut13, lut2)]
    _check("slot_fill_compressed_batch", lib().slot_fill_compressed_batch(
        C.byref(pool), n, C.cast(d, C.c_void_p), C.cast(arrs[0], C.c_void_p), C.cast(cb, C.c_void_p),
        C.cast(arrs[1], C.c_void_p), C.cast(arrs[2], C.c_void_p), _ptr(status), _stream(stream), _event(done_event)))


def slot_fill_compressed(pool: pqe_pool, dest, pinned_comp, comp_bytes, staging, lut13, lut2, status, stream=None,
                         done_event=None):
    _check("slot_fill_compressed", lib().slot_fill_compressed(
        C.byref(pool), dest, _ptr(pinned_comp), comp_bytes, _ptr(staging), _nbytes(staging), _ptr(lut13),
        _ptr(lut2), _ptr(status), _stream(stream), _event(done_event)))


# ---- RAM tier and paging file -----------------------------------------------------

def pqe_paging_file_write(path: str, pages, nbytes) -> list:
    """Write pages (host tensors / numpy arrays, or addresses) into a paging file; returns their offsets."""
    n = len(pages)
    srcs = (C.c_void_p * n)(*[p.ctypes.data if hasattr(p, "ctypes") else _ptr(p) for p in pages])
    b = (C.c_size_t * n)(*[int(x) for x in nbytes])
    offs = (C.c_uint64 * n)()
    _check("pqe_paging_file_write", lib().pqe_paging_file_write(os.fsencode(path), n, C.cast(srcs, C.c_void_p),
                                                                C.cast(b, C.c_void_p), C.cast(offs, C.c_void_p)))
    return list(offs)


class RamTier:
    """The host-RAM tier of one layer over a paging file (pqe_ram_tier).

    ``ram`` is host memory of (S + W) * slot_bytes bytes, 4096-byte aligned: a
    pinned tensor when the GPU reads from it, any aligned buffer otherwise."""

    def __init__(self, path: str, offsets, nbytes, S: int, W: int, ram, slot_bytes: int, n_threads: int = 4,
                 direct_io: bool = True):
        E = len(offsets)
        self.E, self.S, self.W, self.slot_bytes = E, S, W, slot_bytes
        self.cfg = pqe_ram_tier_config(E, S, W, n_threads, int(bool(direct_io)), 0, slot_bytes)
        self._ram = ram
        addr = ram.ctypes.data if hasattr(ram, "ctypes") else _ptr(ram)
        self.ram_addr = addr
        offs = (C.c_uint64 * E)(*[int(o) for o in offsets])
        b = (C.c_size_t * E)(*[int(x) for x in nbytes])
        self._h = lib().pqe_ram_tier_create(C.byref(self.cfg), os.fsencode(path), C.cast(offs, C.c_void_p),
                                            C.cast(b, C.c_void_p), addr)
        if not self._h:
            raise PqeError("pqe_ram_tier_create", PQE_ERR_INVALID_ARG)
        self._page = (C.c_void_p * E)()
        self._queued = (C.c_int32 * E)()

    def close(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pqe_ram_tier_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def request(self, need):
        """need [E] (nonzero = wanted from RAM) -> (RAM addresses [E] (None if not needed), read_queued [E],
        n_read, working)."""
        nd = (C.c_int32 * self.E)(*[int(x) for x in need])
        nr = C.c_int32(0)
        wb = C.c_int32(0)
        _check("pqe_ram_tier_request", lib().pqe_ram_tier_request(self._h, C.cast(nd, C.c_void_p),
                                                                  C.cast(self._page, C.c_void_p),
                                                                  C.cast(self._queued, C.c_void_p), C.byref(nr),
                                                                  C.byref(wb)))
        return list(self._page), list(self._queued), nr.value, bool(wb.value)

    def wait(self):
        _check("pqe_ram_tier_wait", lib().pqe_ram_tier_wait(self._h))

    def state(self):
        se = (C.c_int32 * max(self.S, 1))()
        lu = (C.c_int64 * max(self.S, 1))()
        st = C.c_int64(0)
        stats = (C.c_int64 * 4)()
        _check("pqe_ram_tier_state", lib().pqe_ram_tier_state(self._h, C.cast(se, C.c_void_p),
                                                              C.cast(lu, C.c_void_p), C.byref(st),
                                                              C.cast(stats, C.c_void_p)))
        return (list(se)[:self.S], list(lu)[:self.S], st.value,
                {"reads": stats[0], "bytes": stats[1], "working_steps": stats[2], "direct_io": bool(stats[3])})


# ---- bit-width assignment ---------------------------------------------------------

def pqe_importance_step(m: torch.Tensor, ids: torch.Tensor, gates: torch.Tensor, T, k, E, alpha, step, every,
                        n_hi, fmt: torch.Tensor) -> bool:
    rr = torch.zeros(1, dtype=torch.int32)
    _check("pqe_importance_step", lib().pqe_importance_step(_ptr(m), _ptr(ids), _ptr(gates), T, k, E, alpha, step,
                                                            every, n_hi, _ptr(fmt), _ptr(rr)))
    return bool(rr.item())


def pqe_rank_formats_quality(m: torch.Tensor, q: torch.Tensor, n_hi: int, fmt: torch.Tensor):
    """Top n_hi of importance x 4-bit error keep FP8 (host double m, q; host uint8 fmt)."""
    _check("pqe_rank_formats_quality", lib().pqe_rank_formats_quality(_ptr(m), _ptr(q), m.numel(), n_hi, _ptr(fmt)))


def pqe_quality_workspace_size(n: int, H: int, I: int) -> int:
    return int(lib().pqe_quality_workspace_size(n, H, I))


def pqe_expert_quant_error(x, n, page_fp8, page_fp4, H, I, sums, ws, status, stream=None):
    """sums (device float64 [2]) <- (sum ||y4 - y8||^2, sum ||y8||^2) over the n tokens x."""
    _check("pqe_expert_quant_error", lib().pqe_expert_quant_error(_ptr(x), n, _ptr(page_fp8), _ptr(page_fp4), H, I,
                                                                  _ptr(sums), _ptr(ws), _nbytes(ws), _ptr(status),
                                                                  _stream(stream)))


def pqe_module_batch_size(E, k, H, I, hbm_gbs, fp8_tflops, granule=64) -> int:
    """Tokens to accumulate so that the layer's FFN is compute-bound (0: no knee)."""
    return int(lib().pqe_module_batch_size(E, k, H, I, float(hbm_gbs), float(fp8_tflops), granule))


def pqe_rank_formats(m: torch.Tensor, n_hi: int, fmt: torch.Tensor):
    _check("pqe_rank_formats", lib().pqe_rank_formats(_ptr(m), m.numel(), n_hi, _ptr(fmt)))


def pqe_pack_fp8_page(w13, w2, H, I, page, stream=None):
    _check("pqe_pack_fp8_page", lib().pqe_pack_fp8_page(_ptr(w13), _ptr(w2), H, I, _ptr(page), _stream(stream)))


def pqe_pack_mxfp4_page(fp8_page, H, I, fp4_page, stream=None):
    _check("pqe_pack_mxfp4_page", lib().pqe_pack_mxfp4_page(_ptr(fp8_page), H, I, _ptr(fp4_page),
                                                            _stream(stream)))


# ---- layer runtime ---------------------------------------------------------------

class PagedMoELayer:
    """One MoE layer over its own slot pool (pqe_layer): the public per-step API.

    The caller owns the host tier: ``host_pages`` is a pinned uint8 tensor
    [E, page_stride] (or a list of pinned tensors, one page each) holding each
    expert's page in the library's page layout (compressed pages when
    ``compressed``). Device memory (pool, scratch, code tables, format tags) is
    allocated here with PyTorch and handed to the library.
    """

    def __init__(self, E, H, I, k, S, W, max_T, host_pages, host_page_bytes, compressed=False, luts=None,
                 expert_fmt=None, device="cuda", working_buffer: Optional[torch.Tensor] = None,
                 device_pager=False, overlap_groups=0):
        self.cfg = pqe_layer_config(E, H, I, k, S, W, max_T, int(bool(compressed)), int(bool(device_pager)),
                                    int(overlap_groups))
        self.device_pager = bool(device_pager)
        self.E, self.H, self.I, self.k, self.S, self.W, self.max_T = E, H, I, k, S, W, max_T
        self.pool_mem = torch.zeros(max(S, 1) * slot_stride(H, I), dtype=torch.uint8, device=device)
        # the working buffer holds one step's pages; layers on one stream may share it
        self.wb_mem = working_buffer if working_buffer is not None else alloc_working_buffer(W, H, I, device)
        self.pool = make_pool(self.pool_mem, S, H, I, self.wb_mem, W)
        nbytes = lib().pqe_layer_scratch_bytes(C.byref(self.cfg))
        if nbytes == 0:
            raise PqeError("pqe_layer_scratch_bytes", PQE_ERR_INVALID_ARG)
        self.scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.scratch.data_ptr()) % 256
        self._scratch_ptr = self.scratch.data_ptr() + off
        if isinstance(host_pages, torch.Tensor):
            ptrs = [host_pages[e].data_ptr() for e in range(E)]
        else:
            ptrs = [p.data_ptr() for p in host_pages]
        self._host_keep = host_pages
        self._ptrs = (C.c_void_p * E)(*ptrs)
        self._bytes = (C.c_size_t * E)(*[int(b) for b in host_page_bytes])
        self.luts = luts
        self.expert_fmt = expert_fmt
        self._h = lib().pqe_layer_create(C.byref(self.cfg), C.byref(self.pool), C.cast(self._ptrs, C.c_void_p),
                                         C.cast(self._bytes, C.c_void_p), _ptr(luts), _ptr(expert_fmt),
                                         self._scratch_ptr, nbytes)
        if not self._h:
            raise PqeError("pqe_layer_create", PQE_ERR_INVALID_ARG)
        b = pqe_layer_buffers_t()
        _check("pqe_layer_buffers", lib().pqe_layer_buffers(self._h, C.byref(b)))
        self.buffers = b
        self.info = pqe_step_info()

    def close(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pqe_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def set_host_page(self, expert: int, pinned_page: torch.Tensor, nbytes: int):
        self._host_keep = (self._host_keep, pinned_page) if not isinstance(self._host_keep, list) else \
            self._host_keep + [pinned_page]
        _check("pqe_layer_set_host_page", lib().pqe_layer_set_host_page(self._h, expert, pinned_page.data_ptr(),
                                                                        nbytes))

    def step(self, x, y, T, logits=None, w_router=None, stream=None, side_stream=None) -> pqe_step_info:
        _check("pqe_layer_step", lib().pqe_layer_step(self._h, _ptr(x), _ptr(w_router), _ptr(logits), T, _ptr(y),
                                                      _stream(stream), _stream(side_stream) if side_stream
                                                      is not None else None, C.byref(self.info)))
        return self.info

    def step_host(self, x_host, y_host, T, logits_host=None, w_router=None, stream=None, side_stream=None):
        _check("pqe_layer_step_host", lib().pqe_layer_step_host(
            self._h, _ptr(x_host), _ptr(w_router), _ptr(logits_host), T, _ptr(y_host), _stream(stream),
            _stream(side_stream) if side_stream is not None else None, C.byref(self.info)))
        return self.info

    def attach_ram_tier(self, tier: Optional["RamTier"]):
        """Serve refills from a RAM tier (host pager only); None detaches it."""
        self._ram_tier = tier
        _check("pqe_layer_attach_ram_tier", lib().pqe_layer_attach_ram_tier(self._h, tier._h if tier else None))

    def set_step_graphs(self, enable):
        _check("pqe_layer_set_step_graphs", lib().pqe_layer_set_step_graphs(self._h, 1 if enable else 0))

    def set_ffn_events(self, ev_begin, ev_end):
        _check("pqe_layer_set_ffn_events", lib().pqe_layer_set_ffn_events(self._h, _event(ev_begin),
                                                                          _event(ev_end)))

    def lru_state(self):
        se = torch.empty(self.S, dtype=torch.int32)
        lu = torch.empty(self.S, dtype=torch.int64)
        st = torch.zeros(1, dtype=torch.int64)
        if self.device_pager:
            stats = torch.zeros(4, dtype=torch.int64)
            _check("pqe_layer_device_stats", lib().pqe_layer_device_stats(self._h, _ptr(stats), _ptr(se), _ptr(lu),
                                                                          _ptr(st), _stream(None)))
        else:
            _check("pqe_layer_lru_state", lib().pqe_layer_lru_state(self._h, _ptr(se), _ptr(lu), _ptr(st)))
        return se, lu, int(st.item())

    def device_stats(self, stream=None) -> dict:
        """Device-pager totals since creation (synchronises)."""
        stats = torch.zeros(4, dtype=torch.int64)
        _check("pqe_layer_device_stats", lib().pqe_layer_device_stats(self._h, _ptr(stats), None, None, None,
                                                                      _stream(stream)))
        r, m, w, b = stats.tolist()
        return {"routed": r, "misses": m, "working_buffer_steps": w, "refill_bytes": b}

    def device_view(self, name: str, dtype, shape):
        """A torch view of one of the layer's device buffers (no copy)."""
        ptr = getattr(self.buffers, name)
        n = 1
        for d in shape:
            n *= d
        esize = torch.empty(0, dtype=dtype).element_size()
        base = self.scratch.data_ptr()
        off = ptr - base
        return self.scratch[off:off + n * esize].view(dtype).view(*shape)


def pqe_set_wait_limit(polls: int):
    """Polls of every bounded device wait before it gives up (0: the default)."""
    _check("pqe_set_wait_limit", lib().pqe_set_wait_limit(int(polls)))


def pqe_test_set_phase2_bias(bias: int):
    """Test hook: a nonzero bias makes the weight stream's phase-2 waits expire."""
    _check("pqe_test_set_phase2_bias", lib().pqe_test_set_phase2_bias(int(bias)))


def pqe_test_set_stream_kernel(kind: int):
    """Test hook: the weight-stream kernel, 0 default choice, 1 CUDA cores, 2 tensor cores."""
    _check("pqe_test_set_stream_kernel", lib().pqe_test_set_stream_kernel(int(kind)))


def kernel_launches() -> int:
    """Kernels libpqe has launched in this process."""
    return int(lib().pqe_kernel_launches())


# ---- GPU-resident pager -------------------------------------------------------------

def pqe_lru_device_bytes(E: int, S: int) -> int:
    return lib().pqe_lru_device_bytes(E, S)


def pqe_lru_device_init(state, E, S, stream=None):
    _check("pqe_lru_device_init", lib().pqe_lru_device_init(_ptr(state), E, S, _stream(stream)))


def pqe_lru_device_invalidate(state, E, S, expert, stream=None):
    _check("pqe_lru_device_invalidate", lib().pqe_lru_device_invalidate(_ptr(state), E, S, expert, _stream(stream)))


def pqe_lru_device_state(state, E, S, stream=None):
    se = torch.empty(max(S, 1), dtype=torch.int32)
    lu = torch.empty(max(S, 1), dtype=torch.int64)
    st = torch.zeros(1, dtype=torch.int64)
    stats = torch.zeros(4, dtype=torch.int64)
    _check("pqe_lru_device_state", lib().pqe_lru_device_state(_ptr(state), E, S, _ptr(se), _ptr(lu), _ptr(st),
                                                              _ptr(stats), _stream(stream)))
    return se[:S], lu[:S], int(st.item()), stats


def page_table_update_device(state, E, S, counts, page_bytes, page_table, miss, stream=None):
    _check("page_table_update_device", lib().page_table_update_device(_ptr(state), E, S, _ptr(counts),
                                                                      _ptr(page_bytes), _ptr(page_table), _ptr(miss),
                                                                      _stream(stream)))


def slot_fill_device(pool: pqe_pool, miss, E, host_pages, page_bytes, stream=None):
    _check("slot_fill_device", lib().slot_fill_device(C.byref(pool), _ptr(miss), E, _ptr(host_pages),
                                                      _ptr(page_bytes), _stream(stream)))
