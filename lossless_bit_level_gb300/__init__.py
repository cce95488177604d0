"""Python binding of the GB300 Invariant Bit Packing codec (``include/ibp.h``).

Argument marshalling only: every step of the codec runs in the CUDA kernels of
``_build/libibp_gb300.so``. Tensors are torch tensors used as plain memory
(device memory, or page-locked host memory for rows and slots read or written
zero-copy); calls are enqueued on the current CUDA stream unless one is given.
There is no CPU fallback: importing works without the library, but every call
raises if the shared library has not been built (``build_lib.build()``).

Method: "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
Extended", technical summary, "Core algorithm" and "System integration".

The path, in order:
  build_meta (or meta_count + meta_finalize across holders; build_meta_select for
  the saving-aware mask)       -> 16-byte metadata in device memory
  compress                     -> fixed-size slots + bitmask (+ row sizes)
  decompress_gather            -> the rows an index list names, rebuilt bit for bit
Gather variants: decompress_gather_dedup (each distinct row read once),
decompress_gather_sized (only each row's used bytes), decompress_gather_batched
(several tables in one launch), decompress_range (rows in order). Next to them: the
packed store (pack_offsets, pack, decompress_gather_packed) and per-position or
block-position metadata (build_meta_positions, build_meta_block_positions,
compress_positions, decompress_gather_positions). ``offload.py`` streams compressed
tensors through device buffers; ``sharded.py`` builds the metadata of a table spread
over several processes.
"""
from __future__ import annotations

import ctypes
import os
import struct

import torch

from . import build_lib

FP32, FP16, BF16, W8 = 0, 1, 2, 3
OK = 0
ERR_ARG, ERR_DTYPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_INDEX, ERR_CORRUPT, ERR_META, ERR_TIMEOUT = (
    -1, -2, -3, -4, -5, -6, -7, -8)

_TORCH_DTYPES = {torch.float32: FP32, torch.float16: FP16, torch.bfloat16: BF16}
for _name in ("float8_e4m3fn", "float8_e5m2"):
    if hasattr(torch, _name):
        _TORCH_DTYPES[getattr(torch, _name)] = W8
WIDTH = {FP32: 32, FP16: 16, BF16: 16, W8: 8}

_lib = None


class IBPError(RuntimeError):
    def __init__(self, code: int, call: str):
        self.code = code
        super().__init__(f"{call}: {status_string(code)} ({code})")


class GatherJob(ctypes.Structure):
    """ibp_gather_job: one gather of a batch."""
    _fields_ = [("slots", ctypes.c_void_p), ("slot_bytes", ctypes.c_int64),
                ("n_rows", ctypes.c_int64), ("d_row_bitmask", ctypes.c_void_p),
                ("d_meta", ctypes.c_void_p), ("d_idx", ctypes.c_void_p),
                ("n_idx", ctypes.c_int64), ("out", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("n_compressed", ctypes.c_int64),
                ("raw_bytes", ctypes.c_int64), ("stored_bytes", ctypes.c_int64),
                ("total_bits", ctypes.c_int64)]


SYMBOLS = ("ibp_status_string", "ibp_slot_bytes", "ibp_meta_scratch_bytes", "ibp_build_meta",
           "ibp_compress", "ibp_decompress_gather", "ibp_query", "ibp_probe_read",
           "ibp_build_meta_noalloc", "ibp_meta_select_scratch_bytes", "ibp_build_meta_select",
           "ibp_pack_scratch_bytes", "ibp_pack_offsets", "ibp_pack", "ibp_decompress_gather_packed",
           "ibp_decompress_range", "ibp_meta_positions_scratch_bytes", "ibp_build_meta_positions",
           "ibp_compress_positions", "ibp_decompress_gather_positions",
           "ibp_decompress_gather_sized", "ibp_decompress_gather_batched", "ibp_meta_count",
           "ibp_meta_finalize", "ibp_build_meta_block_positions", "ibp_gather_dedup_scratch_bytes",
           "ibp_decompress_gather_dedup", "ibp_query_async")

# declared in include/ibp_testing.h (a testing hook, not part of the codec)
TESTING_SYMBOLS = ("ibp_testing_set_wait_limit_ns", "ibp_testing_withhold_plans")

MAX_MASK_CANDIDATES = 33


def library_path() -> str:
    return build_lib.LIB


def load() -> ctypes.CDLL:
    """Load the built library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"IBP CUDA library not built ({path}); run "
                           "lossless_bit_level_gb300.build_lib.build() first")
    lib = ctypes.CDLL(path)
    i64, i32, u32, dbl, vp = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_double,
                              ctypes.c_void_p)
    lib.ibp_status_string.argtypes = [i32]
    lib.ibp_status_string.restype = ctypes.c_char_p
    lib.ibp_slot_bytes.argtypes = [i64, i32, ctypes.POINTER(i64)]
    lib.ibp_meta_scratch_bytes.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
    lib.ibp_build_meta.argtypes = [vp, i64, i64, i32, dbl, u32, vp, vp, vp]
    lib.ibp_compress.argtypes = [vp, i64, i64, i32, u32, vp, vp, i64, vp, vp, vp, vp]
    lib.ibp_decompress_gather.argtypes = [vp, i64, i64, i64, i32, u32, vp, vp, vp, i64, vp, vp, vp]
    lib.ibp_query.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.ibp_query_async.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.ibp_probe_read.argtypes = [vp, i64, vp, vp]
    lib.ibp_build_meta_noalloc.argtypes = [vp, i64, i64, i32, dbl, u32, vp, vp]
    lib.ibp_meta_select_scratch_bytes.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
    lib.ibp_build_meta_select.argtypes = [vp, i64, i64, i32, dbl, u32, vp, vp, vp, vp]
    u64 = ctypes.c_uint64
    lib.ibp_meta_positions_scratch_bytes.argtypes = [i64, i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.ibp_build_meta_positions.argtypes = [vp, i64, i64, i32, dbl, u32, vp, vp, vp, vp]
    lib.ibp_compress_positions.argtypes = [vp, i64, i64, i32, u32, vp, vp, vp, i64, vp, vp, vp]
    lib.ibp_decompress_gather_positions.argtypes = [vp, i64, i64, i64, i32, u32, vp, vp, vp, vp,
                                                    i64, vp, vp, vp]
    lib.ibp_meta_count.argtypes = [vp, i64, i64, i32, vp, vp]
    lib.ibp_gather_dedup_scratch_bytes.argtypes = [i64, i64, i32, u32, ctypes.POINTER(ctypes.c_size_t)]
    lib.ibp_decompress_gather_dedup.argtypes = [vp, i64, i64, i64, i32, u32, vp, vp, vp, i64, vp, vp,
                                                ctypes.c_size_t, vp, vp]
    lib.ibp_build_meta_block_positions.argtypes = [vp, i64, i64, i32, dbl, u32, vp, vp, vp, vp]
    lib.ibp_meta_finalize.argtypes = [vp, i64, i32, dbl, u32, vp, vp, vp]
    lib.ibp_decompress_gather_batched.argtypes = [vp, i32, i64, i32, u32, vp, vp]
    lib.ibp_decompress_gather_sized.argtypes = [vp, i64, i64, i64, i32, u32, vp, vp, vp, vp, i64,
                                                vp, vp, vp]
    lib.ibp_decompress_range.argtypes = [vp, i64, i64, i64, i32, u32, vp, vp, i64, i64, vp, vp, vp]
    lib.ibp_pack_scratch_bytes.argtypes = [i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.ibp_pack_offsets.argtypes = [vp, vp, i64, i64, i32, vp, i64, vp, vp, vp, vp]
    lib.ibp_pack.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, i64, vp, vp, u64, vp, vp, vp, vp]
    lib.ibp_decompress_gather_packed.argtypes = [vp, u64, vp, i64, i64, i32, u32, vp, vp, vp, i64,
                                                 vp, vp, vp]
    for name in SYMBOLS[1:]:
        getattr(lib, name).restype = i32
    lib.ibp_testing_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.ibp_testing_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.ibp_testing_withhold_plans.argtypes = [ctypes.c_int]
    lib.ibp_testing_withhold_plans.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().ibp_status_string(int(code)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(rc: int, call: str) -> None:
    if rc != OK:
        raise IBPError(rc, call)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dtype_code(t: torch.Tensor, dtype: int | None = None) -> int:
    if dtype is not None:
        return int(dtype)
    if t.dtype not in _TORCH_DTYPES:
        raise ValueError(f"pass dtype= for element tensors of {t.dtype}")
    return _TORCH_DTYPES[t.dtype]


def slot_bytes(row_elems: int, dtype: int) -> int:
    out = ctypes.c_int64(0)
    _check(load().ibp_slot_bytes(int(row_elems), int(dtype), ctypes.byref(out)), "ibp_slot_bytes")
    return out.value


def meta_scratch_bytes() -> int:
    out = ctypes.c_size_t(0)
    _check(load().ibp_meta_scratch_bytes(ctypes.byref(out)), "ibp_meta_scratch_bytes")
    return out.value


def _rows_shape(rows: torch.Tensor) -> tuple[int, int]:
    if rows.dim() != 2 or not rows.is_contiguous():
        raise ValueError("rows must be a contiguous 2-D tensor [n_rows, row_elems]")
    return rows.shape[0], rows.shape[1]


def build_meta(rows: torch.Tensor, T: float, block_elems: int, meta: torch.Tensor,
               scratch: torch.Tensor, dtype: int | None = None, stream=None) -> None:
    """ibp_build_meta: mask/bitval of ``rows`` into ``meta`` (16 device bytes)."""
    n, L = _rows_shape(rows)
    _check(load().ibp_build_meta(_ptr(rows), n, L, dtype_code(rows, dtype), float(T),
                                 int(block_elems), _ptr(meta), _ptr(scratch), _stream(stream)),
           "ibp_build_meta")


def meta_count(rows: torch.Tensor, counters: torch.Tensor, dtype: int | None = None,
               stream=None) -> None:
    """ibp_meta_count: per-bit 1-counts of ``rows`` into ``counters`` (32 x int64 on
    the device, overwritten); counters of several row sets add up."""
    n, L = _rows_shape(rows)
    _check(load().ibp_meta_count(_ptr(rows), n, L, dtype_code(rows, dtype), _ptr(counters),
                                 _stream(stream)), "ibp_meta_count")


def meta_finalize(counters: torch.Tensor, n_elems: int, dtype: int, T: float, block_elems: int,
                  meta: torch.Tensor, status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_meta_finalize: the threshold rule applied to (summed) ``counters``; counters
    larger than ``n_elems`` give invalid metadata and ERR_META in ``status``."""
    _check(load().ibp_meta_finalize(_ptr(counters), int(n_elems), int(dtype), float(T),
                                    int(block_elems), _ptr(meta), _ptr(status),
                                    _stream(stream)),
           "ibp_meta_finalize")


def build_meta_noalloc(rows: torch.Tensor, T: float, block_elems: int, meta: torch.Tensor,
                       dtype: int | None = None, stream=None) -> None:
    """ibp_build_meta_noalloc: as build_meta, with the library's built-in counter
    array instead of caller scratch (for callers that cannot allocate)."""
    n, L = _rows_shape(rows)
    _check(load().ibp_build_meta_noalloc(_ptr(rows), n, L, dtype_code(rows, dtype), float(T),
                                         int(block_elems), _ptr(meta), _stream(stream)),
           "ibp_build_meta_noalloc")


def meta_select_scratch_bytes() -> int:
    out = ctypes.c_size_t(0)
    _check(load().ibp_meta_select_scratch_bytes(ctypes.byref(out)),
           "ibp_meta_select_scratch_bytes")
    return out.value


def build_meta_select(rows: torch.Tensor, T: float, block_elems: int, meta: torch.Tensor,
                      scratch: torch.Tensor, candidates: torch.Tensor | None = None,
                      dtype: int | None = None, stream=None) -> None:
    """ibp_build_meta_select: the saving-aware mask (the cheapest of the threshold
    mask and its nested reductions) into ``meta``; ``candidates`` (optional,
    MAX_MASK_CANDIDATES x 16 device bytes) receives every candidate and its score."""
    n, L = _rows_shape(rows)
    _check(load().ibp_build_meta_select(_ptr(rows), n, L, dtype_code(rows, dtype), float(T),
                                        int(block_elems), _ptr(meta), _ptr(candidates),
                                        _ptr(scratch), _stream(stream)), "ibp_build_meta_select")


def read_candidates(candidates: torch.Tensor) -> list[tuple[int, int, int]]:
    """(mask, bitval, stored_bytes) of every used entry of a candidate table."""
    raw = candidates.detach().to("cpu").contiguous().view(torch.uint8).numpy().tobytes()
    out = []
    for k in range(MAX_MASK_CANDIDATES):
        mask, bitval, stored = struct.unpack_from("<IIq", raw, 16 * k)
        if stored >= 0:
            out.append((mask, bitval, stored))
    return out


def compress(rows: torch.Tensor, block_elems: int, meta: torch.Tensor, slots: torch.Tensor,
             bitmask: torch.Tensor, row_bits: torch.Tensor | None = None,
             status: torch.Tensor | None = None, dtype: int | None = None,
             stream=None) -> None:
    """ibp_compress: encode ``rows`` into ``slots`` ([n_rows, slot_bytes] bytes)."""
    n, L = _rows_shape(rows)
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(n, 1)
    _check(load().ibp_compress(_ptr(rows), n, L, dtype_code(rows, dtype), int(block_elems),
                               _ptr(meta), _ptr(slots), sb, _ptr(bitmask), _ptr(row_bits),
                               _ptr(status), _stream(stream)), "ibp_compress")


def decompress_gather(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
                      block_elems: int, bitmask: torch.Tensor, meta: torch.Tensor,
                      idx: torch.Tensor, out: torch.Tensor, status: torch.Tensor | None = None,
                      stream=None) -> None:
    """ibp_decompress_gather: rows ``idx`` rebuilt into ``out`` [n_idx, row_elems]."""
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    _check(load().ibp_decompress_gather(_ptr(slots), sb, int(n_rows), int(row_elems), int(dtype),
                                        int(block_elems), _ptr(bitmask), _ptr(meta), _ptr(idx),
                                        idx.numel(), _ptr(out), _ptr(status), _stream(stream)),
           "ibp_decompress_gather")


def gather_dedup_scratch_bytes(n_idx: int, row_elems: int, dtype: int, block_elems: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().ibp_gather_dedup_scratch_bytes(int(n_idx), int(row_elems), int(dtype),
                                                 int(block_elems), ctypes.byref(out)),
           "ibp_gather_dedup_scratch_bytes")
    return out.value


def decompress_gather_dedup(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
                            block_elems: int, bitmask: torch.Tensor, meta: torch.Tensor,
                            idx: torch.Tensor, out: torch.Tensor, scratch: torch.Tensor,
                            status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_decompress_gather_dedup: the result of decompress_gather, each distinct
    row read and decoded once (``scratch``: gather_dedup_scratch_bytes bytes)."""
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    _check(load().ibp_decompress_gather_dedup(
        _ptr(slots), sb, int(n_rows), int(row_elems), int(dtype), int(block_elems), _ptr(bitmask),
        _ptr(meta), _ptr(idx), idx.numel(), _ptr(out), _ptr(scratch),
        scratch.numel() * scratch.element_size(), _ptr(status), _stream(stream)),
        "ibp_decompress_gather_dedup")


def pack_scratch_bytes(n_sel: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().ibp_pack_scratch_bytes(int(n_sel), ctypes.byref(out)), "ibp_pack_scratch_bytes")
    return out.value


def pack_offsets(bitmask: torch.Tensor, row_bits: torch.Tensor, n_rows: int, row_elems: int,
                 dtype: int, offsets: torch.Tensor, scratch: torch.Tensor,
                 sel: torch.Tensor | None = None, n_sel: int | None = None,
                 status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_pack_offsets: entry offsets ([n_sel + 1] int64 on the device) of a packed
    store of rows ``sel`` (all rows when None)."""
    if sel is not None and sel.dtype != torch.int64:
        raise ValueError("sel must be int64")
    ns = int(n_sel) if n_sel is not None else (sel.numel() if sel is not None else int(n_rows))
    _check(load().ibp_pack_offsets(_ptr(bitmask), _ptr(row_bits), int(n_rows), int(row_elems),
                                   int(dtype), _ptr(sel), ns, _ptr(offsets), _ptr(scratch),
                                   _ptr(status), _stream(stream)), "ibp_pack_offsets")


def pack(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int, bitmask: torch.Tensor,
         row_bits: torch.Tensor, offsets: torch.Tensor, packed: torch.Tensor,
         pack_bitmask: torch.Tensor, pack_row_bits: torch.Tensor | None = None,
         sel: torch.Tensor | None = None, n_sel: int | None = None,
         status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_pack: copy the entries of a packed store into ``packed``."""
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    ns = int(n_sel) if n_sel is not None else (sel.numel() if sel is not None else int(n_rows))
    _check(load().ibp_pack(_ptr(slots), sb, int(n_rows), int(row_elems), int(dtype),
                           _ptr(bitmask), _ptr(row_bits), _ptr(sel), ns, _ptr(offsets),
                           _ptr(packed), packed.numel() * packed.element_size(),
                           _ptr(pack_bitmask), _ptr(pack_row_bits), _ptr(status),
                           _stream(stream)), "ibp_pack")


def decompress_gather_packed(packed: torch.Tensor, offsets: torch.Tensor, n_rows: int,
                             row_elems: int, dtype: int, block_elems: int, bitmask: torch.Tensor,
                             meta: torch.Tensor, idx: torch.Tensor, out: torch.Tensor,
                             status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_decompress_gather_packed: rows ``idx`` of a packed store into ``out``."""
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    _check(load().ibp_decompress_gather_packed(
        _ptr(packed), packed.numel() * packed.element_size(), _ptr(offsets), int(n_rows),
        int(row_elems), int(dtype), int(block_elems), _ptr(bitmask), _ptr(meta), _ptr(idx),
        idx.numel(), _ptr(out), _ptr(status), _stream(stream)), "ibp_decompress_gather_packed")


def meta_positions_scratch_bytes(row_elems: int, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().ibp_meta_positions_scratch_bytes(int(row_elems), int(dtype), ctypes.byref(out)),
           "ibp_meta_positions_scratch_bytes")
    return out.value


def build_meta_block_positions(rows: torch.Tensor, T: float, block_elems: int,
                               pmask: torch.Tensor, pbitval: torch.Tensor, scratch: torch.Tensor,
                               dtype: int | None = None, stream=None) -> None:
    """ibp_build_meta_block_positions: one mask/bitval per position within a block,
    written row-sized (entry e holds the pair of position e % block_elems)."""
    n, L = _rows_shape(rows)
    _check(load().ibp_build_meta_block_positions(_ptr(rows), n, L, dtype_code(rows, dtype),
                                                 float(T), int(block_elems), _ptr(pmask),
                                                 _ptr(pbitval), _ptr(scratch), _stream(stream)),
           "ibp_build_meta_block_positions")


def build_meta_positions(rows: torch.Tensor, T: float, block_elems: int, pmask: torch.Tensor,
                         pbitval: torch.Tensor, scratch: torch.Tensor, dtype: int | None = None,
                         stream=None) -> None:
    """ibp_build_meta_positions: one mask/bitval per element position of a row."""
    n, L = _rows_shape(rows)
    _check(load().ibp_build_meta_positions(_ptr(rows), n, L, dtype_code(rows, dtype), float(T),
                                           int(block_elems), _ptr(pmask), _ptr(pbitval),
                                           _ptr(scratch), _stream(stream)),
           "ibp_build_meta_positions")


def compress_positions(rows: torch.Tensor, block_elems: int, pmask: torch.Tensor,
                       pbitval: torch.Tensor, slots: torch.Tensor, bitmask: torch.Tensor,
                       row_bits: torch.Tensor | None = None, dtype: int | None = None,
                       stream=None) -> None:
    """ibp_compress_positions: encode ``rows`` with per-position metadata."""
    n, L = _rows_shape(rows)
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(n, 1)
    _check(load().ibp_compress_positions(_ptr(rows), n, L, dtype_code(rows, dtype),
                                         int(block_elems), _ptr(pmask), _ptr(pbitval),
                                         _ptr(slots), sb, _ptr(bitmask), _ptr(row_bits),
                                         _stream(stream)), "ibp_compress_positions")


def decompress_gather_positions(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
                                block_elems: int, bitmask: torch.Tensor, pmask: torch.Tensor,
                                pbitval: torch.Tensor, idx: torch.Tensor, out: torch.Tensor,
                                status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_decompress_gather_positions: rows ``idx`` rebuilt with per-position metadata."""
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    _check(load().ibp_decompress_gather_positions(
        _ptr(slots), sb, int(n_rows), int(row_elems), int(dtype), int(block_elems),
        _ptr(bitmask), _ptr(pmask), _ptr(pbitval), _ptr(idx), idx.numel(), _ptr(out),
        _ptr(status), _stream(stream)), "ibp_decompress_gather_positions")


def decompress_gather_sized(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
                            block_elems: int, bitmask: torch.Tensor, row_bits: torch.Tensor,
                            meta: torch.Tensor, idx: torch.Tensor, out: torch.Tensor,
                            status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_decompress_gather_sized: as decompress_gather, staging only each row's
    stored bytes (known from ``row_bits``)."""
    if idx.dtype != torch.int64:
        raise ValueError("idx must be int64")
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    _check(load().ibp_decompress_gather_sized(
        _ptr(slots), sb, int(n_rows), int(row_elems), int(dtype), int(block_elems),
        _ptr(bitmask), _ptr(row_bits), _ptr(meta), _ptr(idx), idx.numel(), _ptr(out),
        _ptr(status), _stream(stream)), "ibp_decompress_gather_sized")


def decompress_gather_batched(jobs, row_elems: int, dtype: int, block_elems: int,
                              status: torch.Tensor | None = None, stream=None) -> None:
    """ibp_decompress_gather_batched: ``jobs`` is a list of (slots, n_rows, bitmask, meta,
    idx, out) tuples sharing one row geometry; one launch per 64 jobs."""
    arr = (GatherJob * max(len(jobs), 1))()
    for k, (slots, n_rows, bitmask, meta, idx, out) in enumerate(jobs):
        if idx.dtype != torch.int64:
            raise ValueError("idx must be int64")
        sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
            slots.element_size() // max(int(n_rows), 1)
        arr[k] = GatherJob(slots.data_ptr(), sb, int(n_rows), bitmask.data_ptr(), meta.data_ptr(),
                           idx.data_ptr(), idx.numel(), out.data_ptr())
    _check(load().ibp_decompress_gather_batched(ctypes.cast(arr, ctypes.c_void_p), len(jobs),
                                                int(row_elems), int(dtype), int(block_elems),
                                                _ptr(status), _stream(stream)),
           "ibp_decompress_gather_batched")


def decompress_range(slots: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
                     block_elems: int, bitmask: torch.Tensor, meta: torch.Tensor, row_begin: int,
                     n_out: int, out: torch.Tensor, status: torch.Tensor | None = None,
                     stream=None) -> None:
    """ibp_decompress_range: rows row_begin .. row_begin + n_out - 1 into ``out``."""
    sb = slots.shape[1] * slots.element_size() if slots.dim() == 2 else slots.numel() * \
        slots.element_size() // max(int(n_rows), 1)
    _check(load().ibp_decompress_range(_ptr(slots), sb, int(n_rows), int(row_elems), int(dtype),
                                       int(block_elems), _ptr(bitmask), _ptr(meta),
                                       int(row_begin), int(n_out), _ptr(out), _ptr(status),
                                       _stream(stream)), "ibp_decompress_range")


def query(bitmask: torch.Tensor, row_bits: torch.Tensor, n_rows: int, row_elems: int, dtype: int,
          stream=None) -> Stats:
    """ibp_query: store statistics, returned in host memory (synchronises the stream)."""
    out = Stats()
    _check(load().ibp_query(_ptr(bitmask), _ptr(row_bits), int(n_rows), int(row_elems),
                            int(dtype), ctypes.byref(out), _stream(stream)), "ibp_query")
    return out


def query_async(bitmask: torch.Tensor, row_bits: torch.Tensor, n_rows: int, row_elems: int,
                dtype: int, stats: torch.Tensor, stream=None) -> None:
    """ibp_query_async: store statistics into ``stats`` (40 device bytes, see Stats),
    asynchronously."""
    _check(load().ibp_query_async(_ptr(bitmask), _ptr(row_bits), int(n_rows), int(row_elems),
                                  int(dtype), _ptr(stats), _stream(stream)), "ibp_query_async")


def read_stats(stats: torch.Tensor) -> Stats:
    host = stats.detach().to("cpu").contiguous().view(torch.uint8).numpy().tobytes()
    return Stats.from_buffer_copy(host[:ctypes.sizeof(Stats)])


def probe_read(src: torch.Tensor, sink: torch.Tensor, nbytes: int | None = None,
               stream=None) -> None:
    """ibp_probe_read: stream ``nbytes`` of ``src`` through the GPU (bandwidth probe)."""
    n = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    _check(load().ibp_probe_read(_ptr(src), n, _ptr(sink), _stream(stream)), "ibp_probe_read")


def testing_set_wait_limit_ns(ns: int) -> int:
    """ibp_testing_set_wait_limit_ns (include/ibp_testing.h): the limit of the gather
    kernels' bounded waits, in ns (0: the default 2 s); returns the previous one."""
    return int(load().ibp_testing_set_wait_limit_ns(int(ns)))


def testing_withhold_plans(on: bool) -> bool:
    """ibp_testing_withhold_plans (include/ibp_testing.h): the warp-specialised
    gather's planners keep their plans from the decoders; returns the previous setting."""
    return bool(load().ibp_testing_withhold_plans(1 if on else 0))
