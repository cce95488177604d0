"""Python loader for the plain C++ IBP oracle (``ibp_oracle.cpp``).

TEST INFRASTRUCTURE ONLY. The test suite, the smoke check in ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` may import this module; the GPU codec
package never does, and this module imports nothing from it.

The oracle is a slow, single-threaded, bit-by-bit restatement of Invariant Bit
Packing as described in "Reducing the GPU Memory Bottleneck with Lossless
Compression for ML -- Extended", technical summary, "Core algorithm". The wrapper
below only marshals numpy arrays into the C entry points.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ibp_oracle.cpp")
_HDR = os.path.join(_HERE, "ibp_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libibp_oracle.so")

OK = 0
BAD_ARG = -1
BAD_INDEX = -5
CORRUPT = -6

_default = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libibp_oracle.so`` (plain g++, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """ctypes view of one compiled copy of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, i32, u32, dbl, vp = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_double,
                                  ctypes.c_void_p)
        lib.ibpo_build_meta.argtypes = [vp, i64, i32, dbl, ctypes.POINTER(u32),
                                        ctypes.POINTER(u32)]
        lib.ibpo_build_meta.restype = i32
        lib.ibpo_slot_bytes.argtypes = [i64, i32]
        lib.ibpo_slot_bytes.restype = i64
        lib.ibpo_compress.argtypes = [vp, i64, i64, i32, i64, u32, u32, vp, i64, vp, vp]
        lib.ibpo_compress.restype = i32
        lib.ibpo_decompress_gather.argtypes = [vp, i64, i64, i64, i32, i64, vp, u32, u32, vp,
                                               i64, vp]
        lib.ibpo_decompress_gather.restype = i32
        lib.ibpo_select_meta.argtypes = [vp, i64, i64, i32, dbl, i64, ctypes.POINTER(u32),
                                         ctypes.POINTER(u32), vp, vp, ctypes.POINTER(i32)]
        lib.ibpo_select_meta.restype = i32
        lib.ibpo_build_meta_positions.argtypes = [vp, i64, i64, i32, dbl, vp, vp]
        lib.ibpo_build_meta_block_positions.argtypes = [vp, i64, i64, i32, dbl, i64, vp, vp]
        lib.ibpo_build_meta_block_positions.restype = ctypes.c_int
        lib.ibpo_build_meta_positions.restype = i32
        lib.ibpo_compress_positions.argtypes = [vp, i64, i64, i32, i64, vp, vp, vp, i64, vp, vp]
        lib.ibpo_compress_positions.restype = i32
        lib.ibpo_decompress_gather_positions.argtypes = [vp, i64, i64, i64, i32, i64, vp, vp, vp,
                                                         vp, i64, vp]
        lib.ibpo_decompress_gather_positions.restype = i32
        lib.ibpo_pack.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, i64, vp, vp, vp, vp]
        lib.ibpo_pack.restype = i32
        lib.ibpo_decompress_gather_packed.argtypes = [vp, vp, i64, i64, i32, i64, vp, u32, u32,
                                                      vp, i64, vp]
        lib.ibpo_decompress_gather_packed.restype = i32
        self.lib = lib
        self.path = path

    def slot_bytes(self, row_elems: int, w_bits: int) -> int:
        return int(self.lib.ibpo_slot_bytes(row_elems, w_bits))

    def build_meta(self, elems: np.ndarray, T: float) -> tuple[int, int]:
        """Return (mask, bitval) over every element of ``elems`` (any shape)."""
        a = np.ascontiguousarray(elems)
        w = _width(a)
        mask, bitval = ctypes.c_uint32(0), ctypes.c_uint32(0)
        rc = self.lib.ibpo_build_meta(_ptr(a), a.size, w, float(T), ctypes.byref(mask),
                                      ctypes.byref(bitval))
        if rc != OK:
            raise ValueError(f"oracle build_meta rejected its arguments ({rc})")
        return mask.value, bitval.value

    def build_meta_positions(self, rows: np.ndarray, T: float):
        """Per-position (mask, bitval) arrays, one entry per element position."""
        a = np.ascontiguousarray(rows)
        if a.ndim != 2:
            raise ValueError("rows must be 2-D")
        w = _width(a)
        n, L = a.shape
        pm = np.zeros(L, dtype=np.uint32)
        pb = np.zeros(L, dtype=np.uint32)
        rc = self.lib.ibpo_build_meta_positions(_ptr(a), n, L, w, float(T), _ptr(pm), _ptr(pb))
        if rc != OK:
            raise ValueError(f"oracle build_meta_positions rejected its arguments ({rc})")
        return pm, pb

    def build_meta_block_positions(self, rows: np.ndarray, T: float, block_elems: int):
        """Block-position (mask, bitval) arrays, written one entry per element
        position (entry e holds the pair of block position e % block_elems)."""
        a = np.ascontiguousarray(rows)
        if a.ndim != 2:
            raise ValueError("rows must be 2-D")
        w = _width(a)
        n, L = a.shape
        pm = np.zeros(L, dtype=np.uint32)
        pb = np.zeros(L, dtype=np.uint32)
        rc = self.lib.ibpo_build_meta_block_positions(_ptr(a), n, L, w, float(T),
                                                      int(block_elems), _ptr(pm), _ptr(pb))
        if rc != OK:
            raise ValueError(f"oracle build_meta_block_positions rejected its arguments ({rc})")
        return pm, pb

    def compress_positions(self, rows: np.ndarray, block_elems: int, pmask: np.ndarray,
                           pbitval: np.ndarray, slot_bytes_: int | None = None):
        a = np.ascontiguousarray(rows)
        w = _width(a)
        n, L = a.shape
        pm = np.ascontiguousarray(pmask, dtype=np.uint32)
        pb = np.ascontiguousarray(pbitval, dtype=np.uint32)
        if pm.size != L or pb.size != L:
            raise ValueError("one mask and bitval per element position")
        sb = self.slot_bytes(L, w) if slot_bytes_ is None else int(slot_bytes_)
        slots = np.zeros((n, sb), dtype=np.uint8)
        bitmask = np.zeros(((n + 31) // 32,), dtype=np.uint32)
        row_bits = np.zeros((n,), dtype=np.uint32)
        rc = self.lib.ibpo_compress_positions(_ptr(a), n, L, w, int(block_elems), _ptr(pm),
                                              _ptr(pb), _ptr(slots), sb, _ptr(bitmask),
                                              _ptr(row_bits))
        if rc != OK:
            raise ValueError(f"oracle compress_positions rejected its arguments ({rc})")
        return slots, bitmask, row_bits

    def decompress_gather_positions(self, slots, n_rows, row_elems, dtype, block_elems, bitmask,
                                    pmask, pbitval, idx, out=None):
        dt = np.dtype(dtype)
        w = 8 * dt.itemsize
        s = np.ascontiguousarray(slots)
        ix = np.ascontiguousarray(idx, dtype=np.int64)
        bm = np.ascontiguousarray(bitmask, dtype=np.uint32)
        pm = np.ascontiguousarray(pmask, dtype=np.uint32)
        pb = np.ascontiguousarray(pbitval, dtype=np.uint32)
        if out is None:
            out = np.zeros((ix.size, row_elems), dtype=dt)
        rc = self.lib.ibpo_decompress_gather_positions(_ptr(s), s.shape[1], n_rows, row_elems, w,
                                                       int(block_elems), _ptr(bm), _ptr(pm),
                                                       _ptr(pb), _ptr(ix), ix.size, _ptr(out))
        if rc == BAD_ARG:
            raise ValueError("oracle decompress_gather_positions rejected its arguments")
        return out, rc

    def pack(self, slots: np.ndarray, row_elems: int, dtype, bitmask: np.ndarray,
             row_bits: np.ndarray, sel: np.ndarray | None = None):
        """Packed store of rows ``sel`` (all rows if None) of a 2-D slotted store.
        Returns (offsets i64[n_sel+1], packed u8[total], bitmask u32, row_bits u32)."""
        s = np.ascontiguousarray(slots)
        n = s.shape[0]
        w = 8 * np.dtype(dtype).itemsize
        bm = np.ascontiguousarray(bitmask, dtype=np.uint32)
        rb = np.ascontiguousarray(row_bits, dtype=np.uint32)
        sl = None if sel is None else np.ascontiguousarray(sel, dtype=np.int64)
        n_sel = n if sl is None else sl.size
        offsets = np.zeros(n_sel + 1, dtype=np.int64)
        rc = self.lib.ibpo_pack(_ptr(s), s.shape[1], n, row_elems, w, _ptr(bm), _ptr(rb), _ptr(sl),
                                n_sel, _ptr(offsets), None, None, None)
        if rc != OK:
            raise ValueError(f"oracle pack rejected its arguments ({rc})")
        packed = np.zeros(int(offsets[-1]), dtype=np.uint8)
        pbm = np.zeros((n_sel + 31) // 32, dtype=np.uint32)
        prb = np.zeros(n_sel, dtype=np.uint32)
        rc = self.lib.ibpo_pack(_ptr(s), s.shape[1], n, row_elems, w, _ptr(bm), _ptr(rb), _ptr(sl),
                                n_sel, _ptr(offsets), _ptr(packed), _ptr(pbm), _ptr(prb))
        if rc != OK:
            raise ValueError(f"oracle pack rejected its arguments ({rc})")
        return offsets, packed, pbm, prb

    def decompress_gather_packed(self, packed: np.ndarray, offsets: np.ndarray, row_elems: int,
                                 dtype, block_elems: int, bitmask: np.ndarray, mask: int,
                                 bitval: int, idx: np.ndarray, out: np.ndarray | None = None):
        """Rebuild rows ``idx`` of a packed store. Returns (out, status)."""
        dt = np.dtype(dtype)
        w = 8 * dt.itemsize
        p = np.ascontiguousarray(packed, dtype=np.uint8)
        off = np.ascontiguousarray(offsets, dtype=np.int64)
        ix = np.ascontiguousarray(idx, dtype=np.int64)
        bm = np.ascontiguousarray(bitmask, dtype=np.uint32)
        if out is None:
            out = np.zeros((ix.size, row_elems), dtype=dt)
        rc = self.lib.ibpo_decompress_gather_packed(_ptr(p), _ptr(off), off.size - 1, row_elems, w,
                                                    int(block_elems), _ptr(bm), int(mask),
                                                    int(bitval), _ptr(ix), ix.size, _ptr(out))
        if rc == BAD_ARG:
            raise ValueError("oracle decompress_gather_packed rejected its arguments")
        return out, rc

    def select_meta(self, rows: np.ndarray, T: float, block_elems: int):
        """Saving-aware mask choice over a 2-D array of rows.
        Returns (mask, bitval, [(candidate mask, stored bytes), ...])."""
        a = np.ascontiguousarray(rows)
        if a.ndim != 2:
            raise ValueError("rows must be 2-D")
        w = _width(a)
        n, L = a.shape
        mask, bitval, nc = ctypes.c_uint32(0), ctypes.c_uint32(0), ctypes.c_int(0)
        cm = np.zeros(33, dtype=np.uint32)
        cb = np.zeros(33, dtype=np.int64)
        rc = self.lib.ibpo_select_meta(_ptr(a), n, L, w, float(T), int(block_elems),
                                       ctypes.byref(mask), ctypes.byref(bitval), _ptr(cm),
                                       _ptr(cb), ctypes.byref(nc))
        if rc != OK:
            raise ValueError(f"oracle select_meta rejected its arguments ({rc})")
        cands = [(int(cm[k]), int(cb[k])) for k in range(nc.value)]
        return mask.value, bitval.value, cands

    def compress(self, rows: np.ndarray, block_elems: int, mask: int, bitval: int,
                 slot_bytes_: int | None = None):
        """Compress a 2-D array of rows.
        Returns (slots u8[n, slot_bytes], bitmask u32[ceil(n/32)], row_bits u32[n])."""
        a = np.ascontiguousarray(rows)
        if a.ndim != 2:
            raise ValueError("rows must be 2-D")
        w = _width(a)
        n, L = a.shape
        sb = self.slot_bytes(L, w) if slot_bytes_ is None else int(slot_bytes_)
        slots = np.zeros((n, sb), dtype=np.uint8)
        bitmask = np.zeros(((n + 31) // 32,), dtype=np.uint32)
        row_bits = np.zeros((n,), dtype=np.uint32)
        rc = self.lib.ibpo_compress(_ptr(a), n, L, w, int(block_elems), int(mask), int(bitval),
                                    _ptr(slots), sb, _ptr(bitmask), _ptr(row_bits))
        if rc != OK:
            raise ValueError(f"oracle compress rejected its arguments ({rc})")
        return slots, bitmask, row_bits

    def decompress_gather(self, slots: np.ndarray, n_rows: int, row_elems: int, dtype,
                          block_elems: int, bitmask: np.ndarray, mask: int, bitval: int,
                          idx: np.ndarray, out: np.ndarray | None = None):
        """Rebuild rows ``idx`` from 2-D ``slots``. Returns (out[n_idx, row_elems], status)."""
        dt = np.dtype(dtype)
        w = 8 * dt.itemsize
        s = np.ascontiguousarray(slots)
        ix = np.ascontiguousarray(idx, dtype=np.int64)
        bm = np.ascontiguousarray(bitmask, dtype=np.uint32)
        if out is None:
            out = np.zeros((ix.size, row_elems), dtype=dt)
        rc = self.lib.ibpo_decompress_gather(_ptr(s), s.shape[1], n_rows, row_elems, w,
                                             int(block_elems), _ptr(bm), int(mask), int(bitval),
                                             _ptr(ix), ix.size, _ptr(out))
        if rc == BAD_ARG:
            raise ValueError("oracle decompress_gather rejected its arguments")
        return out, rc


def _width(a: np.ndarray) -> int:
    if a.dtype.itemsize not in (1, 2, 4):
        raise ValueError("elements must be 8-, 16- or 32-bit words")
    return 8 * a.dtype.itemsize


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def compile_variant(source_text: str, workdir: str) -> Oracle:
    """Compile an edited copy of the oracle source (used by tests that plant a
    mistake in the oracle to show that its pins catch it)."""
    os.makedirs(workdir, exist_ok=True)
    src = os.path.join(workdir, "ibp_oracle_variant.cpp")
    with open(os.path.join(workdir, "ibp_oracle.h"), "w") as f:
        f.write(open(_HDR).read())
    with open(src, "w") as f:
        f.write(source_text)
    lib = os.path.join(workdir, "libibp_oracle_variant.so")
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", lib, src])
    return Oracle(lib)


def source_text() -> str:
    return open(_SRC).read()


def slot_bytes(row_elems: int, w_bits: int) -> int:
    return default().slot_bytes(row_elems, w_bits)


def build_meta(elems: np.ndarray, T: float) -> tuple[int, int]:
    return default().build_meta(elems, T)


def build_meta_positions(rows, T):
    return default().build_meta_positions(rows, T)


def build_meta_block_positions(rows, T, block_elems):
    return default().build_meta_block_positions(rows, T, block_elems)


def compress_positions(rows, block_elems, pmask, pbitval, slot_bytes_=None):
    return default().compress_positions(rows, block_elems, pmask, pbitval, slot_bytes_)


def decompress_gather_positions(slots, n_rows, row_elems, dtype, block_elems, bitmask, pmask,
                                pbitval, idx, out=None):
    return default().decompress_gather_positions(slots, n_rows, row_elems, dtype, block_elems,
                                                 bitmask, pmask, pbitval, idx, out)


def pack(slots, row_elems, dtype, bitmask, row_bits, sel=None):
    return default().pack(slots, row_elems, dtype, bitmask, row_bits, sel)


def decompress_gather_packed(packed, offsets, row_elems, dtype, block_elems, bitmask, mask,
                             bitval, idx, out=None):
    return default().decompress_gather_packed(packed, offsets, row_elems, dtype, block_elems,
                                              bitmask, mask, bitval, idx, out)


def select_meta(rows: np.ndarray, T: float, block_elems: int):
    return default().select_meta(rows, T, block_elems)


def compress(rows: np.ndarray, block_elems: int, mask: int, bitval: int,
             slot_bytes_: int | None = None):
    return default().compress(rows, block_elems, mask, bitval, slot_bytes_)


def decompress_gather(slots, n_rows, row_elems, dtype, block_elems, bitmask, mask, bitval, idx,
                      out=None):
    return default().decompress_gather(slots, n_rows, row_elems, dtype, block_elems, bitmask,
                                       mask, bitval, idx, out)


def stored_bytes(row_bits: np.ndarray, bitmask: np.ndarray, raw_bytes: int) -> np.ndarray:
    """Bytes each row occupies in its slot: 4*ceil(bits/32) if compressed, else raw."""
    n = row_bits.size
    flags = (bitmask[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1
    words = (row_bits.astype(np.int64) + 31) // 32
    return np.where(flags == 1, 4 * words, raw_bytes)
