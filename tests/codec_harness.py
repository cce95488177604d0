"""Shared harness of the GPU parity tests: runs the CUDA codec and the oracle on
the same seeded words and compares their outputs."""
from __future__ import annotations

import numpy as np
import torch

import lossless_bit_level_gb300 as ibp
import oracle

INT_VIEW = {np.dtype(np.uint32): (np.int32, torch.int32), np.dtype(np.uint16): (np.int16, torch.int16),
            np.dtype(np.uint8): (np.uint8, torch.uint8)}


def words_of(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.float32:
        return x.view(np.uint32)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    assert x.dtype in (np.uint32, np.uint16, np.uint8), x.dtype
    return x


def to_torch(words: np.ndarray, where: str) -> torch.Tensor:
    npv, _ = INT_VIEW[words.dtype]
    t = torch.from_numpy(np.ascontiguousarray(words).view(npv))
    if where == "device":
        return t.to("cuda")
    if where == "host":
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h
    raise ValueError(where)


def from_torch(t: torch.Tensor, dtype) -> np.ndarray:
    return t.cpu().numpy().view(dtype)


def meta_tensor(mask: int, bitval: int, dtype_code: int, B: int) -> torch.Tensor:
    return torch.tensor(np.array([mask, bitval, dtype_code, B], dtype=np.uint32).view(np.int32),
                        device="cuda")


def meta_values(meta: torch.Tensor) -> tuple[int, int, int, int]:
    v = meta.cpu().numpy().view(np.uint32)
    return int(v[0]), int(v[1]), int(v[2]), int(v[3])


class GpuStore:
    """Slots + bitmask + per-row bits of one compressed table on the GPU side."""

    def __init__(self, n_rows: int, row_elems: int, dtype_code: int, B: int, where: str,
                 slot_bytes: int | None = None):
        self.n_rows, self.row_elems, self.dtype, self.B, self.where = (
            n_rows, row_elems, dtype_code, B, where)
        self.slot_bytes = slot_bytes or ibp.slot_bytes(row_elems, dtype_code)
        shape = (n_rows, self.slot_bytes)
        if where == "device":
            self.slots = torch.zeros(shape, dtype=torch.uint8, device="cuda")
        else:
            self.slots = torch.zeros(shape, dtype=torch.uint8, pin_memory=True)
        self.bitmask = torch.zeros(((n_rows + 31) // 32,), dtype=torch.int32, device="cuda")
        self.row_bits = torch.zeros((max(n_rows, 1),), dtype=torch.int32, device="cuda")
        self.status = torch.zeros((1,), dtype=torch.int32, device="cuda")


def gpu_meta(words_t: torch.Tensor, dtype_code: int, T: float, B: int) -> torch.Tensor:
    meta = torch.zeros((4,), dtype=torch.int32, device="cuda")
    scratch = torch.empty((ibp.meta_scratch_bytes() // 4,), dtype=torch.int32, device="cuda")
    ibp.build_meta(words_t, T, B, meta, scratch, dtype=dtype_code)
    return meta


def gpu_compress(words_t: torch.Tensor, meta: torch.Tensor, store: GpuStore) -> None:
    ibp.compress(words_t, store.B, meta, store.slots, store.bitmask, store.row_bits, store.status,
                 dtype=store.dtype)


def gpu_gather(store: GpuStore, meta: torch.Tensor, idx: np.ndarray,
               out: torch.Tensor | None = None) -> tuple[torch.Tensor, int]:
    idx_t = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int64)).to("cuda")
    wdt = {32: torch.int32, 16: torch.int16, 8: torch.uint8}[ibp.WIDTH[store.dtype]]
    if out is None:
        out = torch.zeros((idx.size, store.row_elems), dtype=wdt, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ibp.decompress_gather(store.slots, store.n_rows, store.row_elems, store.dtype, store.B,
                          store.bitmask, meta, idx_t, out, status)
    torch.cuda.synchronize()
    return out, int(status.item())


def bitmask_np(store: GpuStore) -> np.ndarray:
    return store.bitmask.cpu().numpy().view(np.uint32)


def row_bits_np(store: GpuStore) -> np.ndarray:
    return store.row_bits.cpu().numpy().view(np.uint32)[: store.n_rows]


def slots_np(store: GpuStore) -> np.ndarray:
    return store.slots.cpu().numpy()


def compare_slots(gpu_slots: np.ndarray, ora_slots: np.ndarray, bitmask: np.ndarray,
                  row_bits: np.ndarray, raw_bytes: int, rows: np.ndarray | None = None) -> None:
    """Compressed rows: first 4*ceil(bits/32) bytes equal; raw rows: raw bytes equal."""
    n = row_bits.size
    r = np.arange(n)
    flags = (bitmask[r // 32] >> (r % 32).astype(np.uint32)) & 1
    used = np.where(flags == 1, 4 * ((row_bits.astype(np.int64) + 31) // 32), raw_bytes)
    col = np.arange(gpu_slots.shape[1])[None, :]
    valid = col < used[:, None]
    diff = (gpu_slots != ora_slots) & valid
    if diff.any():
        bad = np.nonzero(diff.any(axis=1))[0]
        raise AssertionError(f"{bad.size} slots differ, first rows {bad[:8].tolist()}")


def oracle_store(words: np.ndarray, T: float, B: int):
    mask, bitval = oracle.build_meta(words, T)
    slots, bitmask, row_bits = oracle.compress(words, B, mask, bitval)
    return mask, bitval, slots, bitmask, row_bits
