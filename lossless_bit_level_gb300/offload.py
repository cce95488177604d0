"""Overlapped offload pipeline: tensors kept compressed in page-locked host memory and
decompressed into device buffers one layer ahead of their consumer.

"Reducing the GPU Memory Bottleneck with Lossless Compression for ML -- Extended",
technical summary: "System integration" (offloaded LLM inference keeps weights and
the KV cache in host memory; they cross the host link compressed, into fixed-size
buffers) and "Core algorithm" (decompression hides behind the transfer). Here the
transfer and the decompression are one kernel (``ibp_decompress_range`` reads the
host slots zero-copy), and this module overlaps it with the consumer's compute:

    loader stream:    [decode layer 0 -> buf 0][decode layer 1 -> buf 1][wait buf 0 free][decode layer 2 -> buf 0] ...
    consumer stream:                 [wait][compute layer 0 (buf 0)][wait][compute layer 1 (buf 1)] ...

Two sets of device buffers alternate; CUDA events order a buffer's reuse after its
consumer and its consumer after its decode. Every byte of a tensor is rebuilt by the
library's CUDA kernels; this module only allocates buffers and orders launches.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import BF16, FP16, FP32, WIDTH
from . import build_meta, build_meta_select, compress, decompress_range, meta_scratch_bytes, \
    meta_select_scratch_bytes, slot_bytes

_WORD = {FP32: (np.int32, torch.int32), FP16: (np.int16, torch.int16),
         BF16: (np.int16, torch.int16)}


@dataclass
class CompressedTensor:
    """One tensor ([n_rows, row_elems] element words) stored as IBP slots."""

    n_rows: int
    row_elems: int
    dtype: int
    block_elems: int
    slots: torch.Tensor     # [n_rows, slot_bytes] uint8, page-locked host (or device)
    bitmask: torch.Tensor   # device
    row_bits: torch.Tensor  # device
    meta: torch.Tensor      # device, 16 bytes
    status: torch.Tensor    # device, first error of the last compress/decompress

    @classmethod
    def from_words(cls, words: np.ndarray, dtype: int, T: float, block_elems: int,
                   device: torch.device, where: str = "host",
                   saving_aware: bool = False) -> "CompressedTensor":
        """Compress a 2-D array of element words (uint16/uint32 bit patterns).
        The rows are staged once in page-locked memory, read zero-copy by the
        metadata and compression kernels, and released; only the slots remain."""
        n, L = words.shape
        npv, tdt = _WORD[dtype]
        src = torch.from_numpy(np.ascontiguousarray(words).view(npv))
        rows = torch.empty(src.shape, dtype=tdt, pin_memory=True)
        rows.copy_(src)
        meta = torch.zeros(4, dtype=torch.int32, device=device)
        if saving_aware:
            scratch = torch.empty(meta_select_scratch_bytes() // 4, dtype=torch.int32,
                                  device=device)
            build_meta_select(rows, T, block_elems, meta, scratch, dtype=dtype)
        else:
            scratch = torch.empty(meta_scratch_bytes() // 4, dtype=torch.int32, device=device)
            build_meta(rows, T, block_elems, meta, scratch, dtype=dtype)
        sb = slot_bytes(L, dtype)
        if where == "host":
            slots = torch.empty((n, sb), dtype=torch.uint8, pin_memory=True)
        else:
            slots = torch.empty((n, sb), dtype=torch.uint8, device=device)
        bitmask = torch.zeros(((n + 31) // 32,), dtype=torch.int32, device=device)
        row_bits = torch.zeros((max(n, 1),), dtype=torch.int32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        compress(rows, block_elems, meta, slots, bitmask, row_bits, status, dtype=dtype)
        torch.cuda.current_stream(device).synchronize()
        del rows
        return cls(n, L, dtype, block_elems, slots, bitmask, row_bits, meta, status)

    @property
    def word_dtype(self) -> torch.dtype:
        return _WORD[self.dtype][1]

    @property
    def raw_bytes(self) -> int:
        return self.n_rows * self.row_elems * WIDTH[self.dtype] // 8

    def stored_bytes(self) -> int:
        """Bytes the rows occupy in their slots (the bytes a full decompression reads)."""
        bits = self.row_bits.cpu().numpy().view(np.uint32)[: self.n_rows].astype(np.int64)
        bm = self.bitmask.cpu().numpy().view(np.uint32)
        r = np.arange(self.n_rows)
        comp = (bm[r // 32] >> (r % 32).astype(np.uint32)) & 1
        raw_row = self.row_elems * WIDTH[self.dtype] // 8
        return int(np.where(comp == 1, 4 * ((bits + 31) // 32), raw_row).sum())

    def empty_like(self, device: torch.device) -> torch.Tensor:
        return torch.empty((self.n_rows, self.row_elems), dtype=self.word_dtype, device=device)

    def decompress_into(self, out: torch.Tensor, stream=None) -> None:
        """Every row, in order, into ``out`` (device memory, [n_rows, row_elems])."""
        decompress_range(self.slots, self.n_rows, self.row_elems, self.dtype, self.block_elems,
                         self.bitmask, self.meta, 0, self.n_rows, out, self.status,
                         stream=stream)


class OffloadPipeline:
    """Double-buffered streaming of layers (lists of same-shaped tensors per layer)
    through device buffers, decoding layer l+1 while the consumer computes layer l.

    ``load(tensor, out, stream)`` fills one device buffer (by default
    ``tensor.decompress_into``; a raw-copy loader gives the uncompressed baseline).
    ``consume(layer, buffers)`` enqueues the consumer's work on the current stream.
    With ``overlap=False`` loads and compute share one stream (no overlap)."""

    def __init__(self, layers: list, device: torch.device, load=None, overlap: bool = True):
        if not layers:
            raise ValueError("no layers")
        self.layers = layers
        self.device = device
        self.load = load or (lambda t, out, stream: t.decompress_into(out, stream=stream))
        self.overlap = overlap
        self.buffers = [[t.empty_like(device) for t in layers[0]] for _ in range(2)]
        # the loader runs at high priority: its CTAs take SMs as soon as they free up,
        # so the decode (which paces the pipeline) is never queued behind compute
        self.loader = torch.cuda.Stream(device=device, priority=-1)
        self.compute = torch.cuda.Stream(device=device) if overlap else self.loader
        self.loaded = [torch.cuda.Event() for _ in range(2)]
        self.consumed = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]  # buffer set b has a consumer (in this or an earlier run)

    def run(self, n_steps: int, consume, order=None) -> None:
        """Stream layers order[0..n_steps) (default: 0, 1, ..., cycling over the
        layers) through the buffers and hand each to ``consume``."""
        seq = [(order[i] if order is not None else i) % len(self.layers) for i in range(n_steps)]
        used = self.used

        def issue_load(step):
            b = step % 2
            with torch.cuda.stream(self.loader):
                if used[b]:
                    self.loader.wait_event(self.consumed[b])
                for t, out in zip(self.layers[seq[step]], self.buffers[b]):
                    self.load(t, out, self.loader)
                self.loaded[b].record(self.loader)

        issue_load(0)
        for step in range(n_steps):
            b = step % 2
            if self.overlap and step + 1 < n_steps:
                issue_load(step + 1)  # the next layer decodes while this one computes
            with torch.cuda.stream(self.compute):
                self.compute.wait_event(self.loaded[b])
                consume(seq[step], self.buffers[b])
                self.consumed[b].record(self.compute)
                used[b] = True
            if not self.overlap and step + 1 < n_steps:
                issue_load(step + 1)

    def synchronize(self) -> None:
        self.loader.synchronize()
        self.compute.synchronize()


def raw_loader(raw_rows: dict):
    """Loader that copies each tensor's raw rows (page-locked host memory, keyed by
    the tensor's id) with cudaMemcpyAsync: the uncompressed baseline."""

    def load(t, out, stream):
        out.copy_(raw_rows[id(t)], non_blocking=True)

    return load
