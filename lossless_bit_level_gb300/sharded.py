"""Metadata for a table whose rows are spread over several processes (one GPU each).

"Reducing the GPU Memory Bottleneck with Lossless Compression for ML -- Extended",
technical summary, "Core algorithm" (preprocessing): the mask and bitval follow
from how often each bit position holds a 1 among the elements, so the per-position
counts of disjoint row sets add up. Each rank counts its own rows with
``ibp_meta_count`` (32 64-bit counters), the ranks sum the counters and their
element counts in one all-reduce, and every rank applies the threshold to the sums
with ``ibp_meta_finalize``. All ranks then hold the metadata that one GPU would
compute over the union of the rows, and each compresses and serves its own rows
with it; nothing else crosses between ranks.

The exchange is 33 integers per rank; ``allreduce_counts`` is the only collective
and works with any ``torch.distributed`` backend (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch

from . import dtype_code, meta_count, meta_finalize

N_COUNTERS = 32  # one per bit position of a 32-bit word


def allreduce_counts(counters: torch.Tensor, n_elems: int, group=None) -> int:
    """Sum ``counters`` (32 int64) over the ranks of ``group`` in place and return
    the total element count. One all-reduce of 33 int64 values."""
    import torch.distributed as dist
    if counters.dtype != torch.int64 or counters.numel() != N_COUNTERS:
        raise ValueError("counters must be 32 int64 values")
    buf = torch.empty(N_COUNTERS + 1, dtype=torch.int64, device=counters.device)
    buf[:N_COUNTERS].copy_(counters)
    buf[N_COUNTERS] = int(n_elems)
    dist.all_reduce(buf, op=dist.ReduceOp.SUM, group=group)
    counters.copy_(buf[:N_COUNTERS])
    return int(buf[N_COUNTERS].item())


def sharded_meta(rows: torch.Tensor, T: float, block_elems: int, meta: torch.Tensor,
                 counters: torch.Tensor, dtype: int | None = None, group=None,
                 stream=None) -> int:
    """Metadata of the union of every rank's ``rows`` (this rank's shard, [n, L] on
    this rank's GPU or in its page-locked host memory) into ``meta``. ``counters`` is
    a 32 x int64 device buffer; on return it holds the summed counts. Returns the
    total number of elements. A rank with no rows passes an empty [0, L] tensor."""
    code = dtype_code(rows, dtype)
    n, L = rows.shape[0], rows.shape[1]
    # with no rows the call only clears the counters, on the same stream as the
    # exchange and the finalize below (so nothing reads them before the clear)
    meta_count(rows, counters, dtype=code, stream=stream)
    if counters.is_cuda:  # the exchange is ordered after the count on the same stream
        s = stream if stream is not None else torch.cuda.current_stream(counters.device)
        with torch.cuda.stream(s):
            total = allreduce_counts(counters, n * L, group)
    else:
        total = allreduce_counts(counters, n * L, group)
    if total <= 0:
        raise ValueError("no rows on any rank")
    meta_finalize(counters, total, code, T, block_elems, meta, stream=stream)
    return total


__all__ = ["allreduce_counts", "sharded_meta", "N_COUNTERS"]
