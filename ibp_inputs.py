"""Seeded synthetic workloads for the IBP codec (inputs only: no codec arithmetic).

Both the test suite (oracle and GPU sides) and ``bench.py`` draw their inputs
from here, so the two sides always see identical bytes. Nothing in this module
computes masks, streams or sizes; it only produces element words and row
indices with the shapes and distributions of the five workloads below.

Every generator uses ``numpy.random.default_rng([seed, workload, part])`` with
seed 0 for data, 1 for indices and 2 for outlier channels, and generates rows in
order, so the first ``n`` rows of a workload are the same whatever ``n_rows`` is
asked for (smaller parity cases are prefixes of the full-size ones).

Workloads (row = one feature vector / embedding row / weight row / token):
  tiny_fp32   4096 x 128 FP32, iid N(0, 0.05)
  gnn_dense   2,000,000 x 128 FP32, column c ~ N(mu_c, sigma_c) with
              mu_c ~ U(-0.1, 0.1), sigma_c ~ U(0.01, 0.2), drawn in float64,
              each row divided by its L2 norm, then cast to FP32
  gnn_sparse  500,000 x 512 FP32, each element 1.0 with prob. 0.01 else 0.0
  dlrm        26 tables x 1,000,000 x 128 FP32, U(-1/sqrt(1e6), 1/sqrt(1e6))
  llm_bf16    BF16 decoder weights ([out, in] rows, N(0, 0.02)) for 32 layers of
              hidden 4096 / FFN 11008, and KV rows ([batch*seq] x 32 heads*128)
              N(0, 1) with 41 seeded channels per tensor scaled by 10
"""
from __future__ import annotations

import numpy as np

DATA, INDEX, OUTLIER = 0, 1, 2

TINY, GNN_DENSE, GNN_SPARSE, DLRM, LLM = 1, 2, 3, 4, 5

LLM_HIDDEN = 4096
LLM_FFN = 11008
LLM_LAYERS = 32
LLM_HEADS = 32
LLM_HEAD_DIM = 128
LLM_MATRICES = {  # name -> (rows = out features, row length = in features)
    "q": (LLM_HIDDEN, LLM_HIDDEN),
    "k": (LLM_HIDDEN, LLM_HIDDEN),
    "v": (LLM_HIDDEN, LLM_HIDDEN),
    "o": (LLM_HIDDEN, LLM_HIDDEN),
    "gate": (LLM_FFN, LLM_HIDDEN),
    "up": (LLM_FFN, LLM_HIDDEN),
    "down": (LLM_HIDDEN, LLM_FFN),
}
_MATRIX_ID = {name: i for i, name in enumerate(LLM_MATRICES)}


def rng(seed: int, workload: int, part: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, workload, part])


def _chunked_rows(n_rows: int, chunk: int, make):
    out = []
    done = 0
    while done < n_rows:
        k = min(chunk, n_rows - done)
        out.append(make(k))
        done += k
    return np.concatenate(out, axis=0) if len(out) > 1 else out[0]


def tiny_fp32(n_rows: int = 4096, row_elems: int = 128) -> np.ndarray:
    g = rng(DATA, TINY)
    return g.normal(0.0, 0.05, size=(n_rows, row_elems)).astype(np.float32)


def gnn_dense(n_rows: int = 2_000_000, row_elems: int = 128) -> np.ndarray:
    g = rng(DATA, GNN_DENSE)
    mu = g.uniform(-0.1, 0.1, size=row_elems)
    sigma = g.uniform(0.01, 0.2, size=row_elems)

    def make(k):
        x = g.normal(mu, sigma, size=(k, row_elems))
        x /= np.sqrt(np.einsum("ij,ij->i", x, x))[:, None]
        return x.astype(np.float32)

    return _chunked_rows(n_rows, 262_144, make)


def gnn_sparse(n_rows: int = 500_000, row_elems: int = 512) -> np.ndarray:
    g = rng(DATA, GNN_SPARSE)

    def make(k):
        return np.where(g.random(size=(k, row_elems)) < 0.01, np.float32(1.0), np.float32(0.0))

    return _chunked_rows(n_rows, 131_072, make)


def dlrm_table(table: int, n_rows: int = 1_000_000, row_elems: int = 128) -> np.ndarray:
    g = rng(DATA, DLRM, table)
    a = 1.0 / np.sqrt(1e6)

    def make(k):
        return g.uniform(-a, a, size=(k, row_elems)).astype(np.float32)

    return _chunked_rows(n_rows, 262_144, make)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round half to even) and return uint16 words.
    Inputs here are finite, so no NaN handling is needed; for finite words the sum
    below stays under 2^32 (at most 0xFF7FFFFF + 0x8000), so 32-bit arithmetic is
    exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def llm_weight(layer: int, name: str, n_rows: int | None = None) -> np.ndarray:
    """BF16 weight rows of one projection as uint16 words, shape [out, in]."""
    rows, cols = LLM_MATRICES[name]
    n = rows if n_rows is None else n_rows
    g = rng(DATA, LLM, layer * 16 + _MATRIX_ID[name])

    def make(k):
        return f32_to_bf16_bits(g.normal(0.0, 0.02, size=(k, cols)).astype(np.float32))

    return _chunked_rows(n, 1024, make)


def llm_kv(layer: int, kv: int, batch: int = 8, seq: int = 4096,
           n_rows: int | None = None) -> np.ndarray:
    """BF16 K (kv=0) or V (kv=1) cache rows of one layer as uint16 words,
    shape [batch*seq, heads*head_dim]; 1% of channels (41 of 4096) scaled by 10."""
    width = LLM_HEADS * LLM_HEAD_DIM
    n = batch * seq if n_rows is None else n_rows
    part = 1000 + layer * 2 + kv
    outliers = rng(OUTLIER, LLM, part).choice(width, size=int(round(0.01 * width)), replace=False)
    scale = np.ones(width, dtype=np.float32)
    scale[outliers] = 10.0
    g = rng(DATA, LLM, part)

    def make(k):
        return f32_to_bf16_bits(g.normal(0.0, 1.0, size=(k, width)).astype(np.float32) * scale)

    return _chunked_rows(n, 2048, make)


def uniform_indices(n_rows: int, count: int, part: int = 0, workload: int = 0) -> np.ndarray:
    g = rng(INDEX, workload, part)
    return g.integers(0, n_rows, size=count, dtype=np.int64)


def zipf_indices(n_rows: int, count: int, alpha: float, part: int = 0,
                 workload: int = 0) -> np.ndarray:
    """Draw ``count`` rows with replacement, rank k (1-based) with probability
    proportional to k**-alpha over a finite population of n_rows (inverse-CDF
    sampling); ranks map to rows through a seeded permutation so that hot rows are
    scattered over the table."""
    g = rng(INDEX, workload, part)
    perm = g.permutation(n_rows)
    weights = np.arange(1, n_rows + 1, dtype=np.float64) ** (-float(alpha))
    cdf = np.cumsum(weights)
    cdf /= cdf[-1]
    u = g.random(size=count)
    rank = np.minimum(np.searchsorted(cdf, u, side="right"), n_rows - 1)
    return perm[rank].astype(np.int64)
