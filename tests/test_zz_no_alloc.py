"""ibp_build_meta_noalloc, the metadata build for callers that cannot allocate
device memory (a plug-in whose host framework owns all device memory, a loop that
must never hit cudaMalloc's implicit synchronisation, a system that forbids
allocation after start-up), called through the C ABI and checked against the
regular ibp_build_meta, which takes caller-allocated scratch.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import ibp_inputs as gen
import lossless_bit_level_gb300 as ibp

pytestmark = pytest.mark.gpu


def _noalloc(rows_t: torch.Tensor, dtype: int, T: float, B: int, meta_t: torch.Tensor) -> int:
    lib = ibp.load()
    n, L = rows_t.shape
    return lib.ibp_build_meta_noalloc(ctypes.c_void_p(rows_t.data_ptr()), n, L, dtype, T, B,
                                      ctypes.c_void_p(meta_t.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _regular(rows_t: torch.Tensor, dtype: int, T: float, B: int) -> np.ndarray:
    meta = torch.zeros(4, dtype=torch.int32, device="cuda")
    scratch = torch.empty(ibp.meta_scratch_bytes() // 4, dtype=torch.int32, device="cuda")
    ibp.build_meta(rows_t, T, B, meta, scratch, dtype=dtype)
    torch.cuda.synchronize()
    return meta.cpu().numpy().view(np.uint32).copy()


def test_noalloc_meta_equals_regular_on_two_calls_in_a_row():
    tiny = gen.tiny_fp32(4096).view(np.uint32)
    kv = gen.llm_kv(0, 1, n_rows=2048)
    cases = [
        (torch.from_numpy(tiny.view(np.int32)).cuda(), ibp.FP32, 0.9, 32),
        (torch.from_numpy(kv.view(np.int16)).cuda(), ibp.BF16, 0.9, 64),
    ]
    # two different inputs back to back: the second call must not keep any of the
    # first call's counts in the shared built-in array
    for rows_t, dtype, T, B in cases + cases[:1]:
        expected = _regular(rows_t, dtype, T, B)
        meta = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(rows_t, dtype, T, B, meta) == ibp.OK
        torch.cuda.synchronize()
        got = meta.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, expected), ([hex(v) for v in got], [hex(v) for v in expected])


def test_noalloc_meta_rejects_bad_arguments():
    rows_t = torch.zeros((4, 32), dtype=torch.int32, device="cuda")
    meta = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert _noalloc(rows_t, ibp.FP32, 1.5, 32, meta) == ibp.ERR_ARG
    assert _noalloc(rows_t, 9, 0.9, 32, meta) == ibp.ERR_DTYPE
