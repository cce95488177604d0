"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks answer before any CUDA work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import lossless_bit_level_gb300 as ibp
from lossless_bit_level_gb300 import build_lib

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "ibp.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return ibp.load()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ibp_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(ibp.SYMBOLS)
    # every header of include/ is covered: the codec's and the testing hook's
    headers = sorted(f for f in os.listdir(INCLUDE) if f.endswith(".h"))
    assert headers == ["ibp.h", "ibp_testing.h"]
    testing = declared_functions(os.path.join(INCLUDE, "ibp_testing.h"))
    assert set(testing) == set(ibp.TESTING_SYMBOLS)
    for name in testing:
        assert hasattr(lib, name), name


def test_testing_wait_limit_hook(lib):
    """Host-side only: returns the previous setting, 0 meaning the default."""
    assert ibp.testing_set_wait_limit_ns(5) == 0
    assert ibp.testing_set_wait_limit_ns(0) == 5
    assert ibp.testing_set_wait_limit_ns(0) == 0
    assert ibp.testing_withhold_plans(True) is False
    assert ibp.testing_withhold_plans(False) is True
    assert ibp.testing_withhold_plans(False) is False


def test_size_queries(lib):
    assert ibp.slot_bytes(128, ibp.FP32) == 512
    assert ibp.slot_bytes(4096, ibp.BF16) == 8192
    assert ibp.slot_bytes(11008, ibp.BF16) == 22016
    assert ibp.slot_bytes(33, ibp.FP16) == 80
    assert ibp.meta_scratch_bytes() == 256
    assert ibp.meta_select_scratch_bytes() == 1024
    assert ibp.pack_scratch_bytes(0) == 8
    assert ibp.pack_scratch_bytes(4096) == 8
    assert ibp.pack_scratch_bytes(4097) == 16
    assert ibp.meta_positions_scratch_bytes(128, ibp.FP32) == 128 * 256
    assert ibp.meta_positions_scratch_bytes(4096, ibp.BF16) == 2048 * 256
    assert ibp.meta_positions_scratch_bytes(64, ibp.W8) == 16 * 256
    with pytest.raises(ibp.IBPError):
        ibp.slot_bytes(0, ibp.FP32)
    with pytest.raises(ibp.IBPError) as e:
        ibp.slot_bytes(128, 7)
    assert e.value.code == ibp.ERR_DTYPE


def test_argument_errors_before_cuda(lib):
    vp = ctypes.c_void_p
    # null pointers, bad T, bad dtype, unsupported block size, ragged row
    assert lib.ibp_build_meta(None, 10, 128, ibp.FP32, 0.9, 32, None, None, None) == ibp.ERR_ARG
    assert lib.ibp_build_meta(vp(16), 10, 128, ibp.FP32, 1.5, 32, vp(16), vp(16), None) == \
        ibp.ERR_ARG
    assert lib.ibp_build_meta(vp(16), 10, 128, 9, 0.9, 32, vp(16), vp(16), None) == ibp.ERR_DTYPE
    assert lib.ibp_compress(None, 10, 98, ibp.FP32, 32, None, None, 400, None, None, None,
                            None) == ibp.ERR_ARG  # shorter last block, row not 16-byte whole
    assert lib.ibp_compress(None, 10, 100, ibp.FP32, 32, None, None, 400, None, None, None,
                            None) == ibp.ERR_ARG  # shorter last block allowed; null pointers
    assert lib.ibp_compress(None, 10, 100, 7, 32, None, None, 400, None, None, None,
                            None) == ibp.ERR_DTYPE
    assert ibp.slot_bytes(40, ibp.W8) == 48
    assert lib.ibp_compress(None, 10, 128, ibp.FP32, 16, None, None, 512, None, None, None,
                            None) == ibp.ERR_UNSUPPORTED
    assert lib.ibp_compress(None, 10, 128, ibp.FP32, 32, None, None, 496, None, None, None,
                            None) == ibp.ERR_ARG  # slot too small
    assert lib.ibp_compress(None, 10, 1 << 21, ibp.FP32, 32, None, None, 1 << 23, None, None,
                            None, None) == ibp.ERR_UNSUPPORTED
    assert lib.ibp_decompress_gather(None, 512, 10, 128, ibp.FP32, 32, None, None, None, 0, None,
                                     None, None) == ibp.OK  # empty gather is a no-op
    assert lib.ibp_decompress_gather(None, 512, 10, 128, ibp.FP32, 32, None, None, None, -1, None,
                                     None, None) == ibp.ERR_ARG
    assert lib.ibp_decompress_gather(None, 512, 10, 128, ibp.FP32, 32, None, None, None, 4, None,
                                     None, None) == ibp.ERR_ARG
    assert lib.ibp_probe_read(None, 17, None, None) == ibp.ERR_ARG
    assert lib.ibp_build_meta_select(None, 10, 128, ibp.FP32, 0.9, 32, None, None, None,
                                     None) == ibp.ERR_ARG
    assert lib.ibp_build_meta_select(vp(16), 0, 128, ibp.FP32, 0.9, 32, vp(16), None, vp(16),
                                     None) == ibp.ERR_ARG
    assert lib.ibp_build_meta_select(vp(16), 10, 128, ibp.FP32, -0.1, 32, vp(16), None, vp(16),
                                     None) == ibp.ERR_ARG
    assert lib.ibp_build_meta_select(vp(16), 10, 128, ibp.FP32, 0.9, 16, vp(16), None, vp(16),
                                     None) == ibp.ERR_UNSUPPORTED
    assert lib.ibp_build_meta_select(vp(16), 10, 128, 5, 0.9, 32, vp(16), None, vp(16),
                                     None) == ibp.ERR_DTYPE
    # packed store: sizes, null pointers, selection count, empty calls
    assert lib.ibp_pack_offsets(None, None, 10, 128, ibp.FP32, None, 11, vp(16), vp(16), None,
                                None) == ibp.ERR_ARG  # n_sel > n_rows without a selection
    assert lib.ibp_pack_offsets(None, None, 10, 128, 4, None, 5, vp(16), vp(16), None,
                                None) == ibp.ERR_DTYPE
    assert lib.ibp_pack(None, 512, 10, 128, ibp.FP32, None, None, None, 0, None, None, 0, None,
                        None, None, None) == ibp.OK  # nothing to pack
    assert lib.ibp_pack(None, 496, 10, 128, ibp.FP32, None, None, None, 4, None, None, 0, None,
                        None, None, None) == ibp.ERR_ARG  # slot smaller than a raw row
    assert lib.ibp_pack(None, 512, 10, 128, ibp.FP32, None, None, None, 4, None, None, 0, None,
                        None, None, None) == ibp.ERR_ARG
    assert lib.ibp_decompress_gather_packed(None, 0, None, 10, 128, ibp.FP32, 32, None, None,
                                            None, 0, None, None, None) == ibp.OK
    assert lib.ibp_decompress_gather_packed(None, 0, None, 10, 128, ibp.FP32, 32, None, None,
                                            None, 3, None, None, None) == ibp.ERR_ARG
    assert lib.ibp_decompress_gather_packed(None, 0, None, 10, 128, ibp.FP32, 48, None, None,
                                            None, 3, None, None, None) == ibp.ERR_UNSUPPORTED
    # per-position metadata: rows over 16 KiB are not handled; empty calls are no-ops
    assert lib.ibp_compress_positions(None, 10, 8200, ibp.BF16, 64, None, None, None, 16400, None,
                                      None, None) == ibp.ERR_UNSUPPORTED
    assert lib.ibp_compress_positions(None, 0, 128, ibp.FP32, 32, None, None, None, 512, None,
                                      None, None) == ibp.OK
    assert lib.ibp_decompress_gather_positions(None, 512, 10, 128, ibp.FP32, 32, None, None, None,
                                               None, 0, None, None, None) == ibp.OK
    assert lib.ibp_decompress_gather_positions(None, 512, 10, 128, ibp.FP32, 32, None, None, None,
                                               None, 2, None, None, None) == ibp.ERR_ARG
    assert lib.ibp_build_meta_positions(None, 10, 128, ibp.FP32, 0.9, 32, None, None, None,
                                        None) == ibp.ERR_ARG
    # split preprocessing: counts of rows not whole 32-bit words, bad T, bad block
    assert lib.ibp_meta_count(vp(16), 3, 3, ibp.W8, vp(16), None) == ibp.ERR_ARG
    assert lib.ibp_meta_finalize(vp(16), 100, ibp.FP32, 1.2, 32, vp(16), None, None) == \
        ibp.ERR_ARG
    assert lib.ibp_meta_finalize(vp(16), 100, ibp.FP32, 0.9, 48, vp(16), None, None) == \
        ibp.ERR_UNSUPPORTED
    assert lib.ibp_meta_finalize(vp(16), 0, ibp.FP32, 0.9, 32, vp(16), None, None) == ibp.ERR_ARG
    assert lib.ibp_meta_finalize(vp(16), 100, 6, 0.9, 32, vp(16), None, None) == ibp.ERR_DTYPE
    # store statistics: host output needs a destination; sizes, dtype, null arrays
    st = ibp.Stats()
    assert lib.ibp_query(None, None, 0, 128, ibp.FP32, None, None) == ibp.ERR_ARG
    assert lib.ibp_query(None, None, -1, 128, ibp.FP32, ctypes.byref(st), None) == ibp.ERR_ARG
    assert lib.ibp_query(None, None, 0, 0, ibp.FP32, ctypes.byref(st), None) == ibp.ERR_ARG
    assert lib.ibp_query(None, None, 5, 128, ibp.FP32, ctypes.byref(st), None) == ibp.ERR_ARG
    assert lib.ibp_query(None, None, 5, 128, 8, ctypes.byref(st), None) == ibp.ERR_DTYPE
    assert lib.ibp_query_async(None, None, 0, 128, ibp.FP32, None, None) == ibp.ERR_ARG
    assert lib.ibp_query_async(None, None, 5, 128, 8, vp(16), None) == ibp.ERR_DTYPE
    assert ctypes.sizeof(ibp.Stats) == 40
    # de-duplicated gather: scratch size query (a hash table of at least 16 bytes per
    # index, then 4 + 8 bytes per index), limits, and an empty list as a no-op
    sz = ctypes.c_size_t(0)
    assert lib.ibp_gather_dedup_scratch_bytes(100_000, 128, ibp.FP32, 32, ctypes.byref(sz)) == ibp.OK
    assert sz.value == 262_144 * 8 + 16 + 100_000 * 4 + 100_000 * 8
    assert lib.ibp_gather_dedup_scratch_bytes(1 << 24, 128, ibp.FP32, 32, ctypes.byref(sz)) == \
        ibp.ERR_UNSUPPORTED
    assert lib.ibp_gather_dedup_scratch_bytes(10, 128, ibp.FP32, 32, None) == ibp.ERR_ARG
    assert lib.ibp_decompress_gather_dedup(vp(16), 512, 10, 128, ibp.FP32, 32, vp(16), vp(16),
                                           vp(16), 0, vp(16), vp(16), 0, None, None) == ibp.OK
    assert lib.ibp_decompress_gather_dedup(vp(16), 512, 1 << 40, 128, ibp.FP32, 32, vp(16),
                                           vp(16), vp(16), 5, vp(16), vp(16), 1 << 20, None,
                                           None) == ibp.ERR_UNSUPPORTED
    # batched gathers: empty batch is a no-op; a null job array with jobs is refused
    assert lib.ibp_decompress_gather_batched(None, 0, 128, ibp.FP32, 32, None, None) == ibp.OK
    assert lib.ibp_decompress_gather_batched(None, 3, 128, ibp.FP32, 32, None, None) == ibp.ERR_ARG
    assert ctypes.sizeof(ibp.GatherJob) == 64
    # contiguous ranges: inside the store, empty is a no-op
    assert lib.ibp_decompress_range(None, 512, 10, 128, ibp.FP32, 32, None, None, 4, 0, None, None,
                                    None) == ibp.OK
    assert lib.ibp_decompress_range(None, 512, 10, 128, ibp.FP32, 32, None, None, 4, 7, None, None,
                                    None) == ibp.ERR_ARG  # past the last row
    assert lib.ibp_decompress_range(None, 512, 10, 128, ibp.FP32, 32, None, None, -1, 2, None,
                                    None, None) == ibp.ERR_ARG
    assert lib.ibp_decompress_range(None, 512, 10, 128, ibp.FP32, 32, None, None, 0, 2, None, None,
                                    None) == ibp.ERR_ARG  # null pointers
    assert ibp.status_string(ibp.ERR_CORRUPT) == "corrupt slot header"
