"""The expert file tier's read engine (TurboFieldfare write-up, "Explicit reads
made expert streaming work": a miss is read from the model file with a bounded
number of parallel pread calls).  No GPU: moe_pread_parallel is the engine the
MOE_FILE_POOL contexts use, exported on its own; the GPU parity of a
file-pool context against a host-pool context is in test_gpu_pool.py."""

import numpy as np
import pytest

import bit_routed_expert_router_gb300 as moe

EXPERT = 3_345_408      # device bytes of one full-shape routed expert


def _file(tmp_path, n, seed=0):
    data = np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)
    p = tmp_path / "experts.bin"
    p.write_bytes(data.tobytes())
    return p, data


@pytest.mark.parametrize("threads,chunk", [(1, 0), (4, 4096), (8, 65536), (3, 12288), (16, 524288)])
def test_reads_exact_bytes(tmp_path, threads, chunk):
    p, data = _file(tmp_path, 2 * EXPERT + 777)
    cases = [(0, EXPERT), (EXPERT, EXPERT), (4096, 1), (123, 100_000), (len(data) - 5, 5), (0, 0),
             (0, len(data))]
    for off, n in cases:
        dst = np.zeros(max(n, 1), np.uint8)
        assert moe.moe_pread_parallel(str(p), off, n, dst.ctypes.data, threads, chunk) == moe.MOE_OK
        assert np.array_equal(dst[:n], data[off:off + n]), (off, n)


def test_chunks_cover_the_range_without_overlap(tmp_path):
    # a chunk size that does not divide the length: the tail chunk is short
    p, data = _file(tmp_path, 1_000_003, seed=3)
    dst = np.full(1_000_003 + 64, 0xAB, np.uint8)
    assert moe.moe_pread_parallel(str(p), 0, 1_000_003, dst.ctypes.data, 7, 4096) == moe.MOE_OK
    assert np.array_equal(dst[:1_000_003], data)
    assert np.all(dst[1_000_003:] == 0xAB)          # nothing written past the range


def test_reading_past_the_end_is_eio(tmp_path):
    p, _ = _file(tmp_path, 10_000)
    dst = np.zeros(20_000, np.uint8)
    assert moe.moe_pread_parallel(str(p), 5_000, 10_000, dst.ctypes.data, 4, 4096) == moe.MOE_EIO


def test_bad_arguments(tmp_path):
    dst = np.zeros(16, np.uint8)
    assert moe.moe_pread_parallel(str(tmp_path / "missing.bin"), 0, 16, dst.ctypes.data, 2, 0) == moe.MOE_EINVAL
    p, _ = _file(tmp_path, 64)
    assert moe.moe_pread_parallel(str(p), 0, 16, dst.ctypes.data, 0, 0) == moe.MOE_EINVAL
    assert moe.moe_pread_parallel(str(p), 0, 16, dst.ctypes.data, 65, 0) == moe.MOE_EINVAL
    assert moe.moe_pread_parallel(None, 0, 16, dst.ctypes.data, 1, 0) == moe.MOE_EINVAL
    assert moe.moe_pread_parallel(str(p), 0, 16, None, 1, 0) == moe.MOE_EINVAL
    assert moe.moe_status_string(moe.MOE_EIO) == "MOE_EIO"
