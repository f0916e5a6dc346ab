"""The allocation-free entry point, vqx_plane_stats_noalloc.

It exists for callers that must not allocate once they run (a real-time
pipeline whose frame budget cannot absorb an allocation that may take driver
locks or wait for the GPU, or an application whose own allocator owns all of
the GPU's memory).  It runs the same kernels as vqx_plane_stats with a fixed
static scratch array, so its records must equal the oracle's, and
vqx_plane_stats' records exactly, call after call, even though the scratch
keeps the previous call's contents.  Batches large enough to leave the
scratch short make every unit write one record instead of one per warp; two
of the cases below take that branch, one of them at the largest batch the
scratch holds.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import parity
from exact_full_reference_gb300 import workloads as wl


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    """More than VQX_NOALLOC_MAX_RECORDS / 2 frames: VQX_EINVAL, before any
    CUDA call (so this runs without a GPU too)."""
    so = lib.library()
    n = lib.VQX_NOALLOC_MAX_RECORDS // 2 + 1
    out = np.zeros(n, lib.FRAME_STATS_DTYPE)
    rc = so.vqx_plane_stats_noalloc(1 << 20, 1 << 20, 16, 16, 32, 16, n, None, out.ctypes.data)
    assert rc == lib.VQX_EINVAL


def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _check(lib, orc, ref, dist, bpc, stride=None):
    """One noalloc call on (n, h, w) planes: records equal to the oracle's and
    to vqx_plane_stats'."""
    torch = _need_gpu()
    n, h, w = ref.shape
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride)
    got = lib.vqx_plane_stats_noalloc(pr, pd, w, h, stride, bpc, n)
    torch.cuda.synchronize()
    sc, un = orc.batch(rb, db, w, h, stride, bpc, n)
    parity.compare(got, sc, un, bpc, w * h, planes=(ref, dist))
    expect = lib.vqx_plane_stats(pr, pd, w, h, stride, bpc, n)
    assert got.tobytes() == expect.tobytes()
    return got


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_and_the_allocating_entry_point(lib, orc):
    _need_gpu()
    # Two calls in a row with different batches: the larger one first, so
    # that stale records from it would show up in the second call.
    cases = [
        (wl.WORKLOADS["3840x2160_16bit_x32"], list(range(6)) + [31]),
        (wl.WORKLOADS["1920x1080_10bit_x48"], [0, 1, 2]),
    ]
    for w, frames in cases:
        ref, dist = w.generate(frames)
        _check(lib, orc, ref, dist, w.bpc)


@pytest.mark.gpu
def test_noalloc_short_scratch_one_record_per_unit(lib, orc):
    """The largest batch the scratch holds, VQX_NOALLOC_MAX_RECORDS / 2 =
    32768 frames, of 64x2 16-bit frames on a padded pitch (the tile path, not
    the warp-per-frame one): one record per frame is left for stage 1, so
    every unit writes a single record.  Then 5000 dense 176x144 8-bit frames
    (the bulk-copy path, 12 records a frame left) take the same branch.  A
    small batch afterwards must not see either call's records."""
    _need_gpu()
    n = lib.VQX_NOALLOC_MAX_RECORDS // 2
    rng = np.random.Generator(np.random.PCG64(4242))
    ref = rng.integers(0, 65536, (n, 2, 64)).astype(np.uint16)
    dist = rng.integers(0, 65536, (n, 2, 64)).astype(np.uint16)
    _check(lib, orc, ref, dist, 16, stride=64 * 2 + 16)
    ref = rng.integers(0, 256, (5000, 144, 176)).astype(np.uint8)
    dist = np.clip(ref.astype(np.int64) + rng.integers(-9, 10, ref.shape), 0, 255).astype(np.uint8)
    _check(lib, orc, ref, dist, 8)
    w = wl.WORKLOADS["576x324_8bit_x1"]
    ref, dist = w.generate()
    _check(lib, orc, ref, dist, 8)
