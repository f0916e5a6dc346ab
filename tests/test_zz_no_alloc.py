"""The allocation-free entry point, vqx_plane_stats_noalloc.

It exists for callers that must not allocate once they run (a real-time
pipeline whose frame budget cannot absorb an allocation that may take driver
locks or wait for the GPU, or an application whose own allocator owns all of
the GPU's memory).  It runs the same kernels as vqx_plane_stats with a fixed
static scratch array, so its records must equal vqx_plane_stats' records
exactly, call after call, even though the scratch keeps the previous call's
contents.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from exact_full_reference_gb300 import workloads as wl


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    """More than VQX_NOALLOC_MAX_RECORDS / 2 frames: VQX_EINVAL, before any
    CUDA call (so this runs without a GPU too)."""
    so = lib.library()
    n = lib.VQX_NOALLOC_MAX_RECORDS // 2 + 1
    out = np.zeros(n, lib.FRAME_STATS_DTYPE)
    rc = so.vqx_plane_stats_noalloc(1 << 20, 1 << 20, 16, 16, 32, 16, n, None, out.ctypes.data)
    assert rc == lib.VQX_EINVAL


@pytest.mark.gpu
def test_noalloc_matches_the_allocating_entry_point(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # Two calls in a row with different batches: the larger one first, so
    # that stale records from it would show up in the second call.
    cases = [
        (wl.WORKLOADS["3840x2160_16bit_x32"], list(range(6)) + [31]),
        (wl.WORKLOADS["1920x1080_10bit_x48"], [0, 1, 2]),
    ]
    for w, frames in cases:
        ref, dist = w.generate(frames)
        n = ref.shape[0]
        dr = torch.from_numpy(ref.reshape(-1).view(np.uint8)).cuda()
        dd = torch.from_numpy(dist.reshape(-1).view(np.uint8)).cuda()
        stride = w.width * w.bytes_per_sample
        expect = lib.vqx_plane_stats(dr, dd, w.width, w.height, stride, w.bpc, n)
        got = lib.vqx_plane_stats_noalloc(dr, dd, w.width, w.height, stride, w.bpc, n)
        torch.cuda.synchronize()
        # the tolerance of every parity test of the integer path: exact
        assert got.tobytes() == expect.tobytes(), w.name
