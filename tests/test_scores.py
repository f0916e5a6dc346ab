"""GPU parity of vqx_plane_scores: float_psnr, float_moment and the integer
psnr of every frame from one read of the planes, against the oracle.

The statistics records follow the rule of every statistics parity test
(``parity.compare``); the integer psnr records the rule of the integer psnr
tests (the SSE exactly, the doubles bit for bit).  Both must also equal, byte
for byte, what the separate entry points (vqx_plane_stats and
vqx_plane_int_psnr) return for the same planes.
"""
import numpy as np
import pytest

import parity
from exact_full_reference_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

INT_FIELDS = ("mse", "psnr", "psnr_uncapped")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def compare_int(rec, want):
    assert len(rec) == len(want)
    for f in range(len(rec)):
        assert int(rec[f]["sse"]) == int(want[f]["sse"]), (f, int(rec[f]["sse"]), int(want[f]["sse"]))
        for k in INT_FIELDS:
            assert rec[f][k].tobytes() == want[f][k].tobytes(), (f, k, rec[f][k], want[f][k])
        assert int(rec[f]["reserved"]) == 0


def run_case(lib, orc, ref, dist, bpc, stride=None, offset_ref=0, offset_dist=0, separate=True):
    n, h, w = ref.shape
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride, offset_ref, offset_dist)
    stats, ints = lib.vqx_plane_scores(pr, pd, w, h, stride, bpc, n)
    torch.cuda.synchronize()
    sc, un = orc.batch(rb, db, w, h, stride, bpc, n)
    parity.compare(stats, sc, un, bpc, w * h, planes=(ref, dist))
    compare_int(ints, orc.int_psnr(rb, db, w, h, stride, bpc, n))
    assert (stats["flags"] == ints["flags"]).all()
    if separate:
        assert stats.tobytes() == lib.vqx_plane_stats(pr, pd, w, h, stride, bpc, n).tobytes()
        assert ints.tobytes() == lib.vqx_plane_int_psnr(pr, pd, w, h, stride, bpc, n).tobytes()
    return stats, ints, un


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_scores(lib, orc, name):
    """Every frame of every workload at full size, the past-2^53 stress
    frames included (the SSE is exact at any size)."""
    w = wl.WORKLOADS[name]
    ref, dist = w.generate()
    run_case(lib, orc, ref, dist, w.bpc)


def test_sse_differs_from_the_float_noise_at_16_bits(lib, orc):
    """Full-range 16-bit differences: the float squares drop bits, so the SSE
    and the noise sum differ on every frame, and the pass must return both."""
    w = wl.WORKLOADS["stress_inverse_4k16"]
    ref, dist = w.generate()
    stats, ints, un = run_case(lib, orc, ref, dist, 16, separate=False)
    assert (ints["sse"] != stats["noise_units"]).all()


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("w,h,pad", [(1, 1, 0), (7, 3, 0), (333, 17, 0), (1000, 97, 48), (1922, 67, 30),
                                     (257, 49, 16), (37, 9, 6), (3840, 64, 256), (64, 64, 0)])
def test_shapes_and_layouts(lib, orc, bpc, w, h, pad):
    """Dense frames, padded rows (row pieces, boxes) and unaligned pitches:
    every stage-1 path of the 16-bit variant that carries the SSE."""
    rng = np.random.Generator(np.random.PCG64(13 * w + h + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    bps = 1 if bpc == 8 else 2
    ref = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    pad += pad % bps
    run_case(lib, orc, ref, dist, bpc, stride=w * bps + pad if pad else None)


def test_many_small_frames_warp_per_frame(lib, orc):
    """2500 dense 64x64 16-bit frames take the warp-per-frame path."""
    rng = np.random.Generator(np.random.PCG64(77))
    ref = rng.integers(0, 65536, (2500, 64, 64)).astype(np.uint16)
    dist = rng.integers(0, 65536, (2500, 64, 64)).astype(np.uint16)
    run_case(lib, orc, ref, dist, 16)


def test_unaligned_bases(lib, orc):
    rng = np.random.Generator(np.random.PCG64(5))
    ref = rng.integers(0, 65536, (2, 40, 300)).astype(np.uint16)
    dist = rng.integers(0, 65536, (2, 40, 300)).astype(np.uint16)
    run_case(lib, orc, ref, dist, 16, offset_ref=2, offset_dist=6)


def test_identical_planes_cap_and_range_flag(lib, orc):
    for bpc in (8, 10, 12, 16):
        dt = np.uint8 if bpc == 8 else np.uint16
        ref = np.random.Generator(np.random.PCG64(bpc)).integers(0, 1 << bpc, (2, 64, 96)).astype(dt)
        stats, ints, _ = run_case(lib, orc, ref, ref.copy(), bpc)
        assert (ints["sse"] == 0).all() and (stats["noise_units"] == 0).all()
        assert (ints["psnr"] == lib.psnr_cap(bpc)).all() and (stats["psnr"] == lib.psnr_cap(bpc)).all()
    rng = np.random.Generator(np.random.PCG64(9))
    ref = rng.integers(0, 4096, (3, 8, 40)).astype(np.uint16)
    dist = rng.integers(0, 4096, (3, 8, 40)).astype(np.uint16)
    dist[1, 2, 3] = 5000
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    stats, ints, rc = lib.vqx_plane_scores(pr, pd, 40, 8, stride, 12, 3, check=False)
    assert rc == lib.VQX_ERANGE
    assert [int(x) for x in stats["flags"]] == [0, 1, 0] == [int(x) for x in ints["flags"]]


def test_headline_batch_pipelined_as_the_benchmark_runs_it(lib, orc):
    """The 3840x2160 16-bit batch as bench.py --op scores times it: batch
    i + 1 submitted with VQX_SUBMIT_PLANES_READY before batch i is finished;
    every batch equals the blocking call, whose records equal the oracle's
    (test_workload_scores)."""
    w = wl.WORKLOADS[wl.HEADLINE]
    ref, dist = w.generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    geo = (w.width, w.height, stride, w.bpc, w.n_frames)
    want_s, want_i = lib.vqx_plane_scores(pr, pd, *geo)
    prev = None
    for _ in range(6):
        cur = lib.vqx_plane_scores_submit(pr, pd, *geo, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            s, i = prev.finish()
            assert s.tobytes() == want_s.tobytes() and i.tobytes() == want_i.tobytes()
        prev = cur
    s, i = prev.finish()
    assert s.tobytes() == want_s.tobytes() and i.tobytes() == want_i.tobytes()
    # a handle of another pair is refused (and released)
    p = lib.vqx_plane_stats_submit(pr, pd, *geo)
    p.kind = "scores"
    assert p.finish(check=False)[2] == lib.VQX_EINVAL
