"""vqx_plane_stats_ordered against the oracle: every double of every frame
bit for bit, also past 2^53 units, where the CPU's running double sum rounds
and vqx_plane_stats only meets the bound of "ADR-1447 ..." (Decision)."""
import numpy as np
import pytest

import parity
from exact_full_reference_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

DOUBLES = ("noise", "mse", "psnr", "psnr_uncapped", "ref_mean", "ref_meansq", "dist_mean",
           "dist_meansq")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def check_identical(rec, sc, un):
    for f in range(len(rec)):
        for k in parity.UNIT_FIELDS:
            assert int(rec[f][k]) == int(un[f][k]), (f, k)
        for k in DOUBLES:
            assert rec[f][k].tobytes() == sc[f][k].tobytes(), (f, k, rec[f][k], sc[f][k])


@pytest.mark.parametrize("name", ["stress_full_range_4k16", "stress_dark_tenth_4k16",
                                  "stress_inverse_4k16", "3840x2160_16bit_x32",
                                  "1920x1080_16bit_x64", "3840x2160_12bit_x32"])
def test_ordered_equals_the_cpu_everywhere(lib, orc, name):
    w = wl.WORKLOADS[name]
    frames = range(w.n_frames) if w.n_frames <= 8 else [0, 1, 2, w.n_frames - 1]
    ref, dist = w.generate(frames)
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    n = ref.shape[0]
    rec = lib.vqx_plane_stats_ordered(pr, pd, w.width, w.height, stride, w.bpc, n)
    sc, un = orc.batch(rb, db, w.width, w.height, stride, w.bpc, n)
    check_identical(rec, sc, un)
    if name.startswith("stress"):
        # these frames do leave the exact range, and there the plain entry
        # point differs from the CPU on at least one output
        plain = lib.vqx_plane_stats(pr, pd, w.width, w.height, stride, w.bpc, n)
        assert parity.exact_count(un) < n
        assert any(plain[f][k].tobytes() != sc[f][k].tobytes() for f in range(n) for k in DOUBLES)


def test_ordered_with_padded_rows_and_odd_sizes(lib, orc):
    """Raster blocks cross rows and the last block is short: 4001 x 2399
    (9.6 M pixels), full-range 16-bit, rows padded; the first frame is a
    plane against its inverse, whose noise passes 2^53 units."""
    rng = np.random.Generator(np.random.PCG64(77))
    ref = rng.integers(0, 65536, (2, 2399, 4001), dtype=np.uint16)
    dist = (65535 - ref).astype(np.uint16)
    dist[1] = rng.integers(0, 65536, (2399, 4001), dtype=np.uint16)
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride=4001 * 2 + 38)
    rec = lib.vqx_plane_stats_ordered(pr, pd, 4001, 2399, stride, 16, 2)
    sc, un = orc.batch(rb, db, 4001, 2399, stride, 16, 2)
    assert int(un[0]["noise_units"]) >= 2 ** 53
    check_identical(rec, sc, un)


def test_ordered_is_plain_below_the_limit(lib):
    """Frames whose sums stay below 2^53 units: the same records as
    vqx_plane_stats."""
    w = wl.WORKLOADS["1920x1080_10bit_x48"]
    ref, dist = w.generate([0, 1])
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    a = lib.vqx_plane_stats(pr, pd, w.width, w.height, stride, w.bpc, 2)
    b = lib.vqx_plane_stats_ordered(pr, pd, w.width, w.height, stride, w.bpc, 2)
    assert a.tobytes() == b.tobytes()


def test_ordered_submit_finish_pipelined(lib, orc):
    """Replay batches enqueued back to back, with and without
    VQX_SUBMIT_PLANES_READY, give the blocking call's records; so does a
    batch that needs no replay (submitted as a plain one)."""
    w = wl.WORKLOADS["stress_full_range_4k16"]
    ref, dist = w.generate()
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    want = lib.vqx_plane_stats_ordered(pr, pd, w.width, w.height, stride, 16, 2)
    for flags in (0, lib.VQX_SUBMIT_PLANES_READY):
        pend = [lib.vqx_plane_stats_ordered_submit(pr, pd, w.width, w.height, stride, 16, 2, flags=flags)
                for _ in range(4)]
        for p in pend[::-1]:
            assert p.finish().tobytes() == want.tobytes()
    small = wl.WORKLOADS["1920x1080_10bit_x48"]
    r2, d2 = small.generate([0, 1])
    k2, p2, q2, s2, _ = parity.place(r2, d2)
    p = lib.vqx_plane_stats_ordered_submit(p2, q2, small.width, small.height, s2, 10, 2)
    assert p.finish().tobytes() == lib.vqx_plane_stats(p2, q2, small.width, small.height, s2, 10, 2).tobytes()


def test_headline_batch_pipelined_as_the_benchmark_runs_it(lib, orc):
    """The 3840x2160 16-bit batch as bench.py --op ordered times it: batch
    i + 1 submitted with VQX_SUBMIT_PLANES_READY before batch i is finished
    (its block sums run beside the previous batch's classification, tables
    and walk); every batch equals the oracle's doubles, checked on the first
    and the last (checkerboard) frame."""
    w = wl.WORKLOADS["3840x2160_16bit_x32"]
    ref, dist = w.generate()
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    geo = (w.width, w.height, stride, w.bpc, w.n_frames)
    want = lib.vqx_plane_stats_ordered(pr, pd, *geo)
    sub_r, sub_d = w.generate([0, w.n_frames - 1])
    k2, p2, q2, s2, (r2, d2) = parity.place(sub_r, sub_d)
    sc, un = orc.batch(r2, d2, w.width, w.height, s2, w.bpc, 2)
    check_identical(want[[0, w.n_frames - 1]], sc, un)
    prev = None
    for _ in range(6):
        cur = lib.vqx_plane_stats_ordered_submit(pr, pd, *geo, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            assert prev.finish().tobytes() == want.tobytes()
        prev = cur
    assert prev.finish().tobytes() == want.tobytes()


def test_ordered_at_the_largest_frame(lib, orc):
    """One 8192x4096 16-bit frame pair (2^25 pixels, the largest frame the
    library takes) of full-range noise: the square sums reach about 2^56
    units, so the replay works at ulps up to 2^4, the most any frame needs
    (the block ORs it tests keep at least the terms' low 16 bits)."""
    rng = np.random.Generator(np.random.PCG64(2025))
    ref = rng.integers(0, 1 << 16, (1, 4096, 8192), dtype=np.uint16)
    dist = rng.integers(0, 1 << 16, (1, 4096, 8192), dtype=np.uint16)
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    rec = lib.vqx_plane_stats_ordered(pr, pd, 8192, 4096, stride, 16, 1)
    sc, un = orc.batch(rb, db, 8192, 4096, stride, 16, 1)
    assert int(un[0]["ref_sumsq"]) > 1 << 55
    check_identical(rec, sc, un)



@pytest.mark.parametrize("w,h,n", [(2048, 1026, 3), (2560, 1440, 2), (4096, 520, 5)])
def test_ordered_whole_block_frames_and_partial_units(lib, orc, w, h, n):
    """Dense frames of whole 4096-pixel blocks just above 2^21 pixels and
    beyond: 2048 x 1026 (513 blocks a frame), 2560 x 1440 (900) and
    4096 x 520 (520); bright samples, every other frame a plane against its
    inverse.  Every double equals the oracle's, and the records equal those
    of the same frames on a padded pitch (sample loads row by row)."""
    rng = np.random.Generator(np.random.PCG64(w + h + n))
    ref = rng.integers(50000, 1 << 16, (n, h, w), dtype=np.uint16)
    dist = rng.integers(50000, 1 << 16, (n, h, w), dtype=np.uint16)
    dist[::2] = 65535 - ref[::2]
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    rec = lib.vqx_plane_stats_ordered(pr, pd, w, h, stride, 16, n)
    sc, un = orc.batch(rb, db, w, h, stride, 16, n)
    check_identical(rec, sc, un)
    if w * h > 3_000_000:  # bright enough and large enough to pass 2^53 units
        assert parity.exact_count(un) < n
    keep2, pr2, pd2, stride2, _ = parity.place(ref, dist, stride=2 * w + 32)
    assert lib.vqx_plane_stats_ordered(pr2, pd2, w, h, stride2, 16, n).tobytes() == rec.tobytes()
