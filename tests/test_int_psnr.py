"""GPU parity of the integer psnr (vqx_plane_int_psnr) against the oracle.

The SSE is an integer and must equal the oracle's exactly; the MSE and the
PSNRs are the same double operations on the same integer and must be equal
bit for bit, on every frame.
"""
import numpy as np
import pytest

import parity
from exact_full_reference_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FIELDS = ("mse", "psnr", "psnr_uncapped")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def compare(rec, want):
    assert len(rec) == len(want)
    for f in range(len(rec)):
        assert int(rec[f]["sse"]) == int(want[f]["sse"]), (f, int(rec[f]["sse"]), int(want[f]["sse"]))
        for k in FIELDS:
            assert rec[f][k].tobytes() == want[f][k].tobytes(), (f, k, rec[f][k], want[f][k])
        assert int(rec[f]["reserved"]) == 0


def run_case(lib, orc, ref, dist, bpc, stride=None, offset_ref=0, offset_dist=0):
    n, h, w = ref.shape
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride, offset_ref, offset_dist)
    rec = lib.vqx_plane_int_psnr(pr, pd, w, h, stride, bpc, n)
    torch.cuda.synchronize()
    compare(rec, orc.int_psnr(rb, db, w, h, stride, bpc, n))
    assert not rec["flags"].any()
    return rec


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_int_psnr(lib, orc, name):
    """Every frame of every workload (the past-2^53 stress frames too: the
    SSE is an integer, exact at any size)."""
    w = wl.WORKLOADS[name]
    ref, dist = w.generate()
    run_case(lib, orc, ref, dist, w.bpc)


def test_full_range_16bit_frames(lib, orc):
    """Full-range 16-bit differences (the float squares round; the SSE must
    not) and the inverse plane (differences up to 65535)."""
    w = wl.WORKLOADS["stress_inverse_4k16"]
    ref, dist = w.generate()
    rec = run_case(lib, orc, ref, dist, 16)
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    fl = lib.vqx_plane_stats(pr, pd, 3840, 2160, stride, 16, len(ref))
    assert (rec["sse"] != fl["noise_units"]).all()  # the float squares drop bits here


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("w,h,pad", [(1, 1, 0), (7, 3, 0), (333, 17, 0), (1000, 97, 48), (1922, 67, 30),
                                     (257, 49, 16), (37, 9, 6), (3840, 64, 256)])
def test_shapes_and_layouts(lib, orc, bpc, w, h, pad):
    """Dense frames, padded rows (row pieces, boxes) and unaligned pitches."""
    rng = np.random.Generator(np.random.PCG64(11 * w + h + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    bps = 1 if bpc == 8 else 2
    ref = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    pad += pad % bps
    run_case(lib, orc, ref, dist, bpc, stride=w * bps + pad if pad else None)


def test_identical_planes_and_cap(lib, orc):
    for bpc in (8, 10, 12, 16):
        dt = np.uint8 if bpc == 8 else np.uint16
        ref = np.random.Generator(np.random.PCG64(bpc)).integers(0, 1 << bpc, (2, 64, 96)).astype(dt)
        rec = run_case(lib, orc, ref, ref.copy(), bpc)
        assert (rec["sse"] == 0).all() and (rec["psnr"] == lib.psnr_cap(bpc)).all()
        assert np.isinf(rec["psnr_uncapped"]).all()


def test_range_flag_10bit(lib, orc):
    rng = np.random.Generator(np.random.PCG64(9))
    ref = rng.integers(0, 1024, (3, 8, 40)).astype(np.uint16)
    dist = rng.integers(0, 1024, (3, 8, 40)).astype(np.uint16)
    dist[2, 1, 1] = 2000
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    rec, rc = lib.vqx_plane_int_psnr(pr, pd, 40, 8, stride, 10, 3, check=False)
    assert rc == lib.VQX_ERANGE and [int(x) for x in rec["flags"]] == [0, 0, 1]


def test_submit_finish_and_kind_check(lib, orc):
    w = wl.WORKLOADS["1920x1080_16bit_x64"]
    ref, dist = w.generate(range(6))
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    want = orc.int_psnr(rb, db, 1920, 1080, stride, 16, 6)
    pend = [lib.vqx_plane_int_psnr_submit(pr, pd, 1920, 1080, stride, 16, 6) for _ in range(3)]
    for p in reversed(pend):
        compare(p.finish(), want)
    # a handle of the other kind is refused (and released)
    p = lib.vqx_plane_stats_submit(pr, pd, 1920, 1080, stride, 16, 6)
    p.kind = "int_psnr"
    out, rc = p.finish(check=False)
    assert rc == lib.VQX_EINVAL


def test_headline_batch_pipelined_as_the_benchmark_runs_it(lib, orc):
    """The 3840x2160 16-bit batch as bench.py --op int_psnr times it: batch
    i + 1 submitted with VQX_SUBMIT_PLANES_READY before batch i is finished;
    every batch equals the blocking call, whose SSE and doubles equal the
    oracle's on the first and last frame."""
    w = wl.WORKLOADS["3840x2160_16bit_x32"]
    ref, dist = w.generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    geo = (w.width, w.height, stride, w.bpc, w.n_frames)
    want = lib.vqx_plane_int_psnr(pr, pd, *geo)
    oracle_rec = orc.int_psnr_frames(ref[[0, -1]], dist[[0, -1]], w.bpc)
    for i, f in enumerate((0, w.n_frames - 1)):
        assert int(want[f]["sse"]) == int(oracle_rec[i]["sse"])
        assert want[f]["psnr"] == oracle_rec[i]["psnr"] and want[f]["mse"] == oracle_rec[i]["mse"]
    prev = None
    for _ in range(6):
        cur = lib.vqx_plane_int_psnr_submit(pr, pd, *geo, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            assert prev.finish().tobytes() == want.tobytes()
        prev = cur
    assert prev.finish().tobytes() == want.tobytes()

