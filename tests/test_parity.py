"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every output of every frame is compared (see ``parity.compare``): the integer
sums always exactly, the scores bit for bit in the exact range and within the
stated bound past it.
"""
import threading

import numpy as np
import pytest

import parity
from exact_full_reference_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_case(lib, orc, ref, dist, bpc, stride=None, offset_ref=0, offset_dist=0):
    n, h, w = ref.shape
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride, offset_ref, offset_dist)
    rec = lib.vqx_plane_stats(pr, pd, w, h, stride, bpc, n)
    torch.cuda.synchronize()
    sc, un = orc.batch(rb, db, w, h, stride, bpc, n)
    parity.compare(rec, sc, un, bpc, w * h, planes=(ref, dist))
    return rec, sc, un


# ------------------------------------------------------------- full workloads
@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_parity(lib, orc, name):
    """The measured configurations at full size (every frame, the launch the
    benchmark times) and the past-2^53 stress frames."""
    w = wl.WORKLOADS[name]
    ref, dist = w.generate()
    rec, sc, un = run_case(lib, orc, ref, dist, w.bpc)
    if name.startswith("stress"):
        # these are chosen to leave the exact range
        assert parity.exact_count(un) < len(un)
    elif w.bpc < 16 or w.width * w.height <= 2 ** 21:
        assert parity.exact_count(un) == len(un)


def test_headline_batch_pipelined_as_the_benchmark_runs_it(lib):
    """The 3840x2160 16-bit batch in the benchmark's launch configuration:
    batch i + 1 submitted with VQX_SUBMIT_PLANES_READY before batch i is
    finished, so consecutive batches' kernels overlap; every batch's records
    equal the blocking call's, which test_workload_parity holds to the
    oracle."""
    w = wl.WORKLOADS[wl.HEADLINE]
    ref, dist = w.generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    geo = (w.width, w.height, stride, w.bpc, w.n_frames)
    want = lib.vqx_plane_stats(pr, pd, *geo).tobytes()
    prev = None
    for _ in range(6):
        cur = lib.vqx_plane_stats_submit(pr, pd, *geo, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            assert prev.finish().tobytes() == want
        prev = cur
    assert prev.finish().tobytes() == want


def test_headline_checkerboard_frame(lib, orc):
    """The checkerboard frame of the 3840x2160 16-bit batch, alone."""
    w = wl.WORKLOADS["3840x2160_16bit_x32"]
    ref, dist = w.generate([w.n_frames - 1])
    rec, sc, un = run_case(lib, orc, ref, dist, 16)
    assert int(rec[0]["noise_units"]) == 3840 * 2160 * 4294836224


# ------------------------------------------------------------- shapes and layouts
SHAPES = [(1, 1), (1, 7), (7, 1), (3, 5), (17, 13), (64, 1), (1, 300), (33, 31), (130, 9),
          (576, 2), (1000, 3), (8, 16), (16, 16), (24, 40)]


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("w,h", SHAPES)
def test_small_shapes_dense(lib, orc, bpc, w, h):
    rng = np.random.Generator(np.random.PCG64(w * 1000 + h * 10 + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (3, h, w)).astype(dt)
    run_case(lib, orc, ref, dist, bpc)


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize(
    "w,h,pad,off_r,off_d",
    [
        (100, 7, 16, 0, 0),     # padded, 16-byte aligned rows: vector path with a tail
        (96, 5, 32, 0, 0),
        (37, 9, 6, 0, 0),       # padded, unaligned rows: scalar path
        (64, 4, 0, 2, 2),       # dense but both bases off a 16-byte boundary
        (64, 4, 0, 0, 6),       # ref aligned, dist not
        (333, 3, 2, 4, 8),
        (1921, 3, 14, 0, 0),
    ],
)
def test_layouts(lib, orc, bpc, w, h, pad, off_r, off_d):
    bps = 1 if bpc == 8 else 2
    rng = np.random.Generator(np.random.PCG64(7 * w + h + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, 1 << bpc, (4, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (4, h, w)).astype(dt)
    if bps == 2:
        pad += pad % 2
    run_case(lib, orc, ref, dist, bpc, stride=w * bps + pad, offset_ref=off_r, offset_dist=off_d)


def test_large_frame_at_the_limit(lib, orc):
    """A single 16-bit frame of exactly 2^25 pixels (8192 x 4096)."""
    rng = np.random.Generator(np.random.PCG64(99))
    ref = rng.integers(0, 1 << 16, (1, 4096, 8192), dtype=np.uint16)
    dist = rng.integers(0, 1 << 16, (1, 4096, 8192), dtype=np.uint16)
    run_case(lib, orc, ref, dist, 16)


def test_many_small_frames(lib, orc):
    rng = np.random.Generator(np.random.PCG64(5))
    ref = rng.integers(0, 1024, (3000, 6, 10)).astype(np.uint16)
    dist = rng.integers(0, 1024, (3000, 6, 10)).astype(np.uint16)
    run_case(lib, orc, ref, dist, 10)


# ------------------------------------------------------------- boundary behaviour
def test_range_flag(lib, orc):
    """A 10-bit frame holding 1024 is flagged; the call reports VQX_ERANGE and
    still fills every record (the integers are the sums of what was read)."""
    rng = np.random.Generator(np.random.PCG64(3))
    ref = rng.integers(0, 1024, (3, 8, 24)).astype(np.uint16)
    dist = rng.integers(0, 1024, (3, 8, 24)).astype(np.uint16)
    ref[1, 5, 7] = 1024
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    rec, rc = lib.vqx_plane_stats(pr, pd, 24, 8, stride, 10, 3, check=False)
    assert rc == lib.VQX_ERANGE
    assert [int(f) for f in rec["flags"]] == [0, 1, 0]
    _, un = orc.batch(rb, db, 24, 8, stride, 10, 3, scores=False)
    for k in parity.UNIT_FIELDS:
        assert [int(x) for x in rec[k]] == [int(x) for x in un[k]]


def test_no_stale_state_between_calls(lib, orc):
    """ADR-1423 (Context, cause 3): a later, larger call must not see an
    earlier call's sums.  Small call, then a larger one on a new stream."""
    a = wl.WORKLOADS["576x324_8bit_x1"]
    ref, dist = a.generate()
    run_case(lib, orc, ref, dist, 8)
    s = torch.cuda.Stream()
    rng = np.random.Generator(np.random.PCG64(17))
    big_r = rng.integers(0, 65536, (5, 1080, 1920), dtype=np.uint16)
    big_d = rng.integers(0, 65536, (5, 1080, 1920), dtype=np.uint16)
    with torch.cuda.stream(s):
        run_case(lib, orc, big_r, big_d, 16)


def test_concurrent_calls_on_two_streams(lib, orc):
    rng = np.random.Generator(np.random.PCG64(21))
    cases = []
    for k in range(2):
        r = rng.integers(0, 4096, (6, 540, 960)).astype(np.uint16)
        d = rng.integers(0, 4096, (6, 540, 960)).astype(np.uint16)
        keep, pr, pd, stride, (rb, db) = parity.place(r, d)
        sc, un = orc.batch(rb, db, 960, 540, stride, 12, 6)
        cases.append((keep, pr, pd, stride, sc, un))
    results = [None, None]

    def worker(k):
        s = torch.cuda.Stream()
        keep, pr, pd, stride, _, _ = cases[k]
        outs = []
        for _ in range(20):
            outs.append(lib.vqx_plane_stats(pr, pd, 960, 540, stride, 12, 6, stream=s.cuda_stream))
        results[k] = outs

    th = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for k in range(2):
        for rec in results[k]:
            parity.compare(rec, cases[k][4], cases[k][5], 12, 960 * 540)


def test_repeat_calls_are_identical(lib):
    w = wl.WORKLOADS["1920x1080_16bit_x64"]
    ref, dist = w.generate(range(8))
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    a = lib.vqx_plane_stats(pr, pd, 1920, 1080, stride, 16, 8)
    b = lib.vqx_plane_stats(pr, pd, 1920, 1080, stride, 16, 8)
    assert a.tobytes() == b.tobytes()


def test_empty_batch(lib):
    rec = lib.vqx_plane_stats(0, 0, 0, 0, 0, 16, 0)
    assert rec.size == 0


def test_host_entry_point_matches(lib, orc):
    """vqx_plane_stats_host (pageable numpy, pinned tensor, padded rows) gives
    the device path's records."""
    w = wl.WORKLOADS["3840x2160_12bit_x32"]
    ref, dist = w.generate(range(6))
    rb, stride = wl.with_layout(ref)
    db, _ = wl.with_layout(dist)
    host = lib.vqx_plane_stats_host(rb, db, 3840, 2160, stride, 12, 6)
    sc, un = orc.batch(rb, db, 3840, 2160, stride, 12, 6)
    parity.compare(host, sc, un, 12, 3840 * 2160)
    pr = torch.from_numpy(rb).pin_memory()
    pdd = torch.from_numpy(db).pin_memory()
    pinned = lib.vqx_plane_stats_host(pr.data_ptr(), pdd.data_ptr(), 3840, 2160, stride, 12, 6)
    assert pinned.tobytes() == host.tobytes()
    rp, stride_p = wl.with_layout(ref[:3], 3840 * 2 + 10)
    dp, _ = wl.with_layout(dist[:3], 3840 * 2 + 10)
    padded = lib.vqx_plane_stats_host(rp, dp, 3840, 2160, stride_p, 12, 3)
    assert padded.tobytes() == host[:3].tobytes()


def test_profile_counts_launches(lib):
    w = wl.WORKLOADS["576x324_8bit_x1"]
    ref, dist = w.generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    lib.profile_enable(True)
    lib.profile_read(reset=True)
    for _ in range(3):
        lib.vqx_plane_stats(pr, pd, 576, 324, stride, 8, 1)
    p = lib.profile_read(reset=True)
    lib.profile_enable(False)
    assert p["calls"] == 3 and p["kernel_launches"] == 6 and p["stage1_launches"] == 3
    assert p["stage1_ms"] > 0 and p["stage1_bytes"] == 3 * 2 * 576 * 324


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
@pytest.mark.parametrize("w,h,pad", [(3840, 2160, 256), (1000, 97, 48), (257, 49, 16), (64, 200, 64),
                                     (1922, 67, 30), (4100, 13, 16), (2052, 3, 40), (4096, 50, 16),
                                     (256, 70, 48), (1024, 33, 16), (1920, 1080, 128)])
def test_padded_aligned_rows(lib, orc, bpc, w, h, pad):
    """Rows on a 16-byte aligned pitch, with padding: bulk copies of row
    pieces where a row is a whole number of 16-byte vectors (and at least
    512 bytes), tensor-map boxes otherwise, including boxes past the last
    column and row (zero-filled by the copy)."""
    bps = 1 if bpc == 8 else 2
    stride = (w * bps + pad + 15) // 16 * 16
    n = 3 if w * h < 1_000_000 else 2
    rng = np.random.Generator(np.random.PCG64(w + 7 * h + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    run_case(lib, orc, ref, dist, bpc, stride=stride)


def test_headline_batch_with_padded_rows(lib, orc):
    """The 3840x2160 16-bit batch with 256 bytes of padding per row."""
    w = wl.WORKLOADS["3840x2160_16bit_x32"]
    ref, dist = w.generate(range(8))
    run_case(lib, orc, ref, dist, 16, stride=3840 * 2 + 256)


def test_submit_finish_matches_the_blocking_call(lib):
    """Batches enqueued back to back (on one stream, then on two) and
    finished in another order give the blocking call's records."""
    rng = np.random.Generator(np.random.PCG64(31))
    cases = []
    for bpc, (n, h, w) in [(16, (4, 540, 960)), (10, (3, 270, 480)), (8, (5, 99, 640))]:
        dt = np.uint8 if bpc == 8 else np.uint16
        ref = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
        dist = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
        keep, pr, pd, stride, _ = parity.place(ref, dist)
        geo = (w, h, stride, bpc, n)
        cases.append((keep, pr, pd, geo, lib.vqx_plane_stats(pr, pd, *geo)))
    pend = [lib.vqx_plane_stats_submit(pr, pd, *geo) for _, pr, pd, geo, _ in cases]
    for k in (2, 0, 1):
        assert pend[k].finish().tobytes() == cases[k][4].tobytes()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    pend = [lib.vqx_plane_stats_submit(pr, pd, *geo, stream=streams[k % 2])
            for k, (_, pr, pd, geo, _) in enumerate(cases * 2)]
    for k in reversed(range(len(pend))):
        assert pend[k].finish().tobytes() == cases[k % 3][4].tobytes()
    with pytest.raises(RuntimeError):
        pend[0].finish()
    # planes written long before: the batches may start reading early
    pend = [lib.vqx_plane_stats_submit(pr, pd, *geo, flags=lib.VQX_SUBMIT_PLANES_READY)
            for _, pr, pd, geo, _ in cases * 3]
    for k, p in enumerate(pend):
        assert p.finish().tobytes() == cases[k % 3][4].tobytes()


def test_submit_profiles_on_the_finishing_thread(lib):
    w = wl.WORKLOADS["576x324_8bit_x1"]
    ref, dist = w.generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    lib.profile_enable(True)
    lib.profile_read(reset=True)
    pend = [lib.vqx_plane_stats_submit(pr, pd, 576, 324, stride, 8, 1) for _ in range(4)]
    for p in pend:
        p.finish()
    prof = lib.profile_read(reset=True)
    lib.profile_enable(False)
    assert prof["calls"] == 4 and prof["stage1_launches"] == 4 and prof["stage1_ms"] > 0


@pytest.mark.parametrize("bpc,w,h,n", [(16, 64, 64, 1300), (8, 96, 64, 2000), (10, 64, 32, 1500),
                                       (12, 32, 48, 1250)])
def test_many_tiny_dense_frames(lib, orc, bpc, w, h, n):
    """Batches of many frames of at most 16 KB per plane: a warp per frame
    (the many-small-frames path), each frame's record written by its warp."""
    rng = np.random.Generator(np.random.PCG64(n + w + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    rec, sc, un = run_case(lib, orc, ref, dist, bpc)
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist)
    ip = lib.vqx_plane_int_psnr(pr, pd, w, h, stride, bpc, n)
    assert [int(x) for x in ip["sse"][:50]] == [int(x) for x in orc.int_psnr(rb, db, w, h, stride, bpc, 50)["sse"]]
    na = lib.vqx_plane_stats_noalloc(pr, pd, w, h, stride, bpc, n)
    assert na.tobytes() == rec.tobytes()


def test_every_kind_from_four_threads(lib, orc):
    """Four threads, four streams, each submitting and finishing its own kind
    of batch (fused, integer psnr, multi-plane, replay) 15 times over; every
    result equals the blocking call's."""
    rng = np.random.Generator(np.random.PCG64(44))
    r16 = rng.integers(0, 65536, (2, 1200, 2000)).astype(np.uint16)  # past 2^21 px: replay
    d16 = rng.integers(0, 65536, (2, 1200, 2000)).astype(np.uint16)
    k16, p16, q16, s16, _ = parity.place(r16, d16)
    r10 = rng.integers(0, 1024, (3, 270, 480)).astype(np.uint16)
    d10 = rng.integers(0, 1024, (3, 270, 480)).astype(np.uint16)
    k10, p10, q10, s10, _ = parity.place(r10, d10)
    descs = [(p10, q10, 480, 270, s10, None), (q10, p10, 480, 270, s10, None)]
    jobs = {
        "stats": (lambda st: lib.vqx_plane_stats_submit(p10, q10, 480, 270, s10, 10, 3, stream=st),
                  lib.vqx_plane_stats(p10, q10, 480, 270, s10, 10, 3)),
        "int_psnr": (lambda st: lib.vqx_plane_int_psnr_submit(p16, q16, 2000, 1200, s16, 16, 2, stream=st),
                     lib.vqx_plane_int_psnr(p16, q16, 2000, 1200, s16, 16, 2)),
        "planes": (lambda st: lib.vqx_planes_stats_submit(descs, 10, 3, stream=st),
                   lib.vqx_planes_stats(descs, 10, 3)),
        "ordered": (lambda st: lib.vqx_plane_stats_ordered_submit(p16, q16, 2000, 1200, s16, 16, 2,
                                                                  stream=st),
                    lib.vqx_plane_stats_ordered(p16, q16, 2000, 1200, s16, 16, 2)),
    }
    torch.cuda.synchronize()
    bad = []

    def worker(name):
        submit, want = jobs[name]
        st = torch.cuda.Stream()
        pend = []
        for i in range(15):
            pend.append(submit(st))
            if i % 3 == 2:  # keep a few in flight, finish out of order
                for p in pend[::-1]:
                    if p.finish().tobytes() != want.tobytes():
                        bad.append(name)
                pend = []
        for p in pend:
            if p.finish().tobytes() != want.tobytes():
                bad.append(name)

    th = [threading.Thread(target=worker, args=(k,)) for k in jobs]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not bad, bad


@pytest.mark.parametrize("w,h,bpc,n", [(512, 512, 16, 400), (512, 512, 8, 400), (1920, 1080, 16, 64),
                                       (1920, 1080, 12, 70), (2000, 1000, 10, 5)])
def test_dense_batches_against_padded_pitches(lib, orc, w, h, bpc, n):
    """Batches of many mid-size dense frames (512x512 x400: more frames than
    CTAs, units of whole frames) and of few large ones: every frame's records
    equal the oracle's and those of the same frames on a padded pitch (row
    pieces instead of whole-frame copies); so do the integer psnr and the
    one-read scores."""
    rng = np.random.Generator(np.random.PCG64(w + 7 * n + bpc))
    dt = np.uint8 if bpc == 8 else np.uint16
    bps = 1 if bpc == 8 else 2
    ref = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bpc, (n, h, w)).astype(dt)
    rec, sc, un = run_case(lib, orc, ref, dist, bpc)
    keep, pr, pd, stride, _ = parity.place(ref, dist, stride=w * bps + 32)
    assert lib.vqx_plane_stats(pr, pd, w, h, stride, bpc, n).tobytes() == rec.tobytes()
    keep2, pr2, pd2, stride2, _ = parity.place(ref, dist)
    ip = lib.vqx_plane_int_psnr(pr2, pd2, w, h, stride2, bpc, n)
    assert ip.tobytes() == lib.vqx_plane_int_psnr(pr, pd, w, h, stride, bpc, n).tobytes()
    st, ip2 = lib.vqx_plane_scores(pr2, pd2, w, h, stride2, bpc, n)
    assert st.tobytes() == rec.tobytes() and ip2.tobytes() == ip.tobytes()
