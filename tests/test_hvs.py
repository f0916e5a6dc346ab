"""GPU parity of the psnr_hvs plane sum (vqx_psnr_hvs_sum) against the oracle.

"ADR-1397: GPU psnr_hvs twins reproduce the CPU's running float sum bit for
bit" makes the comparison an equality: the device's sum and score must equal
the oracle's floats bit for bit, on every plane.
"""
import numpy as np
import pytest

from exact_full_reference_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_device(buf, offset_floats=0):
    """float32 host array -> device copy whose first float sits
    ``offset_floats`` floats past a 256-byte boundary.  Returns (keep, ptr)."""
    flat = np.ascontiguousarray(buf, np.float32).reshape(-1)
    t = torch.empty(flat.size + 64 + offset_floats, dtype=torch.float32, device="cuda")
    start = ((-t.data_ptr()) % 256) // 4 + offset_floats
    t[start : start + flat.size].copy_(torch.from_numpy(flat))
    return t, t.data_ptr() + 4 * start


def check(lib, orc, planes, bpc=8, n_terms=None, pitch=None, offset_floats=0):
    planes = np.atleast_2d(np.asarray(planes, np.float32))
    n_planes, width = planes.shape
    pitch = width if pitch is None else pitch
    n_terms = width if n_terms is None else n_terms
    buf = np.full((n_planes, pitch), np.nan, np.float32)  # padding would poison any sum
    buf[:, :n_terms] = planes[:, :n_terms]
    keep, ptr = to_device(buf, offset_floats)
    rec = lib.vqx_psnr_hvs_sum(ptr, n_terms, pitch, n_planes, bpc)
    torch.cuda.synchronize()
    sums, scores = orc.hvs(buf, bpc, n_terms=n_terms, pitch=pitch, n_planes=n_planes)
    for p in range(n_planes):
        assert rec[p]["sum"].tobytes() == sums[p].tobytes(), (p, rec[p]["sum"], sums[p])
        assert rec[p]["score"].tobytes() == scores[p].tobytes(), (p, rec[p]["score"], scores[p])
    assert not rec["flags"].any()
    return rec


@pytest.mark.parametrize("name", ["hvs_576x324_8bit_x4", "hvs_1920x1080_10bit_x4",
                                  "hvs_3840x2160_10bit_x2", "hvs_ones_2e24", "hvs_ties",
                                  "hvs_drift", "hvs_subnormal", "hvs_wide", "hvs_zeros"])
def test_workload_parity(lib, orc, name):
    w = wl.HVS_WORKLOADS[name]
    check(lib, orc, w.generate(), w.bpc)


def test_headline_batch_every_plane(lib, orc):
    """The 3840x2160 batch of 32 planes, in the launch the benchmark times."""
    w = wl.HVS_WORKLOADS[wl.HVS_HEADLINE]
    rec = check(lib, orc, w.generate(), w.bpc)
    # the guesses hold: under 1 % of the leaves are walked run by run
    leaves = -(-w.n_terms // 1024)
    assert rec["replayed_leaves"].max() < leaves // 100, rec["replayed_leaves"]


def test_headline_batch_pipelined_as_the_benchmark_runs_it(lib, orc):
    """The 3840x2160 batch of 32 planes as the benchmark times it: batch i + 1
    submitted with VQX_SUBMIT_PLANES_READY before batch i is finished, so the
    next batch's tables run beside this batch's walk; every batch equals the
    oracle bit for bit."""
    w = wl.HVS_WORKLOADS[wl.HVS_HEADLINE]
    t = w.generate()
    dev = torch.from_numpy(t).cuda()
    torch.cuda.synchronize()
    sums, scores = orc.hvs(t, w.bpc)
    prev = None
    for _ in range(6):
        cur = lib.vqx_psnr_hvs_sum_submit(dev, bpc=w.bpc, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            rec = prev.finish()
            assert rec["sum"].tobytes() == sums.tobytes() and rec["score"].tobytes() == scores.tobytes()
        prev = cur
    rec = prev.finish()
    assert rec["sum"].tobytes() == sums.tobytes() and rec["score"].tobytes() == scores.tobytes()


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
def test_score_at_every_depth(lib, orc, bpc):
    w = wl.HVS_WORKLOADS["hvs_576x324_8bit_x4"]
    check(lib, orc, w.generate([0, 1]), bpc)


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 1023, 1024, 1025, 8191, 8192, 8193, 16383, 16384, 16385,
                               16384 * 33 + 7, 16384 * 32 * 3 + 1024 * 5 + 3])
def test_ragged_lengths(lib, orc, n):
    rng = np.random.default_rng(n)
    t = wl.HvsWorkload("r", 0, 0, 8, 2, n, "masked", n_terms_override=n).generate()
    t[1] = rng.uniform(0, 3, n).astype(np.float32)
    check(lib, orc, t)


@pytest.mark.parametrize("offset,pitch_extra", [(0, 0), (0, 5), (1, 0), (3, 4), (2, 13)])
def test_layouts_wide_and_scalar_loads(lib, orc, offset, pitch_extra):
    """16-byte aligned planes with a pitch of whole vectors take 16-byte
    loads, anything else single floats; padding (NaN) is never read."""
    w = wl.HvsWorkload("l", 0, 0, 8, 3, 50 + offset, "masked", n_terms_override=70001)
    t = w.generate()
    check(lib, orc, t, n_terms=t.shape[1], pitch=t.shape[1] + pitch_extra, offset_floats=offset)


@pytest.mark.parametrize("n,extra", [(36, 0), (1052, 4), (8220, 0), (16400, 12), (65540, 4),
                                     (540696, 8), (1577988, 0)])
def test_pipeline_partial_rows(lib, orc, n, extra):
    """16-byte aligned planes with a pitch of whole vectors stream through the
    persistent pipeline in boxes of full 32-term rows; a plane whose length is
    not a multiple of 32 ends in a partial row that no box holds (the lane
    whose run it is reads it itself).  NaN padding after every plane would
    poison any sum that read past the plane's end."""
    rng = np.random.default_rng(n)
    t = rng.uniform(0, 5, (3, n)).astype(np.float32)
    t[rng.random(t.shape) < 0.6] = 0.0
    check(lib, orc, t, n_terms=n, pitch=n + extra)


def test_pipeline_many_planes_with_partial_rows(lib, orc):
    """500 planes of 1028 terms (one node each, four terms past the last full
    row) through the pipeline: nodes of many planes interleave in every CTA."""
    rng = np.random.default_rng(11)
    t = rng.uniform(0, 1000, (500, 1028)).astype(np.float32)
    t[rng.random(t.shape) < 0.7] = 0.0
    check(lib, orc, t, n_terms=1028, pitch=1032)


@pytest.mark.parametrize("where", ["row", "partial_row"])
def test_pipeline_term_outside_the_domain(lib, orc, where):
    """A negative term in a full row or in the partial last row flags its
    plane on the pipelined path too; the other planes are unaffected."""
    n = 70004
    rng = np.random.default_rng(5)
    t = rng.uniform(0, 3, (3, n)).astype(np.float32)
    t[1, 31337 if where == "row" else n - 2] = -1.0
    keep, ptr = to_device(t)
    rec, rc = lib.vqx_psnr_hvs_sum(ptr, n, n, 3, 8, check=False)
    torch.cuda.synchronize()
    assert rc == lib.VQX_ERANGE
    assert list(rec["flags"]) == [0, lib.VQX_FLAG_RANGE, 0]
    sums, scores = orc.hvs(t[[0, 2]], 8)
    assert rec[0]["sum"].tobytes() == sums[0].tobytes()
    assert rec[2]["sum"].tobytes() == sums[1].tobytes()


def test_one_plane_with_a_huge_pitch(lib, orc):
    """With one plane the pitch is never stepped over: a pitch of 2^40 floats
    (far more memory than exists) must not matter on the pipelined path."""
    rng = np.random.default_rng(17)
    t = rng.uniform(0, 4, (1, 40004)).astype(np.float32)
    t[rng.random(t.shape) < 0.5] = 0.0
    keep, ptr = to_device(t)
    rec = lib.vqx_psnr_hvs_sum(ptr, t.shape[1], 1 << 40, 1, 8)
    torch.cuda.synchronize()
    sums, scores = orc.hvs(t, 8)
    assert rec["sum"].tobytes() == sums.tobytes() and rec["score"].tobytes() == scores.tobytes()


def test_one_very_long_plane(lib, orc):
    """2^27 terms in one plane (16384 nodes, 4 Mi rows of 32): the row and
    node coordinates of the pipelined path at a large scale."""
    rng = np.random.default_rng(23)
    n = (1 << 27) + 12
    t = rng.uniform(0, 2, n).astype(np.float32)
    t[rng.random(n) < 0.7] = 0.0
    dev = torch.from_numpy(t).cuda()
    rec = lib.vqx_psnr_hvs_sum(dev, bpc=8)
    sums, scores = orc.hvs(t, 8)
    assert rec["sum"].tobytes() == sums.tobytes() and rec["score"].tobytes() == scores.tobytes()


@pytest.mark.parametrize("growth", [2.0, 1.3, "steps"])
def test_walk_crossings_node_after_node(lib, orc, growth):
    """Sums that cross a power of two in node after node (growth 2: every
    node of 8192 terms, over 80 nodes; 1.3: most, over 200; "steps": bursts
    every fifth node, over 200): windows where many nodes are walked leaf by
    leaf in turn, each window rescanned from the node after the last one
    walked, across the walk's register blocks of 64 nodes."""
    rng = np.random.default_rng(41)
    nodes, node = (80 if growth == 2.0 else 200), 8192
    k = np.repeat(np.arange(nodes), node).astype(np.float64)
    if growth == "steps":
        scale = np.where(k % 5 == 0, 2.0 ** (k / 5.0), 2.0 ** (k / 5.0) / 64.0)
    else:
        scale = growth ** k
    t = np.empty((3, nodes * node), np.float32)
    for p in range(3):
        t[p] = (scale * rng.uniform(0.25, 1.0, nodes * node) / node).astype(np.float32)
    t[:, rng.random(t.shape[1]) < 0.3] = 0.0
    rec = check(lib, orc, t)
    assert (rec["replayed_leaves"] > 0).all()


def test_many_small_planes(lib, orc):
    """3000 planes of 37 terms: one node each, 3000 walks."""
    rng = np.random.default_rng(7)
    t = rng.uniform(0, 1000, (3000, 37)).astype(np.float32)
    t[rng.random(t.shape) < 0.7] = 0.0
    check(lib, orc, t)


def test_largest_terms(lib, orc):
    """Terms just below 2^95 and the negative zero are inside the domain."""
    rng = np.random.default_rng(3)
    t = (rng.uniform(0.5, 1.0, 5000) * 2.0 ** 95).astype(np.float32)
    t = np.minimum(t, np.float32(np.nextafter(np.float32(2.0 ** 95), np.float32(0))))
    t[::7] = -0.0
    check(lib, orc, t)


@pytest.mark.parametrize("bad", [-1.0, np.nan, np.inf, 2.0 ** 95, -np.inf])
def test_terms_outside_the_domain(lib, orc, bad):
    """A plane with a negative, NaN, infinite or too large term is flagged and
    gets NaN results; the other planes are unaffected; the status is
    VQX_ERANGE."""
    w = wl.HvsWorkload("b", 0, 0, 8, 3, 9, "masked", n_terms_override=50000)
    t = w.generate()
    t[1, 31337] = bad
    keep, ptr = to_device(t)
    rec, rc = lib.vqx_psnr_hvs_sum(ptr, t.shape[1], t.shape[1], 3, 8, check=False)
    torch.cuda.synchronize()
    assert rc == lib.VQX_ERANGE
    assert list(rec["flags"]) == [0, lib.VQX_FLAG_RANGE, 0]
    assert np.isnan(rec[1]["sum"]) and np.isnan(rec[1]["score"])
    sums, scores = orc.hvs(t[[0, 2]], 8)
    assert rec[0]["sum"].tobytes() == sums[0].tobytes()
    assert rec[2]["sum"].tobytes() == sums[1].tobytes()


def test_submit_finish_overlapping_batches(lib, orc):
    """Two batches in flight on two streams, finished in reverse order."""
    a = wl.HVS_WORKLOADS["hvs_ties"].generate()
    b = wl.HVS_WORKLOADS["hvs_wide"].generate()
    ka, pa = to_device(a)
    kb, pb = to_device(b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ha = lib.vqx_psnr_hvs_sum_submit(pa, a.shape[1], a.shape[1], a.shape[0], 8, stream=s1)
    hb = lib.vqx_psnr_hvs_sum_submit(pb, b.shape[1], b.shape[1], b.shape[0], 10, stream=s2)
    rb = hb.finish()
    ra = ha.finish()
    for rec, t, bpc in ((ra, a, 8), (rb, b, 10)):
        sums, scores = orc.hvs(t, bpc)
        assert rec["sum"].tobytes() == sums.tobytes()
        assert rec["score"].tobytes() == scores.tobytes()


def test_tensor_geometry(lib, orc):
    """A (planes, n) CUDA tensor needs no explicit sizes."""
    t = wl.HVS_WORKLOADS["hvs_576x324_8bit_x4"].generate()
    dev = torch.from_numpy(t).cuda()
    rec = lib.vqx_psnr_hvs_sum(dev, bpc=8)
    sums, scores = orc.hvs(t, 8)
    assert rec["sum"].tobytes() == sums.tobytes() and rec["score"].tobytes() == scores.tobytes()
