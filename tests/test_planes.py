"""vqx_planes_stats: every plane of every frame in one call, against the
oracle plane by plane and against vqx_plane_stats on the same plane."""
import numpy as np
import pytest

import parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def yuv_frames(rng, n, w, h, cw, ch, bpc):
    """n frames of three planes (w x h luma, cw x ch chroma), reference and
    a lightly distorted copy."""
    dt = np.uint8 if bpc == 8 else np.uint16
    top = (1 << bpc) - 1
    planes = []
    for pw, ph in ((w, h), (cw, ch), (cw, ch)):
        ref = rng.integers(0, top + 1, (n, ph, pw)).astype(np.int64)
        dist = np.clip(ref + np.rint(rng.normal(0, 3 << max(bpc - 8, 0), ref.shape)).astype(np.int64), 0, top)
        planes.append((ref.astype(dt), dist.astype(dt)))
    return planes


def check_against_oracle(rec, orc, layouts, bpc, n):
    """layouts[p] = (ref bytes, dist bytes, offset, w, h, stride, pitch)."""
    for p, (rb, db, off, w, h, stride, pitch) in enumerate(layouts):
        for f in range(n):
            sc, un = orc.batch(rb, db, w, h, stride, bpc, 1, offset=off + f * pitch)
            parity.compare(rec[f : f + 1, p], sc, un, bpc, w * h)


@pytest.mark.parametrize("bpc,w,h,cw,ch", [(10, 576, 324, 288, 162), (10, 576, 324, 288, 324),
                                           (8, 333, 17, 167, 17), (16, 1920, 1080, 960, 540),
                                           (12, 64, 48, 32, 24)])
def test_separate_plane_buffers(lib, orc, bpc, w, h, cw, ch):
    """Y, Cb and Cr each in their own buffer of back-to-back frames (4:2:0,
    4:2:2, odd widths)."""
    rng = np.random.Generator(np.random.PCG64(w * h + bpc))
    n = 3
    planes = yuv_frames(rng, n, w, h, cw, ch, bpc)
    keep, descs, layouts = [], [], []
    for ref, dist in planes:
        k, pr, pd, stride, (rb, db) = parity.place(ref, dist)
        keep.append(k)
        ph, pw = ref.shape[1:]
        descs.append((pr, pd, pw, ph, stride, 0))
        layouts.append((rb, db, 0, pw, ph, stride, ph * stride))
    rec = lib.vqx_planes_stats(descs, bpc, n)
    assert rec.shape == (n, 3)
    check_against_oracle(rec, orc, layouts, bpc, n)
    for p, (pr, pd, pw, ph, stride, _) in enumerate(descs):
        alone = lib.vqx_plane_stats(pr, pd, pw, ph, stride, bpc, n)
        assert rec[:, p].tobytes() == alone.tobytes()


@pytest.mark.parametrize("bpc,w,h,cw,ch,pad,align", [(10, 576, 324, 288, 162, 0, True),
                                                     (16, 3840, 64, 1920, 32, 64, True),
                                                     (8, 200, 40, 100, 20, 16, True),
                                                     (10, 130, 9, 65, 5, 6, True),
                                                     (8, 33, 7, 17, 4, 3, False)])
def test_planes_interleaved_in_each_frame(lib, orc, bpc, w, h, cw, ch, pad, align):
    """One buffer per video: frame f holds Y, then Cb, then Cr (rows padded
    by pad bytes, rounded up to 16 with align); each plane's frame pitch is
    the whole frame.  Covers row pieces, tensor-map boxes and sample loads
    with frames that are not back to back."""
    rng = np.random.Generator(np.random.PCG64(3 * w + h + bpc))
    n = 3
    bps = 1 if bpc == 8 else 2
    planes = yuv_frames(rng, n, w, h, cw, ch, bpc)
    strides = [pw * bps + pad for pw in (w, cw, cw)]
    if align:
        strides = [(x + 15) // 16 * 16 for x in strides]
    offs = [0, h * strides[0], h * strides[0] + ch * strides[1]]
    pitch = offs[2] + ch * strides[2]
    pitch += (-pitch) % 16
    bufs = []
    for side in (0, 1):
        buf = np.full(n * pitch, 0xA5, np.uint8)
        for p, (pw, ph) in enumerate(((w, h), (cw, ch), (cw, ch))):
            for f in range(n):
                for y in range(ph):
                    a = f * pitch + offs[p] + y * strides[p]
                    buf[a : a + pw * bps] = planes[p][side][f, y].view(np.uint8)
        bufs.append(buf)
    tr, base_r = parity.device_bytes(bufs[0])
    td, base_d = parity.device_bytes(bufs[1])
    descs = [(base_r + offs[p], base_d + offs[p], pw, ph, strides[p], pitch)
             for p, (pw, ph) in enumerate(((w, h), (cw, ch), (cw, ch)))]
    rec = lib.vqx_planes_stats(descs, bpc, n)
    layouts = [(bufs[0], bufs[1], offs[p], pw, ph, strides[p], pitch)
               for p, (pw, ph) in enumerate(((w, h), (cw, ch), (cw, ch)))]
    check_against_oracle(rec, orc, layouts, bpc, n)


def test_one_plane_is_vqx_plane_stats(lib, orc):
    rng = np.random.Generator(np.random.PCG64(8))
    ref = rng.integers(0, 4096, (4, 270, 480)).astype(np.uint16)
    dist = rng.integers(0, 4096, (4, 270, 480)).astype(np.uint16)
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    rec = lib.vqx_planes_stats([(pr, pd, 480, 270, stride, None)], 12, 4)
    assert rec[:, 0].tobytes() == lib.vqx_plane_stats(pr, pd, 480, 270, stride, 12, 4).tobytes()


def test_planes_submit_finish(lib, orc):
    """The two-half form: batches enqueued back to back (with and without
    VQX_SUBMIT_PLANES_READY) give the blocking call's records; a handle of
    another kind is refused."""
    rng = np.random.Generator(np.random.PCG64(12))
    planes = yuv_frames(rng, 4, 576, 324, 288, 162, 10)
    keep, descs = [], []
    for ref, dist in planes:
        k, pr, pd, stride, _ = parity.place(ref, dist)
        keep.append(k)
        descs.append((pr, pd, ref.shape[2], ref.shape[1], stride, 0))
    want = lib.vqx_planes_stats(descs, 10, 4)
    for flags in (0, lib.VQX_SUBMIT_PLANES_READY):
        pend = [lib.vqx_planes_stats_submit(descs, 10, 4, flags=flags) for _ in range(3)]
        for p in reversed(pend):
            assert p.finish().tobytes() == want.tobytes()
    p = lib.vqx_planes_stats_submit(descs, 10, 4)
    p.kind, p.shape = "stats", 4
    out, rc = p.finish(check=False)
    assert rc == lib.VQX_EINVAL


def test_headline_planes_pipelined_as_the_benchmark_runs_it(lib, orc):
    """Y, Cb and Cr of the 3840x2160 16-bit batch (the chroma planes at half
    size, the same content recipe, their own seeds) as bench.py --op
    planes420 times them: batch i + 1 submitted with VQX_SUBMIT_PLANES_READY
    before batch i is finished.  Every batch equals the blocking call, whose
    records equal vqx_plane_stats plane by plane and the oracle on the first
    and last frame of each plane."""
    import dataclasses

    from exact_full_reference_gb300 import workloads as wl

    w = wl.WORKLOADS[wl.HEADLINE]
    chroma = [dataclasses.replace(w, name=w.name + "_c%d" % k, width=w.width // 2,
                                  height=w.height // 2, seed=w.seed + 1000 * k) for k in (1, 2)]
    keep, descs, frames = [], [], []
    for p_w in [w] + chroma:
        ref, dist = p_w.generate()
        k, pr, pd, stride, (rb, db) = parity.place(ref, dist)
        keep.append(k)
        descs.append((pr, pd, p_w.width, p_w.height, stride, 0))
        frames.append((ref, dist, rb, db, stride, p_w))
    n = w.n_frames
    want = lib.vqx_planes_stats(descs, 16, n)
    for q, (ref, dist, rb, db, stride, p_w) in enumerate(frames):
        plain = lib.vqx_plane_stats(descs[q][0], descs[q][1], p_w.width, p_w.height, stride, 16, n)
        assert want[:, q].tobytes() == plain.tobytes(), q
        sc, un = orc.frames(ref[[0, n - 1]], dist[[0, n - 1]], 16)
        for i, f in enumerate((0, n - 1)):
            for k_u in parity.UNIT_FIELDS:
                assert int(want[f, q][k_u]) == int(un[i][k_u]), (q, f, k_u)
    prev = None
    for _ in range(6):
        cur = lib.vqx_planes_stats_submit(descs, 16, n, flags=lib.VQX_SUBMIT_PLANES_READY)
        if prev is not None:
            assert prev.finish().tobytes() == want.tobytes()
        prev = cur
    assert prev.finish().tobytes() == want.tobytes()

