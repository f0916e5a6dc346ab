"""Seeded random layouts through every entry point, against the oracle.

Each case draws a bit depth, a frame size, a row padding, base offsets and a
frame count (sometimes enough small frames for the warp-per-frame path), and
checks vqx_plane_stats, vqx_plane_int_psnr, vqx_planes_stats (two planes),
vqx_plane_stats_noalloc and vqx_plane_stats_host on the same planes.  The
integer sums must be equal always, the doubles bit for bit (every case stays
in the exact range: 16-bit frames up to 2^21 pixels).
"""
import numpy as np
import pytest

import parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_CASES = 200


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def draw(seed):
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    bpc = int(rng.choice([8, 10, 12, 16]))
    bps = 1 if bpc == 8 else 2
    kind = rng.integers(0, 4)
    if kind == 0:  # many tiny dense frames
        w, h, n = int(rng.choice([16, 32, 64])), int(rng.choice([8, 16, 32])), int(rng.integers(1200, 2600))
    elif kind == 1:  # mid-size
        w, h, n = int(rng.integers(64, 700)), int(rng.integers(8, 200)), int(rng.integers(1, 6))
    elif kind == 2:  # thin
        w, h, n = int(rng.integers(1, 40)), int(rng.integers(1, 40)), int(rng.integers(1, 20))
    else:  # wide rows
        w, h, n = int(rng.integers(700, 2500)), int(rng.integers(1, 12)), int(rng.integers(1, 4))
    pad = int(rng.choice([0, 0, 0, bps, 16, 48, 2 * bps + 6]))
    off_r = int(rng.choice([0, 0, 16, bps * 3]))
    off_d = int(rng.choice([0, 0, 32, bps]))
    lo = int(rng.choice([0, 0, (1 << bpc) - 300])) if bpc > 8 else 0
    ref = rng.integers(lo, 1 << bpc, (n, h, w)).astype(np.uint8 if bpc == 8 else np.uint16)
    dist = rng.integers(lo, 1 << bpc, (n, h, w)).astype(ref.dtype)
    return bpc, ref, dist, w * bps + pad, off_r, off_d


@pytest.mark.parametrize("seed", range(N_CASES))
def test_fuzz_every_entry_point(lib, orc, seed):
    bpc, ref, dist, stride, off_r, off_d = draw(seed)
    n, h, w = ref.shape
    keep, pr, pd, stride, (rb, db) = parity.place(ref, dist, stride, off_r, off_d)
    sc, un = orc.batch(rb, db, w, h, stride, bpc, n)
    rec = lib.vqx_plane_stats(pr, pd, w, h, stride, bpc, n)
    parity.compare(rec, sc, un, bpc, w * h, planes=(ref, dist))
    # integer psnr
    ip = lib.vqx_plane_int_psnr(pr, pd, w, h, stride, bpc, n)
    want = orc.int_psnr(rb, db, w, h, stride, bpc, n)
    assert [int(x) for x in ip["sse"]] == [int(x) for x in want["sse"]]
    assert ip["psnr"].tobytes() == want["psnr"].tobytes()
    # two planes: the pair and the pair swapped
    two = lib.vqx_planes_stats([(pr, pd, w, h, stride, None), (pd, pr, w, h, stride, None)], bpc, n)
    assert two[:, 0].tobytes() == rec.tobytes()
    assert [int(x) for x in two[:, 1]["noise_units"]] == [int(x) for x in rec["noise_units"]]
    assert two[:, 1]["ref_sum"].tobytes() == rec["dist_sum"].tobytes()
    # no allocation, and planes in host memory
    if 2 * n <= lib.VQX_NOALLOC_MAX_RECORDS:
        assert lib.vqx_plane_stats_noalloc(pr, pd, w, h, stride, bpc, n).tobytes() == rec.tobytes()
    if off_r == 0 and off_d == 0:
        assert lib.vqx_plane_stats_host(rb, db, w, h, stride, bpc, n).tobytes() == rec.tobytes()
