"""Pipelined batches of two different inputs in turn.

Every entry point whose kernels are launched as programmatic dependents
(stage 2 after stage 1, the replay's classification, tables and walk, the
psnr_hvs walk after its tables, and each batch's first kernel after the
batch ahead) is run with batch i + 1 submitted before batch i is finished,
inputs A and B alternating, with and without VQX_SUBMIT_PLANES_READY.  Each
batch's records must equal, byte for byte, those of a blocking call on its
own input, which the parity tests compare with the oracle.  A kernel that
read a buffer before the kernel ahead had finished writing it, or that read
a record the batch ahead left in a reused workspace, returns the other
input's values or garbage instead.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROUNDS = 12


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def planes(seed, n, h, w, lo, hi):
    rng = np.random.Generator(np.random.PCG64(seed))
    ref = rng.integers(lo, hi, (n, h, w), dtype=np.uint16)
    dist = np.clip(ref.astype(np.int64) + rng.integers(-(hi - lo) // 8, (hi - lo) // 8, ref.shape),
                   0, 65535).astype(np.uint16)
    return (torch.from_numpy(ref.view(np.int16)).cuda(), torch.from_numpy(dist.view(np.int16)).cuda())


def as_bytes(rec):
    return b"".join(r.tobytes() for r in rec) if isinstance(rec, tuple) else rec.tobytes()


def alternate(submit, inputs, want, flags):
    prev, prev_k = None, None
    for i in range(ROUNDS):
        k = i % 2
        cur = submit(inputs[k], flags)
        if prev is not None:
            assert as_bytes(prev.finish()) == want[prev_k], (i, prev_k, flags)
        prev, prev_k = cur, k
    assert as_bytes(prev.finish()) == want[prev_k]


@pytest.mark.parametrize("op", ["stats", "int_psnr", "scores"])
@pytest.mark.parametrize("flags", [0, 1])
def test_fused_pass_alternating_inputs(lib, op, flags):
    """1920x1080 16-bit x 12 frames, full range against a narrow band."""
    inputs = [planes(1, 12, 1080, 1920, 0, 65536), planes(2, 12, 1080, 1920, 30000, 31000)]
    blocking = {"stats": lib.vqx_plane_stats, "int_psnr": lib.vqx_plane_int_psnr,
                "scores": lib.vqx_plane_scores}[op]
    submit = {"stats": lib.vqx_plane_stats_submit, "int_psnr": lib.vqx_plane_int_psnr_submit,
              "scores": lib.vqx_plane_scores_submit}[op]
    want = [as_bytes(blocking(r, d, bpc=16)) for r, d in inputs]
    assert want[0] != want[1]
    alternate(lambda x, f: submit(x[0], x[1], bpc=16, flags=f), inputs, want,
              lib.VQX_SUBMIT_PLANES_READY if flags else 0)


@pytest.mark.parametrize("flags", [0, 1])
def test_replay_alternating_inputs(lib, flags):
    """Two 3840x2160 16-bit frames (past 2^21 pixels: classification,
    tables and walk all run), full range against a bright narrow band."""
    inputs = [planes(3, 2, 2160, 3840, 0, 65536), planes(4, 2, 2160, 3840, 60000, 65535)]
    want = [as_bytes(lib.vqx_plane_stats_ordered(r, d, bpc=16)) for r, d in inputs]
    assert want[0] != want[1]
    alternate(lambda x, f: lib.vqx_plane_stats_ordered_submit(x[0], x[1], bpc=16, flags=f), inputs,
              want, lib.VQX_SUBMIT_PLANES_READY if flags else 0)


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("pitch", [1048584, 1048587])
def test_psnr_hvs_alternating_inputs(lib, flags, pitch):
    """Four planes of 1,048,583 terms, on the pipelined tables kernel
    (a pitch of whole vectors) and on the one-CTA-per-node kernel (an odd
    pitch)."""
    n = 1048583
    inputs = []
    for seed in (5, 6):
        rng = np.random.Generator(np.random.PCG64(seed))
        t = np.zeros((4, pitch), np.float32)
        t[:, :n] = rng.uniform(0, 2.0 + 100 * (seed - 5), (4, n)).astype(np.float32)
        t[:, :n][rng.random((4, n)) < 0.5] = 0.0
        inputs.append(torch.from_numpy(t).cuda())
    want = [as_bytes(lib.vqx_psnr_hvs_sum(x, n_terms=n, pitch=pitch, n_planes=4)) for x in inputs]
    assert want[0] != want[1]
    alternate(lambda x, f: lib.vqx_psnr_hvs_sum_submit(x, n_terms=n, pitch=pitch, n_planes=4, flags=f),
              inputs, want, lib.VQX_SUBMIT_PLANES_READY if flags else 0)
