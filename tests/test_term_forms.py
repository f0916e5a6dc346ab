"""The library's conversion-free accumulators against the literal per-pixel
form, on the GPU, for every sample pair of every bit depth.

The accumulators (vqx::TermSums<bpc>, and at 16 bits vqx::TermSums16Sse, which
also carries the exact SSE) replace the literal arithmetic (convert to fp32,
subtract, square with round to nearest even, convert back; for the SSE the
integer square) by forms the source argues are value-identical.  This test
runs both on the device, for each reference value against every distorted
value (2^32 pairs at 16 bits), through the vector path and the per-sample
path, and on random word streams that cross many flush boundaries.  The sums
must be equal.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "term_forms.cu")
OUT = os.path.join(HERE, "_build", "libvqx_term_forms.so")


def build_test_library():
    from exact_full_reference_gb300 import build as vb

    deps = [SRC, os.path.join(vb.CSRC, "vqx_kernels.cuh")]
    if os.path.exists(OUT) and all(os.path.getmtime(d) <= os.path.getmtime(OUT) for d in deps):
        return OUT
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    tmp = OUT + ".tmp%d" % os.getpid()
    subprocess.run([vb.nvcc(), vb.ARCH, "-O3", "-std=c++17", "--fmad=false", "-shared",
                    "-Xcompiler=-fPIC", "-I" + vb.CSRC, "-o", tmp, SRC], check=True)
    os.replace(tmp, OUT)
    return OUT


@pytest.fixture(scope="module")
def tf():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctypes.CDLL(build_test_library())
    u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
    lib.vqx_test_exhaustive.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, u64p, u64p]
    lib.vqx_test_exhaustive.restype = ctypes.c_int
    lib.vqx_test_stream.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_uint, ctypes.c_uint, u64p, u64p]
    lib.vqx_test_stream.restype = ctypes.c_int
    lib.vqx_test_wait_timeout.argtypes = [ctypes.c_longlong, np.ctypeslib.ndpointer(np.int64)]
    lib.vqx_test_wait_timeout.restype = ctypes.c_int
    return lib


FIELDS = ["noise", "ref_sum", "dist_sum", "ref_sumsq", "dist_sumsq", "or", "sse-noise", "zero"]
W = len(FIELDS)


def assert_same(fast, lit, bpc, what, sse=False):
    fast = fast.reshape(-1, W)
    lit = lit.reshape(-1, W)
    cols = [0, 1, 2, 3, 4] + ([5] if bpc in (10, 12) else []) + ([6] if sse else [])
    # the last word is always 0; without the SSE form word 6 is 0 too, which
    # is the SSE up to 12 bits, where the float squares are exact (the
    # literal difference is 0 there as well)
    assert not fast[:, 7].any()
    if not sse:
        assert not fast[:, 6].any()
        if bpc <= 12:
            assert not lit[:, 6].any()
    for c in cols:
        bad = np.nonzero(fast[:, c] != lit[:, c])[0]
        assert bad.size == 0, "%s bpc=%d %s: %d threads differ, first %d: %d vs %d" % (
            what, bpc, FIELDS[c], bad.size, bad[0], int(fast[bad[0], c]), int(lit[bad[0], c]))


@pytest.mark.parametrize("use_samples", [0, 1], ids=["vec", "sample"])
@pytest.mark.parametrize("bpc,sse", [(8, 0), (10, 0), (12, 0), (16, 0), (16, 1)],
                         ids=["8", "10", "12", "16", "16sse"])
def test_every_sample_pair(tf, bpc, sse, use_samples):
    n = W << bpc
    fast = np.zeros(n, np.uint64)
    lit = np.zeros(n, np.uint64)
    assert tf.vqx_test_exhaustive(bpc, use_samples, sse, fast, lit) == 0
    assert_same(fast, lit, bpc, "exhaustive", bool(sse))
    assert lit.reshape(-1, W)[:, 0].sum() > 0
    if sse:  # 16-bit squares from 4097^2 on round: the difference is not trivial
        assert lit.reshape(-1, W)[:, 6].any()


@pytest.mark.parametrize("sse", [0, 1], ids=["plain", "sse"])
@pytest.mark.parametrize("bpc,lo,hi", [(16, 0, 65535), (16, 56000, 64000), (16, 60000, 65535),
                                       (12, 0, 4095), (10, 0, 1023), (8, 0, 255)])
def test_random_streams_across_flushes(tf, bpc, lo, hi, sse):
    if sse and bpc != 16:
        pytest.skip("the SSE-carrying form is the 16-bit one")
    threads, n_vec = 1024, 301  # 301 vectors per thread: many flush boundaries
    rng = np.random.Generator(np.random.PCG64(bpc * 1000 + lo))
    dt = np.uint8 if bpc == 8 else np.uint16
    words = 16 // np.dtype(dt).itemsize
    a = rng.integers(lo, hi + 1, threads * n_vec * words).astype(dt)
    b = rng.integers(lo, hi + 1, threads * n_vec * words).astype(dt)
    fast = np.zeros(W * threads, np.uint64)
    lit = np.zeros(W * threads, np.uint64)
    assert tf.vqx_test_stream(bpc, sse, a.ctypes.data, b.ctypes.data, n_vec, threads, fast, lit) == 0
    assert_same(fast, lit, bpc, "stream", bool(sse))


def test_long_runs_of_large_rounding_errors(tf):
    """The SSE form adds the rounding errors of the 16-bit noise squares in
    fp32 lanes, exact while a run between flushes stays below 2^24.  Here
    every pixel pair has one of the two largest errors of any 16-bit
    difference (D = 46347: D^2 - fl(D^2) = +121; D = 46399: -127), one per
    lane, over 8192 vectors a thread (four flushes); the words must still
    equal the literal ones."""
    threads, n_vec = 256, 8192
    a = np.full(threads * n_vec * 8, 65535, np.uint16)
    b = np.empty(threads * n_vec * 8, np.uint16)
    b[0::2] = 65535 - 46347
    b[1::2] = 65535 - 46399
    fast = np.zeros(W * threads, np.uint64)
    lit = np.zeros(W * threads, np.uint64)
    assert tf.vqx_test_stream(16, 1, a.ctypes.data, b.ctypes.data, n_vec, threads, fast, lit) == 0
    assert_same(fast, lit, 16, "long runs", True)
    # per thread: 4 * 8192 pairs of each difference
    want = (4 * n_vec * (121 - 127)) % (1 << 64)
    assert (lit.reshape(-1, W)[:, 6] == want).all()


def test_bounded_wait_gives_up(tf, lib):
    """The kernels' mbarrier waits are bounded: a barrier that nothing ever
    completes makes the wait return after its limit (here 2e6 cycles, about a
    millisecond), and the GPU stays usable for the next call."""
    out = np.zeros(2, np.int64)
    assert tf.vqx_test_wait_timeout(2_000_000, out) == 0
    assert out[0] == 1 and 2_000_000 <= out[1] < 200_000_000
    from exact_full_reference_gb300 import workloads as wl
    import parity

    ref, dist = wl.WORKLOADS["576x324_8bit_x1"].generate()
    keep, pr, pd, stride, _ = parity.place(ref, dist)
    rec = lib.vqx_plane_stats(pr, pd, 576, 324, stride, 8, 1)
    assert int(rec[0]["flags"]) == 0
