"""The C-ABI library builds, loads and exports what include/vqx.h declares;
argument checks that need no GPU (CPU only: no compute call is made)."""
import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(vqx_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("vqx_plane_stats", "vqx_plane_stats_host", "vqx_plane_int_psnr", "vqx_planes_stats",
              "vqx_planes_stats_submit", "vqx_planes_stats_finish",
              "vqx_plane_stats_ordered_submit", "vqx_plane_stats_ordered_finish",
              "vqx_plane_int_psnr_submit", "vqx_plane_int_psnr_finish", "vqx_status_string",
              "vqx_last_cuda_error", "vqx_psnr_cap", "vqx_profile_enable", "vqx_profile_read",
              "vqx_psnr_hvs_sum", "vqx_psnr_hvs_sum_submit", "vqx_psnr_hvs_sum_finish",
              "vqx_plane_scores", "vqx_plane_scores_submit", "vqx_plane_scores_finish"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = lib.library()
    for name in declared_functions():
        assert hasattr(so, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(declared_functions()) <= exported
    # the statically linked CUDA runtime stays private
    assert not any(s.startswith("cuda") for s in exported), sorted(
        s for s in exported if s.startswith("cuda"))[:5]


def test_status_strings_and_caps(lib):
    assert lib.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert lib.status_string(code) not in ("ok", "unknown status")
    assert lib.status_string(-99) == "unknown status"
    assert [lib.psnr_cap(b) for b in (8, 10, 12, 16)] == [60.0, 72.0, 84.0, 108.0]
    assert math.isnan(lib.psnr_cap(9))


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize(
    "args,status",
    [
        (dict(bpc=9), -2),
        (dict(bpc=0), -2),
        (dict(width=0), -1),
        (dict(height=-3), -1),
        (dict(n_frames=-1), -1),
        (dict(stride=2 * 64 - 2), -1),
        (dict(ref=0), -1),
        (dict(dist=0), -1),
        (dict(ref=FAKE + 1), -1),  # odd address, 16-bit samples
        (dict(stride=2 * 64 + 1), -1),  # odd stride, 16-bit samples
        (dict(width=8192, height=4097, stride=8192 * 2), -1),  # over 2^25 pixels
        (dict(bpc=8, width=1 << 13, height=(1 << 12) + 1, stride=1 << 13), -1),
    ],
)
def test_argument_errors_need_no_gpu(lib, args, status):
    a = dict(ref=FAKE, dist=FAKE, width=64, height=4, stride=128, bpc=16, n_frames=2)
    a.update(args)
    out = (ctypes.c_char * (152 * 4))()
    so = lib.library()
    for name in ("vqx_plane_stats", "vqx_plane_stats_host", "vqx_plane_int_psnr"):
        rc = getattr(so, name)(a["ref"] or None, a["dist"] or None, a["width"], a["height"],
                               a["stride"], a["bpc"], a["n_frames"], None, out)
        assert rc == status, (name, args, rc)


@pytest.mark.parametrize("args,status", [(dict(bpc=9), -2), (dict(width=0), -1), (dict(ref=0), -1),
                                         (dict(stride=2 * 64 + 1), -1), (dict(n_frames=-2), -1)])
def test_submit_argument_errors_need_no_gpu(lib, args, status):
    a = dict(ref=FAKE, dist=FAKE, width=64, height=4, stride=128, bpc=16, n_frames=2)
    a.update(args)
    so = lib.library()
    handle = ctypes.c_void_p(1234)
    rc = so.vqx_plane_stats_submit(a["ref"] or None, a["dist"] or None, a["width"], a["height"],
                                   a["stride"], a["bpc"], a["n_frames"], None, 0, ctypes.byref(handle))
    assert rc == status
    assert handle.value is None  # cleared on every error


def test_submit_finish_empty_and_null(lib):
    so = lib.library()
    handle = ctypes.c_void_p(1234)
    assert so.vqx_plane_stats_submit(None, None, 0, 0, 0, 16, 0, None, 0, ctypes.byref(handle)) == 0
    assert handle.value is None
    assert so.vqx_plane_stats_finish(None, None) == 0
    assert so.vqx_plane_stats_submit(FAKE, FAKE, 4, 4, 8, 16, 1, None, 0, None) == -1
    # an unknown flag is refused before anything else
    assert so.vqx_plane_stats_submit(FAKE, FAKE, 4, 4, 8, 16, 1, None, 2, ctypes.byref(handle)) == -1
    assert handle.value is None
    assert so.vqx_plane_int_psnr_submit(None, None, 0, 0, 0, 12, 0, None, 0, ctypes.byref(handle)) == 0
    assert handle.value is None and so.vqx_plane_int_psnr_finish(None, None) == 0
    assert so.vqx_plane_int_psnr(None, None, 0, 0, 0, 8, 0, None, None) == 0
    p = lib.vqx_plane_stats_submit(np.zeros((0, 4, 4), np.uint16), np.zeros((0, 4, 4), np.uint16))
    assert p.finish().size == 0


def test_planes_argument_errors_need_no_gpu(lib):
    so = lib.library()
    out = (ctypes.c_char * (112 * 16))()

    def call(descs, n_planes=None, bpc=16, n_frames=2):
        arr = (lib.PlaneDesc * max(len(descs), 1))(*descs)
        return so.vqx_planes_stats(arr, len(descs) if n_planes is None else n_planes, bpc, n_frames,
                                   None, out)

    y = lib.PlaneDesc(FAKE, FAKE, 64, 4, 128, 0)
    c = lib.PlaneDesc(FAKE, FAKE, 32, 2, 64, 0)
    assert call([y, c, c], n_planes=0) == -1
    assert call([y, c, c, c, c]) == -1  # more than VQX_MAX_PLANES
    assert call([y, c], bpc=9) == -2
    assert call([y, lib.PlaneDesc(FAKE, FAKE, 32, 2, 64, 100)]) == -1  # pitch below height * stride
    assert call([y, lib.PlaneDesc(FAKE, FAKE, 32, 2, 64, 129)]) == -1  # odd pitch at 16 bits
    assert call([y, lib.PlaneDesc(FAKE + 1, FAKE, 32, 2, 64, 0)]) == -1  # odd base at 16 bits
    assert call([y], n_frames=0) == 0
    assert so.vqx_planes_stats(None, 1, 16, 1, None, out) == -1
    assert ctypes.sizeof(lib.PlaneDesc) == 40
    handle = ctypes.c_void_p(99)
    arr = (lib.PlaneDesc * 2)(y, c)
    assert so.vqx_planes_stats_submit(arr, 2, 9, 2, None, 0, ctypes.byref(handle)) == -2
    assert handle.value is None
    assert so.vqx_planes_stats_submit(arr, 2, 16, 2, None, 4, ctypes.byref(handle)) == -1
    assert so.vqx_planes_stats_submit(arr, 2, 16, 0, None, 0, ctypes.byref(handle)) == 0
    assert handle.value is None and so.vqx_planes_stats_finish(None, None) == 0


@pytest.mark.parametrize("args,status", [(dict(bpc=9), -2), (dict(width=0), -1), (dict(ref=0), -1),
                                         (dict(stride=2 * 64 + 1), -1), (dict(n_frames=-2), -1),
                                         (dict(width=8192, height=4097, stride=8192 * 2), -1)])
def test_scores_argument_errors_need_no_gpu(lib, args, status):
    a = dict(ref=FAKE, dist=FAKE, width=64, height=4, stride=128, bpc=16, n_frames=2)
    a.update(args)
    so = lib.library()
    out = (ctypes.c_char * (112 * 2))()
    ints = (ctypes.c_char * (40 * 2))()
    rc = so.vqx_plane_scores(a["ref"] or None, a["dist"] or None, a["width"], a["height"], a["stride"],
                             a["bpc"], a["n_frames"], None, out, ints)
    assert rc == status
    handle = ctypes.c_void_p(1234)
    rc = so.vqx_plane_scores_submit(a["ref"] or None, a["dist"] or None, a["width"], a["height"],
                                    a["stride"], a["bpc"], a["n_frames"], None, 0, ctypes.byref(handle))
    assert rc == status and handle.value is None


def test_scores_outputs_and_empty_batches_without_gpu(lib):
    so = lib.library()
    out = (ctypes.c_char * 112)()
    ints = (ctypes.c_char * 40)()
    # either output missing: refused before anything runs
    assert so.vqx_plane_scores(FAKE, FAKE, 4, 4, 8, 16, 1, None, None, ints) == -1
    assert so.vqx_plane_scores(FAKE, FAKE, 4, 4, 8, 16, 1, None, out, None) == -1
    # empty batches touch nothing and need no outputs
    assert so.vqx_plane_scores(None, None, 0, 0, 0, 16, 0, None, None, None) == 0
    handle = ctypes.c_void_p(1234)
    assert so.vqx_plane_scores_submit(None, None, 0, 0, 0, 10, 0, None, 0, ctypes.byref(handle)) == 0
    assert handle.value is None and so.vqx_plane_scores_finish(None, None, None) == 0
    assert so.vqx_plane_scores_submit(FAKE, FAKE, 4, 4, 8, 16, 1, None, 2, ctypes.byref(handle)) == -1
    stats, ip = lib.vqx_plane_scores(np.zeros((0, 4, 4), np.uint16), np.zeros((0, 4, 4), np.uint16))
    assert stats.size == 0 and ip.size == 0


def test_empty_batch_is_ok_without_gpu(lib):
    so = lib.library()
    assert so.vqx_plane_stats(None, None, 0, 0, 0, 16, 0, None, None) == 0
    assert so.vqx_plane_stats_host(None, None, 0, 0, 0, 8, 0, None, None) == 0


def test_null_output_rejected(lib):
    so = lib.library()
    assert so.vqx_plane_stats(FAKE, FAKE, 4, 4, 8, 16, 1, None, None) == -1


def test_record_layout_matches_header(lib):
    # 5 uint64 + 2 uint32 + 8 doubles = 112 bytes, no padding
    assert lib.FRAME_STATS_DTYPE.itemsize == 112
    # 1 uint64 + 2 uint32 + 3 doubles = 40 bytes
    assert lib.INT_PSNR_DTYPE.itemsize == 40
    assert ctypes.sizeof(lib.VqxProfile) == 48


def test_profile_counters_without_gpu(lib):
    lib.profile_enable(True)
    p = lib.profile_read(reset=True)
    assert p["calls"] == 0 and p["stage1_ms"] == 0.0
    lib.profile_enable(False)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import exact_full_reference_gb300 as vqx

    monkeypatch.setattr(vqx, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(vqx, "_lib", None)
    with pytest.raises(ImportError):
        vqx.library()


@pytest.mark.parametrize(
    "args,status",
    [
        (dict(bpc=9), -2),
        (dict(n_planes=-1), -1),
        (dict(terms=0), -1),
        (dict(terms=FAKE + 2), -1),  # not 4-byte aligned
        (dict(n_terms=0), -1),
        (dict(n_terms=1 << 31, pitch=1 << 31), -1),  # over 2^31 - 1 terms
        (dict(pitch=999), -1),  # pitch below n_terms
        (dict(n_planes=1 << 20, n_terms=(1 << 31) - 1, pitch=(1 << 31) - 1), -1),  # grid too large
    ],
)
def test_hvs_argument_errors_need_no_gpu(lib, args, status):
    a = dict(terms=FAKE, n_terms=1000, pitch=1000, n_planes=2, bpc=8)
    a.update(args)
    so = lib.library()
    out = np.zeros(max(a["n_planes"], 1), lib.HVS_PLANE_DTYPE)
    rc = so.vqx_psnr_hvs_sum(a["terms"], a["n_terms"], a["pitch"], a["n_planes"], a["bpc"], None,
                             out.ctypes.data)
    assert rc == status
    h = ctypes.c_void_p(123)
    rc = so.vqx_psnr_hvs_sum_submit(a["terms"], a["n_terms"], a["pitch"], a["n_planes"], a["bpc"],
                                    None, 0, ctypes.byref(h))
    assert rc == status and h.value is None


def test_hvs_no_planes_and_flags_need_no_gpu(lib):
    so = lib.library()
    out = np.zeros(1, lib.HVS_PLANE_DTYPE)
    assert so.vqx_psnr_hvs_sum(FAKE, 1000, 1000, 0, 8, None, out.ctypes.data) == 0
    assert so.vqx_psnr_hvs_sum(FAKE, 1000, 1000, 0, 8, None, None) == 0
    h = ctypes.c_void_p()
    assert so.vqx_psnr_hvs_sum_submit(FAKE, 1000, 1000, 1, 8, None, 2, ctypes.byref(h)) == -1
    assert so.vqx_psnr_hvs_sum_submit(FAKE, 1000, 1000, 1, 8, None, 0, None) == -1
    assert so.vqx_psnr_hvs_sum_finish(None, out.ctypes.data) == 0
