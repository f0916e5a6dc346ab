"""Python binding of the vqx C ABI (``include/vqx.h``): argument marshalling only.

Every step of the statistics runs in ``libvqx.so`` (CUDA kernels for sm_103a
plus the host conclusion in C++).  This module loads that library with ctypes,
turns tensors / arrays into pointers and sizes, and returns the per-frame
records as a numpy structured array.  There is no fallback: if the library is
missing or a call fails, an exception is raised.

PyTorch is used only as a source of device memory and streams: anything with a
``data_ptr()`` method (a CUDA tensor) or a plain integer address is accepted.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvqx.so")

VQX_OK = 0
VQX_EINVAL = -1
VQX_EBPC = -2
VQX_ERANGE = -3
VQX_ECUDA = -4
VQX_ENOMEM = -5
VQX_ETIMEOUT = -6
VQX_FLAG_RANGE = 1
VQX_FLAG_TIMEOUT = 2
VQX_MAX_FRAME_PIXELS = 1 << 25
VQX_NOALLOC_MAX_RECORDS = 65536

FRAME_STATS_DTYPE = np.dtype(
    [
        ("noise_units", "<u8"),
        ("ref_sum", "<u8"),
        ("dist_sum", "<u8"),
        ("ref_sumsq", "<u8"),
        ("dist_sumsq", "<u8"),
        ("flags", "<u4"),
        ("reserved", "<u4"),
        ("noise", "<f8"),
        ("mse", "<f8"),
        ("psnr", "<f8"),
        ("psnr_uncapped", "<f8"),
        ("ref_mean", "<f8"),
        ("ref_meansq", "<f8"),
        ("dist_mean", "<f8"),
        ("dist_meansq", "<f8"),
    ]
)

INT_PSNR_DTYPE = np.dtype(
    [
        ("sse", "<u8"),
        ("flags", "<u4"),
        ("reserved", "<u4"),
        ("mse", "<f8"),
        ("psnr", "<f8"),
        ("psnr_uncapped", "<f8"),
    ]
)

HVS_PLANE_DTYPE = np.dtype(
    [
        ("sum", "<f4"),
        ("score", "<f4"),
        ("flags", "<u4"),
        ("replayed_leaves", "<u4"),
    ]
)


class VqxProfile(ctypes.Structure):
    _fields_ = [
        ("calls", ctypes.c_uint64),
        ("kernel_launches", ctypes.c_uint64),
        ("stage1_launches", ctypes.c_uint64),
        ("stage1_ms", ctypes.c_double),
        ("stage2_ms", ctypes.c_double),
        ("stage1_bytes", ctypes.c_uint64),
    ]


VQX_MAX_PLANES = 4
VQX_SUBMIT_PLANES_READY = 1


class PlaneDesc(ctypes.Structure):
    """``vqx_plane_desc``: one plane of every frame (device pointers)."""
    _fields_ = [
        ("ref", ctypes.c_void_p),
        ("dist", ctypes.c_void_p),
        ("width", ctypes.c_int),
        ("height", ctypes.c_int),
        ("stride", ctypes.c_size_t),
        ("frame_pitch", ctypes.c_size_t),
    ]


class VqxError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(msg)
        self.status = status


_lib = None


def library():
    """The loaded ``libvqx.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libvqx.so is not built (%s); run exact_full_reference_gb300.build.build_library()"
                % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        for name in ("vqx_plane_stats", "vqx_plane_stats_host", "vqx_plane_stats_noalloc",
                     "vqx_plane_stats_ordered", "vqx_plane_int_psnr"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, i, i, sz, i, i, vp, vp]
            fn.restype = i
        for kind in ("stats", "int_psnr", "stats_ordered", "scores"):
            sub = getattr(lib, "vqx_plane_%s_submit" % kind)
            sub.argtypes = [vp, vp, i, i, sz, i, i, vp, ctypes.c_uint, ctypes.POINTER(vp)]
            sub.restype = i
            fin = getattr(lib, "vqx_plane_%s_finish" % kind)
            fin.argtypes = [vp, vp, vp] if kind == "scores" else [vp, vp]
            fin.restype = i
        lib.vqx_plane_scores.argtypes = [vp, vp, i, i, sz, i, i, vp, vp, vp]
        lib.vqx_plane_scores.restype = i
        lib.vqx_planes_stats.argtypes = [ctypes.POINTER(PlaneDesc), i, i, i, vp, vp]
        lib.vqx_planes_stats.restype = i
        lib.vqx_planes_stats_submit.argtypes = [ctypes.POINTER(PlaneDesc), i, i, i, vp, ctypes.c_uint,
                                                ctypes.POINTER(vp)]
        lib.vqx_planes_stats_submit.restype = i
        lib.vqx_planes_stats_finish.argtypes = [vp, vp]
        lib.vqx_planes_stats_finish.restype = i
        i64 = ctypes.c_int64
        lib.vqx_psnr_hvs_sum.argtypes = [vp, i64, i64, i, i, vp, vp]
        lib.vqx_psnr_hvs_sum.restype = i
        lib.vqx_psnr_hvs_sum_submit.argtypes = [vp, i64, i64, i, i, vp, ctypes.c_uint,
                                                ctypes.POINTER(vp)]
        lib.vqx_psnr_hvs_sum_submit.restype = i
        lib.vqx_psnr_hvs_sum_finish.argtypes = [vp, vp]
        lib.vqx_psnr_hvs_sum_finish.restype = i
        lib.vqx_psnr_cap.argtypes = [i]
        lib.vqx_psnr_cap.restype = ctypes.c_double
        lib.vqx_status_string.argtypes = [i]
        lib.vqx_status_string.restype = ctypes.c_char_p
        lib.vqx_last_cuda_error.argtypes = []
        lib.vqx_last_cuda_error.restype = i
        lib.vqx_profile_enable.argtypes = [i]
        lib.vqx_profile_enable.restype = None
        lib.vqx_profile_read.argtypes = [ctypes.POINTER(VqxProfile), i]
        lib.vqx_profile_read.restype = None
        _lib = lib
    return _lib


def _address(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError("expected a tensor, an ndarray or an integer address, got %r" % type(x))


def _stream_handle(stream):
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _geometry(ref, width, height, stride, n_frames, bpc):
    bps = 1 if bpc == 8 else 2
    shape = tuple(getattr(ref, "shape", ()))
    if width is None or height is None:
        if len(shape) < 2:
            raise ValueError("width and height are needed for a flat buffer")
        height, width = int(shape[-2]), int(shape[-1])
        if n_frames is None:
            n_frames = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
        if stride is None:
            stride = width * bps
    if stride is None:
        stride = width * bps
    if n_frames is None:
        n_frames = 1
    return width, height, stride, n_frames


def status_string(status):
    return library().vqx_status_string(status).decode()


def psnr_cap(bpc):
    return library().vqx_psnr_cap(bpc)


def _raise(name, rc):
    msg = "%s failed: %s (%d)" % (name, status_string(rc), rc)
    if rc == VQX_ECUDA:
        msg += ", cudaError %d" % library().vqx_last_cuda_error()
    raise VqxError(rc, msg)


def _call(name, ref, dist, width, height, stride, bpc, n_frames, stream, out, check,
          dtype=FRAME_STATS_DTYPE):
    width, height, stride, n_frames = _geometry(ref, width, height, stride, n_frames, bpc)
    if out is None:
        out = np.zeros(max(n_frames, 0), dtype)
    rc = getattr(library(), name)(
        _address(ref), _address(dist), width, height, stride, bpc, n_frames, stream,
        out.ctypes.data if out.size else None)
    if check and rc not in (VQX_OK,):
        _raise(name, rc)
    return out, rc


def vqx_plane_stats(ref, dist, width=None, height=None, stride=None, bpc=16, n_frames=None,
                    stream=None, out=None, check=True):
    """Per-frame statistics of device-resident planes.

    ``ref``/``dist``: CUDA tensors (shape (n, h, w) or (h, w); any dtype whose
    bytes hold the samples) or device addresses with explicit geometry.
    ``stride`` is in bytes.  Returns a structured array of ``n_frames``
    records (``FRAME_STATS_DTYPE``).  With ``check=False`` returns
    ``(records, status)`` instead of raising on a non-zero status."""
    out, rc = _call("vqx_plane_stats", ref, dist, width, height, stride, bpc, n_frames,
                    _stream_handle(stream), out, check)
    return out if check else (out, rc)


class Pending:
    """A batch enqueued by ``vqx_plane_stats_submit``; ``finish()`` waits for
    it and returns its records (call it exactly once)."""

    def __init__(self, handle, n_frames, keep, kind="stats", n_planes=None):
        self._handle = handle
        self.n_frames = n_frames
        self.kind = kind
        self.shape = n_frames if n_planes is None else (n_frames, n_planes)
        self._keep = keep  # the planes stay referenced until the batch is finished

    def finish(self, out=None, check=True):
        if self._handle is False:
            raise RuntimeError("this batch was already finished")
        if self.kind == "scores":
            stats = np.zeros(self.shape, FRAME_STATS_DTYPE)
            ints = np.zeros(self.shape, INT_PSNR_DTYPE)
            rc = library().vqx_plane_scores_finish(self._handle, stats.ctypes.data if stats.size else None,
                                                   ints.ctypes.data if ints.size else None)
            self._handle, self._keep = False, None
            if check and rc != VQX_OK:
                _raise("vqx_plane_scores_finish", rc)
            return (stats, ints) if check else (stats, ints, rc)
        if out is None:
            dtype = {"int_psnr": INT_PSNR_DTYPE, "hvs": HVS_PLANE_DTYPE}.get(self.kind, FRAME_STATS_DTYPE)
            out = np.zeros(self.shape, dtype)
        name = {"planes": "vqx_planes_stats_finish", "hvs": "vqx_psnr_hvs_sum_finish"}.get(
            self.kind, "vqx_plane_%s_finish" % self.kind)
        rc = getattr(library(), name)(self._handle, out.ctypes.data if out.size else None)
        self._handle, self._keep = False, None
        if check and rc != VQX_OK:
            _raise(name, rc)
        return out if check else (out, rc)


def _submit(kind, ref, dist, width, height, stride, bpc, n_frames, stream, flags):
    width, height, stride, n_frames = _geometry(ref, width, height, stride, n_frames, bpc)
    handle = ctypes.c_void_p()
    name = "vqx_plane_%s_submit" % kind
    rc = getattr(library(), name)(_address(ref), _address(dist), width, height, stride, bpc,
                                  n_frames, _stream_handle(stream), flags, ctypes.byref(handle))
    if rc != VQX_OK:
        _raise(name, rc)
    return Pending(handle.value, max(n_frames, 0), (ref, dist), kind)


def vqx_plane_stats_submit(ref, dist, width=None, height=None, stride=None, bpc=16,
                           n_frames=None, stream=None, flags=0):
    """Enqueue a batch of device planes without waiting; returns a
    ``Pending`` whose ``finish()`` gives what ``vqx_plane_stats`` would.
    ``flags``: 0 or ``VQX_SUBMIT_PLANES_READY``."""
    return _submit("stats", ref, dist, width, height, stride, bpc, n_frames, stream, flags)


def vqx_plane_stats_ordered_submit(ref, dist, width=None, height=None, stride=None, bpc=16,
                                   n_frames=None, stream=None, flags=0):
    """The same for ``vqx_plane_stats_ordered`` (its workspace is held until
    ``finish()``)."""
    return _submit("stats_ordered", ref, dist, width, height, stride, bpc, n_frames, stream, flags)


def vqx_plane_int_psnr_submit(ref, dist, width=None, height=None, stride=None, bpc=16,
                              n_frames=None, stream=None, flags=0):
    """The same for the integer psnr (``finish()`` gives ``INT_PSNR_DTYPE``)."""
    return _submit("int_psnr", ref, dist, width, height, stride, bpc, n_frames, stream, flags)


def vqx_plane_int_psnr(ref, dist, width=None, height=None, stride=None, bpc=16, n_frames=None,
                       stream=None, out=None, check=True):
    """Integer psnr per frame of device-resident planes: the exact SSE of the
    raw samples, its MSE and the PSNR with peak 2^bpc - 1 (``INT_PSNR_DTYPE``
    records)."""
    out, rc = _call("vqx_plane_int_psnr", ref, dist, width, height, stride, bpc, n_frames,
                    _stream_handle(stream), out, check, INT_PSNR_DTYPE)
    return out if check else (out, rc)


def vqx_plane_scores_submit(ref, dist, width=None, height=None, stride=None, bpc=16,
                            n_frames=None, stream=None, flags=0):
    """The same for ``vqx_plane_scores`` (``finish()`` gives the pair of
    record arrays)."""
    return _submit("scores", ref, dist, width, height, stride, bpc, n_frames, stream, flags)


def vqx_plane_scores(ref, dist, width=None, height=None, stride=None, bpc=16, n_frames=None,
                     stream=None, check=True):
    """float_psnr, float_moment and the integer psnr of device-resident planes
    from one read: returns ``(stats, int_psnr)``, a ``FRAME_STATS_DTYPE`` and
    an ``INT_PSNR_DTYPE`` array of ``n_frames`` records each (with
    ``check=False``, ``(stats, int_psnr, status)``)."""
    width, height, stride, n_frames = _geometry(ref, width, height, stride, n_frames, bpc)
    stats = np.zeros(max(n_frames, 0), FRAME_STATS_DTYPE)
    ints = np.zeros(max(n_frames, 0), INT_PSNR_DTYPE)
    rc = library().vqx_plane_scores(_address(ref), _address(dist), width, height, stride, bpc,
                                    n_frames, _stream_handle(stream),
                                    stats.ctypes.data if stats.size else None,
                                    ints.ctypes.data if ints.size else None)
    if check and rc != VQX_OK:
        _raise("vqx_plane_scores", rc)
    return (stats, ints) if check else (stats, ints, rc)


def vqx_plane_stats_host(ref, dist, width=None, height=None, stride=None, bpc=16,
                         n_frames=None, stream=None, out=None, check=True):
    """The same for planes in host memory (numpy arrays, pinned tensors or
    host addresses): the library copies them to the device in chunks."""
    out, rc = _call("vqx_plane_stats_host", ref, dist, width, height, stride, bpc, n_frames,
                    _stream_handle(stream), out, check)
    return out if check else (out, rc)


def vqx_plane_stats_ordered(ref, dist, width=None, height=None, stride=None, bpc=16,
                            n_frames=None, stream=None, out=None, check=True):
    """Device planes; the doubles equal the CPU's also past 2^53 units (the
    CPU's sequential roundings are replayed on the device)."""
    out, rc = _call("vqx_plane_stats_ordered", ref, dist, width, height, stride, bpc, n_frames,
                    _stream_handle(stream), out, check)
    return out if check else (out, rc)


def vqx_plane_stats_noalloc(ref, dist, width=None, height=None, stride=None, bpc=16,
                            n_frames=None, stream=None, out=None, check=True):
    """The allocation-free variant (device planes, at most
    ``VQX_NOALLOC_MAX_RECORDS // 2`` frames a call; calls must not overlap
    on the GPU)."""
    out, rc = _call("vqx_plane_stats_noalloc", ref, dist, width, height, stride, bpc, n_frames,
                    _stream_handle(stream), out, check)
    return out if check else (out, rc)


def _plane_descs(planes):
    descs = (PlaneDesc * max(len(planes), 1))()
    for k, (r, d, w, h, st, fp) in enumerate(planes):
        descs[k] = PlaneDesc(_address(r), _address(d), w, h, st, fp or 0)
    return descs


def vqx_planes_stats_submit(planes, bpc, n_frames, stream=None, flags=0):
    """Enqueue ``vqx_planes_stats`` without waiting; ``finish()`` gives the
    (n_frames, len(planes)) records."""
    handle = ctypes.c_void_p()
    rc = library().vqx_planes_stats_submit(_plane_descs(planes), len(planes), bpc, n_frames,
                                           _stream_handle(stream), flags, ctypes.byref(handle))
    if rc != VQX_OK:
        _raise("vqx_planes_stats_submit", rc)
    return Pending(handle.value, max(n_frames, 0), [p[:2] for p in planes], "planes", len(planes))


def vqx_planes_stats(planes, bpc, n_frames, stream=None, check=True):
    """Per-frame statistics of several planes of each frame (Y, Cb, Cr ...).

    ``planes``: a sequence of ``(ref, dist, width, height, stride,
    frame_pitch)``; ref/dist are CUDA tensors or device addresses of the
    plane in frame 0, stride and frame_pitch in bytes (frame_pitch 0 or None:
    height * stride).  Returns ``FRAME_STATS_DTYPE`` records of shape
    (n_frames, len(planes))."""
    descs = _plane_descs(planes)
    out = np.zeros((max(n_frames, 0), len(planes)), FRAME_STATS_DTYPE)
    rc = library().vqx_planes_stats(descs, len(planes), bpc, n_frames, _stream_handle(stream),
                                    out.ctypes.data if out.size else None)
    if check and rc != VQX_OK:
        _raise("vqx_planes_stats", rc)
    return out if check else (out, rc)


def profile_enable(on=True):
    library().vqx_profile_enable(1 if on else 0)


def profile_read(reset=False):
    p = VqxProfile()
    library().vqx_profile_read(ctypes.byref(p), 1 if reset else 0)
    return {k: getattr(p, k) for k, _ in VqxProfile._fields_}


def _hvs_geometry(terms, n_terms, pitch, n_planes):
    shape = tuple(getattr(terms, "shape", ()))
    if pitch is None:
        if not shape:
            raise ValueError("plane_pitch is needed for a flat address")
        pitch = int(shape[-1])
    if n_terms is None:
        n_terms = pitch
    if n_planes is None:
        n_planes = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    return int(n_terms), int(pitch), int(n_planes)


def vqx_psnr_hvs_sum(terms, n_terms=None, pitch=None, n_planes=None, bpc=8, stream=None,
                     out=None, check=True):
    """psnr_hvs plane sums of device-resident float32 terms: shape
    (n_planes, pitch) or (n,) for one plane, or an address with explicit
    sizes.  Returns ``HVS_PLANE_DTYPE`` records (the sequential float sum and
    the plane score); with ``check=False``, ``(records, status)``."""
    n_terms, pitch, n_planes = _hvs_geometry(terms, n_terms, pitch, n_planes)
    if out is None:
        out = np.zeros(max(n_planes, 0), HVS_PLANE_DTYPE)
    rc = library().vqx_psnr_hvs_sum(_address(terms), n_terms, pitch, n_planes, bpc,
                                    _stream_handle(stream), out.ctypes.data if out.size else None)
    if check and rc != VQX_OK:
        _raise("vqx_psnr_hvs_sum", rc)
    return out if check else (out, rc)


def vqx_psnr_hvs_sum_submit(terms, n_terms=None, pitch=None, n_planes=None, bpc=8, stream=None,
                            flags=0):
    """The same without waiting: a ``Pending`` whose ``finish()`` gives the
    records."""
    n_terms, pitch, n_planes = _hvs_geometry(terms, n_terms, pitch, n_planes)
    handle = ctypes.c_void_p()
    rc = library().vqx_psnr_hvs_sum_submit(_address(terms), n_terms, pitch, n_planes, bpc,
                                           _stream_handle(stream), flags, ctypes.byref(handle))
    if rc != VQX_OK:
        _raise("vqx_psnr_hvs_sum_submit", rc)
    return Pending(handle.value, max(n_planes, 0), terms, "hvs")
