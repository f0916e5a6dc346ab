"""CPU oracle for the fused float_psnr noise and float_moment statistics, for
the integer psnr and for the psnr_hvs plane sum.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The GPU
library (``exact_full_reference_gb300``) never imports, links or calls it, and
the two share no code.

The arithmetic lives in ``vqx_oracle.c`` (plain C, strict floating point); this
module only marshals numpy arrays to it and states the past-2^53 bound of
"ADR-1447: float_moment_hip adds the float squares the CPU adds ..." (section
Decision).
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

SCORES_DTYPE = np.dtype(
    [
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
UNITS_DTYPE = np.dtype(
    [
        ("noise_units", "<u8"),
        ("ref_sum", "<u8"),
        ("dist_sum", "<u8"),
        ("ref_sumsq", "<u8"),
        ("dist_sumsq", "<u8"),
    ]
)

INT_PSNR_DTYPE = np.dtype(
    [
        ("sse", "<u8"),
        ("mse", "<f8"),
        ("psnr", "<f8"),
        ("psnr_uncapped", "<f8"),
    ]
)


class Oracle:
    """ctypes handle on one build of the oracle library (the real one, or a
    deliberately mutated copy used by the mutation tests)."""

    def __init__(self, lib_path=None):
        if lib_path is None:
            lib_path = _build.build_oracle()
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.vqx_oracle_batch.argtypes = [vp, vp, i, i, sz, i, i, vp, vp]
        lib.vqx_oracle_batch.restype = i
        lib.vqx_oracle_int_psnr_batch.argtypes = [vp, vp, i, i, sz, i, i, vp]
        lib.vqx_oracle_int_psnr_batch.restype = i
        i64 = ctypes.c_int64
        lib.vqx_oracle_hvs_batch.argtypes = [vp, i64, i64, i, i, vp, vp]
        lib.vqx_oracle_hvs_batch.restype = i
        lib.vqx_oracle_psnr_cap.argtypes = [i]
        lib.vqx_oracle_psnr_cap.restype = ctypes.c_double
        self._lib = lib

    def psnr_cap(self, bpc):
        return self._lib.vqx_oracle_psnr_cap(bpc)

    def batch(self, ref, dist, width, height, stride, bpc, n_frames, offset=0,
              scores=True, units=True):
        """Run the oracle over ``n_frames`` frames.

        ``ref``/``dist`` are numpy arrays holding the planes as raw bytes in the
        GPU library's layout (frame f at ``offset + f*height*stride`` bytes, row
        y at ``+ y*stride``).  Returns ``(scores, units)`` structured arrays
        (either may be ``None`` when not requested)."""
        ref = np.ascontiguousarray(ref)
        dist = np.ascontiguousarray(dist)
        need = offset + (n_frames - 1) * height * stride + (height - 1) * stride + width * (
            1 if bpc == 8 else 2) if n_frames > 0 else 0
        if ref.nbytes < need or dist.nbytes < need:
            raise ValueError("plane buffer smaller than the frame geometry needs")
        sc = np.zeros(n_frames, SCORES_DTYPE) if scores else None
        un = np.zeros(n_frames, UNITS_DTYPE) if units else None
        rc = self._lib.vqx_oracle_batch(
            ref.ctypes.data + offset,
            dist.ctypes.data + offset,
            width,
            height,
            stride,
            bpc,
            n_frames,
            sc.ctypes.data if sc is not None else None,
            un.ctypes.data if un is not None else None,
        )
        if rc != 0:
            raise ValueError("oracle rejected the arguments (status %d)" % rc)
        return sc, un

    def int_psnr(self, ref, dist, width, height, stride, bpc, n_frames, offset=0):
        """Integer psnr of ``n_frames`` frames (same layout as ``batch``):
        an ``INT_PSNR_DTYPE`` array."""
        ref = np.ascontiguousarray(ref)
        dist = np.ascontiguousarray(dist)
        need = offset + (n_frames - 1) * height * stride + (height - 1) * stride + width * (
            1 if bpc == 8 else 2) if n_frames > 0 else 0
        if ref.nbytes < need or dist.nbytes < need:
            raise ValueError("plane buffer smaller than the frame geometry needs")
        out = np.zeros(n_frames, INT_PSNR_DTYPE)
        rc = self._lib.vqx_oracle_int_psnr_batch(ref.ctypes.data + offset, dist.ctypes.data + offset,
                                                 width, height, stride, bpc, n_frames,
                                                 out.ctypes.data if n_frames else None)
        if rc != 0:
            raise ValueError("oracle rejected the arguments (status %d)" % rc)
        return out

    def int_psnr_frames(self, ref, dist, bpc):
        """Convenience form for dense arrays of shape (n, h, w) or (h, w)."""
        ref = np.asarray(ref)
        dist = np.asarray(dist)
        if ref.ndim == 2:
            ref = ref[None]
            dist = dist[None]
        n, h, w = ref.shape
        return self.int_psnr(ref, dist, w, h, w * ref.itemsize, bpc, n)

    def hvs(self, terms, bpc, n_terms=None, pitch=None, n_planes=None):
        """psnr_hvs plane sums and scores of float32 terms.

        ``terms`` is a float32 array: shape (n_planes, pitch) or (n,) for one
        plane; ``n_terms`` (default: the last axis) terms of each plane are
        added.  Returns ``(sums, scores)``, float32 arrays of n_planes."""
        terms = np.ascontiguousarray(terms)
        if terms.dtype != np.float32:
            raise ValueError("terms must be float32")
        if terms.ndim == 1:
            terms = terms[None]
        if pitch is None:
            pitch = terms.shape[-1]
        if n_planes is None:
            n_planes = terms.size // pitch if pitch else 0
        if n_terms is None:
            n_terms = pitch
        if n_planes > 0 and (n_planes - 1) * pitch + n_terms > terms.size:
            raise ValueError("term buffer smaller than the planes need")
        sums = np.zeros(n_planes, np.float32)
        scores = np.zeros(n_planes, np.float32)
        rc = self._lib.vqx_oracle_hvs_batch(terms.ctypes.data, n_terms, pitch, n_planes, bpc,
                                            sums.ctypes.data if n_planes else None,
                                            scores.ctypes.data if n_planes else None)
        if rc != 0:
            raise ValueError("oracle rejected the arguments (status %d)" % rc)
        return sums, scores

    def frames(self, ref, dist, bpc, scores=True, units=True):
        """Convenience form for dense arrays of shape (n, h, w) or (h, w)."""
        ref = np.asarray(ref)
        dist = np.asarray(dist)
        if ref.shape != dist.shape:
            raise ValueError("ref and dist shapes differ")
        if ref.ndim == 2:
            ref = ref[None]
            dist = dist[None]
        n, h, w = ref.shape
        return self.batch(ref, dist, w, h, w * ref.itemsize, bpc, n, scores=scores, units=units)


_default = None


def load():
    """The oracle built from ``vqx_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def moment_bound(pixels, e):
    """Bound, as a moment, on the gap between the CPU's sequential double sum
    and the exact sum rounded once, for sums of at least 2^53 units, after
    "ADR-1447 ..." (Decision).  Terms stay below 2^32 units, so the first 2^21
    additions cannot leave the exact range; each of the remaining
    pixels - 2^21 + 1 additions can round by half an ulp of a sum with
    2^e <= sum < 2^(e+1), i.e. 2^(e-53) units, as can the single rounding of
    the exact sum; one unit is 2^-16 / pixels in moment terms (2^(e-69) per
    addition), and the final two divisions contribute at most 2^-37."""
    later = max(pixels - 2 ** 21 + 1, 0)
    return later / pixels * 2.0 ** (e - 69) + 2.0 ** -37


def binade(units):
    """e with 2^e <= units < 2^(e+1) (units > 0)."""
    return int(units).bit_length() - 1


def mse_bound(pixels, noise_units):
    """The same bound for the MSE (noise / pixels): its terms are float squares
    below 2^32 units of 2^-16 too, so the derivation of ``moment_bound`` applies
    unchanged.  Below 2^53 units the CPU's sum is exact and the bound is 0."""
    if noise_units < 2 ** 53:
        return 0.0
    return moment_bound(pixels, binade(noise_units))


def psnr_bound(mse, dmse, psnr):
    """Bound on |PSNR difference| implied by an MSE difference ``dmse``:
    d/dmse of 10 log10(c/mse) is -(10/ln 10)/mse; plus a few ulps of the
    logarithm and the product."""
    if mse == 0.0 or not math.isfinite(psnr):
        return 0.0
    return (10.0 / math.log(10.0)) * dmse / (mse - dmse) + 4.0 * math.ulp(abs(psnr) + 1.0)
