"""Seeded synthetic luma planes for the parity tests and the benchmark.

This module only draws numbers: it holds none of the statistics' arithmetic, so
both the CPU oracle's tests and the GPU path's tests can take their inputs from
it.  The pages measure on fixtures (the Netflix 576x324 pair, Big Buck Bunny at
3840x2160, full-range noise, a bright 16-bit 1920x1080 pair, checkerboards);
none of them is available, so each workload below is a synthetic stand-in with
the shape, bit depth, frame count and value distribution of one such case.

Random numbers: numpy ``PCG64``; frame f of a workload draws from child f of
``SeedSequence(seed)``, so any frame can be regenerated alone.  Rounding of
normal noise is ``np.rint`` (half to even); results are clipped to
``[0, 2^bpc - 1]``.  Planes are returned as arrays of shape (frames, h, w),
``uint8`` at 8 bits and ``uint16`` otherwise.
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    width: int
    height: int
    bpc: int
    n_frames: int
    seed: int
    kind: str
    note: str = ""

    @property
    def dtype(self):
        return np.uint8 if self.bpc == 8 else np.uint16

    @property
    def bytes_per_sample(self):
        return 1 if self.bpc == 8 else 2

    @property
    def frame_bytes(self):
        """Bytes of one plane of one frame (dense rows)."""
        return self.width * self.height * self.bytes_per_sample

    @property
    def pair_bytes(self):
        """Bytes read per frame pair (each plane once)."""
        return 2 * self.frame_bytes

    def generate(self, frames=None):
        """Return ``(ref, dist)`` for the frames listed (default: all)."""
        idx = range(self.n_frames) if frames is None else list(frames)
        children = np.random.SeedSequence(self.seed).spawn(self.n_frames)
        ref = np.empty((len(idx), self.height, self.width), self.dtype)
        dist = np.empty_like(ref)
        for k, f in enumerate(idx):
            rng = np.random.Generator(np.random.PCG64(children[f]))
            ref[k], dist[k] = _FRAME_MAKERS[self.kind](self, rng, f)
        return ref, dist


def _clip(a, bpc, dtype):
    return np.clip(a, 0, (1 << bpc) - 1).astype(dtype)


def _noisy_copy(sigma):
    """8-bit Netflix-pair stand-in: uniform reference, reference plus rounded
    N(0, sigma^2) as the distorted plane."""

    def make(wl, _rng, _f):
        ref = _rng.integers(0, 1 << wl.bpc, (wl.height, wl.width), dtype=np.int64)
        noise = np.rint(_rng.normal(0.0, sigma, (wl.height, wl.width))).astype(np.int64)
        return ref.astype(wl.dtype), _clip(ref + noise, wl.bpc, wl.dtype)

    return make


def _gradient_texture(wl, rng, _f):
    """Natural-content stand-in: a smooth diagonal ramp over the full range
    plus uniform texture of amplitude 64, and a lightly distorted copy
    (rounded N(0, 4^2))."""
    top = (1 << wl.bpc) - 1
    y, x = np.mgrid[0 : wl.height, 0 : wl.width]
    ramp = np.rint(top * (x + y) / max(wl.width + wl.height - 2, 1)).astype(np.int64)
    tex = rng.integers(-64, 65, (wl.height, wl.width), dtype=np.int64)
    ref = np.clip(ramp + tex, 0, top)
    noise = np.rint(rng.normal(0.0, 4.0, (wl.height, wl.width))).astype(np.int64)
    return ref.astype(wl.dtype), _clip(ref + noise, wl.bpc, wl.dtype)


def _uniform_pair(lo, hi):
    """Independent uniform planes over [lo, hi] (full-range noise, or the
    bright 16-bit pair when lo is high)."""

    def make(wl, rng, _f):
        top = (1 << wl.bpc) - 1
        a = lo if lo is not None else 0
        b = hi if hi is not None else top
        ref = rng.integers(a, b + 1, (wl.height, wl.width), dtype=wl.dtype, endpoint=False)
        dist = rng.integers(a, b + 1, (wl.height, wl.width), dtype=wl.dtype, endpoint=False)
        return ref, dist

    return make


def checkerboard(width, height, cell, bpc):
    """Cells of ``cell`` x ``cell`` samples: 0 where (x//cell + y//cell) is
    even, the top code value elsewhere."""
    y, x = np.mgrid[0:height, 0:width]
    top = (1 << bpc) - 1
    return np.where(((x // cell) + (y // cell)) % 2 == 0, 0, top)


def _bright_with_checker(wl, rng, f):
    """Bright 16-bit 4K stand-in: independent U{60000..65535} planes, except
    the last frame, a 64x64-cell checkerboard against its inverse."""
    top = (1 << wl.bpc) - 1
    if f == wl.n_frames - 1:
        ref = checkerboard(wl.width, wl.height, 64, wl.bpc)
        return ref.astype(wl.dtype), (top - ref).astype(wl.dtype)
    return _uniform_pair(60000, 65535)(wl, rng, f)


def _dark_tenth(wl, rng, _f):
    """Full-range 16-bit noise with a tenth of the samples (same positions in
    both planes) drawn from U{0..4095} instead."""
    ref, dist = _uniform_pair(None, None)(wl, rng, _f)
    mask = rng.random((wl.height, wl.width)) < 0.1
    ref[mask] = rng.integers(0, 4096, int(mask.sum()), dtype=wl.dtype)
    dist[mask] = rng.integers(0, 4096, int(mask.sum()), dtype=wl.dtype)
    return ref, dist


def _inverse_pair(wl, rng, _f):
    """Full-range reference against its inverse: the largest differences."""
    top = (1 << wl.bpc) - 1
    ref = rng.integers(0, top + 1, (wl.height, wl.width), dtype=wl.dtype)
    return ref, (top - ref).astype(wl.dtype)


def _eight_bit_widened(how):
    """8-bit content (the noisy-copy pair at sigma 8) carried in a wider
    container: shifted left by bpc - 8 bits, or multiplied by 257 to span the
    16-bit range."""

    def make(wl, rng, _f):
        ref = rng.integers(0, 256, (wl.height, wl.width), dtype=np.int64)
        noise = np.rint(rng.normal(0.0, 8.0, (wl.height, wl.width))).astype(np.int64)
        dist = np.clip(ref + noise, 0, 255)
        if how == "shift":
            k = wl.bpc - 8
            return (ref << k).astype(wl.dtype), (dist << k).astype(wl.dtype)
        return (ref * 257).astype(wl.dtype), (dist * 257).astype(wl.dtype)

    return make


_FRAME_MAKERS = {
    "noisy_copy_8": _noisy_copy(8.0),
    "gradient_texture": _gradient_texture,
    "uniform_full": _uniform_pair(None, None),
    "uniform_bright": _uniform_pair(56000, 64000),
    "bright_checker": _bright_with_checker,
    "dark_tenth": _dark_tenth,
    "inverse": _inverse_pair,
    "shifted_8": _eight_bit_widened("shift"),
    "times_257": _eight_bit_widened("257"),
}

# The five measured configurations, then the stress frames used only for
# parity past 2^53 units.
WORKLOADS = {
    "576x324_8bit_x1": Workload("576x324_8bit_x1", 576, 324, 8, 1, 1, "noisy_copy_8",
                                "Netflix 576x324 pair stand-in"),
    "1920x1080_10bit_x48": Workload("1920x1080_10bit_x48", 1920, 1080, 10, 48, 2,
                                    "gradient_texture", "natural 10-bit content stand-in"),
    "3840x2160_12bit_x32": Workload("3840x2160_12bit_x32", 3840, 2160, 12, 32, 3,
                                    "uniform_full", "full-range 12-bit noise"),
    "1920x1080_16bit_x64": Workload("1920x1080_16bit_x64", 1920, 1080, 16, 64, 4,
                                    "uniform_bright", "bright 16-bit 1080p pair stand-in"),
    "3840x2160_16bit_x32": Workload("3840x2160_16bit_x32", 3840, 2160, 16, 32, 5,
                                    "bright_checker", "bright 16-bit 4K batch + checkerboard"),
    # Other plane shapes and containers the pages run their twins on: 8-bit
    # content shifted left to 10, 12 and 16 bits, 8-bit content scaled by 257
    # to 16 bits, and 10-bit chroma planes of 4:2:2 and 4:2:0 576x324 video.
    "576x324_8bit_shifted_10": Workload("576x324_8bit_shifted_10", 576, 324, 10, 2, 21, "shifted_8",
                                        "8-bit clip shifted to 10 bits"),
    "576x324_8bit_shifted_12": Workload("576x324_8bit_shifted_12", 576, 324, 12, 2, 22, "shifted_8",
                                        "8-bit clip shifted to 12 bits"),
    "576x324_8bit_shifted_16": Workload("576x324_8bit_shifted_16", 576, 324, 16, 2, 23, "shifted_8",
                                        "8-bit clip shifted to 16 bits"),
    "1920x1080_8bit_x257_16": Workload("1920x1080_8bit_x257_16", 1920, 1080, 16, 4, 24, "times_257",
                                       "8-bit content times 257 as 16 bits"),
    "288x324_10bit_chroma422": Workload("288x324_10bit_chroma422", 288, 324, 10, 4, 25,
                                        "gradient_texture", "4:2:2 chroma plane, 10 bits"),
    "288x162_10bit_chroma420": Workload("288x162_10bit_chroma420", 288, 162, 10, 4, 26,
                                        "gradient_texture", "4:2:0 chroma plane, 10 bits"),
    "stress_full_range_4k16": Workload("stress_full_range_4k16", 3840, 2160, 16, 2, 11,
                                       "uniform_full", "full-range 16-bit 4K noise"),
    "stress_dark_tenth_4k16": Workload("stress_dark_tenth_4k16", 3840, 2160, 16, 2, 12,
                                       "dark_tenth", "a tenth of the samples below 4096"),
    "stress_inverse_4k16": Workload("stress_inverse_4k16", 3840, 2160, 16, 2, 13,
                                    "inverse", "reference against its inverse"),
}

HEADLINE = "3840x2160_16bit_x32"
# The measured configurations, in order: the Netflix-sized 8-bit pair, 1080p
# 10-bit, 4K 12-bit, 1080p 16-bit and the 4K 16-bit headline batch.
BENCH_CONFIGS = ("576x324_8bit_x1", "1920x1080_10bit_x48", "3840x2160_12bit_x32",
                 "1920x1080_16bit_x64", "3840x2160_16bit_x32")


# ---------------------------------------------------------------- psnr_hvs terms
# "ADR-1397: GPU psnr_hvs twins reproduce the CPU's running float sum bit for
# bit" gives 64 terms per 8x8 block and 10 802 176 terms for a 3840x2160 luma
# plane (Context), of which 15 to 32 % are nonzero (Consequences).  Blocks
# every 7 samples in each direction give exactly that count (548 x 308 blocks
# at 3840x2160), so term counts of other sizes follow the same grid.  The
# terms themselves (transform, CSF and masking) are not on the pages: the
# stand-in below draws non-negative float32 values of the same shape.


def hvs_blocks(width, height):
    """8x8 blocks at a step of 7 samples: ((w - 8) // 7 + 1) * ((h - 8) // 7 + 1)."""
    if width < 8 or height < 8:
        return 0
    return ((width - 8) // 7 + 1) * ((height - 8) // 7 + 1)


def hvs_term_count(width, height):
    return 64 * hvs_blocks(width, height)


# A fixed stand-in for a frequency weighting of the 64 positions of a block:
# 1 / (1 + (u + v) / 2) for coefficient (u, v), row order.  Not a CSF table.
_HVS_POS_WEIGHT = np.array([1.0 / (1.0 + (u + v) / 2.0) for v in range(8) for u in range(8)],
                           np.float32)


def _hvs_masked(wl, rng, n):
    """Masked-coefficient-error stand-in: the nonzero share q is drawn from
    U[0.15, 0.32] per plane; a nonzero term is fl(fl(e * w)^2) with e =
    fl(k - thr), k an integer error 1 + Geometric(0.3) scaled by 2^(bpc-8),
    thr ~ U[0, 1), and w the block position's weight times U[0.5, 1)."""
    q = rng.uniform(0.15, 0.32)
    nz = rng.random(n) < q
    k = (1 + rng.geometric(0.3, n)).astype(np.float32) * np.float32(1 << (wl.bpc - 8))
    thr = rng.random(n, dtype=np.float32)
    e = (k - thr).astype(np.float32)
    pos = np.arange(n) % 64
    w = (_HVS_POS_WEIGHT[pos] * rng.uniform(0.5, 1.0, n).astype(np.float32)).astype(np.float32)
    ew = (e * w).astype(np.float32)
    t = (ew * ew).astype(np.float32)
    return np.where(nz, t, np.float32(0)).astype(np.float32)


def _hvs_ones(_wl, _rng, n):
    """Every term 1.0: the running float sum stops at 2^24."""
    return np.ones(n, np.float32)


def _hvs_ties(_wl, rng, n):
    """Terms from {0.5, 1, 1.5, 2, 3} times a power of two drawn from
    2^-2..2^2: many additions land exactly halfway between two floats."""
    base = rng.choice(np.array([0.5, 1.0, 1.5, 2.0, 3.0], np.float32), n)
    return (base * np.exp2(rng.integers(-2, 3, n)).astype(np.float32)).astype(np.float32)


def _hvs_drift(_wl, rng, n):
    """2000 terms from U[16000, 16600] (a sum near 1.94 * 2^24, where the
    float sum's ulp is 2), then terms from U[0.8, 0.999], below half that ulp:
    the float sum stalls under 2^25 while the exact sum passes it."""
    head = min(2000, n)
    t = np.empty(n, np.float32)
    t[:head] = rng.uniform(16000.0, 16600.0, head).astype(np.float32)
    t[head:] = rng.uniform(0.8, 0.999, n - head).astype(np.float32)
    return t


def _hvs_subnormal(_wl, rng, n):
    """Subnormal terms (multiples of 2^-149 below 2^-126): the sum starts in
    the subnormal range and crosses into the normal one."""
    return (rng.integers(0, 1 << 10, n).astype(np.float64) * 2.0 ** -149).astype(np.float32)


def _hvs_wide(_wl, rng, n):
    """Log-uniform magnitudes over 2^-40..2^40, a third of them zero: jumps
    over many binades at once."""
    t = np.exp2(rng.uniform(-40.0, 40.0, n)).astype(np.float32)
    t[rng.random(n) < 1.0 / 3.0] = 0.0
    return t


def _hvs_zeros(_wl, _rng, n):
    return np.zeros(n, np.float32)


_HVS_MAKERS = {
    "masked": _hvs_masked,
    "ones": _hvs_ones,
    "ties": _hvs_ties,
    "drift": _hvs_drift,
    "subnormal": _hvs_subnormal,
    "wide": _hvs_wide,
    "zeros": _hvs_zeros,
}


@dataclass(frozen=True)
class HvsWorkload:
    """``n_planes`` planes of psnr_hvs terms of a width x height luma plane
    (or ``n_terms`` terms when given).  Plane p draws from child p of
    ``SeedSequence(seed)``."""

    name: str
    width: int
    height: int
    bpc: int
    n_planes: int
    seed: int
    kind: str
    n_terms_override: int = 0
    note: str = ""

    @property
    def n_terms(self):
        return self.n_terms_override or hvs_term_count(self.width, self.height)

    @property
    def plane_bytes(self):
        return 4 * self.n_terms

    def generate(self, planes=None):
        """float32 array (len(planes), n_terms)."""
        idx = range(self.n_planes) if planes is None else list(planes)
        children = np.random.SeedSequence(self.seed).spawn(self.n_planes)
        out = np.empty((len(idx), self.n_terms), np.float32)
        for k, p in enumerate(idx):
            rng = np.random.Generator(np.random.PCG64(children[p]))
            out[k] = _HVS_MAKERS[self.kind](self, rng, self.n_terms)
        return out


HVS_WORKLOADS = {
    "hvs_576x324_8bit_x4": HvsWorkload("hvs_576x324_8bit_x4", 576, 324, 8, 4, 31, "masked",
                                       note="Netflix 576x324 luma stand-in"),
    "hvs_1920x1080_10bit_x4": HvsWorkload("hvs_1920x1080_10bit_x4", 1920, 1080, 10, 4, 32,
                                          "masked", note="1920x1080 10-bit luma stand-in"),
    "hvs_3840x2160_8bit_x32": HvsWorkload("hvs_3840x2160_8bit_x32", 3840, 2160, 8, 32, 33,
                                          "masked", note="3840x2160 luma batch (BBB stand-in)"),
    "hvs_3840x2160_10bit_x2": HvsWorkload("hvs_3840x2160_10bit_x2", 3840, 2160, 10, 2, 34,
                                          "masked", note="3840x2160 10-bit luma"),
    "hvs_ones_2e24": HvsWorkload("hvs_ones_2e24", 0, 0, 8, 1, 35, "ones",
                                 n_terms_override=(1 << 24) + 4096 + 77,
                                 note="stalls at 2^24"),
    "hvs_ties": HvsWorkload("hvs_ties", 0, 0, 8, 2, 36, "ties", n_terms_override=3_000_017),
    "hvs_drift": HvsWorkload("hvs_drift", 0, 0, 8, 2, 37, "drift", n_terms_override=2_000_003),
    "hvs_subnormal": HvsWorkload("hvs_subnormal", 0, 0, 8, 2, 38, "subnormal",
                                 n_terms_override=1_000_033),
    "hvs_wide": HvsWorkload("hvs_wide", 0, 0, 8, 2, 39, "wide", n_terms_override=1_500_007),
    "hvs_zeros": HvsWorkload("hvs_zeros", 0, 0, 8, 1, 40, "zeros", n_terms_override=70_001),
}

HVS_HEADLINE = "hvs_3840x2160_8bit_x32"


def with_layout(planes, stride_bytes=None, offset_bytes=0):
    """Copy dense planes (n, h, w) into a flat byte buffer with row pitch
    ``stride_bytes`` and ``offset_bytes`` of lead-in, the layout the library
    takes (frame f at ``offset + f*h*stride``).  Padding bytes are filled with
    0xA5 so that reading them would show up in the sums."""
    n, h, w = planes.shape
    bps = planes.itemsize
    stride = w * bps if stride_bytes is None else stride_bytes
    if stride < w * bps:
        raise ValueError("stride shorter than a row")
    buf = np.full(offset_bytes + n * h * stride, 0xA5, np.uint8)
    rows = planes.reshape(n * h, w).view(np.uint8).reshape(n * h, w * bps)
    view = buf[offset_bytes:].reshape(n * h, stride)
    view[:, : w * bps] = rows
    return buf, stride
