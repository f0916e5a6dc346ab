"""Helpers for the GPU parity tests: device placement and the comparison rule.

The rule (per frame, per output):
- the five integer sums must equal the oracle's exact integer sums, always;
- a score whose CPU double sum is exact (its integer sum below 2^53 units,
  "ADR-1440 ...", Consequences; "ADR-1447 ...", Decision) must equal the
  oracle's double bit for bit;
- past 2^53 units it must lie within the bound "ADR-1447 ..." (Decision)
  states, for the moments, and the analogous bound for the MSE and PSNR.
"""
import math

import numpy as np

import oracle

EXACT_LIMIT = 2 ** 53
UNIT_FIELDS = ("noise_units", "ref_sum", "dist_sum", "ref_sumsq", "dist_sumsq")


def device_bytes(buf, offset=0, align=256):
    """Copy a flat uint8 numpy buffer to the GPU so that its first byte sits
    ``offset`` bytes past an ``align``-byte boundary.  Returns (tensor, ptr)."""
    import torch

    buf = np.ascontiguousarray(buf).view(np.uint8).reshape(-1)
    t = torch.empty(buf.size + align + offset, dtype=torch.uint8, device="cuda")
    base = t.data_ptr()
    start = (-base) % align + offset
    t[start : start + buf.size].copy_(torch.from_numpy(buf))
    return t, base + start


def place(ref, dist, stride=None, offset_ref=0, offset_dist=0):
    """Dense planes (n, h, w) -> device buffers with the given row pitch and
    base offsets.  Returns (keepalive, ref_ptr, dist_ptr, stride, host bytes)."""
    from exact_full_reference_gb300 import workloads as wl

    rb, stride = wl.with_layout(ref, stride)
    db, _ = wl.with_layout(dist, stride)
    tr, pr = device_bytes(rb, offset_ref)
    td, pd = device_bytes(db, offset_dist)
    return (tr, td), pr, pd, stride, (rb, db)


def range_flags(ref, dist, bpc):
    """Per frame, 1 where a sample of either plane (n, h, w) is 2^bpc or more
    (the library's VQX_FLAG_RANGE), else 0."""
    top = (1 << bpc) - 1
    n = ref.shape[0]
    over = (ref.reshape(n, -1) > top).any(axis=1) | (dist.reshape(n, -1) > top).any(axis=1)
    return [int(x) for x in over]


def compare(rec, sc, un, bpc, pixels, planes=None):
    """Assert the GPU records ``rec`` match the oracle's ``sc``/``un``.

    ``planes``: the (ref, dist) sample arrays (n, h, w) the records come
    from; the range flag of each frame must then be set exactly where a
    sample is 2^bpc or more.  Without them every frame's flags must be 0 (the
    callers pass in-range samples)."""
    assert len(rec) == len(sc) == len(un)
    want_flags = range_flags(planes[0], planes[1], bpc) if planes is not None else [0] * len(rec)
    for f in range(len(rec)):
        g, s, u = rec[f], sc[f], un[f]
        for k in UNIT_FIELDS:
            assert int(g[k]) == int(u[k]), (f, k, int(g[k]), int(u[k]))
        noise_exact = int(u["noise_units"]) < EXACT_LIMIT
        if noise_exact:
            for k in ("noise", "mse", "psnr", "psnr_uncapped"):
                assert g[k].tobytes() == s[k].tobytes(), (f, k, g[k], s[k])
        else:
            dm = oracle.mse_bound(pixels, int(u["noise_units"]))
            assert abs(g["mse"] - s["mse"]) <= dm, (f, g["mse"], s["mse"], dm)
            dp = oracle.psnr_bound(s["mse"], dm, s["psnr_uncapped"])
            assert abs(g["psnr_uncapped"] - s["psnr_uncapped"]) <= dp
            assert abs(g["psnr"] - s["psnr"]) <= dp
        for plane in ("ref", "dist"):
            assert g[plane + "_mean"].tobytes() == s[plane + "_mean"].tobytes(), (f, plane)
            units = int(u[plane + "_sumsq"])
            if units < EXACT_LIMIT:
                assert g[plane + "_meansq"].tobytes() == s[plane + "_meansq"].tobytes(), (
                    f, plane, g[plane + "_meansq"], s[plane + "_meansq"])
            else:
                bound = oracle.moment_bound(pixels, oracle.binade(units))
                assert abs(g[plane + "_meansq"] - s[plane + "_meansq"]) <= bound
        # and the flags: only out-of-range samples set one
        assert int(g["flags"]) == want_flags[f], (f, int(g["flags"]), want_flags[f])
    return True


def exact_count(un):
    """How many frames are entirely in the exact range."""
    return sum(
        1 for u in un if all(int(u[k]) < EXACT_LIMIT for k in ("noise_units", "ref_sumsq", "dist_sumsq")))


def assert_finite_or_cap(rec):
    for g in rec:
        assert not math.isnan(g["psnr"])
