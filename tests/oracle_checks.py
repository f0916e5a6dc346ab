"""Pins for the CPU oracle, written as functions of an oracle handle.

Each ``check_*`` raises ``AssertionError`` when the oracle breaks the property.
``test_oracle_pins.py`` runs them on the real oracle (all must pass) and
``test_oracle_mutants.py`` runs them on deliberately broken copies (each copy
must fail at least one), which shows that a plausible mistake anywhere in the
oracle is caught.

Nothing here re-types the oracle's arithmetic.  The independent facts used are:
- integer arithmetic in Python (exact sums of samples and squares);
- a pure-integer statement of IEEE-754 binary32 rounding to nearest even
  (``rne24``), which never touches the float hardware;
- correctly rounded conversions of exact rationals (``float(Fraction)``);
- closed forms (identical planes, swaps, hand-derived one-pixel values);
- for the psnr_hvs plane sum: exact rationals rounded to binary32 by an
  integer-only rule (``f32_round``), numpy's sequential float32 running sum,
  and hand-worked sums (``tests/golden/hvs_sums.txt``);
- the figures the pages print (``tests/golden/page_figures.txt``).
"""
import math
import os
from fractions import Fraction

import numpy as np

from exact_full_reference_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CAPS = {8: 60.0, 10: 72.0, 12: 84.0, 16: 108.0}


# ---------------------------------------------------------------- helpers
def bit_length(x):
    """Bit length of each element of a uint64 array, by integer steps only."""
    x = np.asarray(x, np.uint64)
    nb = np.zeros(x.shape, np.int64)
    v = x.copy()
    for sh in (32, 16, 8, 4, 2, 1):
        m = v >= np.uint64(1 << sh)
        nb += np.where(m, sh, 0)
        v = np.where(m, v >> np.uint64(sh), v)
    return nb + (v > 0)


def rne24(x):
    """Round non-negative integers (< 2^53) to 24 significant bits, ties to
    even: the IEEE-754 binary32 rule for an exact product, in integers."""
    x = np.asarray(x, np.uint64)
    s = np.maximum(bit_length(x) - 24, 0).astype(np.uint64)
    one = np.uint64(1)
    q = x >> s
    rem = x - (q << s)
    half = (one << s) >> one  # 2^(s-1), or 0 when nothing is dropped
    up = (rem > half) | ((rem == half) & (half > 0) & ((q & one) == one))
    return (q + up.astype(np.uint64)) << s


def exact_units(ref, dist, chunk=1 << 20):
    """Independent exact sums (Python integers) of one frame: the rounded
    squares of the raw differences and of the raw samples, and the samples.
    Taken a chunk of pixels at a time (small temporaries)."""
    rr = np.asarray(ref).ravel()
    dd = np.asarray(dist).ravel()
    out = dict.fromkeys(("noise_units", "ref_sum", "dist_sum", "ref_sumsq", "dist_sumsq"), 0)
    for i in range(0, rr.size, chunk):
        r = rr[i : i + chunk].astype(np.int64)
        d = dd[i : i + chunk].astype(np.int64)
        D = np.abs(r - d).astype(np.uint64)
        out["noise_units"] += int(rne24(D * D).sum(dtype=np.uint64))
        out["ref_sum"] += int(r.sum())
        out["dist_sum"] += int(d.sum())
        out["ref_sumsq"] += int(rne24(r.astype(np.uint64) ** 2).sum(dtype=np.uint64))
        out["dist_sumsq"] += int(rne24(d.astype(np.uint64) ** 2).sum(dtype=np.uint64))
    return out


def correctly_rounded(num, den):
    return float(Fraction(num, den))


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def page_figures():
    return {r[0]: r[1] for r in read_table("page_figures.txt")}


def run(orc, ref, dist, bpc):
    sc, un = orc.frames(ref, dist, bpc)
    return sc, un


_cache = {}


def cached(key, fn):
    if key not in _cache:
        _cache[key] = fn()
    return _cache[key]


def small_random(bpc, seed, h=37, w=53, lo=0, hi=None):
    rng = np.random.Generator(np.random.PCG64(seed))
    top = (1 << bpc) - 1 if hi is None else hi
    dt = np.uint8 if bpc == 8 else np.uint16
    ref = rng.integers(lo, top + 1, (h, w)).astype(dt)
    dist = rng.integers(lo, top + 1, (h, w)).astype(dt)
    return ref, dist


# ---------------------------------------------------------------- checks
def check_single_pixel_golden(orc):
    """Hand-derived one-pixel terms (tests/golden/single_pixel_terms.txt) and
    the scores they imply."""
    for bpc, r, d, nu, rss, dss in (map(int, row) for row in read_table("single_pixel_terms.txt")):
        dt = np.uint8 if bpc == 8 else np.uint16
        sc, un = run(orc, np.array([[r]], dt), np.array([[d]], dt), bpc)
        u = un[0]
        assert int(u["noise_units"]) == nu, (bpc, r, d, int(u["noise_units"]), nu)
        assert int(u["ref_sumsq"]) == rss and int(u["dist_sumsq"]) == dss, (bpc, r, d)
        assert int(u["ref_sum"]) == r and int(u["dist_sum"]) == d
        S = 1 << (bpc - 8)
        s = sc[0]
        assert s["noise"] == correctly_rounded(nu, S * S), (bpc, r, d, s["noise"])
        assert s["mse"] == s["noise"]
        assert s["ref_mean"] == correctly_rounded(r, S) and s["dist_mean"] == correctly_rounded(d, S)
        assert s["ref_meansq"] == correctly_rounded(rss, S * S)
        assert s["dist_meansq"] == correctly_rounded(dss, S * S)


def check_psnr_closed_forms(orc):
    """Frames whose MSE is 65025 / 10^k give PSNR = 10 k dB exactly (peak 255,
    ADR-1440 Consequences); MSE 0 gives the cap; large PSNR is capped."""
    # 8 bit, 4 pixels: squared differences 255^2 each -> MSE 65025 -> 0 dB.
    z = np.zeros((2, 2), np.uint8)
    sc, _ = run(orc, np.full((2, 2), 255, np.uint8), z, 8)
    assert sc[0]["mse"] == 65025.0 and sc[0]["psnr_uncapped"] == 0.0 and sc[0]["psnr"] == 0.0
    # 8 bit, 4 pixels, differences (51, 51, 51, 51): MSE 2601 -> 10 log10(25).
    sc, _ = run(orc, np.full((2, 2), 51, np.uint8), z, 8)
    assert sc[0]["mse"] == 2601.0
    assert abs(sc[0]["psnr_uncapped"] - 10 * math.log10(25.0)) <= 1e-12
    # 16 bit: difference 256*51 is 51 on the 8-bit scale: MSE 2601 again.
    z16 = np.zeros((2, 2), np.uint16)
    sc, _ = run(orc, np.full((2, 2), 256 * 51, np.uint16), z16, 16)
    assert sc[0]["mse"] == 2601.0
    # One code value of difference in 100 pixels at 8 bits: MSE 0.01 ->
    # 10 log10(6502500) = 68.13 dB, above the 8-bit cap of 60.
    r = np.zeros((10, 10), np.uint8)
    r[3, 7] = 1
    sc, _ = run(orc, r, np.zeros_like(r), 8)
    assert sc[0]["mse"] == 0.01
    assert abs(sc[0]["psnr_uncapped"] - 10 * math.log10(6502500.0)) <= 1e-12
    assert sc[0]["psnr"] == CAPS[8]


def check_identical_planes(orc):
    """Identical planes: noise 0, PSNR at the cap, uncapped PSNR infinite."""
    for bpc in (8, 10, 12, 16):
        ref, _ = small_random(bpc, 100 + bpc)
        sc, un = run(orc, ref, ref.copy(), bpc)
        assert int(un[0]["noise_units"]) == 0 and sc[0]["noise"] == 0.0 and sc[0]["mse"] == 0.0
        assert sc[0]["psnr"] == CAPS[bpc] and sc[0]["psnr"] == orc.psnr_cap(bpc)
        assert math.isinf(sc[0]["psnr_uncapped"]) and sc[0]["psnr_uncapped"] > 0
        assert sc[0]["ref_mean"] == sc[0]["dist_mean"] and sc[0]["ref_meansq"] == sc[0]["dist_meansq"]


def check_swap_symmetry(orc):
    """Swapping the planes keeps the noise and swaps the moments."""
    for bpc in (8, 10, 12, 16):
        ref, dist = small_random(bpc, 200 + bpc)
        a, ua = run(orc, ref, dist, bpc)
        b, ub = run(orc, dist, ref, bpc)
        assert a[0]["noise"] == b[0]["noise"] and a[0]["psnr"] == b[0]["psnr"]
        assert a[0]["ref_mean"] == b[0]["dist_mean"] and a[0]["ref_meansq"] == b[0]["dist_meansq"]
        assert a[0]["dist_mean"] == b[0]["ref_mean"] and a[0]["dist_meansq"] == b[0]["ref_meansq"]
        assert ua[0]["ref_sumsq"] == ub[0]["dist_sumsq"] and ua[0]["noise_units"] == ub[0]["noise_units"]


def check_units_integer_identity_le12(orc):
    """Below 13 bits every square is smaller than 2^24, so fp32 holds it and
    the float square equals the integer one (ADR-1440 Decision, ADR-1447
    Context)."""
    for bpc in (8, 10, 12):
        for seed in range(3):
            ref, dist = small_random(bpc, 300 + 10 * bpc + seed)
            _, un = run(orc, ref, dist, bpc)
            r = ref.astype(np.int64)
            d = dist.astype(np.int64)
            assert int(un[0]["noise_units"]) == int(((r - d) ** 2).sum())
            assert int(un[0]["ref_sumsq"]) == int((r * r).sum())
            assert int(un[0]["dist_sumsq"]) == int((d * d).sum())
            assert int(un[0]["ref_sum"]) == int(r.sum()) and int(un[0]["dist_sum"]) == int(d.sum())


def check_units_rne24_16bit(orc):
    """With 16-bit samples a square can need up to 32 bits, and fp32 keeps the
    24 leading ones, rounding to nearest with ties to even (ADR-1447
    Decision); checked against the pure-integer rounding on full-range,
    bright and small-difference frames."""
    cases = [
        small_random(16, 400),
        small_random(16, 401, lo=56000, hi=64000),
        small_random(16, 402, lo=30000, hi=36000),
    ]
    # Exact ties at every scale: differences 2^k + 1 for k = 12..15 and 32776.
    ties = np.array([[4097, 8193, 16385, 32769, 32776, 65535]], np.uint16)
    cases.append((ties, np.zeros_like(ties)))
    for ref, dist in cases:
        _, un = run(orc, ref, dist, 16)
        ex = exact_units(ref, dist)
        for k, v in ex.items():
            assert int(un[0][k]) == v, (k, int(un[0][k]), v)


def check_scores_equal_exact_sums(orc):
    """Below 2^53 units a double holds every partial sum exactly (ADR-1440
    Consequences, ADR-1447 Decision), so every score must equal the correctly
    rounded quotient of the independent exact integer sums."""
    cases = [(bpc, None) + small_random(bpc, 500 + bpc) for bpc in (8, 10, 12, 16)]
    cases += [(16, None) + small_random(16, 520, lo=56000, hi=64000)]
    b4 = cached("bright1080p0", lambda: wl.WORKLOADS["1920x1080_16bit_x64"].generate([0]))
    cases += [(16, "bright1080p0_ex", b4[0][0], b4[1][0])]
    for bpc, key, ref, dist in cases:
        sc, _ = run(orc, ref, dist, bpc)
        if key is None:
            ex = exact_units(ref, dist)
        else:
            ex = cached(key, lambda: exact_units(ref, dist))
        S = 1 << (bpc - 8)
        N = ref.size
        s = sc[0]
        assert ex["noise_units"] < 2 ** 53
        assert s["noise"] == correctly_rounded(ex["noise_units"], S * S)
        assert s["mse"] == correctly_rounded(ex["noise_units"], S * S * N)
        assert s["ref_mean"] == correctly_rounded(ex["ref_sum"], S * N)
        assert s["dist_mean"] == correctly_rounded(ex["dist_sum"], S * N)
        if ex["ref_sumsq"] < 2 ** 53:
            assert s["ref_meansq"] == correctly_rounded(ex["ref_sumsq"], S * S * N)
        if ex["dist_sumsq"] < 2 ** 53:
            assert s["dist_meansq"] == correctly_rounded(ex["dist_sumsq"], S * S * N)


def check_stride_and_batch_layout(orc):
    """Padding between rows and frame order do not change a frame's results."""
    ref, dist = small_random(10, 600, h=9, w=13)
    ref3 = np.stack([ref, dist, ref])
    dist3 = np.stack([dist, dist, ref])
    dense_s, dense_u = orc.frames(ref3, dist3, 10)
    rb, stride = wl.with_layout(ref3, stride_bytes=13 * 2 + 6, offset_bytes=4)
    db, _ = wl.with_layout(dist3, stride_bytes=13 * 2 + 6, offset_bytes=4)
    pad_s, pad_u = orc.batch(rb, db, 13, 9, stride, 10, 3, offset=4)
    assert (dense_s.tobytes() == pad_s.tobytes()) and (dense_u.tobytes() == pad_u.tobytes())
    one_s, _ = orc.frames(ref3[1:2], dist3[1:2], 10)
    assert one_s.tobytes() == dense_s[1:2].tobytes()
    assert dense_s[1]["noise"] == 0.0


def check_past_2_53_page_measurements(orc):
    """ADR-1447 Consequences reports, beyond 2^53 units, a gap of about 1.2e-7
    between the CPU's rounded total and the exact one on full-range 3840x2160
    noise, and no gap when all samples exceed 60000; both are reproduced here
    on synthetic frames, within the bound."""
    import oracle as _o

    figs = page_figures()
    full = cached("full4k", lambda: wl.WORKLOADS["stress_full_range_4k16"].generate([0]))
    ex = cached("full4k_ex", lambda: exact_units(full[0][0], full[1][0]))
    sc, un = run(orc, full[0][0], full[1][0], 16)
    N = full[0][0].size
    assert int(un[0]["ref_sumsq"]) == ex["ref_sumsq"] and ex["ref_sumsq"] >= 2 ** 53
    exact = Fraction(ex["ref_sumsq"], 65536 * N)
    diff = abs(float(Fraction(sc[0]["ref_meansq"]) - exact))
    bound = _o.moment_bound(N, _o.binade(ex["ref_sumsq"]))
    page = float(figs["measured_full_range_3840x2160"])
    assert 0 < diff <= bound
    assert page / 10 < diff < page * 10, diff  # the page's magnitude
    bright = cached("bright4k0", lambda: wl.WORKLOADS["3840x2160_16bit_x32"].generate([0]))
    exb = cached("bright4k0_ex", lambda: exact_units(bright[0][0], bright[1][0]))
    scb, _ = run(orc, bright[0][0], bright[1][0], 16)
    assert exb["ref_sumsq"] >= 2 ** 53 and bright[0][0].min() >= 60000
    assert float(figs["measured_all_above_60000"]) == 0.0
    # distance 0: the CPU's value is the exact sum's correctly rounded quotient
    assert scb[0]["ref_meansq"] == correctly_rounded(exb["ref_sumsq"], 65536 * N)
    assert scb[0]["dist_meansq"] == correctly_rounded(exb["dist_sumsq"], 65536 * N)


def check_noise_limit_2_53(orc):
    """ADR-1440 Consequences: the CPU's 16-bit noise total stops being exact
    once it reaches 2^53 units (of 2^-16 each); the inverse pair (MSE far
    above the 16570 limit at 3840x2160) crosses that point, so its double sum
    rounds, and stays within the analogous bound."""
    import oracle as _o

    inv = cached("inv4k", lambda: wl.WORKLOADS["stress_inverse_4k16"].generate([0]))
    ex = cached("inv4k_ex", lambda: exact_units(inv[0][0], inv[1][0]))
    sc, un = run(orc, inv[0][0], inv[1][0], 16)
    N = inv[0][0].size
    assert int(un[0]["noise_units"]) == ex["noise_units"] and ex["noise_units"] > 2 ** 53
    limit = 2 ** 37 / N
    assert sc[0]["mse"] > limit
    exact_mse = Fraction(ex["noise_units"], 65536 * N)
    diff = abs(float(Fraction(sc[0]["mse"]) - exact_mse))
    assert diff <= _o.mse_bound(N, ex["noise_units"])


# ---------------------------------------------------------------- integer psnr
def int_run(orc, ref, dist, bpc):
    return orc.int_psnr_frames(ref, dist, bpc)[0]


def check_int_psnr_closed_forms(orc):
    """A constant difference k: SSE = N k^2, and the uncapped PSNR is
    20 log10((2^bpc - 1) / k) (the peak reading: the largest sample); a
    PSNR above the cap is capped.  Full-scale differences on many pixels
    need all 64 bits of the sum (64 (2^16 - 1)^2 > 2^32)."""
    for bpc in (8, 10, 12, 16):
        top = (1 << bpc) - 1
        dt = np.uint8 if bpc == 8 else np.uint16
        for k in (1, 3, top):
            h, w = 8, 8
            ref = np.full((h, w), k, dt) if k == top else np.arange(h * w, dtype=np.int64).reshape(h, w) % (top - k) + k
            dist = (ref.astype(np.int64) - k).astype(dt)
            out = int_run(orc, ref.astype(dt), dist, bpc)
            assert int(out["sse"]) == h * w * k * k, (bpc, k, int(out["sse"]))
            assert out["mse"] == float(k * k)
            want = 20.0 * math.log10(top / k)
            assert abs(out["psnr_uncapped"] - want) <= 1e-12 * max(1.0, want), (bpc, k, out["psnr_uncapped"], want)
            assert out["psnr"] == min(out["psnr_uncapped"], CAPS[bpc])
    # one code value in 10^4 pixels at 16 bits: 10 log10(65535^2 * 10^4) dB, capped at 108
    r = np.zeros((100, 100), np.uint16)
    r[5, 5] = 1
    out = int_run(orc, r, np.zeros_like(r), 16)
    assert int(out["sse"]) == 1 and out["mse"] == 1e-4
    assert abs(out["psnr_uncapped"] - 10 * math.log10(65535.0 ** 2 * 1e4)) <= 1e-12 * 200
    assert out["psnr"] == CAPS[16]


def check_int_psnr_identical_and_swap(orc):
    """Identical planes: SSE 0, PSNR at the cap, uncapped infinite; swapping
    the planes changes nothing."""
    for bpc in (8, 10, 12, 16):
        ref, dist = small_random(bpc, 500 + bpc)
        same = int_run(orc, ref, ref.copy(), bpc)
        assert int(same["sse"]) == 0 and same["mse"] == 0.0 and same["psnr"] == CAPS[bpc]
        assert math.isinf(same["psnr_uncapped"]) and same["psnr_uncapped"] > 0
        a, b = int_run(orc, ref, dist, bpc), int_run(orc, dist, ref, bpc)
        assert a.tobytes() == b.tobytes()


def check_int_psnr_against_float_units(orc):
    """Up to 12 bits the float square of a difference is the integer square
    (below 2^24), so the SSE equals float_psnr's exact noise units (pinned on
    their own above); at 16 bits the SSE exceeds them by the rounding the
    float squares drop, which the pure-integer rounding gives term by term,
    and the one-pixel golden values show it (4097^2 - 16785408 = 1)."""
    for bpc in (8, 10, 12, 16):
        for seed in range(2):
            ref, dist = small_random(bpc, 600 + 10 * bpc + seed)
            _, un = run(orc, ref, dist, bpc)
            out = int_run(orc, ref, dist, bpc)
            e2 = ((ref.astype(np.int64) - dist.astype(np.int64)) ** 2).astype(np.uint64)
            dropped = int((e2 - rne24(e2)).astype(np.int64).sum())
            assert int(out["sse"]) == int(un[0]["noise_units"]) + dropped, (bpc, seed)
            if bpc <= 12:
                assert dropped == 0 and int(out["sse"]) == int(un[0]["noise_units"])
            n = ref.size
            assert out["mse"] == correctly_rounded(int(out["sse"]), n)
    for bpc, r, d, nu, _, _ in (map(int, row) for row in read_table("single_pixel_terms.txt")):
        dt = np.uint8 if bpc == 8 else np.uint16
        out = int_run(orc, np.array([[r]], dt), np.array([[d]], dt), bpc)
        assert int(out["sse"]) == (r - d) ** 2 and (r - d) ** 2 - nu >= 0, (bpc, r, d)


def check_int_psnr_layout(orc):
    """Padded rows and frames of a batch: the padding is never read, and frame
    f of the batch is the frame alone."""
    for bpc in (8, 16):
        bps = 1 if bpc == 8 else 2
        ref, dist = small_random(bpc, 700 + bpc, h=9, w=13)
        alone = int_run(orc, ref, dist, bpc)
        pad = 7 * bps
        stride = 13 * bps + pad
        rb = np.full((3, 9, stride), 0xA5, np.uint8)
        db = np.full((3, 9, stride), 0x5A, np.uint8)
        for f in range(3):
            rb[f, :, : 13 * bps] = ref.view(np.uint8).reshape(9, 13 * bps)
            db[f, :, : 13 * bps] = dist.view(np.uint8).reshape(9, 13 * bps)
        out = orc.int_psnr(rb, db, 13, 9, stride, bpc, 3)
        for f in range(3):
            assert out[f].tobytes() == alone.tobytes()


# ---------------------------------------------------------------- psnr_hvs plane sum
def f32_round(x):
    """Round an exact rational to IEEE-754 binary32, to nearest with ties to
    the even significand, subnormals kept (exponent floor -126), in integer
    arithmetic only."""
    x = Fraction(x)
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q = x / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def _hvs_value(tok):
    """A golden-file token: a decimal, or m*s<k> / s<k> for m * 2^k.  The
    decimals are rounded to float32 exactly as a C float literal is."""
    if "s" in tok:
        m, _, k = tok.partition("s")
        m = int(m.rstrip("*")) if m else 1
        return Fraction(m) * Fraction(2) ** int(k)
    return f32_round(Fraction(tok))


def _exact_running_sum(terms):
    s = Fraction(0)
    for t in terms:
        s = f32_round(s + Fraction(float(t)))
    return s


def _hvs_sets(n=3000):
    """Seeded term sets of several shapes (small, for the rational reference)."""
    out = []
    for kind in ("masked", "ties", "subnormal", "wide", "drift"):
        w = wl.HvsWorkload("pin_" + kind, 0, 0, 10, 1, 90 + len(out), kind, n_terms_override=n)
        out.append(w.generate()[0])
    return out


def check_hvs_sum_exact_rounding(orc):
    """The oracle's plane sum equals the running sum taken with exact
    rationals and an explicit binary32 rounding after every addition."""
    for t in _hvs_sets():
        s, _ = orc.hvs(t, 10)
        assert Fraction(float(s[0])) == _exact_running_sum(t)


def check_hvs_sum_matches_numpy_accumulate(orc):
    """The plane sum is the last element of numpy's float32 running sum
    (``np.add.accumulate``, a strictly sequential float32 loop), on larger
    sets and on a 4:2:0-sized plane of the masked stand-in."""
    sets = [wl.HvsWorkload("acc_" + k, 0, 0, 8, 1, 70 + i, k, n_terms_override=200_003).generate()[0]
            for i, k in enumerate(("masked", "ties", "wide", "subnormal", "drift"))]
    sets.append(wl.HVS_WORKLOADS["hvs_576x324_8bit_x4"].generate([1])[0])
    for t in sets:
        s, _ = orc.hvs(t, 8)
        ref = np.add.accumulate(t, dtype=np.float32)[-1]
        assert s[0].tobytes() == ref.tobytes(), (s[0], ref)


def check_hvs_golden_sums(orc):
    """Hand-worked running sums (ties to even, lost quarter-ulps, order,
    subnormals, 0.1 + 0.2): ``tests/golden/hvs_sums.txt``."""
    for row in read_table("hvs_sums.txt"):
        want = _hvs_value(row[0])
        terms = np.array([float(_hvs_value(x)) for x in row[1:]], np.float32)
        s, _ = orc.hvs(terms, 8)
        assert Fraction(float(s[0])) == want, (row, float(s[0]))


def check_hvs_ones_stall_at_2_24(orc):
    """A plane of ones: the float sum reaches 2^24 and stays there (every
    later addition is a tie resolved to the even 2^24)."""
    n = (1 << 24) + 77
    s, sc = orc.hvs(np.ones(n, np.float32), 8)
    assert float(s[0]) == 2.0 ** 24


def check_hvs_score_closed_forms(orc):
    """score = (sum / count) / peak^2 in float.  Terms equal to peak^2 give
    exactly 1 at 8, 10 and 12 bits (every step exact); a plane whose sum is
    3 and count 3 gives the float nearest 1 / 65025 at 8 bits; and on
    sums where the order of the two divisions matters, the count comes first."""
    for bpc in (8, 10, 12):
        peak = (1 << bpc) - 1
        n = 5 if bpc < 12 else 1
        s, sc = orc.hvs(np.full(n, peak * peak, np.float32), bpc)
        assert float(s[0]) == n * peak * peak and float(sc[0]) == 1.0, (bpc, s, sc)
    s, sc = orc.hvs(np.ones(3, np.float32), 8)
    assert Fraction(float(sc[0])) == f32_round(Fraction(1, 65025))
    rng = np.random.default_rng(5)
    found = 0
    for _ in range(4000):
        v = f32_round(Fraction(int(rng.integers(1, 1 << 24))) / int(rng.integers(1, 1 << 10)))
        n = int(rng.integers(2, 2000))
        count_first = f32_round(f32_round(v / n) / 65025)
        one_division = f32_round(v / f32_round(Fraction(n * 65025)))
        if count_first == one_division:
            continue
        terms = np.zeros(n, np.float32)
        terms[0] = float(v)
        s, sc = orc.hvs(terms, 8)
        assert Fraction(float(sc[0])) == count_first, (v, n)
        found += 1
        if found == 8:
            break
    assert found == 8


def check_hvs_batch_layout(orc):
    """Planes sit ``pitch`` floats apart; only the first n_terms of each are
    added (the padding holds values that would change any sum), and each
    plane's result equals the plane taken alone."""
    rng = np.random.default_rng(11)
    n, pitch, planes = 1001, 1100, 3
    buf = np.full((planes, pitch), 1.0e6, np.float32)
    buf[:, :n] = rng.uniform(0, 100, (planes, n)).astype(np.float32)
    s, sc = orc.hvs(buf, 10, n_terms=n, pitch=pitch, n_planes=planes)
    for p in range(planes):
        s1, sc1 = orc.hvs(np.ascontiguousarray(buf[p, :n]), 10)
        assert s[p].tobytes() == s1[0].tobytes() and sc[p].tobytes() == sc1[0].tobytes()
        assert Fraction(float(s1[0])) == _exact_running_sum(buf[p, :n])


ALL_CHECKS = [
    check_hvs_sum_exact_rounding,
    check_hvs_sum_matches_numpy_accumulate,
    check_hvs_golden_sums,
    check_hvs_ones_stall_at_2_24,
    check_hvs_score_closed_forms,
    check_hvs_batch_layout,
    check_int_psnr_closed_forms,
    check_int_psnr_identical_and_swap,
    check_int_psnr_against_float_units,
    check_int_psnr_layout,
    check_single_pixel_golden,
    check_psnr_closed_forms,
    check_identical_planes,
    check_swap_symmetry,
    check_units_integer_identity_le12,
    check_units_rne24_16bit,
    check_scores_equal_exact_sums,
    check_stride_and_batch_layout,
    check_past_2_53_page_measurements,
    check_noise_limit_2_53,
]
