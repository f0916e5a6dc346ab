"""The oracle against facts that do not come from the oracle (CPU only)."""
import pytest

import oracle
import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    check(orc)


def test_rne24_helper_against_golden():
    """The pure-integer rounding used by the pins reproduces the hand-derived
    one-pixel values (so it is itself pinned to the golden file)."""
    import numpy as np

    for bpc, r, d, nu, rss, dss in (map(int, row) for row in oc.read_table("single_pixel_terms.txt")):
        assert int(oc.rne24(np.array([(r - d) ** 2], np.uint64))[0]) == nu
        assert int(oc.rne24(np.array([r * r], np.uint64))[0]) == rss
        assert int(oc.rne24(np.array([d * d], np.uint64))[0]) == dss


def test_page_figures_limits():
    """ADR-1440 Consequences and Decision, ADR-1447 Decision: the limits the
    pages print follow from 2^53 units of 2^-16 and from term sizes."""
    f = oc.page_figures()
    import math

    assert 256 * 4095 ** 2 == int(f["block_sum_12bit_max"]) < 2 ** 32
    lim4k = 2 ** 37 / (3840 * 2160)
    assert round(lim4k) == int(f["mse_limit_3840x2160"])
    assert 10 * math.log10(255.0 ** 2 / lim4k) < float(f["psnr_at_limit_3840x2160_below"])
    lim1080 = 2 ** 37 / (1920 * 1080)
    assert abs(lim1080 - float(f["mse_limit_1920x1080"])) / lim1080 < 0.01
    assert lim1080 > 65535.0 ** 2 / 65536  # above the largest possible error
    assert 2 ** 21 == int(f["exact_pixels_16bit"]) and 1920 * 1080 == int(f["pixels_1920x1080"])
    assert 2 ** 21 * (2 ** 32 - 1) < 2 ** 53  # 2^21 terms below 2^32 cannot reach 2^53


def test_page_figures_bound():
    """ADR-1447: the bound formula reproduces the three values the page prints."""
    f = oc.page_figures()
    n4k = 3840 * 2160

    def two_digits(x):
        return float(f"{x:.1e}")

    assert two_digits(oracle.moment_bound(n4k, 54)) == float(f["bound_3840x2160_e54"])
    # full-range 3840x2160 noise: the second-moment sum lies in [2^53, 2^54)
    assert two_digits(oracle.moment_bound(n4k, 53)) == float(f["bound_3840x2160_full_range"])
    assert two_digits(oracle.moment_bound(2560 * 1440, 53)) == float(f["bound_2560x1440"])
    assert oracle.mse_bound(n4k, 2 ** 53 - 1) == 0.0


def test_hvs_workload_matches_page_figures():
    """ADR-1397: the term count of a 3840x2160 plane and the share of nonzero
    terms that the synthetic psnr_hvs planes are built to."""
    import numpy as np

    from exact_full_reference_gb300 import workloads as wl

    f = oc.page_figures()
    assert wl.hvs_term_count(3840, 2160) == int(f["hvs_terms_3840x2160"])
    assert wl.hvs_term_count(3840, 2160) % int(f["hvs_terms_per_block"]) == 0
    lo, hi = float(f["hvs_nonzero_min"]), float(f["hvs_nonzero_max"])
    for name in ("hvs_576x324_8bit_x4", "hvs_1920x1080_10bit_x4"):
        w = wl.HVS_WORKLOADS[name]
        for t in w.generate():
            share = np.count_nonzero(t) / t.size
            assert lo - 0.01 <= share <= hi + 0.01, (name, share)
