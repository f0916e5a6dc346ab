"""Plant a mistake in a copy of the oracle and show that a pin catches it.

Each mutant is a textual change of ``oracle/vqx_oracle.c`` that a careless
implementation of the pages could plausibly contain.  The copy is compiled with
the oracle's own flags into a temporary directory and every pin of
``oracle_checks`` is run on it: at least one must fail.  (CPU only; the planted
mistakes live in the oracle copy, never in the GPU path.)
"""
import os

import pytest

import oracle
import oracle_checks as oc
from oracle import build as obuild

MUTANTS = [
    ("exact integer difference square",
     "float dsq = diff * diff;\n            noise += (uint64_t)dsq;",
     "noise += (uint64_t)((long long)(r - d) * (long long)(r - d));"),
    ("exact integer sample squares",
     "float rsq = (float)r * (float)r;",
     "double rsq = (double)r * (double)r;"),
    ("noise square taken in double",
     "float sq = e * e;",
     "double sq = (double)e * (double)e;"),
    ("noise accumulated in float",
     "double noise = 0.0;",
     "float noise = 0.0f;"),
    ("moment accumulated in float",
     "double sum = 0.0, sum2 = 0.0;",
     "float sum = 0.0f, sum2 = 0.0f;"),
    ("scaler 2^bpc in the noise",
     "const float scaler = (float)(1u << (bpc - 8));\n    double noise",
     "const float scaler = (float)(1u << bpc);\n    double noise"),
    ("scaler 2^bpc in the moments",
     "const float scaler = (float)(1u << (bpc - 8));\n    double sum",
     "const float scaler = (float)(1u << bpc);\n    double sum"),
    ("sum instead of difference",
     "float e = r - d;",
     "float e = r + d;"),
    ("second moment without the square",
     "const float term = pic * pic;",
     "const float term = pic;"),
    ("first moment divided by n - 1",
     "*mean = sum / n;",
     "*mean = sum / (n - 1.0);"),
    ("MSE divided by the width only",
     "out->mse = out->noise / ((double)w * (double)h);",
     "out->mse = out->noise / (double)w;"),
    ("peak 2^bpc - 1 instead of 255",
     "10.0 * log10(255.0 * 255.0 / out->mse)",
     "10.0 * log10(1023.0 * 1023.0 / out->mse)"),
    ("no PSNR cap",
     "out->psnr = out->psnr_uncapped < cap ? out->psnr_uncapped : cap;\n\n    plane_moments",
     "out->psnr = out->psnr_uncapped;\n\n    plane_moments"),
    ("distorted moments taken from the reference",
     "plane_moments(d, w, h, stride, bpc, &out->dist_mean, &out->dist_meansq);",
     "plane_moments(r, w, h, stride, bpc, &out->dist_mean, &out->dist_meansq);"),
    ("row pitch ignored",
     "const unsigned char *rrow = ref + (size_t)y * stride;",
     "const unsigned char *rrow = ref + (size_t)y * (size_t)w * (bpc == 8 ? 1u : 2u);"),
    ("integer psnr: peak 2^bpc",
     "const double peak = (double)((1u << bpc) - 1);",
     "const double peak = (double)(1u << bpc);"),
    ("integer psnr: peak 255 at every depth",
     "const double peak = (double)((1u << bpc) - 1);",
     "const double peak = 255.0;"),
    ("integer psnr: 32-bit sum",
     "uint64_t sse = 0;",
     "uint32_t sse = 0;"),
    ("integer psnr: float squares",
     "sse += (uint64_t)(e * e);",
     "sse += (uint64_t)((float)e * (float)e);"),
    ("integer psnr: absolute differences",
     "sse += (uint64_t)(e * e);",
     "sse += (uint64_t)(e < 0 ? -e : e);"),
    ("integer psnr: MSE over n - 1",
     "out->mse = (double)sse / ((double)w * (double)h);",
     "out->mse = (double)sse / ((double)w * (double)h - 1.0);"),
    ("integer psnr: no cap",
     "out->psnr = out->psnr_uncapped < cap ? out->psnr_uncapped : cap;\n    return VQX_ORACLE_OK;\n}\n\nint vqx_oracle_int_psnr_batch",
     "out->psnr = out->psnr_uncapped;\n    return VQX_ORACLE_OK;\n}\n\nint vqx_oracle_int_psnr_batch"),
    ("integer psnr: distorted plane read as the reference",
     "(int64_t)sample_at(rrow, x, bpc) - (int64_t)sample_at(drow, x, bpc)",
     "(int64_t)sample_at(rrow, x, bpc) - (int64_t)sample_at(rrow, x, bpc)"),
    ("hvs: double accumulator",
     "float s = 0.0f;\n    for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];",
     "double s = 0.0;\n    for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];"),
    ("hvs: terms added last to first",
     "for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];",
     "for (int64_t i = n_terms - 1; i >= 0; i--) s = s + terms[i];"),
    ("hvs: two halves summed apart",
     "for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];",
     "float s2 = 0.0f;\n    for (int64_t i = 0; i < n_terms; i++) { if (i < n_terms / 2) s = s + terms[i]; else s2 = s2 + terms[i]; }\n    s = s + s2;"),
    ("hvs: first term skipped",
     "for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];",
     "for (int64_t i = 1; i < n_terms; i++) s = s + terms[i];"),
    ("hvs: one division by count times peak^2",
     "float q = s / (float)n_terms;\n    q = q / (peak * peak);",
     "float q = s / ((float)n_terms * (peak * peak));"),
    ("hvs: divided by the block count",
     "float q = s / (float)n_terms;",
     "float q = s / (float)(n_terms / 64 > 0 ? n_terms / 64 : 1);"),
    ("hvs: peak 2^bpc",
     "const float peak = (float)((1u << bpc) - 1u);",
     "const float peak = (float)(1u << bpc);"),
    ("hvs: plane pitch ignored",
     "terms + (size_t)p * (size_t)pitch, n_terms",
     "terms + (size_t)p * (size_t)n_terms, n_terms"),
    ("sample byte order swapped",
     "memcpy(&v, row + 2 * (size_t)x, sizeof v);\n    return v;",
     "memcpy(&v, row + 2 * (size_t)x, sizeof v);\n    return (uint16_t)((v >> 8) | (v << 8));"),
]


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation anchor must occur exactly once: %r" % old
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return obuild.build_oracle(src=path, out=os.path.join(tmp_path, "libmutant.so"), force=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    mut = oracle.Oracle(_build_mutant(str(tmp_path), old, new))
    caught = None
    for check in oc.ALL_CHECKS:
        try:
            check(mut)
        except (AssertionError, ValueError, OverflowError, ZeroDivisionError):
            caught = check.__name__
            break
    assert caught, "no pin catches the planted mistake: " + name
