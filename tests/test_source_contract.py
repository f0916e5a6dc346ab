"""Device-free contract checks of the library's build and sources.

The pages guard their exact twins with source-level contract tests: each
names a regression that would silently change a result and fails on a copy
of the code with that regression planted ("ADR-1447: float_moment_hip adds
the float squares the CPU adds, ...", Consequences: four planted regressions
in the contract test).  These do the same for the four things here that the
GPU parity tests could only catch on a GPU, and only for inputs that happen
to exercise them:

- the compiler must not merge a product into a following add (device code
  built with --fmad=false, host code with -ffp-contract=off, no fast-math
  anywhere; the oracle additionally without auto-vectorisation, which would
  reorder its double running sums);
- every 32-bit accumulator run must hold its worst-case terms;
- the packed fp32 square must stay one fused multiply-add with a +0 addend
  (a plain packed multiply was found fused into the add that consumes it);
- kernels launched as programmatic dependents must not read through the
  read-only data path (a walk that did returned an earlier call's records),
  and the psnr_hvs walk must keep its register bound.

Each check returns the problems it finds; every test also plants the
regression in a copy of the text and asserts that the check reports it.
"""
import os
import re

import pytest

from exact_full_reference_gb300 import build as vb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNELS = os.path.join(ROOT, "exact_full_reference_gb300", "csrc", "vqx_kernels.cuh")
CSRC = os.path.join(ROOT, "exact_full_reference_gb300", "csrc")

FAST_MATH = ("--use_fast_math", "-use_fast_math", "--ftz=true", "-ftz=true", "--prec-div=false",
             "-prec-div=false", "--prec-sqrt=false", "-prec-sqrt=false", "-ffast-math", "-Ofast",
             "--fmad=true", "-fmad=true", "-ffp-contract=fast", "-ffp-contract=on")


def check_library_flags(cmd):
    problems = []
    if "--fmad=false" not in cmd:
        problems.append("device code without --fmad=false")
    host = " ".join(a for a in cmd if a.startswith("-Xcompiler"))
    for flag in ("-ffp-contract=off", "-fno-fast-math"):
        if flag not in host:
            problems.append("host code without " + flag)
    for arg in cmd:
        for bad in FAST_MATH:
            if bad in arg:
                problems.append("fast-math or contraction flag " + bad)
    return problems


def check_oracle_flags(cflags):
    problems = []
    for flag in ("-ffp-contract=off", "-fno-fast-math", "-fno-tree-vectorize"):
        if flag not in cflags:
            problems.append("oracle without " + flag)
    for bad in FAST_MATH + ("-O3", "-march=native", "-ftree-vectorize"):
        if bad in cflags:
            problems.append("oracle with " + bad)
    return problems


def strip_comments(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def constant(src, struct_head, name):
    """The value of `static constexpr uint32_t name = N;` inside the struct
    whose declaration starts with struct_head."""
    i = src.index(struct_head)
    m = re.compile(r"static constexpr uint32_t %s = (\d+)u?;" % name).search(src, i)
    return int(m.group(1))


U32 = (1 << 32) - 1


def check_run_bounds(src):
    """Worst cases of the 32-bit runs between flushes (a vector is 16 bytes of
    each plane; samples in a uint16 container may hold any 16-bit value)."""
    problems = []
    f8 = constant(src, "struct TermSums<8> {", "kFlushVecs")
    # 8 bits: four dp4a words a vector, each adding at most 4 * 255^2
    if f8 * 4 * 4 * 255 * 255 > U32:
        problems.append("8-bit square runs overflow: %d vectors" % f8)
    f1012 = constant(src, "struct TermSums {", "kFlushVecs")
    # 10 and 12 bits: 8 samples a vector into the 32-bit sample sums
    if f1012 * 8 * 0xFFFF > U32:
        problems.append("10/12-bit sample-sum runs overflow: %d vectors" % f1012)
    f16 = constant(src, "struct Sums16 {", "kFlushVecs")
    max_terms = constant(src, "struct SplitSum2 {", "kMaxTerms")
    if f16 * 8 * 0xFFFF > U32:
        problems.append("16-bit sample-sum runs overflow: %d vectors" % f16)
    if 8 * f16 > max_terms:
        problems.append("16-bit square runs exceed SplitSum2's bound")
    # the SSE form's fp32 lanes add one rounding error (at most 128 in
    # magnitude) per word of a vector: exact while below 2^24
    if 4 * f16 * 128 > (1 << 24):
        problems.append("16-bit rounding-error runs leave fp32's exact integers")
    # SplitSum2: sum(h) / 2^16 below 2^32 and |sum(l)| below 2^31
    if max_terms * (1 << 16) > U32 or max_terms * (1 << 15) >= (1 << 31):
        problems.append("SplitSum2 bound too large: %d terms" % max_terms)
    return problems


def check_square_form(src):
    code = strip_comments(src)
    problems = []
    if re.search(r"\bmul(\.rn)?\.f32x2\b", code):
        problems.append("a plain packed multiply")
    m = re.search(r"f32x2 f2_square\(f32x2 a\) \{(.*?)\n\}", code, re.S)
    if not m:
        problems.append("f2_square missing")
    else:
        body = m.group(1)
        if "fma.rn.f32x2 %0, %1, %1, %2;" not in body or '"l"(0ull)' not in body:
            problems.append("f2_square is not one fma with a +0 addend")
    return problems


def kernel_sources():
    out = {}
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, name)) as f:
                out[name] = f.read()
    return out


# --------------------------------------------------------------------- the real files
def test_library_build_keeps_products_apart():
    assert check_library_flags(vb.command("libvqx.so")) == []


def test_oracle_build_keeps_the_pages_arithmetic():
    import oracle.build as ob

    assert check_oracle_flags(ob.CFLAGS) == []


def test_accumulator_runs_hold_their_worst_case():
    with open(KERNELS) as f:
        assert check_run_bounds(f.read()) == []


def test_fp32_squares_are_single_roundings_everywhere():
    for name, src in kernel_sources().items():
        problems = check_square_form(src) if name == "vqx_kernels.cuh" else [
            p for p in check_square_form(src) if p == "a plain packed multiply"]
        assert problems == [], (name, problems)


# --------------------------------------------------------------------- planted regressions
@pytest.mark.parametrize("plant", [
    lambda c: [a for a in c if a != "--fmad=false"],
    lambda c: c + ["--use_fast_math"],
    lambda c: [a.replace("-ffp-contract=off", "-ffp-contract=fast") for a in c],
    lambda c: [a.replace(",-fno-fast-math", "") for a in c],
], ids=["fmad", "fast-math", "host-contraction", "host-fast-math"])
def test_planted_library_flag_regressions_are_caught(plant):
    assert check_library_flags(plant(vb.command("libvqx.so")))


@pytest.mark.parametrize("plant", [
    lambda f: [a for a in f if a != "-ffp-contract=off"],
    lambda f: [a for a in f if a != "-fno-tree-vectorize"],
    lambda f: [a.replace("-O2", "-O3") for a in f],
    lambda f: f + ["-ffast-math"],
], ids=["contraction", "vectorise", "O3", "fast-math"])
def test_planted_oracle_flag_regressions_are_caught(plant):
    import oracle.build as ob

    assert check_oracle_flags(plant(list(ob.CFLAGS)))


@pytest.mark.parametrize("struct_head,new", [
    ("struct TermSums<8> {", 8192),
    ("struct TermSums {", 16384),
    ("struct Sums16 {", 8192),
], ids=["8-bit", "10-12-bit", "16-bit"])
def test_planted_run_length_overflows_are_caught(struct_head, new):
    with open(KERNELS) as f:
        src = f.read()
    i = src.index(struct_head)
    j = src.index("kFlushVecs = ", i)
    k = src.index(";", j)
    planted = src[:j] + "kFlushVecs = %d" % new + src[k:]
    assert check_run_bounds(planted)


def test_planted_error_run_overflow_is_caught():
    with open(KERNELS) as f:
        src = f.read()
    i = src.index("struct Sums16 {")
    j = src.index("kFlushVecs = ", i)
    k = src.index(";", j)
    planted = src[:j] + "kFlushVecs = 65536" + src[k:]
    assert "16-bit rounding-error runs leave fp32's exact integers" in check_run_bounds(planted)


def test_planted_split_bound_overflow_is_caught():
    with open(KERNELS) as f:
        src = f.read()
    planted = src.replace("kMaxTerms = 32768;", "kMaxTerms = 131072;")
    assert planted != src and check_run_bounds(planted)


@pytest.mark.parametrize("old,new", [
    ('asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(d) : "l"(a), "l"(0ull));',
     'asm("mul.rn.f32x2 %0, %1, %1;" : "=l"(d) : "l"(a));'),
    ('"l"(0ull));', '"l"(c));'),
], ids=["plain-multiply", "nonzero-addend"])
def test_planted_square_regressions_are_caught(old, new):
    with open(KERNELS) as f:
        src = f.read()
    planted = src.replace(old, new, 1)
    assert planted != src and check_square_form(planted)


# ---------------------------------------------------------------- dependent launches
# Kernels launched as programmatic dependents start before the kernel ahead
# has ended; the read-only data path (__ldg, ld.global.nc) needs data
# unchanged for the reading kernel's whole run, and a psnr_hvs walk that read
# the tables' records through it returned records of an earlier call.  Every
# kernel of the replay and psnr_hvs files is such a dependent, and so is
# stage 2 (frame_sums) in the fused file.
DEPENDENT_FILES = ("vqx_ordered.cuh", "vqx_hvs.cuh")


def function_body(text, signature):
    """The text of the function whose definition starts with ``signature``
    (from its opening brace to the matching closing brace)."""
    start = text.index(signature)
    i = text.index("{", start)
    depth = 0
    for j in range(i, len(text)):
        depth += {"{": 1, "}": -1}.get(text[j], 0)
        if depth == 0:
            return text[i : j + 1]
    raise ValueError("unbalanced braces after %r" % signature)


def check_dependent_loads(texts):
    """texts: file name -> source.  Returns the problems found."""
    problems = []
    for name in DEPENDENT_FILES:
        for m in re.finditer(r"__ldg\s*\(|ld\.global\.nc", texts[name]):
            line = texts[name].count("\n", 0, m.start()) + 1
            problems.append("%s:%d reads through the read-only data path" % (name, line))
    body = function_body(texts["vqx_kernels.cuh"], "frame_sums(const Partial")
    if re.search(r"__ldg\s*\(|ld\.global\.nc", body) or "__ldcg" not in body:
        problems.append("frame_sums does not read the records through L2")
    if not re.search(r"__launch_bounds__\(32,\s*24\)\s*hvs_walk", texts["vqx_hvs.cuh"]):
        problems.append("hvs_walk lost its bound of 80 registers (it must fit beside a tables CTA)")
    return problems


def dependent_sources():
    names = DEPENDENT_FILES + ("vqx_kernels.cuh",)
    return {n: open(os.path.join(CSRC, n)).read() for n in names}


def test_dependent_kernels_read_through_l2():
    assert check_dependent_loads(dependent_sources()) == []


@pytest.mark.parametrize("plant", ["walk_ldg", "ordered_ldg", "frame_sums_plain", "walk_bound"])
def test_planted_dependent_load_regressions_are_caught(plant):
    texts = dependent_sources()
    if plant == "walk_ldg":
        texts["vqx_hvs.cuh"] = texts["vqx_hvs.cuh"].replace("r.k = __ldcg(", "r.k = __ldg(", 1)
    elif plant == "ordered_ldg":
        texts["vqx_ordered.cuh"] = texts["vqx_ordered.cuh"].replace(
            "return __ldcg(reinterpret_cast<const uint4 *>(p));",
            "return __ldg(reinterpret_cast<const uint4 *>(p));", 1)
    elif plant == "frame_sums_plain":
        body = function_body(texts["vqx_kernels.cuh"], "frame_sums(const Partial")
        texts["vqx_kernels.cuh"] = texts["vqx_kernels.cuh"].replace(body, body.replace("__ldcg", "__ldg"))
    else:
        texts["vqx_hvs.cuh"] = texts["vqx_hvs.cuh"].replace("__launch_bounds__(32, 24) hvs_walk",
                                                            "__launch_bounds__(32) hvs_walk", 1)
    assert texts != dependent_sources(), "the plant did not apply"
    assert check_dependent_loads(texts), plant
