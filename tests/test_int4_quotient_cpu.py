"""Host checks of the division-free quotients in the INT4 encode kernels.

The kernels form the group scale RN(D/15) and the element quotients RN(d/sc) of the
INT4 format ("vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual
reconstruction", Purpose: codes from the FP32 minimum and scale) without dividing:
a correctly rounded reciprocal and FMA residual steps (Markstein's theorem).  This
test restates that arithmetic in C (tests/int4_quotient_check.c, the C library's
fmaf and IEEE division) and compares it with the division:

- the scale for every binary32 D in [2^-64, FLT_MAX] (1.6e9 values, about 15 s);
- the element quotient on structured random pairs: bf16 groups, exact half-integer
  ties of bf16 data, quotients a few ulps from a half-integer, and uniform pairs.

A planted error (no residual step) must be caught, so the check can fail.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    out = tmp_path_factory.mktemp("q") / "int4_quotient_check"
    src = os.path.join(HERE, "int4_quotient_check.c")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(out), src, "-lm"], check=True)
    planted = tmp_path_factory.mktemp("q") / "planted"
    text = open(src).read().replace("return fmaf(fmaf(-q0, 15.0f, D), y15, q0);", "return q0;")
    text = text.replace("return fmaf(fmaf(-q1, sc, d), y, q1);", "return q0;")
    psrc = planted.with_suffix(".c")
    psrc.write_text(text)
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(planted), str(psrc), "-lm"], check=True)
    return str(out), str(planted)


def run(exe, *args):
    r = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout


def test_scale_equals_division_everywhere(checker):
    rc, out = run(checker[0], "scale-range")
    assert rc == 0, out
    assert out.split()[1] == str(0x7F800000 - 0x1F800000)  # every value from 2^-64 up


def test_element_quotient_equals_division(checker):
    rc, out = run(checker[0], "quotient", 3_000_000, 7)
    assert rc == 0, out
    assert int(out.split()[1]) > 2_000_000  # most draws are in the domain


def test_planted_error_is_caught(checker):
    _, planted = checker
    rc, out = run(planted, "scale-binades", 0, 1)
    assert rc == 1 and "mismatches 0" not in out
    rc, out = run(planted, "quotient", 300_000, 7)
    assert rc == 1 and "mismatches 0" not in out
