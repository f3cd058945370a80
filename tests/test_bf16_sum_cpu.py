"""Host check of the bf16 residual arithmetic the kernels use.

Residuals are bf16(cur - prev) and reconstructions bf16(prev + y), defined with a
binary32 subtraction (addition) then a rounding to bf16 ("vllm-rlt PR #166: INT4 KV
packing/unpacking and cross-loop residual reconstruction", Purpose: residuals in the
input dtype).  The kernels use one bf16x2 subtraction (addition), which rounds the
exact result once.  tests/bf16_sum_check.c compares the two for every pair of finite
bf16 values (4.3e9 pairs, about 75 s); a planted error (truncation instead of
rounding) must be caught.
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
    d = tmp_path_factory.mktemp("bf16")
    src = os.path.join(HERE, "bf16_sum_check.c")
    out = d / "bf16_sum_check"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(out), src, "-lm"], check=True)
    text = open(src).read().replace("return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);",
                                    "return (uint16_t)(u >> 16);")
    psrc = d / "planted.c"
    psrc.write_text(text)
    planted = d / "planted"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(planted), str(psrc), "-lm"], check=True)
    return str(out), str(planted)


def test_one_rounding_equals_the_binary32_path_for_every_pair(checker):
    r = subprocess.run([checker[0]], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout
    assert r.stdout.split()[1] == "4261478400"  # every ordered pair of finite bf16 values


def test_planted_error_is_caught(checker):
    r = subprocess.run([checker[1], "97"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 1 and "mismatches 0" not in r.stdout
