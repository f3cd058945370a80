"""Host check of the NVFP4 block-scale shortcut of the encode kernels.

The block scale is the E4M3 code of t = min((vb / 6) / rs, 448) ("feat(kvcache): add
nvfp4 kv quantization (FreeToken PR #408)", codec-delta port note).  The kernels
first bracket t by te = (vb * RN(1/6)) * RN(1/rs) widened by 2^-20 either side and
take the code directly when both ends of the bracket agree, dividing only
otherwise.  tests/block_scale_check.c checks on 27.5 M structured pairs (uniform
fractions of the row maximum, and t within 8 ulps of every E4M3 rounding midpoint)
that an agreeing bracket always gives the code of t.  Its E4M3 encoder is a
brute-force nearest search written from the format definition.  A collapsed bracket
must be caught.
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
    out = tmp_path_factory.mktemp("bs") / "block_scale_check"
    subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-o", str(out),
                    os.path.join(HERE, "block_scale_check.c"), "-lm"], check=True)
    return str(out)


def test_agreeing_bracket_gives_the_defined_code(checker):
    r = subprocess.run([checker], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert ", 0 wrong" in r.stdout


def test_collapsed_bracket_is_caught(checker):
    r = subprocess.run([checker, "plant"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, r.stdout + r.stderr
