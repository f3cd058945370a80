"""Host check of the multiply-shift division (kvq::FastDiv in kvq_params.h) that the
kernels use to split flat row and task indices (Granlund & Montgomery, "Division by
invariant integers using multiplication", PLDI 1994).  tests/fastdiv_check.cpp
compiles the header's host path and compares quotient and remainder with the
hardware division for numerators below 2^31 (the host checks keep every index the
kernels split below that bound).  A planted off-by-one in the multiplier must be
caught, so the check can fail.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_kv_cache_nvfp4_gb300", "csrc")


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        inc = os.path.join(d, "include") if d else ""
        if inc and os.path.exists(os.path.join(inc, "cuda_runtime.h")):
            return inc
    return None


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("no C++ compiler or CUDA headers")
    out = tmp_path_factory.mktemp("fd") / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-I", inc, "-o", str(out),
                    os.path.join(HERE, "fastdiv_check.cpp")], check=True)
    return str(out)


def test_fastdiv_matches_division(checker):
    r = subprocess.run([checker], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert ", 0 wrong" in r.stdout


def test_planted_multiplier_error_is_caught(checker):
    r = subprocess.run([checker, "plant"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, r.stdout + r.stderr
