"""Build step for libkvq.so (sm_103a only).

Each .cu under csrc/ is compiled by nvcc in parallel into _build/, then linked into
quantized_kv_cache_nvfp4_gb300/libkvq.so with the CUDA runtime linked statically.
Codec arithmetic is compiled without FMA contraction, flush-to-zero or fast
division (-fmad=false -ftz=false -prec-div=true), which the bit-exact contract
with the CPU definition of the codec needs.

    python -m quantized_kv_cache_nvfp4_gb300.build
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", platform.machine())
LIB = os.path.join(PKG, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH, "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(INCLUDE, "kvq.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, verbose: bool, checked: bool = False) -> str:
    bdir = BUILD_DIR + ("-checked" if checked else "")
    obj = os.path.join(bdir, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) > max(os.path.getmtime(src), _headers_mtime()):
        return obj
    cmd = [nvcc(), *NVCC_FLAGS, *(["-DKVQ_CHECKED"] if checked else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libkvq.so; returns its path.

    checked=True builds libkvq_checked.so instead: a debugging variant in which
    every global access of every kernel is tested against the buffer ranges of its
    launch, recorded and skipped when out of range, and each launch is followed by
    a synchronisation and a one-line report on stderr."""
    os.makedirs(BUILD_DIR + ("-checked" if checked else ""), exist_ok=True)
    out = LIB.replace("libkvq.so", "libkvq_checked.so") if checked else LIB
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, checked), srcs))
    if os.path.exists(out) and os.path.getmtime(out) > max(os.path.getmtime(o) for o in objs):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libkvq.so failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checked="--checked" in sys.argv))
