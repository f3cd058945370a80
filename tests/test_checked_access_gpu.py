"""Every kernel under the checked build, which tests each global access against the
byte ranges the host registered for the launch (and its alignment), counts bad ones
and skips them.  One small call of every entry point and kernel family runs in a
child process against libkvq_checked.so; every launch must report a clean sync and
no bad access.  compute-sanitizer is not used: the range check is the library's own."""

import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import math, sys, torch
sys.path.insert(0, sys.argv[1])
from quantized_kv_cache_nvfp4_gb300 import _abi, build
_abi.load(build.build(checked=True))
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth

dev = torch.device("cuda", 0)
T, H, D, bs = 300, 8, 128, 16
k = synth.normal_bf16((T, H, D), 1, synth.STREAM_K, device="cuda")
v = synth.normal_bf16((T, H, D), 1, synth.STREAM_V, device="cuda")
nblk = (T + bs - 1) // bs
perm = synth.block_permutation(nblk, 1).to(dev)
t = torch.arange(T, device=dev)
slots = (perm[t // bs].long() * bs + t % bs).contiguous()
table = perm.view(1, nblk).to(torch.int32).contiguous()
lens = torch.tensor([T], dtype=torch.int32, device=dev)

# paged pools: NVFP4, FP8, and the split FP8 K / NVFP4 V pool
for fk, fv in ((kvq.FMT_NVFP4, None), (kvq.FMT_FP8, None), (kvq.FMT_FP8, kvq.FMT_NVFP4)):
    pool = kvq.KvPool.empty(nblk * bs, H, D, bs, fmt=fk, v_fmt=fv)
    kvq.kvq_quant_scatter(k, v, slots, pool)
    ko = torch.empty((1, T, H, D), dtype=torch.bfloat16, device=dev)
    vo = torch.empty_like(ko)
    kvq.kvq_restore(pool, table, lens, T, ko, vo)

# logical codecs, both kinds; INT4 with a partial group
for fmt in (kvq.FMT_NVFP4, kvq.FMT_FP8, kvq.FMT_INT4, kvq.FMT_NVFP4_TENSOR):
    for kind in (kvq.KIND_KEY, kvq.KIND_VALUE):
        pk = kvq.Packed.empty(fmt, kind, T, H, D, 64, device=dev)
        kvq.kvq_pack(k, pk)
        kvq.kvq_unpack(pk, torch.empty_like(k))

# residuals against a predecessor, 25% of rows kept: copy and in place
cur, prev = synth.layer_kv(T, H, D, seed=2, device="cuda")
pos = synth.sorted_positions(T, T // 4, 2).to(dev)
for fmt in (kvq.FMT_INT4, kvq.FMT_NVFP4, kvq.FMT_FP8):
    for kind in (kvq.KIND_KEY, kvq.KIND_VALUE):
        pay = kvq.Packed.empty(fmt, kind, T // 4, H, D, 64, device=dev)
        kvq.kvq_encode_residual(cur, prev, pos, pay)
        kvq.kvq_decode_residual(pay, pos, prev, torch.empty_like(prev))
        y = prev.clone()
        kvq.kvq_decode_residual(pay, pos, y, y)

# decode attention: the page-major kernel (block size 16, H 8), the head-major one
# (block size 8), with split sequences merged
lens4 = [1, 77, 0, 600]
for bsz in (16, 8):
    Tm = max(lens4)
    nb = (Tm + bsz - 1) // bsz
    S = len(lens4)
    pool = kvq.KvPool.empty(S * nb * bsz, H, D, bsz)
    kk = synth.normal_bf16((S * nb * bsz, H, D), 3, synth.STREAM_K, device="cuda")
    vv = synth.normal_bf16((S * nb * bsz, H, D), 3, synth.STREAM_V, device="cuda")
    kvq.kvq_quant_scatter(kk, vv, torch.arange(S * nb * bsz, device=dev), pool)
    tab = synth.block_permutation(S * nb, 4).to(dev).view(S, nb).to(torch.int32).contiguous()
    lt = torch.tensor(lens4, dtype=torch.int32, device=dev)
    q = synth.normal_bf16((S, 4 * H, D), 3, 9, device="cuda")
    kvq.kvq_decode_attention(pool, tab, lt, Tm, q, 1.0 / math.sqrt(D), torch.empty_like(q))
torch.cuda.synchronize()
print("done")
"""

# kernels every run must have launched (and so checked)
_EXPECTED = {
    "nvfp4_encode_kernel", "nvfp4_decode_kernel", "payload_kernel", "int4_key_kernel", "int4_value_kernel",
    "int4_key_decode_kernel", "tensor_amax_kernel", "tensor_key_encode_kernel", "tensor_value_encode_kernel",
    "tensor_key_decode_kernel", "decode_attn_page_kernel", "decode_attn_kernel", "decode_attn_merge_kernel",
}


@pytest.mark.gpu
def test_every_kernel_stays_inside_its_registered_buffers():
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "done" in r.stdout, r.stderr[-3000:]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[kvq checked]")]
    seen = {re.match(r"\[kvq checked\] (\w+):", ln).group(1) for ln in lines}
    assert _EXPECTED <= seen, sorted(_EXPECTED - seen)
    bad = [ln for ln in lines if "sync=no error bad=0" not in ln]
    assert not bad, bad[:5]
