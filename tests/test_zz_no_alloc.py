"""kvq_decode_attention_noalloc: decode attention for callers that cannot allocate.

Some callers cannot hand the library a workspace: an engine whose memory planner has
already given all free HBM to the KV pool, or a host runtime that passes in only the
tensors it owns.  For them this entry point puts the split partials in a scratch
array that is part of the library image (48 MiB per device), so no call allocates.
These tests call it through the C ABI and compare it with kvq_decode_attention given
a caller workspace.  The two run the same kernels on the same split plan, so the
outputs must be bit-identical, which is inside the attention tests' tolerance.

The file name sorts last, so a run that stops at the first failure has already run
every other test.  Each test passes alone in a fresh process and after the others.
"""

import os
import subprocess
import sys

import pytest
import torch

import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import _abi, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pool_case(lens, H=1, group=8, D=128, bs=16, seed=15):
    """A pool holding N(0,1) K/V rows (1% x20 outliers) of each sequence behind a
    shuffled block table, and two different query sets."""
    S, Tmax = len(lens), max(max(lens), 1)
    mb = -(-Tmax // bs)
    table = synth.block_permutation(S * mb + 3, seed)[: S * mb].view(S, mb).contiguous()
    pool = kvq.KvPool.empty((S * mb + 3) * bs, H, D, bs, fill=0)
    k = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_K, 0.01, 20.0)
    v = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_V, 0.01, 20.0)
    for s, n in enumerate(lens):
        t = torch.arange(n)
        slots = (table[s, t // bs].long() * bs + t % bs).to(DEV)
        kvq.kvq_quant_scatter(k[s, :n].to(DEV), v[s, :n].to(DEV), slots, pool)
    q1 = synth.normal_bf16((S, H * group, D), seed, 9).to(DEV)
    q2 = synth.normal_bf16((S, H * group, D), seed, 10).to(DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return pool, table.to(DEV), lens_d, q1, q2, Tmax


def _poisoned(shape):
    t = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    t.view(torch.uint8).fill_(0xA5)
    return t


@pytest.mark.parametrize("lens,max_len", [([4096, 1500], None), ([40], 8192), ([300, 77], None)])
def test_noalloc_two_calls_in_a_row_match_the_workspace_entry_point(lens, max_len):
    """Two calls in a row with different queries (a leftover of the first call's
    partials would show in the second) against the workspace entry point."""
    pool, table, lens_d, q1, q2, Tmax = _pool_case(lens)
    ml = max_len or Tmax
    S, Hq = q1.shape[0], q1.shape[1]
    assert kvq.kvq_decode_attention_workspace(S, 1, Hq, 128, ml) > 0 or lens == [300, 77]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for q in (q1, q2):
        b = _poisoned(tuple(q.shape))
        kvq.kvq_decode_attention_noalloc(pool, table, lens_d, ml, q, 0.1, b, dev_status=st)
        outs.append(b)
    refs = []
    for q in (q1, q2):
        a = _poisoned(tuple(q.shape))
        kvq.kvq_decode_attention(pool, table, lens_d, ml, q, 0.1, a)
        refs.append(a)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a, b in zip(refs, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


_FRESH = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from test_zz_no_alloc import _pool_case, _poisoned
import quantized_kv_cache_nvfp4_gb300 as kvq
torch.cuda.set_device(0)
pool, table, lens_d, q1, q2, Tmax = _pool_case([4096, 1500])
outs = []
for q in (q1, q2):   # the first library call on this device that needs the scratch
    b = _poisoned(tuple(q.shape))
    kvq.kvq_decode_attention_noalloc(pool, table, lens_d, Tmax, q, 0.1, b)
    outs.append(b)
for q, b in zip((q1, q2), outs):
    a = _poisoned(tuple(q.shape))
    kvq.kvq_decode_attention(pool, table, lens_d, Tmax, q, 0.1, a)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
print("fresh-process noalloc ok")
"""


def test_noalloc_first_call_in_a_fresh_process():
    """In a new process the first call does the one-time look-up of the scratch
    array's device address; its results must already match."""
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process noalloc ok" in r.stdout


def test_noalloc_worst_case_partials_fit_the_scratch_on_this_device():
    """On the real device (its own SM count), the largest split workspace over the
    supported shapes stays within the 48 MiB scratch."""
    lib = _abi.load()
    torch.cuda.init()
    worst = 0
    for S in (1, 2, 7, 32, 75, 151, 152, 300, 455, 456, 607, 608, 1000, 4096):
        for H in (1, 2, 4, 8):
            for D in (64, 128, 256):
                for T in (256, 4096, 65536, 1 << 20):
                    worst = max(worst, lib.kvq_decode_attention_workspace(S, H, H * 16, D, T))
    assert 0 < worst <= 48 << 20
