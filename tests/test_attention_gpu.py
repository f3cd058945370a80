"""Paged decode attention over the quantised pool on the GPU through the C ABI,
compared with the oracle's fp64 attention of the same pool rows.

Tolerance, from the kernel's arithmetic: K and V decode exactly, Q enters f16
exactly (a power-of-two prescale), products and sums run in fp32; the softmax
weights are rounded once to f16 (relative 2^-11) relative to a reference of V's
row scales, and the output once to bf16 (relative 2^-9).  Numerator and denominator
see different weight roundings, so the weights contribute at most 2^-11 * vmax
(vmax = the largest |v| the row attends to).  The test allows twice each term:
|o - o_ref| <= 2^-8 |o_ref| + 2^-10 vmax (+ 1e-30 for exact zeros)."""

import math

import numpy as np
import pytest
import torch

import oracle as O
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth
from kvq_testutil import POISON, bits, poison_bf16, status_word, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
NV, F8 = kvq.FMT_NVFP4, kvq.FMT_FP8


def _case(S, H, group, D, lens, fmt_k=NV, fmt_v=NV, bs=16, seed=0, spare=3, q_scale=1.0):
    """Token rows N(0,1) (1% x20 outliers) scattered through a shuffled block table."""
    Tmax = max(max(lens), 1)
    mb = -(-Tmax // bs)
    nblocks = S * mb + spare
    table = synth.block_permutation(nblocks, seed)[: S * mb].view(S, mb).contiguous()
    pool = kvq.KvPool.empty(nblocks * bs, H, D, bs, fill=0, fmt=fmt_k, v_fmt=fmt_v)
    k = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_K, 0.01, 20.0)
    v = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_V, 0.01, 20.0)
    for s, n in enumerate(lens):
        if n == 0:
            continue
        t = torch.arange(n)
        slots = (table[s, t // bs].long() * bs + t % bs).to(DEV)
        kvq.kvq_quant_scatter(k[s, :n].to(DEV), v[s, :n].to(DEV), slots, pool)
    q = (synth.normal_bf16((S, H * group, D), seed, 9).float() * q_scale).to(torch.bfloat16)
    return pool, table, torch.tensor(lens, dtype=torch.int32), q, v, Tmax


def _planes(pool):
    kb = None if pool.k_bscale is None else np.ascontiguousarray(u8(pool.k_bscale))
    vb = None if pool.v_bscale is None else np.ascontiguousarray(u8(pool.v_bscale))
    return ((np.ascontiguousarray(u8(pool.k_codes)), kb, pool.k_rscale.cpu().numpy()),
            (np.ascontiguousarray(u8(pool.v_codes)), vb, pool.v_rscale.cpu().numpy()))


def _run(pool, table, lens, q, Tmax, scale, max_seq_len=None, out=None):
    st = status_word()
    out = poison_bf16(tuple(q.shape)) if out is None else out
    kvq.kvq_decode_attention(pool, table.to(DEV), lens.to(DEV), max_seq_len or Tmax, q.to(DEV), scale, out,
                             dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _check(out, ref, v, lens, group):
    got = out.float().cpu().numpy().astype(np.float64)
    S, Hq, D = ref.shape
    for s, n in enumerate(lens):
        if n == 0:
            assert (got[s] == 0).all()
            continue
        vmax = v[s, :n].float().abs().amax(dim=(0, 2)).numpy().astype(np.float64)  # per KV head
        vmax = np.repeat(vmax, group) * 1.01  # the decoded rows stay within 1% of the inputs' maximum
        bound = 2.0 ** -8 * np.abs(ref[s]) + 2.0 ** -10 * vmax[:, None] + 1e-30
        err = np.abs(got[s] - ref[s])
        assert (err <= bound).all(), f"seq {s}: max err/bound {np.max(err / bound):.3f}"


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("group", [1, 4, 7, 8, 9, 16])  # one head n-tile up to 8, two from 9
def test_matches_oracle_nvfp4(D, group):
    lens = [1, 37, 200, 0, 16]
    pool, table, lt, q, v, Tmax = _case(5, 2, group, D, lens, seed=D + group)
    scale = 1.0 / math.sqrt(D)
    out, st = _run(pool, table, lt, q, Tmax, scale)
    assert st == 0
    pk, pv = _planes(pool)
    ref, ost = O.decode_attention(pk, pv, NV, NV, 16, table.numpy(), lt.numpy(), bits(q), scale)
    assert ost == 0
    _check(out, ref, v, lens, group)


@pytest.mark.parametrize("fmt_k,fmt_v", [(F8, F8), (F8, NV), (NV, F8)])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("group", [4, 12])
def test_matches_oracle_fp8_and_split_formats(fmt_k, fmt_v, D, group):
    lens = [130, 5, 64]
    pool, table, lt, q, v, Tmax = _case(3, 2, group, D, lens, fmt_k, fmt_v,
                                        seed=3 * D + fmt_k + 2 * fmt_v + group)
    scale = 1.0 / math.sqrt(D)
    out, st = _run(pool, table, lt, q, Tmax, scale)
    assert st == 0
    pk, pv = _planes(pool)
    ref, ost = O.decode_attention(pk, pv, fmt_k, fmt_v, 16, table.numpy(), lt.numpy(), bits(q), scale)
    assert ost == 0
    _check(out, ref, v, lens, group)


@pytest.mark.parametrize("group", [8, 16])  # one and two head n-tiles
def test_long_sequences_merge_several_splits(group):
    """Two sequences on one KV head: many splits per sequence, merged in the workspace."""
    lens = [4096, 1500]
    pool, table, lt, q, v, Tmax = _case(2, 1, group, 128, lens, seed=11)
    assert kvq.kvq_decode_attention_workspace(2, 1, group, 128, Tmax) > 0
    out, st = _run(pool, table, lt, q, Tmax, 0.0883883)
    assert st == 0
    pk, pv = _planes(pool)
    ref, _ = O.decode_attention(pk, pv, NV, NV, 16, table.numpy(), lt.numpy(), bits(q), 0.0883883)
    _check(out, ref, v, lens, group)


@pytest.mark.parametrize("H,bs,fmts", [
    (4, 16, (NV, NV)), (8, 16, (F8, NV)), (16, 16, (NV, NV)), (16, 32, (F8, F8)),  # page-major kernel
    (4, 64, (NV, F8)), (1, 32, (NV, NV)), (2, 16, (F8, NV)), (8, 16, (NV, NV)),
    (8, 256, (NV, NV)),
    (3, 16, (NV, NV)), (8, 8, (NV, NV)), (2, 1, (F8, NV)),  # head-major kernel: H = 3, block sizes 8, 1
])
def test_kv_head_counts_and_block_sizes(H, bs, fmts):
    """Both attention kernels against the oracle: the page-major kernel (block sizes that
    are multiples of 16, H in {1, 2, 4, 8, 16}: one to eight 16-token chunks a stage,
    warps of one head merging through shared memory) and the head-major one (other
    shapes).  Lengths with partial chunks and pages, one empty sequence, and a sequence
    long enough to be split."""
    fk, fv = fmts
    lens = [1, 77, 0, 600, 3000]
    pool, table, lt, q, v, Tmax = _case(5, H, 4, 128, lens, fk, fv, bs=bs, seed=20 + H + bs)
    scale = 1.0 / math.sqrt(128)
    out, st = _run(pool, table, lt, q, Tmax, scale)
    assert st == 0
    pk, pv = _planes(pool)
    ref, ost = O.decode_attention(pk, pv, fk, fv, bs, table.numpy(), lt.numpy(), bits(q), scale)
    assert ost == 0
    _check(out, ref, v, lens, 4)


@pytest.mark.parametrize("q_scale", [1e-30, 3e4])
def test_query_magnitudes_outside_f16(q_scale):
    """Queries far below and above the f16 range enter the MMA through the power-of-two
    prescale; the softmax of huge scores is one-hot-like."""
    lens = [40, 17]
    pool, table, lt, q, v, Tmax = _case(2, 2, 2, 128, lens, seed=12, q_scale=q_scale)
    out, st = _run(pool, table, lt, q, Tmax, 0.0883883)
    assert st == 0
    pk, pv = _planes(pool)
    ref, _ = O.decode_attention(pk, pv, NV, NV, 16, table.numpy(), lt.numpy(), bits(q), 0.0883883)
    _check(out, ref, v, lens, 2)


def test_bad_length_and_bad_block_leave_the_output_untouched():
    lens = [20, 40, 9]
    pool, table, lt, q, v, Tmax = _case(3, 2, 2, 128, lens, seed=13)
    bad_lens = torch.tensor([20, 10 ** 6, 9], dtype=torch.int32)
    out, st = _run(pool, table, bad_lens, q, Tmax, 0.1)
    assert st == kvq.DEV_BAD_SEQLEN
    assert (bits(out[1]) == 0xA5A5).all() and not (bits(out[0]) == 0xA5A5).any()
    bad_table = table.clone()
    bad_table[2, 0] = 10 ** 6
    out, st = _run(pool, bad_table, lt, q, Tmax, 0.1)
    assert st == kvq.DEV_BAD_BLOCK
    assert (bits(out[2]) == 0xA5A5).all() and not (bits(out[1]) == 0xA5A5).any()
    # the same with several splits per sequence (the merge leaves it untouched too)
    out, st = _run(pool, bad_table, lt, q, Tmax, 0.1, max_seq_len=4096)
    assert st == kvq.DEV_BAD_BLOCK and (bits(out[2]) == 0xA5A5).all()


def test_graph_capture_matches_eager():
    lens = [300, 77]
    pool, table, lt, q, v, Tmax = _case(2, 2, 4, 128, lens, seed=14)
    td, ld, qd = table.to(DEV), lt.to(DEV), q.to(DEV)
    ws = torch.empty(max(kvq.kvq_decode_attention_workspace(2, 2, 8, 128, Tmax), 16), dtype=torch.uint8, device=DEV)
    eager = poison_bf16(tuple(q.shape))
    kvq.kvq_decode_attention(pool, td, ld, Tmax, qd, 0.1, eager, workspace=ws)
    graphed = poison_bf16(tuple(q.shape))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_decode_attention(pool, td, ld, Tmax, qd, 0.1, graphed, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), graphed.view(torch.int16))


def test_paged_32_sequences_of_8192_tokens_sampled():
    """The restore workload's pool (32 x 8192 tokens, 8 KV heads, D128, 16,384 shuffled
    blocks) read by 32 query heads (GQA 4); 4 sequences checked against the oracle,
    and all 32 against attention of the restored bf16 rows (within bf16 noise)."""
    S, Tmax, H, D, bs, Hq = 32, 8192, 8, 128, 16, 32
    nblocks = S * Tmax // bs
    perm = synth.block_permutation(nblocks, seed=3).to(DEV)
    table = perm.view(S, Tmax // bs).contiguous()
    k = synth.normal_bf16((S * Tmax, H, D), 3, synth.STREAM_K, device=DEV)
    v = synth.normal_bf16((S * Tmax, H, D), 3, synth.STREAM_V, device=DEV)
    t = torch.arange(Tmax, device=DEV)
    slots = (table[:, t // bs].long() * bs + t % bs).reshape(-1)
    pool = kvq.KvPool.empty(nblocks * bs, H, D, bs)
    kvq.kvq_quant_scatter(k, v, slots, pool)
    q = synth.normal_bf16((S, Hq, D), 3, 9, device=DEV)
    lens = torch.full((S,), Tmax, dtype=torch.int32, device=DEV)
    out = poison_bf16((S, Hq, D))
    st = status_word()
    kvq.kvq_decode_attention(pool, table, lens, Tmax, q, 1.0 / math.sqrt(D), out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pk, pv = _planes(pool)
    pick = [0, 7, 19, 31]
    ref, _ = O.decode_attention(pk, pv, NV, NV, bs, table.cpu().numpy()[pick], lens.cpu().numpy()[pick],
                                bits(q[pick]), 1.0 / math.sqrt(D))
    vv = v.view(S, Tmax, H, D)
    _check(out[pick], ref, vv[pick].cpu(), [Tmax] * 4, Hq // H)
    # all sequences against torch attention of the restored bf16 rows
    ko, vo = torch.empty((S, Tmax, H, D), dtype=torch.bfloat16, device=DEV), torch.empty((S, Tmax, H, D), dtype=torch.bfloat16, device=DEV)
    kvq.kvq_restore(pool, table, lens, Tmax, ko, vo)
    kr = ko.permute(0, 2, 1, 3).repeat_interleave(Hq // H, dim=1).float()
    vr = vo.permute(0, 2, 1, 3).repeat_interleave(Hq // H, dim=1).float()
    ref2 = torch.nn.functional.scaled_dot_product_attention(q.float()[:, :, None], kr, vr,
                                                            scale=1.0 / math.sqrt(D))[:, :, 0]
    assert (out.float() - ref2).abs().max().item() < 0.02


@pytest.mark.parametrize("bs,fmts", [(16, (NV, NV)), (16, (F8, NV)), (8, (NV, F8))])
def test_many_short_sequences(bs, fmts):
    """A decode batch of 300 short sequences (0 to 200 tokens, a tenth of them empty):
    few or no splits, so most outputs are written by the attention kernel itself.
    Block size 16 runs the page-major kernel, 8 the head-major one."""
    rng = np.random.default_rng(31 + bs)
    lens = [0 if rng.random() < 0.1 else int(rng.integers(1, 201)) for _ in range(300)]
    fk, fv = fmts
    pool, table, lt, q, v, Tmax = _case(300, 8, 4, 128, lens, fk, fv, bs=bs, seed=40 + bs)
    scale = 1.0 / math.sqrt(128)
    out, st = _run(pool, table, lt, q, Tmax, scale)
    assert st == 0
    pk, pv = _planes(pool)
    ref, ost = O.decode_attention(pk, pv, fk, fv, bs, table.numpy(), lt.numpy(), bits(q), scale)
    assert ost == 0
    _check(out, ref, v, lens, 4)
