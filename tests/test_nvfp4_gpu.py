"""NVFP4 quant-scatter and paged restore on the GPU, through the C ABI, compared
element by element with the CPU oracle (bit-exact: codes, block scales, row
scales and restored bf16)."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth
from kvq_testutil import (POISON, assert_rows_equal, bits, f32bits, oracle_on_all_cores, oracle_rows,
                          poison_bf16, status_word, u8)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def scatter_and_check(k, v, slots, pool, sample_tokens=None):
    """Scatter on the GPU, then compare the written slots with the oracle's rows."""
    st = status_word()
    kvq.kvq_quant_scatter(k, v, slots, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sl = slots.cpu().numpy()
    toks = np.arange(len(sl)) if sample_tokens is None else sample_tokens
    for x, codes, bsc, rsc, what in ((k, pool.k_codes, pool.k_bscale, pool.k_rscale, "K"),
                                     (v, pool.v_codes, pool.v_bscale, pool.v_rscale, "V")):
        if x is None:
            continue
        idx = torch.as_tensor(toks, device=x.device)
        c, b, r = oracle_rows(x.index_select(0, idx))
        s = torch.as_tensor(sl[toks], device=codes.device)
        assert_rows_equal(u8(codes.index_select(0, s)), u8(bsc.index_select(0, s)),
                          rsc.index_select(0, s), c, b, r, what)
    return sl


def test_one_layer_round_trip_contiguous_slots():
    """K, V [256, 8, 128], N(0,1) with 1% x20 outliers, seed 0, slots 0..255."""
    k, v, slots = synth.one_layer_case(seed=0)
    kd, vd, sd = k.to(DEV), v.to(DEV), slots.to(DEV)
    pool = kvq.Nvfp4Pool.empty(256, 8, 128, 16, fill=POISON)
    scatter_and_check(kd, vd, sd, pool)
    table = torch.arange(16, dtype=torch.int32, device=DEV).view(1, 16)
    lens = torch.tensor([256], dtype=torch.int32, device=DEV)
    ko, vo = poison_bf16((1, 256, 8, 128)), poison_bf16((1, 256, 8, 128))
    st = status_word()
    kvq.kvq_restore(pool, table, lens, 256, ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, out in ((k, ko), (v, vo)):
        want = O.nvfp4_decode_rows(*O.nvfp4_encode_rows(bits(x)))
        np.testing.assert_array_equal(bits(out[0]), want)
    # the logical pack/unpack pair gives the same bytes
    pk = kvq.Packed.empty(kvq.FMT_NVFP4, kvq.KIND_KEY, 256, 8, 128)
    kvq.kvq_pack(kd, pk)
    y = poison_bf16((256, 8, 128))
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    c, b, r = O.nvfp4_encode_rows(bits(k))
    assert_rows_equal(u8(pk.codes), u8(pk.meta0), pk.rscale, c, b, r, "pack")
    np.testing.assert_array_equal(bits(y), O.nvfp4_decode_rows(c, b, r))
    # reconstruction RMSE (information): a few percent of the N(0,1) scale
    err = (y.float() - kd.float()).pow(2).mean().sqrt().item()
    assert err < 0.2


def _decode_step_inputs():
    qkv, k, v, slots = synth.decode_step_case(seed=2)
    qkv = qkv.to(DEV)
    kd = qkv[:, :1024].unflatten(1, (8, 128))
    assert kd.stride(0) == 1152 and kd.stride(1) == 128
    vd = v.to(DEV)
    assert vd.stride(0) == 1024
    return k, v, kd, vd, slots.to(DEV)


def test_decode_step_strided_k_separate_v_pitch_under_graph_capture():
    """256 one-token appends into a 65,536-slot pool; K a view of a fused qkv (row
    pitch 1152), V its own tensor (pitch 1024); captured in a CUDA graph."""
    k, v, kd, vd, sd = _decode_step_inputs()
    pool = kvq.Nvfp4Pool.empty(65536, 8, 128, 16, fill=POISON)
    st = status_word()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        kvq.kvq_quant_scatter(kd, vd, sd, pool, st)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    pool2 = kvq.Nvfp4Pool.empty(65536, 8, 128, 16, fill=POISON)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_quant_scatter(kd, vd, sd, pool2, st)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sl = sd.cpu().numpy()
    for x, P in ((k, (pool2.k_codes, pool2.k_bscale, pool2.k_rscale)),
                 (v, (pool2.v_codes, pool2.v_bscale, pool2.v_rscale))):
        c, b, r = oracle_rows(x)
        assert_rows_equal(u8(P[0])[sl], u8(P[1])[sl], P[2].cpu()[sl], c, b, r)
    # untouched slots keep the poison bytes; the eager warm-up pool is identical
    mask = np.ones(65536, bool)
    mask[sl] = False
    assert (u8(pool2.k_codes)[mask] == POISON).all() and (u8(pool2.v_bscale)[mask] == POISON).all()
    assert (f32bits(pool2.v_rscale)[mask] == 0xA5A5A5A5).all()
    for a, b2 in ((pool.k_codes, pool2.k_codes), (pool.v_rscale, pool2.v_rscale)):
        assert torch.equal(a.view(torch.uint8), b2.view(torch.uint8))


def test_shared_pitch_regression_geometry():
    """The V-pitch bug geometry: 8 tokens, 3 KV heads, D128; K = qkv[:, 384:768] of a
    [8, 1152] fused tensor (pitch 1152), V contiguous (pitch 384)."""
    qkv = synth.normal_bf16((8, 1152), seed=30, stream=1).to(DEV)
    kd = qkv[:, 384:768].unflatten(1, (3, 128))
    vd = synth.normal_bf16((8, 3, 128), seed=30, stream=2).to(DEV)
    slots = torch.arange(8, dtype=torch.int64, device=DEV).flip(0) * 2
    pool = kvq.Nvfp4Pool.empty(16, 3, 128, 16, fill=POISON)
    scatter_and_check(kd, vd, slots, pool)


def test_restore_under_graph_capture_matches_eager():
    H, D, bs = 2, 64, 16
    k, v = synth.layer_kv(96, H, D, seed=31)
    perm = synth.block_permutation(8, seed=31).to(DEV)
    t = torch.arange(96, device=DEV)
    slots = perm[t // bs].long() * bs + t % bs
    pool = kvq.Nvfp4Pool.empty(128, H, D, bs, fill=0)
    kvq.kvq_quant_scatter(k.to(DEV), v.to(DEV), slots, pool)
    table = perm[:6].view(1, 6).contiguous()
    lens = torch.tensor([96], dtype=torch.int32, device=DEV)
    ko, vo = poison_bf16((1, 96, H, D)), poison_bf16((1, 96, H, D))
    kvq.kvq_restore(pool, table, lens, 96, ko, vo)
    ko2, vo2 = poison_bf16((1, 96, H, D)), poison_bf16((1, 96, H, D))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_restore(pool, table, lens, 96, ko2, vo2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ko.view(torch.int16), ko2.view(torch.int16))
    want = O.nvfp4_decode_rows(*O.nvfp4_encode_rows(bits(v)))
    np.testing.assert_array_equal(bits(vo2[0]), want)


def _paged_case(S, Tmax, H, D, lens, seed, bs=16, spare_blocks=3, outliers=(0.0, 1.0)):
    mb = -(-Tmax // bs)
    nblocks = S * mb + spare_blocks
    perm = synth.block_permutation(nblocks, seed)
    table = perm[: S * mb].view(S, mb).contiguous()
    k = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_K, *outliers)
    v = synth.normal_bf16((S, Tmax, H, D), seed, synth.STREAM_V, *outliers)
    return k, v, table, nblocks


@pytest.mark.parametrize("H,D", [(1, 16), (3, 48), (2, 96), (8, 128), (4, 256), (1, 512)])
def test_ragged_paged_round_trip_all_shapes(H, D):
    S, Tmax, bs = 3, 70, 16
    lens = torch.tensor([70, 33, 1], dtype=torch.int32)
    k, v, table, nblocks = _paged_case(S, Tmax, H, D, lens, seed=40 + D, outliers=(0.02, 30.0))
    pool = kvq.Nvfp4Pool.empty(nblocks * bs, H, D, bs, fill=POISON)
    for s in range(S):
        n = int(lens[s])
        t = torch.arange(n)
        slots = (table[s, t // bs].long() * bs + t % bs).to(DEV)
        scatter_and_check(k[s, :n].to(DEV), v[s, :n].to(DEV), slots, pool)
    ko, vo = poison_bf16((S, Tmax, H, D)), poison_bf16((S, Tmax, H, D))
    st = status_word()
    kvq.kvq_restore(pool, table.to(DEV), lens.to(DEV), Tmax, ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    opool = tuple(np.ascontiguousarray(a) for a in (u8(pool.k_codes), u8(pool.k_bscale), pool.k_rscale.cpu().numpy()))
    want, ost = O.nvfp4_restore(opool, bs, table.numpy(), lens.numpy(), Tmax,
                                out=np.full((S, Tmax, H, D), 0xA5A5, np.uint16))
    assert ost == 0
    np.testing.assert_array_equal(bits(ko), want)
    for s in range(S):  # rows past the sequence length are not written
        assert (bits(vo[s, int(lens[s]):]) == 0xA5A5).all()


@pytest.mark.parametrize("bs", [1, 8, 32, 64, 256])
def test_ragged_paged_round_trip_block_sizes(bs):
    """The restore's block-table arithmetic at block sizes other than 16, with a
    sequence that ends inside a block and one shorter than a block."""
    S, Tmax, H, D = 3, 300, 4, 128
    lens = torch.tensor([300, 129, 5], dtype=torch.int32)
    k, v, table, nblocks = _paged_case(S, Tmax, H, D, lens, seed=60 + bs, bs=bs)
    pool = kvq.Nvfp4Pool.empty(nblocks * bs, H, D, bs, fill=POISON)
    for s in range(S):
        n = int(lens[s])
        t = torch.arange(n)
        slots = (table[s, t // bs].long() * bs + t % bs).to(DEV)
        scatter_and_check(k[s, :n].to(DEV), v[s, :n].to(DEV), slots, pool)
    ko, vo = poison_bf16((S, Tmax, H, D)), poison_bf16((S, Tmax, H, D))
    st = status_word()
    kvq.kvq_restore(pool, table.to(DEV), lens.to(DEV), Tmax, ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for plane, got in (((pool.k_codes, pool.k_bscale, pool.k_rscale), ko),
                       ((pool.v_codes, pool.v_bscale, pool.v_rscale), vo)):
        opool = tuple(np.ascontiguousarray(a) for a in (u8(plane[0]), u8(plane[1]), plane[2].cpu().numpy()))
        want, ost = O.nvfp4_restore(opool, bs, table.numpy(), lens.numpy(), Tmax,
                                    out=np.full((S, Tmax, H, D), 0xA5A5, np.uint16))
        assert ost == 0
        np.testing.assert_array_equal(bits(got), want)


def test_unaligned_to_32_bytes_takes_the_16_byte_path():
    """A view 16 bytes off a 32-byte boundary (pitch 8 mod 16) is still exact."""
    T, H, D = 50, 2, 64
    base = synth.normal_bf16((T, H * D + 8), seed=41, stream=1).to(DEV)
    kd = base[:, 8:].unflatten(1, (H, D))
    assert kd.data_ptr() % 32 == 16
    pool = kvq.Nvfp4Pool.empty(64, H, D, 16, fill=POISON)
    scatter_and_check(kd, None, torch.arange(T, device=DEV).long(), pool)
    table = torch.arange(4, dtype=torch.int32, device=DEV).view(1, 4)
    y = poison_bf16((64, H, D + 8))[:, :, 8:]
    kvq.kvq_restore(pool, table, torch.tensor([T], dtype=torch.int32, device=DEV), 64, y, None)
    torch.cuda.synchronize()
    want = O.nvfp4_decode_rows(*oracle_rows(kd))
    np.testing.assert_array_equal(bits(y[:T]), want)


# ---------------------------------------------------------------------------
# constructed rows: rounding sweeps and the special cases the method has
# ---------------------------------------------------------------------------
def _gpu_pack_rows(x_bits: np.ndarray):
    """x [n, D] bf16 bits -> GPU (codes, bscale, rscale) through the scatter path."""
    n, D = x_bits.shape
    x = synth.from_bits(x_bits).to(DEV).view(n, 1, D)
    pool = kvq.Nvfp4Pool.empty(-(-n // 16) * 16, 1, D, 16, fill=POISON)
    kvq.kvq_quant_scatter(x, None, torch.arange(n, device=DEV).long(), pool)
    y = poison_bf16((pool.num_slots, 1, D))
    table = torch.arange(pool.num_slots // 16, dtype=torch.int32, device=DEV).view(1, -1)
    kvq.kvq_restore(pool, table, torch.tensor([n], dtype=torch.int32, device=DEV), pool.num_slots, y, None)
    torch.cuda.synchronize()
    return u8(pool.k_codes)[:n, 0], u8(pool.k_bscale)[:n, 0], pool.k_rscale.cpu()[:n, 0], bits(y)[:n, 0]


def _check_constructed(rows: np.ndarray):
    xb = O.f32_to_bf16(rows.astype(np.float32))
    c, b, r, y = _gpu_pack_rows(xb)
    wc, wb, wr = O.nvfp4_encode_rows(xb)
    assert_rows_equal(c, b, r, wc, wb, wr, "constructed")
    np.testing.assert_array_equal(y, O.nvfp4_decode_rows(wc, wb, wr))


def test_e2m1_rounding_of_every_bf16_value_in_range():
    """rs = 1 and block scale 1 make q = x exactly: every bf16 value in [-6.5, 6.5]
    goes through the hardware E2M1 rounding once."""
    allb = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f32(allb)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 6.5)]
    per_block = 15
    nblk = 15
    chunks = [vals[i:i + per_block] for i in range(0, len(vals), per_block)]
    rows = []
    for j in range(0, len(chunks), nblk):
        r = np.zeros(16 * (nblk + 1), np.float32)
        r[0] = 2688.0
        for bi, ch in enumerate(chunks[j:j + nblk], start=1):
            r[16 * bi] = 6.0
            r[16 * bi + 1:16 * bi + 1 + len(ch)] = ch
        rows.append(r)
    _check_constructed(np.array(rows))


def test_e4m3_rounding_sweep_of_block_scales():
    """rs = 1: block maxima over every bf16 value in the E4M3 range (t = vb / 6),
    plus every exact E4M3 midpoint; and rows with non-power-of-two row scales."""
    allb = np.arange(0, 1 << 15, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f32(allb)
    vals = vals[(vals >= 6 * 2.0 ** -11) & (vals <= 2688.0)]
    tab = np.array([O.e4m3_value(c) for c in range(127)], np.float64)
    mids = 6 * (tab[:-1] + tab[1:]) / 2
    vals = np.concatenate([vals, mids[mids <= 2688].astype(np.float32)])
    rows = []
    for j in range(0, len(vals), 15):
        r = np.zeros(256, np.float32)
        r[0] = 2688.0
        for bi, vb in enumerate(vals[j:j + 15], start=1):
            r[16 * bi] = vb
            r[16 * bi + 3] = -vb * 0.37
        rows.append(r)
    rng = np.random.default_rng(3)
    for _ in range(200):  # random row maxima: inexact rs and t
        r = (rng.standard_normal(256) * np.exp2(rng.uniform(-20, 20, 16)).repeat(16)).astype(np.float32)
        rows.append(r)
    _check_constructed(np.array(rows))


def test_special_rows_zero_signed_tiny_fallback_and_huge():
    rows = np.zeros((8, 64), np.float64)
    rows[1] = -0.0
    rows[2, ::3] = 2.0 ** -133                    # smallest bf16 subnormal: rs subnormal
    rows[2, 1::3] = -(2.0 ** -133)
    rows[3, 0] = 2.0 ** -110                      # reciprocal of s overflows: direct division
    rows[3, 16], rows[3, 17], rows[3, 18] = 2.0 ** -126, 2.0 ** -127, -(2.0 ** -128)
    rows[4, 0] = 1e4                              # a block far below the row maximum
    rows[4, 16:32] = 1e-4 * np.array([1, -1] * 8)
    rows[5] = 3.0e38 * np.linspace(-1, 1, 64)     # near the bf16 maximum
    rows[6] = np.where(np.arange(64) % 2, 1.0, -1.0) * 6 * 448 * 2.0 ** -20
    rows[7, 5] = -1.0                             # a single negative value
    _check_constructed(rows)


def test_exact_rows_round_trip_identically():
    rng = np.random.default_rng(5)
    e4 = np.array([O.e4m3_value(c) for c in range(40, 127)])
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    rows = []
    for k in (-90, -5, 0, 9, 70):
        for _ in range(8):
            r = np.zeros(128)
            for bi in range(8):
                e = 448.0 if bi == 0 else rng.choice(e4)
                c = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
                c[rng.integers(0, 16)] = 6.0
                r[16 * bi:16 * bi + 16] = c * e
            rows.append(r * 2.0 ** k)
    rows = np.array(rows)
    xb = O.f32_to_bf16(rows.astype(np.float32))
    _, _, _, y = _gpu_pack_rows(xb)
    np.testing.assert_array_equal(y, xb)


# ---------------------------------------------------------------------------
# device-side error reporting and host-side rejections
# ---------------------------------------------------------------------------
def test_bad_slot_block_and_length_are_flagged_not_trapped():
    H, D = 2, 32
    k, v = synth.layer_kv(5, H, D, seed=42)
    kd, vd = k.to(DEV), v.to(DEV)
    pool = kvq.Nvfp4Pool.empty(32, H, D, 16, fill=0)
    st = status_word()
    slots = torch.tensor([0, -1, 32, 5, 10**12], dtype=torch.int64, device=DEV)
    kvq.kvq_quant_scatter(kd, vd, slots, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_SLOT
    rs = pool.k_rscale.cpu()
    assert rs[0].abs().sum() > 0 and rs[5].abs().sum() > 0
    assert rs[[1, 2, 3, 4, 6]].abs().sum() == 0  # skipped tokens wrote nothing
    # the context is still usable: a correct call after the flagged one works
    st.zero_()
    table = torch.tensor([[0, 7], [1, -1]], dtype=torch.int32, device=DEV)
    out = poison_bf16((2, 32, H, D))
    kvq.kvq_restore(pool, table, torch.tensor([20, 10], dtype=torch.int32, device=DEV), 32, out, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_BLOCK
    assert (bits(out[0, 16:20]) == 0xA5A5).all()  # rows of the bad block skipped
    st.zero_()
    kvq.kvq_restore(pool, table, torch.tensor([33, 3], dtype=torch.int32, device=DEV), 32, out, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_SEQLEN


def test_host_side_rejections():
    H, D = 2, 32
    x = torch.zeros((4, H, D), dtype=torch.bfloat16, device=DEV)
    pool = kvq.Nvfp4Pool.empty(16, H, D, 16, fill=0)
    slots = torch.arange(4, device=DEV).long()
    with pytest.raises(kvq.KvqError, match="NOT_DEVICE_PTR"):
        kvq.kvq_quant_scatter(x.cpu(), None, slots, pool)
    with pytest.raises(kvq.KvqError, match="NOT_DEVICE_PTR"):
        kvq.kvq_quant_scatter(x, None, slots.cpu(), pool)
    flat = torch.zeros(4 * H * D + 4, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(kvq.KvqError, match="MISALIGNED"):
        kvq.kvq_quant_scatter(flat[4:].view(4, H, D), None, slots, pool)
    wide = torch.zeros((4, H * D + 4), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(kvq.KvqError, match="MISALIGNED"):
        kvq.kvq_quant_scatter(wide[:, :H * D].unflatten(1, (H, D)), None, slots, pool)
    kvq.kvq_quant_scatter(x[:0], None, slots[:0], pool)  # empty: a no-op


# ---------------------------------------------------------------------------
# the two full-size workloads, every row against the oracle
# ---------------------------------------------------------------------------
def _check_every_row(x, slots, planes, out_rows):
    """Codes, block scales and row scales of every (token, head) row of x, read from
    the pool at its slot, and the restored bf16 of every row, against the oracle run
    on all of x (on every host core)."""
    xb = bits(x)
    c, b, r = oracle_on_all_cores(O.nvfp4_encode_rows, xb)
    del xb
    assert_rows_equal(u8(planes[0].index_select(0, slots)), u8(planes[1].index_select(0, slots)),
                      planes[2].index_select(0, slots), c, b, r)
    want = oracle_on_all_cores(O.nvfp4_decode_rows, c, b, r)
    np.testing.assert_array_equal(bits(out_rows), want)


def test_paged_restore_32_sequences_of_8192_tokens_every_row():
    """32 sequences x 8192 tokens, 8 KV heads, D128, block tables a seeded permutation
    of 16,384 physical blocks: every pool row and every restored row of K and V equals
    the oracle's (FreeToken PR #408, fp8 store notes: only an exact-code check caught
    the V-pitch bug)."""
    S, Tmax, H, D, bs = 32, 8192, 8, 128, 16
    nblocks = S * Tmax // bs
    perm = synth.block_permutation(nblocks, seed=3).to(DEV)
    table = perm.view(S, Tmax // bs).contiguous()
    k = synth.normal_bf16((S * Tmax, H, D), 3, synth.STREAM_K, device=DEV)
    v = synth.normal_bf16((S * Tmax, H, D), 3, synth.STREAM_V, device=DEV)
    t = torch.arange(Tmax, device=DEV)
    slots = (table[:, t // bs].long() * bs + t % bs).reshape(-1)
    pool = kvq.Nvfp4Pool.empty(nblocks * bs, H, D, bs)
    st = status_word()
    kvq.kvq_quant_scatter(k, v, slots, pool, st)
    ko, vo = poison_bf16((S, Tmax, H, D)), poison_bf16((S, Tmax, H, D))
    lens = torch.full((S,), Tmax, dtype=torch.int32, device=DEV)
    kvq.kvq_restore(pool, table, lens, Tmax, ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_every_row(k, slots, (pool.k_codes, pool.k_bscale, pool.k_rscale), ko.view(-1, H, D))
    _check_every_row(v, slots, (pool.v_codes, pool.v_bscale, pool.v_rscale), vo.view(-1, H, D))


def test_long_context_one_million_tokens_every_row():
    """1,048,576 tokens x 4 KV heads x D256 with 0.5% x50 outliers into a 1,048,576-slot
    pool with block-shuffled slots, then a full paged restore (the bench workload):
    every pool row and every restored row of K and V equals the oracle's."""
    T, H, D, bs = 1 << 20, 4, 256, 16
    nblocks = T // bs
    perm = synth.block_permutation(nblocks, seed=5).to(DEV)
    t = torch.arange(T, device=DEV)
    slots = perm[t // bs].long() * bs + t % bs
    k = synth.normal_bf16((T, H, D), 5, synth.STREAM_K, 0.005, 50.0, device=DEV)
    v = synth.normal_bf16((T, H, D), 5, synth.STREAM_V, 0.005, 50.0, device=DEV)
    pool = kvq.Nvfp4Pool.empty(T, H, D, bs)
    st = status_word()
    kvq.kvq_quant_scatter(k, v, slots, pool, st)
    ko, vo = poison_bf16((1, T, H, D)), poison_bf16((1, T, H, D))
    kvq.kvq_restore(pool, perm.view(1, -1), torch.tensor([T], dtype=torch.int32, device=DEV), T,
                    ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_every_row(k, slots, (pool.k_codes, pool.k_bscale, pool.k_rscale), ko[0])
    _check_every_row(v, slots, (pool.v_codes, pool.v_bscale, pool.v_rscale), vo[0])
