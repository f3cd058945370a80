"""Pins of the oracle's paged decode attention (fp64) against torch's
scaled_dot_product_attention on the same K/V values.

The pools are built from rows the codecs represent exactly (format-grid values with
the row's largest code present; the round trip of such rows is pinned in
test_oracle_pins.py), so the decoded K/V are known without decoding them here."""

import numpy as np
import pytest
import torch

import oracle as O

NVFP4, FP8 = O.FMT_NVFP4, O.FMT_FP8


def _exact_nvfp4_rows(rng, n, D, lo=-6, hi=6):
    """n rows [D] of e2m1 * e4m3 * 2^k values: every 16-block holds code 6 (so its
    block scale is exact) and block 0 has scale 448 (so the row scale is 2^k)."""
    e4 = np.array([O.e4m3_value(c) for c in range(40, 127)])
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    rows = np.zeros((n, D))
    for i in range(n):
        k = rng.integers(lo, hi + 1)
        for b in range(D // 16):
            e = 448.0 if b == 0 else rng.choice(e4)
            c = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
            c[rng.integers(0, 16)] = 6.0 * rng.choice([-1, 1])
            rows[i, 16 * b:16 * b + 16] = c * e
        rows[i] *= 2.0 ** k
    return rows


def _exact_fp8_rows(rng, n, D, lo=-6, hi=6):
    e4 = np.array([O.e4m3_value(c) for c in range(0, 127)])
    rows = rng.choice(e4, (n, D)) * rng.choice([-1, 1], (n, D))
    rows[np.arange(n), rng.integers(0, D, n)] = 448.0
    return rows * (2.0 ** rng.integers(lo, hi + 1, (n, 1)))


def _pool(rows_k, rows_v, fmt_k, fmt_v, H, D, slots_of, num_slots):
    """Encode token rows [T][H][D] into pool planes at slots_of[t]."""
    planes = []
    for rows, fmt in ((rows_k, fmt_k), (rows_v, fmt_v)):
        xb = O.f32_to_bf16(rows.astype(np.float32))
        assert (O.bf16_to_f32(xb) == rows).all()  # the rows are exact in bf16 too
        if fmt == FP8:
            c, r = O.fp8_encode_rows(xb)
            codes = np.zeros((num_slots, H, D), np.uint8)
            bs = None
        else:
            c, b, r = O.nvfp4_encode_rows(xb)
            codes = np.zeros((num_slots, H, D // 2), np.uint8)
            bs = np.zeros((num_slots, H, D // 16), np.uint8)
            bs[slots_of] = b
        rs = np.zeros((num_slots, H), np.float32)
        codes[slots_of] = c
        rs[slots_of] = r
        # the pool rows decode back to the rows exactly
        dec = O.fp8_decode_rows(c, r) if fmt == FP8 else O.nvfp4_decode_rows(c, b, r)
        np.testing.assert_array_equal(O.bf16_to_f32(dec), rows)
        planes.append((codes, bs, rs))
    return planes


def _sdpa(q, k, v, scale):
    """torch reference, float64: q [Hq, D], k/v [T, Hq, D] (already expanded per query head)."""
    qt = torch.from_numpy(q)[:, None, :]                     # [Hq, 1, D]
    kt = torch.from_numpy(k).permute(1, 0, 2)                # [Hq, T, D]
    vt = torch.from_numpy(v).permute(1, 0, 2)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[:, 0].numpy()


def _case(fmt_k, fmt_v, H=2, Hq=4, D=64, bs=16, lens=(37, 16, 1), seed=0):
    rng = np.random.default_rng(seed)
    S = len(lens)
    mb = -(-max(lens) // bs)
    nblocks = S * mb + 2
    perm = rng.permutation(nblocks).astype(np.int32)
    table = perm[:S * mb].reshape(S, mb)
    T = sum(lens)
    gen = {NVFP4: _exact_nvfp4_rows, FP8: _exact_fp8_rows}
    rows_k = gen[fmt_k](rng, T * H, D).reshape(T, H, D)
    rows_v = gen[fmt_v](rng, T * H, D).reshape(T, H, D)
    slots = []
    for s, n in enumerate(lens):
        t = np.arange(n)
        slots.append(table[s, t // bs].astype(np.int64) * bs + t % bs)
    slots = np.concatenate(slots)
    planes = _pool(rows_k, rows_v, fmt_k, fmt_v, H, D, slots, nblocks * bs)
    q = O.f32_to_bf16(rng.standard_normal((S, Hq, D)).astype(np.float32))
    return planes, table, np.array(lens, np.int32), q, rows_k, rows_v, H, Hq, D, bs


@pytest.mark.parametrize("fmt_k,fmt_v", [(NVFP4, NVFP4), (FP8, FP8), (FP8, NVFP4)])
@pytest.mark.parametrize("H,Hq", [(2, 4), (1, 16), (2, 18)])  # GQA 2, 16 and 9
def test_attention_equals_torch_sdpa_on_the_decoded_rows(fmt_k, fmt_v, H, Hq):
    planes, table, lens, q, rk, rv, H, Hq, D, bs = _case(fmt_k, fmt_v, H=H, Hq=Hq, seed=H + Hq)
    scale = 0.125
    out, st = O.decode_attention(planes[0], planes[1], fmt_k, fmt_v, bs, table, lens, q, scale)
    assert st == 0
    qf = O.bf16_to_f32(q).astype(np.float64)
    t0 = 0
    for s, n in enumerate(lens):
        k = np.repeat(rk[t0:t0 + n], Hq // H, axis=1)  # query head qh reads KV head qh // (Hq/H)
        v = np.repeat(rv[t0:t0 + n], Hq // H, axis=1)
        np.testing.assert_allclose(out[s], _sdpa(qf[s], k, v, scale), rtol=1e-12, atol=1e-12)
        t0 += n


def test_one_token_returns_its_value_row_and_zero_scale_averages():
    planes, table, lens, q, rk, rv, H, Hq, D, bs = _case(NVFP4, NVFP4, lens=(1, 20), seed=1)
    out, st = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, table, lens, q, 0.3)
    assert st == 0
    np.testing.assert_array_equal(out[0], np.repeat(rv[0], Hq // H, axis=0))  # p = 1 exactly
    out, _ = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, table, lens, q, 0.0)
    mean = rv[1:21].mean(axis=0)
    np.testing.assert_allclose(out[1], np.repeat(mean, Hq // H, axis=0), rtol=1e-13, atol=1e-300)


def test_empty_bad_length_and_bad_block():
    planes, table, lens, q, rk, rv, H, Hq, D, bs = _case(NVFP4, NVFP4, lens=(5, 16, 3), seed=2)
    untouched = lambda: np.full((3, Hq, D), np.nan)
    lens = np.array([0, 16, 3], np.int32)
    out, st = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, table, lens, q, 1.0, out=untouched())
    assert st == 0 and (out[0] == 0).all() and np.isfinite(out[1:]).all()
    bad_len = np.array([5, 10 ** 6, 3], np.int32)
    out, st = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, table, bad_len, q, 1.0, out=untouched())
    assert st == O.BAD_SEQLEN and np.isnan(out[1]).all() and np.isfinite(out[[0, 2]]).all()
    bad_tab = table.copy()
    bad_tab[2, 0] = 10 ** 6
    out, st = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, bad_tab, lens, q, 1.0, out=untouched())
    assert st == O.BAD_BLOCK and np.isnan(out[2]).all() and np.isfinite(out[1]).all()


def test_token_order_and_block_placement_do_not_matter():
    """Permuting a sequence's tokens (through a different block table and slot layout)
    leaves the output unchanged: the page mapping is only addressing."""
    rng = np.random.default_rng(3)
    H, Hq, D, bs, n = 1, 2, 32, 16, 32
    rk = _exact_nvfp4_rows(rng, n, D).reshape(n, H, D)
    rv = _exact_nvfp4_rows(rng, n, D).reshape(n, H, D)
    q = O.f32_to_bf16(rng.standard_normal((1, Hq, D)).astype(np.float32))
    outs = []
    for order in (np.arange(n), rng.permutation(n)):
        table = rng.permutation(6)[:2].astype(np.int32).reshape(1, 2)
        t = np.arange(n)
        slots = table[0, t // bs].astype(np.int64) * bs + t % bs
        planes = _pool(rk[order], rv[order], NVFP4, NVFP4, H, D, slots, 6 * bs)
        o, st = O.decode_attention(planes[0], planes[1], NVFP4, NVFP4, bs, table, np.array([n], np.int32), q, 0.2)
        assert st == 0
        outs.append(o)
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-13, atol=0)
