"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these re-types the oracle's formulas.  They use enumeration of the two
small float formats, the e4m3 -> fp16 bit identity printed on the FreeToken page,
library conversions (torch bf16, numpy fp16), exact round trips of representable
inputs, scale invariance, error bounds, brute force on small inputs, and the
storage figures printed on the pages (tests/golden/storage_bytes.txt).
"""

import os

import numpy as np
import pytest
import torch

import oracle as O
from quantized_kv_cache_nvfp4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def brute_nearest_even(a, table):
    """Index of the table entry nearest to each |a| (float64); ties -> even index;
    beyond the last entry saturates.  Brute force over the whole table."""
    a = np.abs(np.asarray(a, np.float64))[..., None]
    d = np.abs(a - table[None, :])
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    idx = np.arange(table.size)
    # among tied candidates prefer the even index
    score = np.where(cand, np.where(idx % 2 == 0, 0, 1) * table.size + idx, 10**9)
    out = score.argmin(axis=-1)
    out = np.where(a[..., 0] >= table[-1], table.size - 1, out)
    return out


def e4m3_table():
    return np.array([O.e4m3_value(c) for c in range(127)], np.float64)


# ---------------------------------------------------------------------------
# E2M1
# ---------------------------------------------------------------------------
def test_host_keeps_subnormals():
    """The oracle's binary32 definitions assume subnormals are kept (no FTZ/DAZ): the
    library's own run-time probe agrees with numpy's float32 arithmetic on this host."""
    assert O.lib().orc_subnormals_kept() == 1
    assert np.float32(2.0 ** -126) * np.float32(0.5) == np.float32(2.0 ** -127)


def test_e2m1_values_are_the_fp4_grid():
    got = [O.e2m1_value(c) for c in range(16)]
    assert got[:8] == list(E2M1_MAGS)
    assert got[8:] == [-v for v in E2M1_MAGS]
    assert np.signbit(got[8])  # code 0x8 is -0


def test_e2m1_round_trip_every_code():
    vals = np.array([O.e2m1_value(c) for c in range(16)], np.float32)
    assert list(O.e2m1_encode(vals)) == list(range(16))


@pytest.mark.parametrize("mid,code", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)])
def test_e2m1_midpoints_tie_to_even_and_nextafter(mid, code):
    m = np.float32(mid)
    lo_code = int(np.searchsorted(E2M1_MAGS, mid) - 1)
    assert int(O.e2m1_encode([m])[0]) == code
    assert int(O.e2m1_encode([-m])[0]) == code | 8
    below = np.nextafter(m, np.float32(0))
    above = np.nextafter(m, np.float32(10))
    assert int(O.e2m1_encode([below])[0]) == lo_code
    assert int(O.e2m1_encode([above])[0]) == lo_code + 1


def test_e2m1_saturates_and_keeps_sign_of_zero():
    big = np.array([6.0, 6.5, 7.0, 1e30, np.inf], np.float32)
    assert list(O.e2m1_encode(big)) == [7] * 5
    assert list(O.e2m1_encode(-big)) == [15] * 5
    assert list(O.e2m1_encode(np.array([0.0, -0.0, 1e-30, -1e-30], np.float32))) == [0, 8, 0, 8]


def test_e2m1_brute_force_sweep():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-8, 8, 200000).astype(np.float32),
        (np.arange(-8 * 64, 8 * 64 + 1) / 64.0).astype(np.float32),  # a dense grid incl. midpoints
    ])
    got = O.e2m1_encode(x)
    want = brute_nearest_even(x, E2M1_MAGS) | np.where(np.signbit(x), 8, 0)
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------
def test_e4m3_decode_matches_the_fp16_bit_identity():
    """FreeToken PR #408, fp8 tile-loader commit: for an e4m3 byte v the fp16 bit
    pattern (v + (v & 0x80)) << 7 holds the value / 256, on every code."""
    for v in range(256):
        if (v & 0x7F) == 0x7F:
            assert np.isnan(O.e4m3_value(v))
            continue
        bits = np.array([((v + (v & 0x80)) << 7) & 0xFFFF], np.uint16)
        via_fp16 = float(bits.view(np.float16)[0]) * 256.0
        got = O.e4m3_value(v)
        assert got == via_fp16 and np.signbit(got) == np.signbit(via_fp16), v


def test_e4m3_known_points():
    assert O.e4m3_value(0x7E) == 448.0
    assert O.e4m3_value(0x01) == 2.0 ** -9
    assert O.e4m3_value(0x08) == 2.0 ** -6
    assert O.e4m3_value(0x38) == 1.0


def test_e4m3_round_trip_every_finite_code():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    assert len(codes) == 254
    vals = np.array([O.e4m3_value(c) for c in codes], np.float32)
    assert list(O.e4m3_encode(vals)) == codes


def test_e4m3_midpoints_tie_to_even_and_nextafter():
    tab = e4m3_table()
    for i in range(126):
        mid = np.float32((tab[i] + tab[i + 1]) / 2)
        assert float(mid) == (tab[i] + tab[i + 1]) / 2  # exactly representable
        even = i if i % 2 == 0 else i + 1
        assert int(O.e4m3_encode([mid])[0]) == even, i
        assert int(O.e4m3_encode([np.nextafter(mid, np.float32(0))])[0]) == i
        assert int(O.e4m3_encode([np.nextafter(mid, np.float32(1e9))])[0]) == i + 1


def test_e4m3_saturates_and_subnormals():
    assert list(O.e4m3_encode(np.array([448, 460, 464, 480, 1e30, np.inf], np.float32))) == [0x7E] * 6
    sub = (np.arange(8) * 2.0 ** -9).astype(np.float32)
    assert list(O.e4m3_encode(sub)) == list(range(8))
    assert int(O.e4m3_encode([2.0 ** -10])[0]) == 0  # tie between 0 and 2^-9 -> even (0)
    assert int(O.e4m3_encode([3 * 2.0 ** -10])[0]) == 2  # tie between 1 and 2 (x 2^-9) -> 2
    assert int(O.e4m3_encode([np.float32(1e-30)])[0]) == 0


def test_e4m3_brute_force_sweep():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        np.exp2(rng.uniform(-14, 9.2, 100000)).astype(np.float32),
        rng.uniform(0, 500, 50000).astype(np.float32),
    ])
    np.testing.assert_array_equal(O.e4m3_encode(x), brute_nearest_even(x, e4m3_table()))


# ---------------------------------------------------------------------------
# bf16 / fp16 narrowing (pinned against library casts)
# ---------------------------------------------------------------------------
def _interesting_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    extra = np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-45, 65504, 65519.99, 65520, 6e-8,
                      2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 1.00048828125], np.float32)
    return np.concatenate([x, extra, rng.normal(0, 1, n).astype(np.float32)])


def test_bf16_matches_torch_cast():
    x = _interesting_f32(300000, 3)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f32_to_bf16(x), want)
    # midpoints between neighbouring bf16 values: ties to even
    base = np.arange(0x3F80, 0x3F90, dtype=np.uint32)
    mids = ((base << 16) | 0x8000).view(np.float32)
    want = torch.from_numpy(mids).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f32_to_bf16(mids), want)


def test_f16_matches_numpy_cast():
    x = _interesting_f32(300000, 4)
    x = x[np.abs(x) < 1e6]
    x = np.concatenate([x, np.float32(np.exp2(np.random.default_rng(5).uniform(-27, 17, 100000)))])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.f32_to_f16(x), want)
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    h = h[(h & 0x7C00) != 0x7C00]
    np.testing.assert_array_equal(O.f16_to_f32(h[::37]), h[::37].view(np.float16).astype(np.float32))


# ---------------------------------------------------------------------------
# NVFP4 row codec
# ---------------------------------------------------------------------------
def _bits(x):
    return O.f32_to_bf16(np.asarray(x, np.float32))


def _exact_rows(rng, n, D, k):
    """Rows x = c * e * 2^k with c on the E2M1 grid, e an E4M3 value per block,
    each block holding a |c| = 6 entry, and one block at e = 448."""
    tab = e4m3_table()
    rows = np.zeros((n, D), np.float64)
    for r in range(n):
        for b in range(D // 16):
            e = tab[rng.integers(40, 127)] if b != r % (D // 16) else 448.0
            c = E2M1_MAGS[rng.integers(0, 8, 16)] * rng.choice([-1, 1], 16)
            c[rng.integers(0, 16)] = 6.0 * rng.choice([-1, 1])
            rows[r, 16 * b:16 * b + 16] = c * e
    return rows * 2.0 ** k


@pytest.mark.parametrize("D", [16, 64, 128, 256])
@pytest.mark.parametrize("k", [-100, -20, -11, 0, 7, 60])
def test_row_codec_identity_on_exact_inputs(D, k):
    rng = np.random.default_rng(D * 1000 + k + 500)
    x = _exact_rows(rng, 24, D, k)
    xb = _bits(x)
    assert np.array_equal(O.bf16_to_f32(xb).astype(np.float64), x)  # inputs representable
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    np.testing.assert_array_equal(rscale, np.float32(2.0 ** k))
    y = O.nvfp4_decode_rows(codes, bscale, rscale)
    np.testing.assert_array_equal(y, xb)


def test_row_layout_low_nibble_first_and_sizes():
    x = np.zeros(16, np.float32)
    x[0], x[1], x[15] = 6.0 * 448 / 448, -1.0, 0.5  # amax 6 -> rs = 6/2688
    codes, bscale, rscale = O.nvfp4_encode_rows(_bits(x)[None])
    assert codes.shape == (1, 8) and bscale.shape == (1, 1) and rscale.shape == (1,)
    # block max 6 with rs = amax/2688 gives the block scale 448, so q = x exactly
    assert bscale[0, 0] == 0x7E
    assert codes[0, 0] == (0x7 | (0xA << 4))  # x0 = 6 (code 7) low, x1 = -1 (code 0xA) high
    assert codes[0, 7] >> 4 == 0x1  # x15 = 0.5 in the high nibble of byte 7


@pytest.mark.parametrize("k", [-40, -3, 5, 30])
def test_scale_invariance_by_powers_of_two(k):
    x = synth.normal_bf16((64, 128), seed=11, stream=1, outlier_frac=0.01, outlier_scale=20.0)
    xb = synth.bf16_bits(x)
    xs = _bits(O.bf16_to_f32(xb).astype(np.float64) * 2.0 ** k)
    c0, b0, r0 = O.nvfp4_encode_rows(xb)
    c1, b1, r1 = O.nvfp4_encode_rows(xs)
    np.testing.assert_array_equal(c0, c1)
    np.testing.assert_array_equal(b0, b1)
    np.testing.assert_array_equal(r1.astype(np.float64), r0.astype(np.float64) * 2.0 ** k)


def _decode_scales(bscale, rscale):
    bs = np.array([O.e4m3_value(int(c)) for c in range(256)], np.float64)[bscale]
    return bs, rscale.astype(np.float64)


def test_codes_are_nearest_against_the_stored_block_scale():
    """Random rows: each code is the nearest-even E2M1 value of x / (bs * rs) computed
    in float64 from the STORED scales (ties within fp32 rounding excepted)."""
    x = synth.normal_bf16((512, 128), seed=12, stream=1, outlier_frac=0.01, outlier_scale=20.0)
    xb = synth.bf16_bits(x)
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    bs, rs = _decode_scales(bscale, rscale)
    xf = O.bf16_to_f32(xb).astype(np.float64).reshape(512, 8, 16)
    s = bs[..., None] * rs[:, None, None]
    q = np.where(s > 0, xf / np.where(s > 0, s, 1), 0.0)
    want = brute_nearest_even(q, E2M1_MAGS) | np.where(np.signbit(xf), 8, 0)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(512, 8, 16)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near_tie = np.abs(np.abs(q)[..., None] - mids).min(-1) <= 1e-6 * np.abs(q)
    bad = (nib != want) & ~near_tie
    assert not bad.any()
    # error bound: |q - value(code)| <= half the local grid spacing (non-saturated)
    val = np.where(nib & 8, -1, 1) * E2M1_MAGS[nib & 7]
    spacing = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])[nib & 7]
    ok = (np.abs(q) > 6) | (np.abs(q - val) <= spacing / 2 * (1 + 1e-6))
    assert ok.all()


def test_block_scale_rounds_to_nearest_even_e4m3():
    """amax = 2688 gives rs = 1, so a block whose max is 6m has t = m exactly; m at
    every E4M3 midpoint (representable in bf16) must take the even neighbour."""
    tab = e4m3_table()
    mids = [(tab[i] + tab[i + 1]) / 2 for i in range(126) if tab[i] >= 2.0 ** -9]
    nb = 16
    rows = []
    for j in range(0, len(mids), nb - 1):
        r = np.zeros(16 * nb)
        r[0] = 2688.0
        for b, m in enumerate(mids[j:j + nb - 1], start=1):
            r[16 * b] = 6 * m
            r[16 * b + 1] = -3 * m
        rows.append(r)
    rows = np.array(rows)
    xb = _bits(rows)
    assert np.array_equal(O.bf16_to_f32(xb).astype(np.float64), rows)
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    assert (rscale == 1.0).all()
    got = bscale[:, 1:].ravel()
    want = []
    for j in range(0, len(mids), nb - 1):
        chunk = mids[j:j + nb - 1]
        want += [int(brute_nearest_even([m], tab)[0]) for m in chunk] + [0] * (nb - 1 - len(chunk))
    np.testing.assert_array_equal(got, np.array(want))


def test_zero_rows_keep_signed_zeros():
    x = np.zeros((2, 32), np.float32)
    x[1] = -0.0
    xb = _bits(x)
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    assert (rscale == 0).all() and (bscale == 0).all()
    assert (codes[0] == 0x00).all() and (codes[1] == 0x88).all()
    np.testing.assert_array_equal(O.nvfp4_decode_rows(codes, bscale, rscale), xb)


def test_block_far_below_row_max_decodes_to_signed_zero():
    x = np.zeros(32, np.float32)
    x[0] = 1e4
    x[16:] = 1e-4 * np.array([1, -1] * 8)
    codes, bscale, rscale = O.nvfp4_encode_rows(_bits(x)[None])
    assert bscale[0, 1] == 0
    assert list(codes[0, 8:]) == [0x80] * 8  # +0 low, -0 high
    y = O.bf16_to_f32(O.nvfp4_decode_rows(codes, bscale, rscale))[0, 16:]
    assert (y == 0).all() and list(np.signbit(y)) == [False, True] * 8


def test_smallest_subnormal_row_round_trips():
    """amax = 2^-133, the smallest bf16 subnormal: the row scale is an fp32
    subnormal, the block scale saturates at 448 and the reciprocal of s overflows."""
    x = np.zeros(16, np.float64)
    x[::3] = 2.0 ** -133
    x[1::3] = -(2.0 ** -133)
    xb = _bits(x)[None]
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    assert 0 < rscale[0] < np.finfo(np.float32).tiny
    assert bscale[0, 0] == 0x7E
    s = np.float32(448.0) * rscale[0]
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(1.0) / s)
    np.testing.assert_array_equal(O.nvfp4_decode_rows(codes, bscale, rscale), xb)


def test_direct_division_fallback_when_the_reciprocal_overflows():
    """A tiny row scale and a tiny block: 1/(bs*rs) overflows, yet the codes must be
    the nearest values of x / (bs*rs), not the saturated x * inf."""
    x = np.zeros(32, np.float64)
    x[0] = 2.0 ** -110
    x[16] = 2.0 ** -126
    x[17] = 2.0 ** -127
    x[18] = -(2.0 ** -128)
    xb = _bits(x)[None]
    assert np.array_equal(O.bf16_to_f32(xb)[0].astype(np.float64), x)
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    bs, rs = _decode_scales(bscale, rscale)
    s32 = np.float32(bs[0, 1]) * rscale[0]
    assert s32 > 0
    with np.errstate(over="ignore", divide="ignore"):
        assert np.isinf(np.float32(1.0) / s32)
    q = x[16:19] / float(s32)
    want = brute_nearest_even(q, E2M1_MAGS) | np.where(q < 0, 8, 0)
    nib = [codes[0, 8] & 15, codes[0, 8] >> 4, codes[0, 9] & 15]
    assert list(nib) == list(want)
    assert (np.abs(q) < 6).any()  # at least one code is not the saturated one


# ---------------------------------------------------------------------------
# storage accounting (golden: figures printed on the pages)
# ---------------------------------------------------------------------------
def _golden_storage():
    rows = []
    with open(os.path.join(GOLDEN, "storage_bytes.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, spec, expected, cite = [p.strip() for p in line.split("|")]
            fmt, kind, G, T, H, D = spec.split()
            rows.append((name, fmt, kind, int(G), int(T), int(H), int(D), float(expected), cite))
    return rows


@pytest.mark.parametrize("case", _golden_storage(), ids=lambda c: c[0])
def test_storage_figures_printed_on_the_pages(case):
    name, fmt, kind, G, T, H, D, expected, cite = case
    k = O.KIND_KEY if kind == "key" else O.KIND_VALUE
    if fmt == "bf16":
        got = T * H * D * 2
    else:
        f = {"nvfp4": O.FMT_NVFP4, "int4": O.FMT_INT4, "fp8": O.FMT_FP8, "nvfp4t": O.FMT_NVFP4_TENSOR}[fmt]
        got = O.storage_bytes(f, k, G, T, H, D)
    if name.endswith("_bits"):
        got = 8.0 * got / (T * H * D)
    assert got == expected, cite


def test_storage_matches_allocated_bytes():
    """The accounting equals the bytes of the buffers the oracle actually fills."""
    for (T, H, D) in [(256, 8, 128), (4100, 2, 96), (33, 4, 256)]:
        pool = O.new_pool(T, H, D)
        assert sum(a.nbytes for a in pool) == O.storage_bytes(O.FMT_NVFP4, 0, 16, T, H, D)
        for kind in (O.KIND_KEY, O.KIND_VALUE):
            x = synth.bf16_bits(synth.normal_bf16((T, H, D), 1, 1))
            codes, mn, sc = O.int4_pack(x, kind, 64)
            assert codes.nbytes + mn.nbytes + sc.nbytes == O.storage_bytes(O.FMT_INT4, kind, 64, T, H, D)


# ---------------------------------------------------------------------------
# INT4 affine codec
# ---------------------------------------------------------------------------
def _f16_exact(v):
    return np.float64(np.float16(v))


@pytest.mark.parametrize("kind", [O.KIND_KEY, O.KIND_VALUE])
def test_int4_exact_grid_round_trips(kind):
    """x = mn + c*sc with fp16-exact mn, sc (and every grid value bf16-exact and the
    fp32 arithmetic exact) decodes to x exactly; codes equal c."""
    rng = np.random.default_rng(7)
    G, T, H, D = 64, 128, 2, 128
    c = rng.integers(0, 16, (T, H, D))
    if kind == O.KIND_KEY:
        c[0::64] = 0
        c[1::64] = 15
        mn = np.array([_f16_exact(v) for v in rng.choice([-4.0, -2.0, -1.0, 0.5, 1.0], (2, H, D)).ravel()]).reshape(2, H, D)
        sc = np.array([_f16_exact(v) for v in rng.choice([0.125, 0.25, 0.5, 1.0], (2, H, D)).ravel()]).reshape(2, H, D)
        x = mn[np.arange(T) // 64] + c * sc[np.arange(T) // 64]
    else:
        c[..., 0::64] = 0
        c[..., 1::64] = 15
        mn = rng.choice([-4.0, -2.0, -1.0, 0.5, 1.0], (T, H, 2))
        sc = rng.choice([0.125, 0.25, 0.5, 1.0], (T, H, 2))
        x = mn[..., np.arange(D) // 64] + c * sc[..., np.arange(D) // 64]
    xb = _bits(x)
    assert np.array_equal(O.bf16_to_f32(xb).astype(np.float64), x)
    codes, m16, s16 = O.int4_pack(xb, kind, G)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(T, H, D)
    np.testing.assert_array_equal(nib, c)
    np.testing.assert_array_equal(O.int4_unpack(codes, m16, s16, kind, G), xb)


def test_int4_constant_group_decodes_to_its_value():
    x = np.full((64, 1, 16), 0.3, np.float32)
    xb = _bits(x)
    for kind in (O.KIND_KEY, O.KIND_VALUE):
        codes, mn, sc = O.int4_pack(xb, kind, 64)
        assert (codes == 0).all() and (sc == 0).all()
        y = O.int4_unpack(codes, mn, sc, kind, 64)
        want = _bits(np.float32(np.float16(O.bf16_to_f32(xb[0, 0, 0]))))
        assert (y == want).all()


def _f16bits(x):
    """fp16 bits by numpy's own conversion (round to nearest even)."""
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def test_int4_signed_zero_groups_order_minus_zero_first():
    """A group whose minimum or maximum is a zero holding both signs: -0 orders below +0
    whatever the order of the elements (IEEE 754-2019 minimum/maximum), so the stored
    FP16 minimum is -0 (0x8000) and the maximum gives sc = (+0 - -0) / 15 = 0."""
    for order in ((0x0000, 0x8000), (0x8000, 0x0000)):
        xb = np.zeros((1, 1, 64), np.uint16)
        xb[0, 0, :32] = order[0]
        xb[0, 0, 32:] = order[1]
        codes, mn, sc = O.int4_pack(xb, O.KIND_VALUE, 64)
        assert mn[0, 0, 0] == 0x8000 and sc[0, 0, 0] == 0 and (codes == 0).all()
        y = O.int4_unpack(codes, mn, sc, O.KIND_VALUE, 64)
        assert (y == 0).all()  # (0 * 0) + (-0) = (+0) + (-0) = +0 in round-to-nearest
        # a positive value above the zeros: min is -0, the codes are those of mn = 0
        xb[0, 0, 7] = 0x3FC0  # bf16 1.5
        codes, mn, sc = O.int4_pack(xb, O.KIND_VALUE, 64)
        assert mn[0, 0, 0] == 0x8000 and sc[0, 0, 0] == _f16bits(np.float32(0.1))
        assert (codes.reshape(-1) == np.where(np.arange(32) == 3, 0xF0, 0)).all()
        # max over {-0, +0, negatives} is +0
        xb[0, 0, 7] = 0xBFC0  # bf16 -1.5
        codes, mn, sc = O.int4_pack(xb, O.KIND_VALUE, 64)
        assert mn[0, 0, 0] == _f16bits(np.float32(-1.5)) and sc[0, 0, 0] == _f16bits(np.float32(0.1))


def test_int4_nibble_order_low_is_even_channel():
    x = np.zeros((1, 1, 64), np.float32)
    x[0, 0, 1] = 15.0  # mn 0, sc 1: channel 1 -> code 15, channel 0 -> 0
    x[0, 0, 2] = 7.0
    codes, mn, sc = O.int4_pack(_bits(x), O.KIND_VALUE, 64)
    assert codes[0, 0, 0] == 0xF0 and codes[0, 0, 1] == 0x07


def test_int4_codes_are_nearest_and_invariants():
    rng = np.random.default_rng(8)
    x = synth.normal_bf16((200, 2, 96), seed=13, stream=1)
    xb = synth.bf16_bits(x)
    xf = O.bf16_to_f32(xb).astype(np.float64)
    for kind, G in [(O.KIND_KEY, 64), (O.KIND_VALUE, 64), (O.KIND_KEY, 16), (O.KIND_VALUE, 16)]:
        codes, mn16, sc16 = O.int4_pack(xb, kind, G)
        nib = np.stack([codes & 15, codes >> 4], -1).reshape(xf.shape)
        if kind == O.KIND_KEY:
            gid = np.arange(200) // G
            grp = [(xf[gid == g], nib[gid == g]) for g in range(gid.max() + 1)]
            groups = [(a[:, h, d], b[:, h, d]) for a, b in grp for h in range(2) for d in range(96)]
        else:
            gid = np.arange(96) // G
            groups = [(xf[t, h, gid == g], nib[t, h, gid == g]) for t in range(0, 200, 7) for h in range(2)
                      for g in range(gid.max() + 1)]
        for vals, cs in groups:
            lo, hi = vals.min(), vals.max()
            sc = (hi - lo) / 15
            assert cs[vals.argmin()] == 0 and cs[vals.argmax()] == 15
            assert (np.abs((vals - lo) / sc - cs) <= 0.5 + 1e-5).all()


def test_int4_partial_last_groups_are_independent():
    """T = 4100 with K over 64-row groups: the 4-row tail group equals packing those
    4 rows alone; D = 96 with V over 64 channels: the 32-channel tail likewise."""
    x = synth.bf16_bits(synth.normal_bf16((4100, 2, 32), seed=14, stream=1))
    codes, mn, sc = O.int4_pack(x, O.KIND_KEY, 64)
    assert mn.shape == (65, 2, 32)
    c2, m2, s2 = O.int4_pack(x[4096:], O.KIND_KEY, 64)
    np.testing.assert_array_equal(codes[4096:], c2)
    np.testing.assert_array_equal(mn[64], m2[0])
    np.testing.assert_array_equal(sc[64], s2[0])
    y = synth.bf16_bits(synth.normal_bf16((5, 3, 96), seed=15, stream=1))
    codes, mn, sc = O.int4_pack(y, O.KIND_VALUE, 64)
    assert mn.shape == (5, 3, 2)
    c2, m2, s2 = O.int4_pack(np.ascontiguousarray(y[..., 64:]), O.KIND_VALUE, 64)
    np.testing.assert_array_equal(codes[..., 32:], c2)
    np.testing.assert_array_equal(mn[..., 1], m2[..., 0])


def test_int4_key_groups_run_over_token_rows():
    x = synth.bf16_bits(synth.normal_bf16((128, 2, 8), seed=16, stream=1))
    _, mn0, sc0 = O.int4_pack(x, O.KIND_KEY, 64)
    x2 = x.copy()
    x2[70, 1, 3] = _bits(np.array([50.0], np.float32))[0]
    _, mn1, sc1 = O.int4_pack(x2, O.KIND_KEY, 64)
    changed = np.argwhere((sc0 != sc1) | (mn0 != mn1))
    assert changed.tolist() == [[1, 1, 3]]


# ---------------------------------------------------------------------------
# residual encode / decode
# ---------------------------------------------------------------------------
FORMATS = [(O.FMT_INT4, O.KIND_KEY), (O.FMT_INT4, O.KIND_VALUE), (O.FMT_NVFP4, O.KIND_KEY)]


def _recon(x, fmt, kind):
    if fmt == O.FMT_INT4:
        return O.int4_unpack(*O.int4_pack(x, kind, 64), kind, 64)
    c, b, r = O.nvfp4_encode_rows(x)
    return O.nvfp4_decode_rows(c, b, r)


@pytest.mark.parametrize("fmt,kind", FORMATS)
def test_zero_residual_returns_prev_bitwise(fmt, kind):
    prev = synth.bf16_bits(synth.normal_bf16((96, 2, 64), 17, 1))
    pay, st = O.residual_encode(prev, prev, None, fmt, kind)
    out, _ = O.residual_decode(pay, prev)
    assert st == 0
    np.testing.assert_array_equal(out, prev)


@pytest.mark.parametrize("fmt,kind", FORMATS)
def test_sparse_with_every_row_equals_dense_and_empty_is_identity(fmt, kind):
    cur = synth.bf16_bits(synth.normal_bf16((130, 2, 64), 18, 1))
    prev = synth.bf16_bits(synth.normal_bf16((130, 2, 64), 18, 2))
    dense, _ = O.residual_encode(cur, prev, None, fmt, kind)
    sparse, st = O.residual_encode(cur, prev, np.arange(130, dtype=np.int32), fmt, kind)
    assert st == 0
    np.testing.assert_array_equal(O.residual_decode(dense, prev)[0], O.residual_decode(sparse, prev)[0])
    empty, st = O.residual_encode(cur, prev, np.zeros(0, np.int32), fmt, kind)
    assert st == 0
    np.testing.assert_array_equal(O.residual_decode(empty, prev)[0], prev)


@pytest.mark.parametrize("fmt,kind", FORMATS)
def test_absent_rows_inherit_and_kept_rows_follow_compact_order(fmt, kind):
    T = 200
    cur = synth.bf16_bits(synth.normal_bf16((T, 2, 64), 19, 1))
    prev = synth.bf16_bits(synth.normal_bf16((T, 2, 64), 19, 2))
    pos = synth.sorted_positions(T, 70, 19).numpy()
    pay, st = O.residual_encode(cur, prev, pos, fmt, kind)
    assert st == 0 and list(pay["pos"]) == list(pos)
    out, _ = O.residual_decode(pay, prev)
    absent = np.setdiff1d(np.arange(T), pos)
    np.testing.assert_array_equal(out[absent], prev[absent])
    # compact payload == dense codec of the gathered residual rows
    r = O.f32_to_bf16(O.bf16_to_f32(cur[pos]) - O.bf16_to_f32(prev[pos]))
    if fmt == O.FMT_INT4:
        c, mn, sc = O.int4_pack(r, kind, 64)
        np.testing.assert_array_equal(pay["codes"], c)
        np.testing.assert_array_equal(pay["meta_a"], mn)
    # in-place decode gives the same bytes
    inplace = prev.copy()
    O.residual_decode(pay, inplace, out=inplace)
    np.testing.assert_array_equal(inplace, out)


@pytest.mark.parametrize("fmt,kind", FORMATS)
def test_chain_against_reconstructed_predecessors_does_not_compound(fmt, kind):
    """vllm-rlt PR #166: encoding against the reconstructed predecessor keeps the
    error from compounding across depths.  Each depth's reconstruction error equals
    that depth's residual quantisation error alone, while a chain encoded against the
    ORIGINAL predecessors drifts further with depth."""
    loops = synth.residual_loops(T=128, H=2, D=64, loops=4, seed=20)
    L = [synth.bf16_bits(x) for x in loops]
    f = lambda a: O.bf16_to_f32(a).astype(np.float64)
    recon = _recon(L[0], fmt, kind)
    naive = recon.copy()
    err_good, err_naive = [], []
    for i in range(1, 4):
        pay, _ = O.residual_encode(L[i], recon, None, fmt, kind)
        recon, _ = O.residual_decode(pay, recon)
        payn, _ = O.residual_encode(L[i], L[i - 1], None, fmt, kind)
        naive, _ = O.residual_decode(payn, naive)
        err_good.append(np.sqrt(np.mean((f(recon) - f(L[i])) ** 2)))
        err_naive.append(np.sqrt(np.mean((f(naive) - f(L[i])) ** 2)))
    assert max(err_good) < 0.1 * err_naive[0] + min(err_good) * 1.5
    assert err_naive[-1] > err_good[-1] * 1.5


def test_bad_positions_are_flagged():
    cur = synth.bf16_bits(synth.normal_bf16((16, 1, 16), 21, 1))
    for pos in ([3, 2], [1, 1], [-1, 4], [4, 16]):
        _, st = O.residual_encode(cur, cur, np.array(pos, np.int32), O.FMT_NVFP4, 0)
        assert st & O.BAD_POS


# ---------------------------------------------------------------------------
# paged store / restore
# ---------------------------------------------------------------------------
def test_restore_of_scatter_equals_row_round_trip_through_random_blocks():
    S, Tmax, H, D, bsz = 3, 80, 2, 64, 16
    lens = np.array([80, 37, 1], np.int32)
    mb = Tmax // bsz
    nblocks = S * mb + 4
    perm = synth.block_permutation(nblocks, 22).numpy()
    table = perm[: S * mb].reshape(S, mb).astype(np.int32)
    k = synth.bf16_bits(synth.normal_bf16((S, Tmax, H, D), 22, 1, 0.01, 20.0))
    pool = O.new_pool(nblocks * bsz, H, D)
    for s in range(S):
        t = np.arange(lens[s])
        slots = table[s, t // bsz].astype(np.int64) * bsz + t % bsz
        st = O.nvfp4_scatter(k[s], H * D, D, int(lens[s]), H, D, slots, pool)
        assert st == 0
    out, st = O.nvfp4_restore(pool, bsz, table, lens, Tmax)
    assert st == 0
    for s in range(S):
        n = lens[s]
        want = O.nvfp4_decode_rows(*O.nvfp4_encode_rows(k[s, :n]))
        np.testing.assert_array_equal(out[s, :n], want)
        assert (out[s, n:] == 0).all()


def test_scatter_reads_each_tensor_with_its_own_pitch():
    """FreeToken PR #408, the V-pitch fix: K a view of a fused qkv (row pitch 1152,
    column offset 384) and V contiguous (pitch 384), 8 tokens x 3 heads x 128."""
    T, H, D = 8, 3, 128
    qkv = synth.bf16_bits(synth.normal_bf16((T, 1152), 23, 1))
    v = synth.bf16_bits(synth.normal_bf16((T, H * D), 23, 2))
    poolk, poolv = O.new_pool(16, H, D), O.new_pool(16, H, D)
    slots = np.arange(T, dtype=np.int64)[::-1].copy()
    assert O.nvfp4_scatter(qkv.ravel()[384:], 1152, D, T, H, D, slots, poolk) == 0
    assert O.nvfp4_scatter(v, H * D, D, T, H, D, slots, poolv) == 0
    kc = np.ascontiguousarray(qkv[:, 384:384 + H * D]).reshape(T, H, D)
    ck, bk, rk = O.nvfp4_encode_rows(kc)
    cv, bv, rv = O.nvfp4_encode_rows(v.reshape(T, H, D))
    np.testing.assert_array_equal(poolk[0][slots], ck)
    np.testing.assert_array_equal(poolk[1][slots], bk)
    np.testing.assert_array_equal(poolv[0][slots], cv)
    np.testing.assert_array_equal(poolv[2][slots], rv)


def test_negative_slot_skips_and_bad_ids_are_flagged():
    T, H, D = 4, 1, 16
    x = synth.bf16_bits(synth.normal_bf16((T, H, D), 24, 1))
    pool = O.new_pool(8, H, D)
    st = O.nvfp4_scatter(x, H * D, D, T, H, D, np.array([0, -1, 9, 3], np.int64), pool)
    assert st == O.BAD_SLOT
    assert (pool[2][[1, 2, 4, 5, 6, 7]] == 0).all() and pool[2][0, 0] > 0 and pool[2][3, 0] > 0
    table = np.array([[0, 7]], np.int32)
    _, st = O.nvfp4_restore(pool, 4, table, np.array([8], np.int32), 8)
    assert st == O.BAD_BLOCK
    _, st = O.nvfp4_restore(pool, 4, table, np.array([9], np.int32), 8)
    assert st == O.BAD_SEQLEN


# ---------------------------------------------------------------------------
# FP8 E4M3 row codec
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D", [16, 128, 256])
@pytest.mark.parametrize("k", [-100, 0, 40])
def test_fp8_identity_on_exact_inputs(D, k):
    """Rows of E4M3 values times 2^k with one entry at +-448 * 2^k decode exactly and
    carry the row scale 2^k."""
    rng = np.random.default_rng(D + 7 * k + 900)
    tab = e4m3_table()
    x = tab[rng.integers(0, 127, (16, D))] * rng.choice([-1, 1], (16, D))
    x[np.arange(16), rng.integers(0, D, 16)] = 448.0 * rng.choice([-1, 1], 16)
    x = x * 2.0 ** k
    xb = _bits(x)
    assert np.array_equal(O.bf16_to_f32(xb).astype(np.float64), x)
    codes, rs = O.fp8_encode_rows(xb)
    np.testing.assert_array_equal(rs, np.float32(2.0 ** k))
    np.testing.assert_array_equal(O.fp8_decode_rows(codes, rs), xb)


def test_fp8_codes_are_nearest_e4m3_of_x_over_scale():
    x = synth.bf16_bits(synth.normal_bf16((256, 128), seed=31, stream=1, outlier_frac=0.01, outlier_scale=20.0))
    codes, rs = O.fp8_encode_rows(x)
    xf = O.bf16_to_f32(x).astype(np.float64)
    q = xf / rs[:, None].astype(np.float64)
    tab = e4m3_table()
    want = brute_nearest_even(q, tab) | np.where(np.signbit(xf), 0x80, 0)
    mids = (tab[:-1] + tab[1:]) / 2
    near = np.abs(np.abs(q)[..., None] - mids).min(-1) <= 1e-6 * np.abs(q)
    assert not ((codes != want) & ~near).any()
    # the row maximum lands on 448 exactly (rs = amax / 448)
    assert (codes.max(axis=1) & 0x7F).max() == 0x7E


def test_fp8_zero_and_tiny_rows():
    x = np.zeros((3, 32))
    x[1] = -0.0
    x[2, 0] = 2.0 ** -125          # rs subnormal: its reciprocal overflows
    x[2, 1] = 2.0 ** -126
    x[2, 2] = -(2.0 ** -127)
    xb = _bits(x)
    codes, rs = O.fp8_encode_rows(xb)
    assert rs[0] == 0 and (codes[0] == 0).all() and (codes[1] == 0x80).all()
    assert 0 < rs[2] < np.finfo(np.float32).tiny
    with np.errstate(over="ignore", divide="ignore"):
        assert np.isinf(np.float32(1.0) / rs[2])
    q = x[2, :3] / float(rs[2])
    want = brute_nearest_even(q, e4m3_table()) | np.where(q < 0, 0x80, 0)
    assert list(codes[2, :3]) == list(want) and (np.abs(q) < 448).any()
    np.testing.assert_array_equal(O.fp8_decode_rows(codes[:2], rs[:2]), xb[:2])


def test_fp8_paged_round_trip_and_residuals():
    S, Tmax, H, D, bsz = 2, 48, 2, 32, 16
    lens = np.array([48, 20], np.int32)
    perm = synth.block_permutation(8, 32).numpy()
    table = perm[:6].reshape(2, 3).astype(np.int32)
    k = synth.bf16_bits(synth.normal_bf16((S, Tmax, H, D), 32, 1))
    pool = O.new_fp8_pool(8 * bsz, H, D)
    for s in range(S):
        t = np.arange(lens[s])
        assert O.fp8_scatter(k[s], H * D, D, int(lens[s]), H, D, table[s, t // bsz].astype(np.int64) * bsz + t % bsz, pool) == 0
    out, st = O.fp8_restore(pool, bsz, table, lens, Tmax)
    assert st == 0
    for s in range(S):
        n = lens[s]
        np.testing.assert_array_equal(out[s, :n], O.fp8_decode_rows(*O.fp8_encode_rows(k[s, :n])))
    prev = synth.bf16_bits(synth.normal_bf16((40, H, D), 33, 1))
    pay, st = O.residual_encode(prev, prev, None, O.FMT_FP8, 0)
    np.testing.assert_array_equal(O.residual_decode(pay, prev)[0], prev)
    cur = synth.bf16_bits(synth.normal_bf16((40, H, D), 33, 2))
    a, _ = O.residual_encode(cur, prev, np.arange(40, dtype=np.int32), O.FMT_FP8, 0)
    b, _ = O.residual_encode(cur, prev, None, O.FMT_FP8, 0)
    np.testing.assert_array_equal(O.residual_decode(a, prev)[0], O.residual_decode(b, prev)[0])


# ---------------------------------------------------------------------------
# decode rounding order on inexact scales, and INT4 half-integer ties
# ---------------------------------------------------------------------------
def _e4m3_via_fp16_identity(codes):
    """E4M3 bytes -> float32 values by the fp16 bit identity printed on the FreeToken
    page (fp8 store notes), not by the oracle's table: fp16 bits (v + (v & 0x80)) << 7
    hold the value / 256."""
    v = np.asarray(codes).astype(np.uint32)
    h = (((v + (v & 0x80)) << 7) & 0xFFFF).astype(np.uint16)
    return h.view(np.float16).astype(np.float32) * np.float32(256.0)


def _torch_bf16(x32):
    """float32 -> bf16 bit patterns by torch's own cast (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_nvfp4_decode_is_exact_block_product_then_one_float32_product_by_rs():
    """Reading R4 on rows whose row scales are not powers of two: the decoded value is
    (e2m1 * bs), exact in float32, times rs rounded once in float32, then torch's bf16
    cast.  Grouping the other way, e2m1 * (bs * rs), gives other bits on some elements
    of these rows, so this pin fixes the order (FreeToken PR #408, codec-delta port
    note: quantise against the stored block scale; decode multiplies both scales)."""
    n, D = 2000, 128
    xb = synth.bf16_bits(synth.normal_bf16((n, D), seed=41, stream=1, outlier_frac=0.01, outlier_scale=20.0))
    codes, bscale, rscale = O.nvfp4_encode_rows(xb)
    mant = np.frexp(rscale.astype(np.float64))[0]
    assert (mant != 0.5).mean() > 0.95  # the row scales are inexact
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(n, D)
    e2m1 = (np.where(nib & 8, -1.0, 1.0) * E2M1_MAGS[nib & 7]).astype(np.float32)
    bs = np.repeat(_e4m3_via_fp16_identity(bscale), 16, axis=1)
    prod = e2m1 * bs
    assert np.array_equal(prod.astype(np.float64), e2m1.astype(np.float64) * bs.astype(np.float64))
    want = _torch_bf16(prod * rscale[:, None])
    np.testing.assert_array_equal(O.nvfp4_decode_rows(codes, bscale, rscale), want)
    other_order = _torch_bf16(e2m1 * (bs * rscale[:, None]))
    assert (other_order != want).sum() > 20  # the pin tells the two orders apart


def test_fp8_decode_is_one_float32_product_then_bf16():
    """Reading R8's decode on inexact row scales: bf16(e4m3 * rs) with the product
    rounded in float32 (numpy) and the narrowing done by torch's cast."""
    xb = synth.bf16_bits(synth.normal_bf16((2000, 128), seed=42, stream=1, outlier_frac=0.01, outlier_scale=20.0))
    codes, rscale = O.fp8_encode_rows(xb)
    assert (np.frexp(rscale.astype(np.float64))[0] != 0.5).mean() > 0.95
    want = _torch_bf16(_e4m3_via_fp16_identity(codes) * rscale[:, None])
    np.testing.assert_array_equal(O.fp8_decode_rows(codes, rscale), want)


@pytest.mark.parametrize("kind,G", [(O.KIND_KEY, 64), (O.KIND_VALUE, 64), (O.KIND_VALUE, 16)])
def test_int4_decode_is_float32_mul_then_add_then_bf16(kind, G):
    """Reading R5's decode on random groups (metadata not on any grid): numpy float32
    code * sc16, then + mn16, then torch's bf16 cast; the FP16 metadata is widened by
    numpy's own fp16 conversion (vllm-rlt PR #166, Purpose: FP32 arithmetic with FP16
    min/scale)."""
    T, H, D = 256, 3, 128
    xb = synth.bf16_bits(synth.normal_bf16((T, H, D), seed=43, stream=1, outlier_frac=0.01, outlier_scale=20.0))
    codes, mn16, sc16 = O.int4_pack(xb, kind, G)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(T, H, D).astype(np.float32)
    mn = mn16.view(np.float16).astype(np.float32)
    sc = sc16.view(np.float16).astype(np.float32)
    if kind == O.KIND_KEY:
        mn, sc = mn[np.arange(T) // G], sc[np.arange(T) // G]
    else:
        mn, sc = mn[..., np.arange(D) // G], sc[..., np.arange(D) // G]
    want = _torch_bf16(nib * sc + mn)
    np.testing.assert_array_equal(O.int4_unpack(codes, mn16, sc16, kind, G), want)


def test_int4_decode_product_is_exact_so_a_fused_multiply_add_agrees():
    """A code has 4 significant bits and an FP16 scale 11, so code * sc16 is exact in
    float32 for every code and every finite FP16 scale; the decode's only rounding is
    the add, and a fused multiply-add rounds the same exact sum.  (This is why no pin
    can tell mul-then-add from an FMA here: the two are the same function.)"""
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    h = h[(h & 0x7C00) != 0x7C00]
    sc = h.view(np.float16)
    c = np.arange(16, dtype=np.float32)[:, None]
    p32 = c * sc.astype(np.float32)[None, :]
    p64 = c.astype(np.float64) * sc.astype(np.float64)[None, :]
    assert np.array_equal(p32.astype(np.float64), p64)
    # fused: the exact sum (exact in float64: at most 45 significant bits) rounded once
    rng = np.random.default_rng(44)
    mn = h[rng.integers(0, h.size, 200000)].view(np.float16)
    scs = h[rng.integers(0, h.size, 200000)].view(np.float16)
    cs = rng.integers(0, 16, 200000).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        mul_add = cs * scs.astype(np.float32) + mn.astype(np.float32)
        fused = (cs.astype(np.float64) * scs.astype(np.float64) + mn.astype(np.float64)).astype(np.float32)
    ok = np.isfinite(fused)
    np.testing.assert_array_equal(mul_add[ok].view(np.uint32), fused[ok].view(np.uint32))


def _tie_groups(mn, mx, ties):
    """One 64-element group: mn, mx, then the tie values, padded with mn."""
    g = np.full(64, mn, np.float64)
    g[1] = mx
    g[2:2 + len(ties)] = ties
    return g


@pytest.mark.parametrize("kind", [O.KIND_KEY, O.KIND_VALUE])
def test_int4_half_integer_quotients_round_to_the_even_code(kind):
    """Reading R5's rounding: groups whose scale (mx - mn)/15 is exact and whose
    quotients (x - mn)/sc are exact half-integers.  Each code must be the even
    neighbour (0.5 -> 0, 1.5 -> 2, 2.5 -> 2, 3.5 -> 4, ...), which is torch.round's
    half-to-even; rounding half away from zero would give the odd one."""
    half = np.arange(15) + 0.5
    cases = [
        (0.0, 15.0, half),              # sc = 1
        (-8.0, 7.0, half - 8.0),        # sc = 1, negative minimum
        (0.0, 30.0, 2.0 * half),        # sc = 2
        (0.0, 7.5, 0.5 * half),         # sc = 0.5
        (-3.0, 0.75, -3.0 + 0.25 * half),  # sc = 0.25
    ]
    groups = np.stack([_tie_groups(*c) for c in cases])        # [5, 64]
    if kind == O.KIND_KEY:
        x = groups.T[:, None, :]                                # [64 rows, 1 head, 5 channels] -> pad D
        x = np.concatenate([x, np.zeros((64, 1, 11))], axis=2)  # D = 16
    else:
        x = groups[:, None, :]                                  # [5 rows, 1 head, 64 channels]
    xb = _bits(x)
    assert np.array_equal(O.bf16_to_f32(xb).astype(np.float64), x)
    codes, mn16, sc16 = O.int4_pack(xb, kind, 64)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(x.shape)
    for i, (mn, mx, ties) in enumerate(cases):
        sc = (mx - mn) / 15.0
        q = (ties - mn) / sc
        assert np.array_equal(q, np.arange(15) + 0.5)           # exact half-integers
        want = torch.round(torch.from_numpy(q)).numpy().astype(np.int64)
        got = nib[2:17, 0, i] if kind == O.KIND_KEY else nib[i, 0, 2:17]
        np.testing.assert_array_equal(got, want)
        assert (got % 2 == 0).all()


def _double_rounding_scales(a, n, seed):
    """Row scales rs for which the exact product a * rs (exact in float64) rounds in
    float32 onto a bf16 midpoint without being one: there rounding once in float32 and
    then to bf16 can differ from rounding the exact product to bf16 directly."""
    rng = np.random.default_rng(seed)
    rs = rng.uniform(0.5, 1.0, 4_000_000).astype(np.float32) * np.float32(2.0 ** -10)
    e = np.float64(a) * rs.astype(np.float64)
    hi = e.astype(np.float32)
    hit = ((hi.view(np.uint32) & 0xFFFF) == 0x8000) & (hi.astype(np.float64) != e)
    assert hit.sum() >= n
    return rs[hit][:n]


def _bf16_direct(e64):
    """The exact float64 value rounded straight to bf16 (8 significant bits, ties to
    even), as bit patterns."""
    m, ex = np.frexp(e64)
    r = np.ldexp(np.rint(m * 256.0) / 256.0, ex).astype(np.float32)
    return _torch_bf16(r)


def test_decode_rounds_in_float32_first_on_double_rounding_cases():
    """Rows built so that the decode product lands, after its float32 rounding, exactly
    on a bf16 midpoint: the oracle's result is the float32 product narrowed by torch's
    cast (reading R4 and R8: one float32 rounding, then bf16), and on some of these
    elements that differs from rounding the exact product to bf16 in one step."""
    # FP8: code 0x39 = 1.125; NVFP4: code 7 (6.0) with block scale 0x39 (1.125) = 6.75
    rs8 = _double_rounding_scales(1.125, 48, 45)
    codes8 = np.full((48, 16), 0x39, np.uint8)
    got8 = O.fp8_decode_rows(codes8, rs8)
    want8 = _torch_bf16(np.float32(1.125) * rs8[:, None] * np.ones((1, 16), np.float32))
    np.testing.assert_array_equal(got8, want8)
    direct8 = _bf16_direct(1.125 * rs8.astype(np.float64))
    assert (direct8 != want8[:, 0]).sum() >= 8

    rs4 = _double_rounding_scales(6.75, 48, 46)
    codes4 = np.full((48, 8), 0x77, np.uint8)
    bscale4 = np.full((48, 1), 0x39, np.uint8)
    got4 = O.nvfp4_decode_rows(codes4, bscale4, rs4)
    want4 = _torch_bf16(np.float32(6.75) * rs4[:, None] * np.ones((1, 16), np.float32))
    np.testing.assert_array_equal(got4, want4)
    direct4 = _bf16_direct(6.75 * rs4.astype(np.float64))
    assert (direct4 != want4[:, 0]).sum() >= 8
