"""Pins of the oracle's per-tensor NVFP4 codec (one FP32 scale per tensor, G16 blocks
along the kind's axis: K over token rows, V over channels), each against something
other than itself: the pinned row codec, the transposition that maps one kind onto
the other, exact grid tensors, scale invariance, zero padding and zero tensors."""

import numpy as np
import pytest

import oracle as O
from quantized_kv_cache_nvfp4_gb300 import synth

K, V = O.KIND_KEY, O.KIND_VALUE


def _rand(shape, seed, outliers=True):
    return synth.bf16_bits(synth.normal_bf16(shape, seed, 1, 0.01 if outliers else 0.0, 20.0))


def test_one_row_tensor_is_the_row_codec():
    for seed, D in [(1, 128), (2, 64), (3, 512)]:
        x = _rand((1, 1, D), seed)
        c, b, r = O.nvfp4t_pack(x, V)
        rc, rb, rr = O.nvfp4_encode_rows(x)
        np.testing.assert_array_equal(c, rc)
        np.testing.assert_array_equal(b, rb)
        assert r[0].view(np.uint32) == rr.reshape(-1)[0].view(np.uint32)
        np.testing.assert_array_equal(O.nvfp4t_unpack(c, b, r, V), O.nvfp4_decode_rows(rc, rb, rr))


def _transpose_codes(codes, T, H, D):
    """Nibble codes [T][H][D/2] -> per-element codes [T][H][D]."""
    e = np.empty((T, H, D), np.uint8)
    e[..., 0::2] = codes & 15
    e[..., 1::2] = codes >> 4
    return e


def test_key_kind_is_the_value_kind_of_the_transposed_tensor():
    """Blocks over 16 token rows at (h, d) are blocks over 16 channels of x'[d][h][t]."""
    T, H, D = 48, 3, 32
    x = _rand((T, H, D), 4)
    ck, bk, rk = O.nvfp4t_pack(x, K)
    xt = np.ascontiguousarray(x.transpose(2, 1, 0))  # [D][H][T]
    cv, bv, rv = O.nvfp4t_pack(xt, V)
    assert rk[0] == rv[0]
    np.testing.assert_array_equal(_transpose_codes(ck, T, H, D), _transpose_codes(cv, D, H, T).transpose(2, 1, 0))
    np.testing.assert_array_equal(bk, bv.transpose(2, 1, 0))  # [T/16][H][D] vs [D][H][T/16]
    yk = O.nvfp4t_unpack(ck, bk, rk, K)
    yv = O.nvfp4t_unpack(cv, bv, rv, V)
    np.testing.assert_array_equal(yk, yv.transpose(2, 1, 0))


@pytest.mark.parametrize("kind", [K, V])
def test_exact_grid_tensors_round_trip(kind):
    """Values e2m1 * e4m3 * 2^k with one block holding 6 * 448 * 2^k and every block
    holding its 6 * bs: rs = 2^k, every block scale exact, so decode(encode(x)) = x."""
    rng = np.random.default_rng(5)
    T, H, D = 32, 2, 64
    e4 = np.array([O.e4m3_value(c) for c in range(40, 127)])
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for k in (-60, -3, 0, 7, 60):
        x = np.zeros((T, H, D))
        if kind == V:
            for t in range(T):
                for h in range(H):
                    for b in range(D // 16):
                        bs = rng.choice(e4)
                        c = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
                        c[rng.integers(0, 16)] = 6.0
                        x[t, h, 16 * b:16 * b + 16] = c * bs
        else:
            for g in range(T // 16):
                for h in range(H):
                    for d in range(D):
                        bs = rng.choice(e4)
                        c = rng.choice(mags, 16) * rng.choice([-1, 1], 16)
                        c[rng.integers(0, 16)] = -6.0
                        x[16 * g:16 * g + 16, h, d] = c * bs
        # block 0 (channels 0..15 of row 0 for V, rows 0..15 of channel 0 for K) holds the
        # tensor's maximum 6 * 448 and zeros: rs = 2^k exactly, its block scale 448
        if kind == V:
            x[0, 0, :16] = 0.0
        else:
            x[:16, 0, 0] = 0.0
        x[0, 0, 0] = 6 * 448.0
        xb = O.f32_to_bf16((x * 2.0 ** k).astype(np.float32))
        assert (O.bf16_to_f32(xb) == (x * 2.0 ** k)).all()
        c, b, r = O.nvfp4t_pack(xb, kind)
        assert r[0] == np.float32(2.0 ** k)
        np.testing.assert_array_equal(O.nvfp4t_unpack(c, b, r, kind), xb)


@pytest.mark.parametrize("kind", [K, V])
def test_scale_invariance(kind):
    x = _rand((40, 2, 64), 6)
    c0, b0, r0 = O.nvfp4t_pack(x, kind)
    for j in (-20, 9):
        xs = O.f32_to_bf16(O.bf16_to_f32(x) * np.float32(2.0 ** j))
        c, b, r = O.nvfp4t_pack(xs, kind)
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(b, b0)
        assert r[0] == r0[0] * np.float32(2.0 ** j)


def test_partial_key_group_equals_zero_padding():
    """T = 20: the last K group holds 4 rows; padding it with zero rows to T = 32
    changes no code and no block scale (|0| never raises a block's or the tensor's max)."""
    T, H, D = 20, 2, 32
    x = _rand((T, H, D), 7)
    c, b, r = O.nvfp4t_pack(x, K)
    xp = np.zeros((32, H, D), np.uint16)
    xp[:T] = x
    cp, bp, rp = O.nvfp4t_pack(xp, K)
    assert r[0] == rp[0]
    np.testing.assert_array_equal(c, cp[:T])
    np.testing.assert_array_equal(b, bp)
    assert b.shape == (2, H, D)


@pytest.mark.parametrize("kind", [K, V])
def test_zero_tensor_gives_signed_zero_codes(kind):
    x = np.zeros((16, 1, 32), np.uint16)
    x[3, 0, 5] = 0x8000  # -0
    c, b, r = O.nvfp4t_pack(x, kind)
    assert r[0] == 0 and (b == 0).all()
    e = _transpose_codes(c, 16, 1, 32)
    assert e[3, 0, 5] == 8 and (np.delete(e.reshape(-1), 3 * 32 + 5) == 0).all()
    y = O.nvfp4t_unpack(c, b, r, kind)
    assert y[3, 0, 5] == 0x8000 and (np.delete(y.reshape(-1), 3 * 32 + 5) == 0).all()


def test_storage_accounting_matches_the_buffers():
    for kind in (K, V):
        for (T, H, D) in [(16, 1, 128), (20, 3, 64), (300, 8, 128)]:
            c, b, r = O.nvfp4t_pack(_rand((T, H, D), 8), kind)
            assert c.nbytes + b.nbytes + r.nbytes == O.storage_bytes(O.FMT_NVFP4_TENSOR, kind, 16, T, H, D)
