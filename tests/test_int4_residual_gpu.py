"""INT4 affine codec and residual encode/decode on the GPU through the C ABI,
compared bit for bit with the CPU oracle (codes, FP16 metadata, position maps and
reconstructed bf16)."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth
from kvq_testutil import POISON, bits, f16bits, f32bits, poison_bf16, status_word, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_int4_pack(x, kind, G=64):
    T, H, D = x.shape
    pk = kvq.Packed.empty(kvq.FMT_INT4, kind, T, H, D, G)
    kvq.kvq_pack(x, pk)
    y = poison_bf16((T, H, D))
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    return pk, y


def check_int4(pk, codes, mn, sc):
    np.testing.assert_array_equal(u8(pk.codes), codes, err_msg="codes")
    np.testing.assert_array_equal(f16bits(pk.meta0), mn, err_msg="fp16 minimum")
    np.testing.assert_array_equal(f16bits(pk.meta1), sc, err_msg="fp16 scale")


def check_payload(pay, opay):
    np.testing.assert_array_equal(u8(pay.codes), opay["codes"], err_msg="payload codes")
    if pay.fmt == kvq.FMT_INT4:
        np.testing.assert_array_equal(f16bits(pay.meta0), opay["meta_a"], err_msg="payload min")
        np.testing.assert_array_equal(f16bits(pay.meta1), opay["meta_b"], err_msg="payload scale")
    elif pay.fmt == kvq.FMT_FP8:
        np.testing.assert_array_equal(f32bits(pay.rscale), f32bits(opay["rscale"]), err_msg="row scales")
    else:
        np.testing.assert_array_equal(u8(pay.meta0), opay["meta_a"], err_msg="payload block scales")
        np.testing.assert_array_equal(f32bits(pay.rscale), f32bits(opay["rscale"]), err_msg="row scales")


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
@pytest.mark.parametrize("T,H,D,G", [(256, 8, 128, 64), (4100, 2, 128, 64), (130, 3, 96, 64),
                                     (64, 2, 32, 64), (200, 2, 128, 16), (77, 1, 512, 512),
                                     (100, 3, 96, 32), (50, 2, 224, 64), (40, 1, 480, 128),
                                     (33, 5, 80, 32), (9, 1, 256, 32)])
def test_int4_pack_unpack_matches_oracle(kind, T, H, D, G):
    x = synth.normal_bf16((T, H, D), seed=50 + T, stream=1, outlier_frac=0.01, outlier_scale=20.0)
    pk, y = gpu_int4_pack(x.to(DEV), kind, G)
    codes, mn, sc = O.int4_pack(bits(x), kind, G)
    check_int4(pk, codes, mn, sc)
    np.testing.assert_array_equal(bits(y), O.int4_unpack(codes, mn, sc, kind, G))


def test_int4_constant_and_exact_groups():
    x = torch.full((64, 2, 32), 0.3, dtype=torch.bfloat16)
    x[:, 1] = torch.arange(32, dtype=torch.float32).remainder(16).to(torch.bfloat16)  # exact grid
    for kind in (kvq.KIND_KEY, kvq.KIND_VALUE):
        pk, y = gpu_int4_pack(x.to(DEV), kind)
        codes, mn, sc = O.int4_pack(bits(x), kind, 64)
        check_int4(pk, codes, mn, sc)
        np.testing.assert_array_equal(bits(y), O.int4_unpack(codes, mn, sc, kind, 64))


def _chain(kind, fmt_res, T=4096, H=8, D=128, P=1024, loops=4, seed=4, inplace_check=True, G=64):
    """Base INT4 pack of loop 0, then loops 1.. residual-encoded against the
    reconstructed predecessor with P kept rows; every step checked against the oracle."""
    stream = synth.STREAM_K if kind == kvq.KIND_KEY else synth.STREAM_V
    L = synth.residual_loops(T, H, D, loops, seed, stream=stream)
    pk, recon = gpu_int4_pack(L[0].to(DEV), kind, G)
    codes, mn, sc = O.int4_pack(bits(L[0]), kind, G)
    check_int4(pk, codes, mn, sc)
    recon_o = O.int4_unpack(codes, mn, sc, kind, G)
    np.testing.assert_array_equal(bits(recon), recon_o)
    st = status_word()
    for i in range(1, loops):
        pos = synth.sorted_positions(T, P, seed, stream=synth.STREAM_POS + i) if P is not None else None
        n = T if pos is None else P
        pay = kvq.Packed.empty(fmt_res, kind, n, H, D, G)
        pos_out = torch.full((max(n, 1),), -7, dtype=torch.int32, device=DEV)[:n]
        posd = pos.to(DEV) if pos is not None else None
        kvq.kvq_encode_residual(L[i].to(DEV), recon, posd, pay, pos_out if pos is not None else None, st)
        nxt = poison_bf16((T, H, D))
        kvq.kvq_decode_residual(pay, posd, recon, nxt, st)
        if inplace_check:
            ip = recon.clone()
            kvq.kvq_decode_residual(pay, posd, ip, ip, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        opay, ost = O.residual_encode(bits(L[i]), recon_o, None if pos is None else pos.numpy(), fmt_res, kind, G)
        assert ost == 0
        check_payload(pay, opay)
        if pos is not None:
            np.testing.assert_array_equal(pos_out.cpu().numpy(), pos.numpy())
        recon_o, _ = O.residual_decode(opay, recon_o)
        np.testing.assert_array_equal(bits(nxt), recon_o, err_msg=f"loop {i} reconstruction")
        if inplace_check:
            assert torch.equal(ip.view(torch.int16), nxt.view(torch.int16))
        recon = nxt
    return recon


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_g64_residual_chain_sparse_quarter_rows(kind):
    """4 loops of [4096, 8, 128]; loops 1-3 keep 25% of rows (int32 position map)."""
    _chain(kind, kvq.FMT_INT4)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_dense_residual_chain(kind):
    _chain(kind, kvq.FMT_INT4, T=1000, H=2, D=64, P=None)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_base_nvfp4_residual_chain(kind):
    """A mixed chain: INT4 base, NVFP4 residual rows."""
    _chain(kind, kvq.FMT_NVFP4, T=600, H=3, D=96, P=150)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_base_fp8_residual_chain(kind):
    """A mixed chain: INT4 base, FP8 E4M3 residual rows."""
    _chain(kind, kvq.FMT_FP8, T=600, H=3, D=96, P=150)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
@pytest.mark.parametrize("G", [16, 32, 128, 256, 512])
def test_int4_residual_chain_every_group_size(kind, G):
    """The other group sizes the encode and decode kernels specialise, with ragged
    compact groups: 1100 tokens, 300 kept a loop (every size leaves a partial group)."""
    _chain(kind, kvq.FMT_INT4, T=1100, H=2, D=128, P=300, loops=3, G=G)


@pytest.mark.parametrize("fmt", [kvq.FMT_NVFP4, kvq.FMT_FP8])
@pytest.mark.parametrize("D", [64, 256, 512])
def test_row_codec_residual_chain_head_dims(fmt, D):
    """NVFP4 and FP8 residual rows at the head dims that change the decode kernels' lane
    layout (4, 16 and 32 blocks of 16 a row), on an INT4 base."""
    _chain(kvq.KIND_VALUE, fmt, T=400, H=2, D=D, P=100, loops=3)


def test_ragged_compact_groups_and_odd_sizes():
    _chain(kvq.KIND_KEY, kvq.FMT_INT4, T=777, H=1, D=48, P=333, loops=3)


def test_empty_and_full_position_maps_and_bad_maps():
    T, H, D = 128, 2, 32
    cur = synth.normal_bf16((T, H, D), 60, 1).to(DEV)
    prev = synth.normal_bf16((T, H, D), 60, 2).to(DEV)
    st = status_word()
    # empty map: nothing kept, out == prev (copy and in place)
    empty = torch.zeros(0, dtype=torch.int32, device=DEV)
    pay = kvq.Packed.empty(kvq.FMT_INT4, kvq.KIND_KEY, 0, H, D, 64)
    kvq.kvq_encode_residual(cur, prev, empty, pay, None, st)
    out = poison_bf16((T, H, D))
    kvq.kvq_decode_residual(pay, empty, prev, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.int16), prev.view(torch.int16))
    # every row kept == dense, bitwise
    allpos = torch.arange(T, dtype=torch.int32, device=DEV)
    for fmt, kind in ((kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_INT4, kvq.KIND_VALUE), (kvq.FMT_NVFP4, 0)):
        a = kvq.Packed.empty(fmt, kind, T, H, D, 64)
        b = kvq.Packed.empty(fmt, kind, T, H, D, 64)
        kvq.kvq_encode_residual(cur, prev, allpos, a, None, st)
        kvq.kvq_encode_residual(cur, prev, None, b, None, st)
        oa, ob = poison_bf16((T, H, D)), poison_bf16((T, H, D))
        kvq.kvq_decode_residual(a, allpos, prev, oa, st)
        kvq.kvq_decode_residual(b, None, prev, ob, st)
        torch.cuda.synchronize()
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
        assert torch.equal(a.codes, b.codes)
    assert int(st.item()) == 0
    # unsorted / out-of-range maps are flagged, and nothing faults
    for bad in ([5, 3, 9], [1, 1, 2], [-1, 4, 6], [2, 4, T]):
        st.zero_()
        pos = torch.tensor(bad, dtype=torch.int32, device=DEV)
        for fmt, kind in ((kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_INT4, kvq.KIND_VALUE), (kvq.FMT_NVFP4, 0)):
            pay = kvq.Packed.empty(fmt, kind, 3, H, D, 64)
            kvq.kvq_encode_residual(cur, prev, pos, pay, None, st)
            o = prev.clone()
            kvq.kvq_decode_residual(pay, pos, o, o, st)
            o2 = poison_bf16((T, H, D))
            kvq.kvq_decode_residual(pay, pos, prev, o2, st)
        torch.cuda.synchronize()
        assert int(st.item()) & kvq.DEV_BAD_POS, bad
    # the context is still healthy
    torch.cuda.synchronize()


def test_zero_residual_reproduces_prev_bitwise():
    T, H, D = 300, 2, 64
    prev = synth.normal_bf16((T, H, D), 61, 1).to(DEV)
    pos = synth.sorted_positions(T, 100, 61).to(DEV)
    for fmt, kind in ((kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_INT4, kvq.KIND_VALUE), (kvq.FMT_NVFP4, 0)):
        pay = kvq.Packed.empty(fmt, kind, 100, H, D, 64)
        kvq.kvq_encode_residual(prev, prev, pos, pay)
        out = poison_bf16((T, H, D))
        kvq.kvq_decode_residual(pay, pos, prev, out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), prev.view(torch.int16))


def test_residual_with_strided_views():
    """cur a strided view (row pitch 3*H*D), prev contiguous, out a strided view."""
    T, H, D = 200, 2, 64
    big = synth.normal_bf16((T, 3 * H * D), 62, 1).to(DEV)
    cur = big[:, H * D:2 * H * D].unflatten(1, (H, D))
    prev = synth.normal_bf16((T, H, D), 62, 2).to(DEV)
    pos = synth.sorted_positions(T, 64, 62).to(DEV)
    for fmt, kind in ((kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_NVFP4, 0)):
        pay = kvq.Packed.empty(fmt, kind, 64, H, D, 64)
        kvq.kvq_encode_residual(cur, prev, pos, pay)
        outbig = poison_bf16((T, 2 * H * D))
        out = outbig[:, H * D:].unflatten(1, (H, D))
        kvq.kvq_decode_residual(pay, pos, prev, out)
        torch.cuda.synchronize()
        opay, _ = O.residual_encode(bits(cur), bits(prev), pos.cpu().numpy(), fmt, kind, 64)
        check_payload(pay, opay)
        want, _ = O.residual_decode(opay, bits(prev))
        np.testing.assert_array_equal(bits(out), want)
        assert (bits(outbig[:, :H * D]) == 0xA5A5).all()


def _tie_rows(scale, n_rows=64):
    """Channel groups (V kind, G = 64 channels) with min 0 and max 15 * scale, so the
    scale is `scale` up to rounding and (x - min) / scale hits every k + 1/2 (a tie,
    where rint must go to even), its bf16 neighbours, and the integers."""
    import numpy as np

    vals = []
    for k in range(15):
        m = (k + 0.5) * scale
        vals += [m, np.nextafter(np.float32(m), np.float32(0)), np.nextafter(np.float32(m), np.float32(99)),
                 k * scale, (k + 0.49) * scale, (k + 0.51) * scale]
    vals = np.array(vals, np.float64)
    rows = []
    for r in range(n_rows):
        body = np.roll(vals, r)[:62]
        rows.append(np.concatenate([[0.0, 15.0 * scale], body]))
    return np.array(rows)


@pytest.mark.parametrize("scale", [1.0, 0.25, 0.3, 1.7, 3e-3, 1e-30])
def test_int4_half_integer_quotients_round_to_even(scale):
    import numpy as np

    rows = _tie_rows(scale)
    xb = O.f32_to_bf16(rows.astype(np.float32)).reshape(-1, 1, 64)
    x = synth.from_bits(xb).to(DEV)
    for kind in (kvq.KIND_VALUE, kvq.KIND_KEY):
        pk, y = gpu_int4_pack(x, kind)
        codes, mn, sc = O.int4_pack(xb, kind, 64)
        check_int4(pk, codes, mn, sc)
        np.testing.assert_array_equal(bits(y), O.int4_unpack(codes, mn, sc, kind, 64))


def _signed_zero_mix(T, H, D, seed):
    """bf16 bits: every element a zero of random sign, then 30% of the elements a
    positive value, and in the second head's last 64 rows the values negative; the
    first 64 rows of head 0 stay zeros only."""
    rng = np.random.default_rng(seed)
    xb = (rng.integers(0, 2, size=(T, H, D)).astype(np.uint16) << 15).astype(np.uint16)
    mag = O.f32_to_bf16(np.abs(rng.standard_normal((T, H, D))).astype(np.float32) + 0.01)
    pick = rng.random((T, H, D)) < 0.3
    pick[:64, 0] = False
    xb[pick] = mag[pick]
    neg = pick.copy()
    neg[:-64] = False
    neg[:, 0] = False
    xb[neg] |= 0x8000
    return xb


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_signed_zero_groups_match_the_oracle(kind):
    """Groups whose minimum is a zero held with both signs: the stored FP16 minimum is
    -0 (the -0 < +0 order), in the plain pack and in the residual pack."""
    T, H, D = 256, 2, 128
    xb = _signed_zero_mix(T, H, D, seed=12)
    x = synth.from_bits(xb).to(DEV)
    pk, y = gpu_int4_pack(x, kind)
    codes, mn, sc = O.int4_pack(xb, kind, 64)
    assert (mn == 0x8000).any()
    check_int4(pk, codes, mn, sc)
    np.testing.assert_array_equal(bits(y), O.int4_unpack(codes, mn, sc, kind, 64))
    # residual: cur - prev gives -0 where cur is -0 and prev is +0
    prev_b = np.zeros_like(xb)
    pos = torch.arange(0, T, 2, dtype=torch.int32)
    pay = kvq.Packed.empty(kvq.FMT_INT4, kind, T // 2, H, D, 64)
    kvq.kvq_encode_residual(x, synth.from_bits(prev_b).to(DEV), pos.to(DEV), pay)
    torch.cuda.synchronize()
    opay, ost = O.residual_encode(xb, prev_b, pos.numpy(), kvq.FMT_INT4, kind, 64)
    assert ost == 0
    check_payload(pay, opay)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
@pytest.mark.parametrize("exps", [(-140, -133, -128, -126, -120, -110, -100, 0),
                                  (-80, -70, -67, -66, -65, -63, -60, -40)])
def test_int4_tiny_and_subnormal_groups(kind, exps):
    """Groups at scales 2^-140 .. 2^-100 (bf16 subnormals, subnormal and tiny normal
    scales) and around 2^-64 (where the kernels switch from dividing to the reciprocal
    and residual steps) beside ordinary groups, against the oracle."""
    T, H, D = 512, 2, 128
    x = synth.normal_bf16((T, H, D), seed=13, stream=1).float()
    exps = torch.tensor(exps, dtype=torch.float32)
    if kind == kvq.KIND_KEY:  # one scale per 64-row group
        s = exps.repeat_interleave(64)[:T].view(T, 1, 1)
    else:  # one scale per 64-channel group
        s = exps[torch.arange(T) % 8].view(T, 1, 1).repeat(1, H, 1)
        s = torch.cat([s.expand(T, H, 64), torch.zeros(T, H, 64)], dim=2)
    xb = (x * torch.exp2(s)).to(torch.bfloat16)
    bits_in = bits(xb)
    if float(exps.min()) < -126:  # subnormals present
        assert (((bits_in & 0x7F80) == 0) & ((bits_in & 0x7FFF) != 0)).any()
    pk, y = gpu_int4_pack(xb.to(DEV), kind)
    codes, mn, sc = O.int4_pack(bits_in, kind, 64)
    check_int4(pk, codes, mn, sc)
    np.testing.assert_array_equal(bits(y), O.int4_unpack(codes, mn, sc, kind, 64))


def test_int4_pack_unpack_at_the_bench_size_sampled():
    """[262144, 8, 128] G64 (the size bench.py times, in the same launch shapes), both
    kinds: 24 sampled K groups (64 rows x 8 heads x 128 channels each) and 256 sampled
    V rows against the oracle run on just those rows, codes, metadata and the unpack."""
    T, H, D, G = 262144, 8, 128, 64
    x = synth.normal_bf16((T, H, D), seed=21, stream=1, outlier_frac=0.01, outlier_scale=20.0, device=DEV)
    rng = np.random.default_rng(21)
    y = torch.empty_like(x)
    for kind in (kvq.KIND_KEY, kvq.KIND_VALUE):
        pk = kvq.Packed.empty(kvq.FMT_INT4, kind, T, H, D, G)
        kvq.kvq_pack(x, pk)
        kvq.kvq_unpack(pk, y)
        torch.cuda.synchronize()
        if kind == kvq.KIND_KEY:
            for g in rng.choice(T // G, 24, replace=False):
                rows = slice(int(g) * G, (int(g) + 1) * G)
                xb = bits(x[rows])
                codes, mn, sc = O.int4_pack(xb, kind, G)
                np.testing.assert_array_equal(u8(pk.codes[rows]), codes)
                np.testing.assert_array_equal(f16bits(pk.meta0[int(g):int(g) + 1]), mn)
                np.testing.assert_array_equal(f16bits(pk.meta1[int(g):int(g) + 1]), sc)
                np.testing.assert_array_equal(bits(y[rows]), O.int4_unpack(codes, mn, sc, kind, G))
        else:
            idx = np.sort(rng.choice(T, 256, replace=False))
            it = torch.from_numpy(idx).to(DEV)
            xb = bits(x[it])
            codes, mn, sc = O.int4_pack(xb, kind, G)
            np.testing.assert_array_equal(u8(pk.codes[it]), codes)
            np.testing.assert_array_equal(f16bits(pk.meta0[it]), mn)
            np.testing.assert_array_equal(f16bits(pk.meta1[it]), sc)
            np.testing.assert_array_equal(bits(y[it]), O.int4_unpack(codes, mn, sc, kind, G))


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_residual_encode_at_the_bench_size_sampled(kind):
    """Residual encode over [262144, 8, 128] with 25% of rows kept (65,536 compact rows),
    as bench.py times it: 16 sampled K groups of 64 compact rows (V: 256 compact rows)
    against the oracle's residual encode of just those rows."""
    T, H, D, G = 262144, 8, 128, 64
    cur = synth.normal_bf16((T, H, D), seed=22, stream=1, device=DEV)
    prev = synth.normal_bf16((T, H, D), seed=22, stream=2, device=DEV)
    pos = synth.sorted_positions(T, T // 4, 22, stream=synth.STREAM_POS).to(DEV)
    P = pos.numel()
    pay = kvq.Packed.empty(kvq.FMT_INT4, kind, P, H, D, G)
    kvq.kvq_encode_residual(cur, prev, pos, pay)
    torch.cuda.synchronize()
    rng = np.random.default_rng(22)
    if kind == kvq.KIND_KEY:
        picks = [slice(int(g) * G, (int(g) + 1) * G) for g in rng.choice(P // G, 16, replace=False)]
    else:
        picks = [torch.from_numpy(np.sort(rng.choice(P, 256, replace=False))).to(DEV)]
    for sel in picks:
        src = pos[sel].long()
        n = src.numel()
        opay, ost = O.residual_encode(bits(cur[src]), bits(prev[src]), np.arange(n, dtype=np.int32), kvq.FMT_INT4,
                                      kind, G)
        assert ost == 0
        np.testing.assert_array_equal(u8(pay.codes[sel]), opay["codes"])
        if kind == kvq.KIND_KEY:
            g = sel.start // G
            np.testing.assert_array_equal(f16bits(pay.meta0[g:g + 1]), opay["meta_a"])
            np.testing.assert_array_equal(f16bits(pay.meta1[g:g + 1]), opay["meta_b"])
        else:
            np.testing.assert_array_equal(f16bits(pay.meta0[sel]), opay["meta_a"])
            np.testing.assert_array_equal(f16bits(pay.meta1[sel]), opay["meta_b"])


@pytest.mark.parametrize("fmt,kind", [(kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_INT4, kvq.KIND_VALUE),
                                      (kvq.FMT_NVFP4, kvq.KIND_VALUE), (kvq.FMT_FP8, kvq.KIND_VALUE)])
def test_residual_arithmetic_across_exponent_gaps(fmt, kind):
    """cur and prev at magnitudes 2^-30 .. 2^30 apart (per token), so bf16(cur - prev)
    and bf16(prev + y) cross the regime where the binary32 result stops being exact;
    payload and reconstruction against the oracle, copy and in place."""
    T, H, D = 640, 2, 128
    gaps = torch.tensor([-30, -17, -16, -9, -8, 0, 8, 9, 16, 17, 30], dtype=torch.float32)
    e = gaps[torch.arange(T) % gaps.numel()].view(T, 1, 1)
    cur = (synth.normal_bf16((T, H, D), 71, 1).float() * torch.exp2(e / 2)).to(torch.bfloat16)
    prev = (synth.normal_bf16((T, H, D), 71, 2).float() * torch.exp2(-e / 2)).to(torch.bfloat16)
    pos = synth.sorted_positions(T, T // 2, 71)
    pay = kvq.Packed.empty(fmt, kind, pos.numel(), H, D, 64)
    kvq.kvq_encode_residual(cur.to(DEV), prev.to(DEV), pos.to(DEV), pay)
    out = poison_bf16((T, H, D))
    kvq.kvq_decode_residual(pay, pos.to(DEV), prev.to(DEV), out)
    ip = prev.to(DEV).clone()
    kvq.kvq_decode_residual(pay, pos.to(DEV), ip, ip)
    torch.cuda.synchronize()
    opay, ost = O.residual_encode(bits(cur), bits(prev), pos.numpy(), fmt, kind, 64)
    assert ost == 0
    check_payload(pay, opay)
    ref, dst = O.residual_decode(opay, bits(prev))
    assert dst == 0
    np.testing.assert_array_equal(bits(out), ref)
    np.testing.assert_array_equal(bits(ip), ref)


# ---------------------------------------------------------------------------
# CUDA Graph capture of pack / unpack and the residual entry points
# (FreeToken PR #408, Summary: the KV writes are safe under CUDA Graph capture)
# ---------------------------------------------------------------------------
def _poison_packed(pk):
    for t in (pk.codes, pk.meta0, pk.meta1, pk.rscale):
        if t is not None:
            t.view(torch.uint8).fill_(POISON)


def _same_packed(a, b):
    for x, y in ((a.codes, b.codes), (a.meta0, b.meta0), (a.meta1, b.meta1), (a.rscale, b.rscale)):
        if x is not None:
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_int4_pack_unpack_under_graph_capture(kind):
    """kvq_pack and kvq_unpack (INT4 G64, a partial last K group) captured in one graph
    and replayed twice: bit-identical to the eager calls and to the oracle."""
    T, H, D, G = 4100, 8, 128, 64
    x = synth.normal_bf16((T, H, D), seed=60, stream=1, outlier_frac=0.01, outlier_scale=20.0)
    xd = x.to(DEV)
    pk, y = gpu_int4_pack(xd, kind, G)
    pk2 = kvq.Packed.empty(kvq.FMT_INT4, kind, T, H, D, G)
    y2 = torch.empty_like(y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_pack(xd, pk2)
        kvq.kvq_unpack(pk2, y2)
    for _ in range(2):
        _poison_packed(pk2)
        y2.view(torch.uint8).fill_(POISON)
        g.replay()
        torch.cuda.synchronize()
        _same_packed(pk2, pk)
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    codes, mn, sc = O.int4_pack(bits(x), kind, G)
    check_int4(pk2, codes, mn, sc)
    np.testing.assert_array_equal(bits(y2), O.int4_unpack(codes, mn, sc, kind, G))


@pytest.mark.parametrize("fmt,kind", [(kvq.FMT_INT4, kvq.KIND_KEY), (kvq.FMT_INT4, kvq.KIND_VALUE),
                                      (kvq.FMT_NVFP4, kvq.KIND_KEY), (kvq.FMT_FP8, kvq.KIND_VALUE)])
def test_residual_encode_decode_under_graph_capture(fmt, kind):
    """kvq_encode_residual with 25% of rows kept, then kvq_decode_residual into a
    separate output and in place, captured in one graph and replayed: payload, owned
    position map and both reconstructions bit-identical to the eager calls and to the
    oracle."""
    T, H, D, P = 4096, 8, 128, 1024
    prev = synth.normal_bf16((T, H, D), seed=61, stream=1)
    cur = synth.normal_bf16((T, H, D), seed=61, stream=2)
    pos = synth.sorted_positions(T, P, seed=61)
    cd, pd, posd = cur.to(DEV), prev.to(DEV), pos.to(DEV)
    st = status_word()

    def run(pay, pos_out, out, ip):
        kvq.kvq_encode_residual(cd, pd, posd, pay, pos_out, st)
        kvq.kvq_decode_residual(pay, posd, pd, out, st)
        kvq.kvq_decode_residual(pay, posd, ip, ip, st)

    pay = kvq.Packed.empty(fmt, kind, P, H, D, 64)
    pos_out = torch.empty(P, dtype=torch.int32, device=DEV)
    out, ip = poison_bf16((T, H, D)), pd.clone()
    run(pay, pos_out, out, ip)
    pay2 = kvq.Packed.empty(fmt, kind, P, H, D, 64)
    pos_out2 = torch.empty(P, dtype=torch.int32, device=DEV)
    out2, ip2 = poison_bf16((T, H, D)), pd.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(pay2, pos_out2, out2, ip2)
    for _ in range(2):
        _poison_packed(pay2)
        pos_out2.fill_(-7)
        out2.view(torch.uint8).fill_(POISON)
        ip2.copy_(pd)
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        _same_packed(pay2, pay)
        assert torch.equal(pos_out2, pos_out)
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(ip2.view(torch.int16), out.view(torch.int16))
    opay, ost = O.residual_encode(bits(cur), bits(prev), pos.numpy(), fmt, kind, 64)
    assert ost == 0
    check_payload(pay2, opay)
    np.testing.assert_array_equal(pos_out2.cpu().numpy(), pos.numpy())
    np.testing.assert_array_equal(bits(out2), O.residual_decode(opay, bits(prev))[0])
