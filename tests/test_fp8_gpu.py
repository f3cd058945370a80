"""FP8 E4M3 row codec on the GPU through the C ABI (quant-scatter into paged slots,
paged restore, pack/unpack and residual payloads), compared element by element with
the CPU oracle: E4M3 code bytes, FP32 row scales and restored bf16 are bit-exact."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth
from kvq_testutil import POISON, bits, f32bits, poison_bf16, status_word, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8 = kvq.FMT_FP8


def fp8_pool(num_slots, H, D, bs=16, fill=POISON):
    return kvq.KvPool.empty(num_slots, H, D, bs, fill=fill, fmt=FP8)


def assert_fp8_rows(got_codes, got_rs, want_codes, want_rs, what=""):
    np.testing.assert_array_equal(got_codes, want_codes, err_msg=f"{what} codes")
    np.testing.assert_array_equal(f32bits(got_rs), f32bits(want_rs), err_msg=f"{what} row scales")


def scatter_and_check(k, v, slots, pool):
    st = status_word()
    kvq.kvq_quant_scatter(k, v, slots, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sl = slots.cpu().numpy()
    for x, codes, rsc, what in ((k, pool.k_codes, pool.k_rscale, "K"), (v, pool.v_codes, pool.v_rscale, "V")):
        if x is None:
            continue
        c, r = O.fp8_encode_rows(bits(x.contiguous()))
        s = torch.as_tensor(sl, device=codes.device)
        assert_fp8_rows(u8(codes.index_select(0, s)), rsc.index_select(0, s), c, r, what)


def test_fp8_pool_layout_and_storage():
    pool = fp8_pool(32, 4, 128)
    assert pool.k_bscale is None and pool.k_codes.shape == (32, 4, 128)
    assert pool.nbytes() == 2 * kvq.kvq_storage_bytes(FP8, 0, 0, 32, 4, 128) == 2 * 32 * 4 * 132


def test_fp8_one_layer_round_trip():
    """K, V [256, 8, 128], N(0,1) with 1% x20 outliers, slots 0..255; pack/unpack too."""
    k, v, slots = synth.one_layer_case(seed=0)
    kd, vd = k.to(DEV), v.to(DEV)
    pool = fp8_pool(256, 8, 128)
    scatter_and_check(kd, vd, slots.to(DEV), pool)
    table = torch.arange(16, dtype=torch.int32, device=DEV).view(1, 16)
    lens = torch.tensor([256], dtype=torch.int32, device=DEV)
    ko, vo = poison_bf16((1, 256, 8, 128)), poison_bf16((1, 256, 8, 128))
    st = status_word()
    kvq.kvq_restore(pool, table, lens, 256, ko, vo, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, out in ((k, ko), (v, vo)):
        np.testing.assert_array_equal(bits(out[0]), O.fp8_decode_rows(*O.fp8_encode_rows(bits(x))))
    pk = kvq.Packed.empty(FP8, kvq.KIND_VALUE, 256, 8, 128)
    kvq.kvq_pack(vd, pk)
    y = poison_bf16((256, 8, 128))
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    c, r = O.fp8_encode_rows(bits(v))
    assert_fp8_rows(u8(pk.codes), pk.rscale, c, r, "pack")
    np.testing.assert_array_equal(bits(y), O.fp8_decode_rows(c, r))
    # FP8 keeps 3 mantissa bits: the error is far below NVFP4's on the same data
    err = (y.float() - vd.float()).pow(2).mean().sqrt().item()
    assert err < 0.1


@pytest.mark.parametrize("H,D", [(1, 16), (3, 48), (2, 96), (8, 128), (4, 256), (1, 512)])
def test_fp8_ragged_paged_round_trip_all_shapes(H, D):
    S, Tmax, bs = 3, 70, 16
    lens = torch.tensor([70, 33, 1], dtype=torch.int32)
    mb = -(-Tmax // bs)
    nblocks = S * mb + 3
    table = synth.block_permutation(nblocks, 60 + D)[: S * mb].view(S, mb).contiguous()
    k = synth.normal_bf16((S, Tmax, H, D), 60 + D, synth.STREAM_K, 0.02, 30.0)
    v = synth.normal_bf16((S, Tmax, H, D), 60 + D, synth.STREAM_V, 0.02, 30.0)
    pool = fp8_pool(nblocks * bs, H, D, bs)
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
    for P, out in (((pool.k_codes, pool.k_rscale), ko), ((pool.v_codes, pool.v_rscale), vo)):
        opool = (np.ascontiguousarray(u8(P[0])), np.ascontiguousarray(P[1].cpu().numpy()))
        want, ost = O.fp8_restore(opool, bs, table.numpy(), lens.numpy(), Tmax,
                                  out=np.full((S, Tmax, H, D), 0xA5A5, np.uint16))
        assert ost == 0
        np.testing.assert_array_equal(bits(out), want)


@pytest.mark.parametrize("bs", [1, 8, 32, 64, 256])
def test_fp8_ragged_paged_round_trip_block_sizes(bs):
    """The FP8 restore reads each row's sequence length and block-table entry an
    iteration ahead; block sizes other than 16, with sequences ending inside a block
    and one shorter than a block."""
    S, Tmax, H, D = 3, 300, 4, 128
    lens = torch.tensor([300, 129, 5], dtype=torch.int32)
    mb = -(-Tmax // bs)
    nblocks = S * mb + 3
    table = synth.block_permutation(nblocks, 70 + bs)[: S * mb].view(S, mb).contiguous()
    k = synth.normal_bf16((S, Tmax, H, D), 70 + bs, synth.STREAM_K)
    v = synth.normal_bf16((S, Tmax, H, D), 70 + bs, synth.STREAM_V)
    pool = fp8_pool(nblocks * bs, H, D, bs)
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
    for P, out in (((pool.k_codes, pool.k_rscale), ko), ((pool.v_codes, pool.v_rscale), vo)):
        opool = (np.ascontiguousarray(u8(P[0])), np.ascontiguousarray(P[1].cpu().numpy()))
        want, ost = O.fp8_restore(opool, bs, table.numpy(), lens.numpy(), Tmax,
                                  out=np.full((S, Tmax, H, D), 0xA5A5, np.uint16))
        assert ost == 0
        np.testing.assert_array_equal(bits(out), want)


def test_fp8_strided_k_under_graph_capture():
    """One-token appends: K a view of a fused qkv (row pitch 1152), V its own tensor,
    captured in a CUDA graph and replayed."""
    qkv, k, v, slots = synth.decode_step_case(seed=2)
    kd = qkv.to(DEV)[:, :1024].unflatten(1, (8, 128))
    vd, sd = v.to(DEV), slots.to(DEV)
    pool = fp8_pool(65536, 8, 128)
    st = status_word()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kvq.kvq_quant_scatter(kd, vd, sd, pool, st)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    pool2 = fp8_pool(65536, 8, 128)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_quant_scatter(kd, vd, sd, pool2, st)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sl = sd.cpu().numpy()
    for x, P in ((k, (pool2.k_codes, pool2.k_rscale)), (v, (pool2.v_codes, pool2.v_rscale))):
        c, r = O.fp8_encode_rows(bits(x))
        assert_fp8_rows(u8(P[0])[sl], P[1].cpu()[sl], c, r)
    mask = np.ones(65536, bool)
    mask[sl] = False
    assert (u8(pool2.v_codes)[mask] == POISON).all()
    assert torch.equal(pool.k_codes, pool2.k_codes)


# ---------------------------------------------------------------------------
# constructed rows
# ---------------------------------------------------------------------------
def _gpu_rows(x_bits: np.ndarray):
    n, D = x_bits.shape
    x = synth.from_bits(x_bits).to(DEV).view(n, 1, D)
    pk = kvq.Packed.empty(FP8, kvq.KIND_KEY, n, 1, D)
    kvq.kvq_pack(x, pk)
    y = poison_bf16((n, 1, D))
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    return u8(pk.codes)[:, 0], pk.rscale.cpu()[:, 0], bits(y)[:, 0]


def _check_constructed(rows: np.ndarray):
    xb = O.f32_to_bf16(rows.astype(np.float32))
    c, r, y = _gpu_rows(xb)
    wc, wr = O.fp8_encode_rows(xb)
    assert_fp8_rows(c, r, wc, wr, "constructed")
    np.testing.assert_array_equal(y, O.fp8_decode_rows(wc, wr))
    return c


def test_e4m3_rounding_of_every_bf16_value_in_range():
    """A row holding 448 has rs = 1 and q = x exactly, so every bf16 value in
    [-448, 448] passes through the hardware E4M3 rounding once; the codes must
    equal the oracle's nearest-even E4M3 encoding."""
    allb = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f32(allb)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    D = 256
    rows = []
    for j in range(0, len(vals), D - 1):
        r = np.zeros(D, np.float32)
        r[0] = 448.0
        ch = vals[j:j + D - 1]
        r[1:1 + len(ch)] = ch
        rows.append(r)
    c = _check_constructed(np.array(rows))
    want = O.e4m3_encode(np.array(rows, np.float32)).reshape(c.shape)
    np.testing.assert_array_equal(c, want)


def test_fp8_special_rows():
    D = 64
    rows = np.zeros((9, D), np.float64)
    rows[1] = -0.0                                  # signed zeros keep their sign bit
    rows[2, ::3] = 2.0 ** -133                      # rs subnormal: divide directly
    rows[2, 1::3] = -(2.0 ** -133)
    rows[3, 0] = 2.0 ** -120
    rows[3, 1:4] = [2.0 ** -126, -(2.0 ** -129), 2.0 ** -131]
    rows[4, 0] = 1e4                                # values far below the row maximum underflow
    rows[4, 1:17] = 1e-4 * np.array([1, -1] * 8)
    rows[5] = 3.0e38 * np.linspace(-1, 1, D)        # near the bf16 maximum
    rows[6, 5] = -1.0                               # a single negative value
    rng = np.random.default_rng(6)
    rows[7] = rng.standard_normal(D) * 2.0 ** 40
    rows[8] = rng.standard_normal(D) * 2.0 ** -40
    _check_constructed(rows)


def test_fp8_exact_rows_round_trip_identically():
    """Rows of E4M3 values scaled by 2^k with 448 * 2^k present reconstruct exactly."""
    rng = np.random.default_rng(7)
    e4 = np.array([O.e4m3_value(c) for c in range(0, 127)])
    rows = []
    for k in (-100, -8, 0, 12, 100):
        for _ in range(6):
            r = rng.choice(e4, 128) * rng.choice([-1, 1], 128)
            r[rng.integers(0, 128)] = 448.0
            rows.append(r * 2.0 ** k)
    xb = O.f32_to_bf16(np.array(rows, np.float32))
    _, _, y = _gpu_rows(xb)
    np.testing.assert_array_equal(y, xb)


# ---------------------------------------------------------------------------
# residual payloads in FP8, and the device status word
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("P", [None, 300])
def test_fp8_base_fp8_residual_chain(P):
    """FP8 base of loop 0, then FP8 residual rows (dense, or 300 of 1200 kept)."""
    T, H, D, loops, seed = 1200, 4, 128, 4, 8
    L = synth.residual_loops(T, H, D, loops, seed, stream=synth.STREAM_V)
    pk = kvq.Packed.empty(FP8, kvq.KIND_VALUE, T, H, D)
    kvq.kvq_pack(L[0].to(DEV), pk)
    recon = poison_bf16((T, H, D))
    kvq.kvq_unpack(pk, recon)
    recon_o = O.fp8_decode_rows(*O.fp8_encode_rows(bits(L[0])))
    st = status_word()
    for i in range(1, loops):
        pos = None if P is None else synth.sorted_positions(T, P, seed, stream=synth.STREAM_POS + i)
        n = T if pos is None else P
        pay = kvq.Packed.empty(FP8, kvq.KIND_VALUE, n, H, D)
        posd = None if pos is None else pos.to(DEV)
        pos_out = None if pos is None else torch.full((n,), -7, dtype=torch.int32, device=DEV)
        kvq.kvq_encode_residual(L[i].to(DEV), recon, posd, pay, pos_out, st)
        nxt = poison_bf16((T, H, D))
        kvq.kvq_decode_residual(pay, posd, recon, nxt, st)
        ip = recon.clone()
        kvq.kvq_decode_residual(pay, posd, ip, ip, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        opay, ost = O.residual_encode(bits(L[i]), recon_o, None if pos is None else pos.numpy(), FP8,
                                      kvq.KIND_VALUE)
        assert ost == 0
        assert_fp8_rows(u8(pay.codes), pay.rscale, opay["codes"], opay["rscale"], f"loop {i} payload")
        if pos is not None:
            np.testing.assert_array_equal(pos_out.cpu().numpy(), pos.numpy())
        recon_o, _ = O.residual_decode(opay, recon_o)
        np.testing.assert_array_equal(bits(nxt), recon_o, err_msg=f"loop {i}")
        assert torch.equal(ip.view(torch.int16), nxt.view(torch.int16))
        recon = nxt


def test_fp8_bad_slots_are_flagged():
    H, D = 2, 32
    k, v = synth.layer_kv(5, H, D, seed=42)
    pool = fp8_pool(32, H, D, fill=0)
    st = status_word()
    slots = torch.tensor([0, -1, 32, 5, 10**12], dtype=torch.int64, device=DEV)
    kvq.kvq_quant_scatter(k.to(DEV), v.to(DEV), slots, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_SLOT
    rs = pool.v_rscale.cpu()
    assert rs[0].abs().sum() > 0 and rs[5].abs().sum() > 0
    assert rs[[1, 2, 3, 4, 6]].abs().sum() == 0
    st.zero_()
    table = torch.tensor([[0, 7]], dtype=torch.int32, device=DEV)
    out = poison_bf16((1, 32, H, D))
    kvq.kvq_restore(pool, table, torch.tensor([20], dtype=torch.int32, device=DEV), 32, out, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.DEV_BAD_BLOCK


def test_fp8_long_context_sampled():
    """262,144 tokens x 4 KV heads x D256 with 0.5% x50 outliers, block-shuffled slots,
    full paged restore; a sample of rows checked against the oracle, and the pack path
    must give the same bytes as the paged path."""
    T, H, D, bs = 1 << 18, 4, 256, 16
    perm = synth.block_permutation(T // bs, seed=9).to(DEV)
    t = torch.arange(T, device=DEV)
    slots = perm[t // bs].long() * bs + t % bs
    k = synth.normal_bf16((T, H, D), 9, synth.STREAM_K, 0.005, 50.0, device=DEV)
    v = synth.normal_bf16((T, H, D), 9, synth.STREAM_V, 0.005, 50.0, device=DEV)
    pool = fp8_pool(T, H, D, bs, fill=None)
    st = status_word()
    kvq.kvq_quant_scatter(k, v, slots, pool, st)
    ko = poison_bf16((1, T, H, D))
    kvq.kvq_restore(pool, perm.view(1, -1), torch.tensor([T], dtype=torch.int32, device=DEV), T,
                    ko, None, st)
    pk = kvq.Packed.empty(FP8, kvq.KIND_KEY, T, H, D)
    kvq.kvq_pack(k, pk)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pool.k_codes.index_select(0, slots), pk.codes)
    rng = np.random.default_rng(9)
    toks = np.unique(np.concatenate([rng.choice(T, 3000, replace=False), [0, 15, 16, T - 1]]))
    ti = torch.as_tensor(toks, device=DEV)
    c, r = O.fp8_encode_rows(bits(k.index_select(0, ti)))
    assert_fp8_rows(u8(pk.codes.index_select(0, ti)), pk.rscale.index_select(0, ti), c, r)
    np.testing.assert_array_equal(bits(ko[0].index_select(0, ti)), O.fp8_decode_rows(c, r))


# ---------------------------------------------------------------------------
# k8v4: FP8 K beside NVFP4 V in one pool
# ---------------------------------------------------------------------------
def test_k8v4_split_pool_scatter_restore_and_graph():
    """FP8 E4M3 keys and NVFP4 values in one pool (two launches per call), ragged
    sequences through a shuffled block table; eager and graph-captured calls agree."""
    H, D, bs, S, Tmax = 4, 128, 16, 3, 90
    lens = torch.tensor([90, 47, 16], dtype=torch.int32)
    mb = -(-Tmax // bs)
    nblocks = S * mb + 2
    table = synth.block_permutation(nblocks, 71)[: S * mb].view(S, mb).contiguous()
    k = synth.normal_bf16((S, Tmax, H, D), 71, synth.STREAM_K, 0.01, 20.0)
    v = synth.normal_bf16((S, Tmax, H, D), 71, synth.STREAM_V, 0.01, 20.0)
    pool = kvq.KvPool.empty(nblocks * bs, H, D, bs, fill=POISON, fmt=FP8, v_fmt=kvq.FMT_NVFP4)
    assert pool.k_bscale is None and pool.v_bscale.shape == (nblocks * bs, H, D // 16)
    assert pool.nbytes() == nblocks * bs * H * ((D + 4) + (D // 2 + D // 16 + 4))
    st = status_word()
    for s in range(S):
        n = int(lens[s])
        t = torch.arange(n)
        slots = (table[s, t // bs].long() * bs + t % bs).to(DEV)
        kvq.kvq_quant_scatter(k[s, :n].to(DEV), v[s, :n].to(DEV), slots, pool, st)
    ko, vo = poison_bf16((S, Tmax, H, D)), poison_bf16((S, Tmax, H, D))
    td, ld = table.to(DEV), lens.to(DEV)  # device inputs before capture (no copies inside it)
    kvq.kvq_restore(pool, td, ld, Tmax, ko, vo, st)
    ko2, vo2 = poison_bf16((S, Tmax, H, D)), poison_bf16((S, Tmax, H, D))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kvq.kvq_restore(pool, td, ld, Tmax, ko2, vo2, st)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kpool = (np.ascontiguousarray(u8(pool.k_codes)), np.ascontiguousarray(pool.k_rscale.cpu().numpy()))
    vpool = (np.ascontiguousarray(u8(pool.v_codes)), np.ascontiguousarray(u8(pool.v_bscale)),
             np.ascontiguousarray(pool.v_rscale.cpu().numpy()))
    for s in range(S):  # the pool rows are the oracle's encodings of the tokens
        n = int(lens[s])
        t = np.arange(n)
        sl = table.numpy()[s, t // bs].astype(np.int64) * bs + t % bs
        c, r = O.fp8_encode_rows(bits(k[s, :n]))
        assert_fp8_rows(kpool[0][sl], kpool[1][sl], c, r, "K")
        c, b, r = O.nvfp4_encode_rows(bits(v[s, :n]))
        np.testing.assert_array_equal(vpool[0][sl], c)
        np.testing.assert_array_equal(vpool[1][sl], b)
        np.testing.assert_array_equal(f32bits(vpool[2][sl]), f32bits(r))
    blank = lambda: np.full((S, Tmax, H, D), 0xA5A5, np.uint16)
    wk, ost = O.fp8_restore(kpool, bs, table.numpy(), lens.numpy(), Tmax, out=blank())
    assert ost == 0
    wv, ost = O.nvfp4_restore(vpool, bs, table.numpy(), lens.numpy(), Tmax, out=blank())
    assert ost == 0
    for out in (ko, ko2):
        np.testing.assert_array_equal(bits(out), wk)
    for out in (vo, vo2):
        np.testing.assert_array_equal(bits(out), wv)
