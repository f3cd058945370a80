"""NVFP4 with one FP32 scale per tensor (G16 blocks along the kind's axis) on the GPU
through kvq_pack / kvq_unpack, bit-exact against the oracle: codes, block scales,
the tensor scale and the decoded bf16."""

import numpy as np
import pytest
import torch

import oracle as O
import quantized_kv_cache_nvfp4_gb300 as kvq
from quantized_kv_cache_nvfp4_gb300 import synth
from kvq_testutil import bits, f32bits, poison_bf16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
T4 = kvq.FMT_NVFP4_TENSOR


def gpu_pack(x, kind):
    T, H, D = x.shape
    pk = kvq.Packed.empty(T4, kind, T, H, D)
    kvq.kvq_pack(x, pk)
    y = poison_bf16((T, H, D))
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    return pk, y


def check(x_cpu, pk, y, kind):
    c, b, r = O.nvfp4t_pack(bits(x_cpu), kind)
    np.testing.assert_array_equal(u8(pk.codes), c, err_msg="codes")
    np.testing.assert_array_equal(u8(pk.meta0), b, err_msg="block scales")
    np.testing.assert_array_equal(f32bits(pk.rscale), f32bits(r), err_msg="tensor scale")
    np.testing.assert_array_equal(bits(y), O.nvfp4t_unpack(c, b, r, kind), err_msg="decoded")


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
@pytest.mark.parametrize("T,H,D", [(256, 8, 128), (20, 3, 64), (4100, 2, 96), (1, 1, 512), (17, 4, 256),
                                   (33, 2, 16), (50, 1, 32)])
def test_matches_oracle(kind, T, H, D):
    x = synth.normal_bf16((T, H, D), seed=T + D, stream=1, outlier_frac=0.01, outlier_scale=20.0)
    pk, y = gpu_pack(x.to(DEV), kind)
    check(x, pk, y, kind)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_tiny_huge_zero_and_strided(kind):
    """A tiny tensor (subnormal scale: the direct-division path), a huge one, an all-zero
    one with a -0, and a strided view (K of a fused qkv)."""
    base = synth.normal_bf16((64, 2, 64), seed=3, stream=1)
    for x in (base.float() * 2.0 ** -125, base.float() * 2.0 ** 120, torch.zeros(64, 2, 64)):
        xb = x.to(torch.bfloat16)
        if not xb.float().abs().max() > 0:
            xb[5, 1, 7] = -0.0
        pk, y = gpu_pack(xb.to(DEV), kind)
        check(xb, pk, y, kind)
    qkv = synth.normal_bf16((48, 3 * 128), seed=4, stream=1).to(DEV)
    xv = qkv[:, 128:256].unflatten(1, (2, 64))
    pk, y = gpu_pack(xv, kind)
    check(xv.cpu(), pk, y, kind)


def test_one_row_value_tensor_equals_the_row_codec():
    x = synth.normal_bf16((1, 1, 128), seed=5, stream=1).to(DEV)
    pk, _ = gpu_pack(x, kvq.KIND_VALUE)
    row = kvq.Packed.empty(kvq.FMT_NVFP4, 0, 1, 1, 128)
    kvq.kvq_pack(x, row)
    torch.cuda.synchronize()
    assert torch.equal(pk.codes, row.codes) and torch.equal(pk.meta0, row.meta0)
    assert torch.equal(pk.rscale.view(torch.int32), row.rscale.view(-1).view(torch.int32))


def test_storage_and_graph_capture():
    T, H, D = 300, 8, 128
    x = synth.normal_bf16((T, H, D), seed=6, stream=1).to(DEV)
    for kind in (kvq.KIND_KEY, kvq.KIND_VALUE):
        pk = kvq.Packed.empty(T4, kind, T, H, D)
        assert pk.nbytes() == kvq.kvq_storage_bytes(T4, kind, 16, T, H, D) == O.storage_bytes(T4, kind, 16, T, H, D)
        kvq.kvq_pack(x, pk)
        pk2 = kvq.Packed.empty(T4, kind, T, H, D)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            kvq.kvq_pack(x, pk2)
        g.replay()
        g.replay()  # replays re-zero the scale slot first: same result
        torch.cuda.synchronize()
        assert torch.equal(pk.codes, pk2.codes) and torch.equal(pk.meta0, pk2.meta0)
        assert torch.equal(pk.rscale, pk2.rscale)


def test_residual_payloads_are_rejected():
    x = torch.zeros((16, 1, 64), dtype=torch.bfloat16, device=DEV)
    pay = kvq.Packed.empty(T4, kvq.KIND_VALUE, 16, 1, 64)
    with pytest.raises(kvq.KvqError, match="UNSUPPORTED"):
        kvq.kvq_encode_residual(x, x, None, pay)


@pytest.mark.parametrize("kind", [kvq.KIND_KEY, kvq.KIND_VALUE])
def test_full_size_sampled(kind):
    """[131072, 8, 128] (the size the per-tensor encoders are timed at), sampled: the
    tensor's largest magnitude is planted in row 0, so row 0's group (K: rows 0-15; V:
    row 0) with 12 sampled K groups (V: 255 sampled rows) reproduces the tensor scale,
    and the oracle runs on just those rows."""
    T, H, D = 131072, 8, 128
    x = synth.normal_bf16((T, H, D), seed=31, stream=1, outlier_frac=0.01, outlier_scale=20.0, device=DEV)
    x[0, 3, 17] = -1000.0  # the tensor's amax (|N(0,1)| x 20 stays far below)
    pk = kvq.Packed.empty(T4, kind, T, H, D)
    kvq.kvq_pack(x, pk)
    y = torch.empty_like(x)
    kvq.kvq_unpack(pk, y)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    if kind == kvq.KIND_KEY:
        groups = [0] + [int(g) for g in rng.choice(np.arange(1, T // 16), 12, replace=False)]
        rows = torch.cat([torch.arange(16 * g, 16 * g + 16) for g in groups]).to(DEV)
        sel_b = torch.tensor(groups, device=DEV)
    else:
        rows = torch.from_numpy(np.concatenate([[0], np.sort(rng.choice(np.arange(1, T), 255, replace=False))])).to(DEV)
        sel_b = rows
    c, b, r = O.nvfp4t_pack(bits(x[rows]), kind)
    np.testing.assert_array_equal(f32bits(pk.rscale), f32bits(r), err_msg="tensor scale")
    np.testing.assert_array_equal(u8(pk.codes[rows]), c, err_msg="codes")
    np.testing.assert_array_equal(u8(pk.meta0[sel_b]), b, err_msg="block scales")
    np.testing.assert_array_equal(bits(y[rows]), O.nvfp4t_unpack(c, b, r, kind), err_msg="decoded")
