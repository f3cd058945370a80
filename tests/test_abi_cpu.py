"""The C ABI without a GPU: the library loads, exports every symbol include/kvq.h
declares, and its host-only calls (storage accounting, status names, argument
checks that fail before any CUDA call) behave as documented."""

import ctypes
import os
import re
import subprocess

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_six_codec_calls():
    names = declared_symbols()
    for n in ["kvq_pack", "kvq_unpack", "kvq_encode_residual", "kvq_decode_residual",
              "kvq_quant_scatter", "kvq_restore", "kvq_storage_bytes", "kvq_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(kvq_lib_path):
    lib = ctypes.CDLL(kvq_lib_path)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", kvq_lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    assert set(declared_symbols()) <= exported
    # nothing but the ABI is exported from our own code
    ours = {s for s in exported if s.startswith("kvq") or "kvq" in s}
    assert ours == set(declared_symbols())


def test_storage_bytes_agrees_with_the_oracle(kvq_lib_path):
    import quantized_kv_cache_nvfp4_gb300 as kvq

    for fmt in (1, 2, 3, 4):
        for kind in (0, 1):
            for G in (16, 64):
                for (T, H, D) in [(1, 1, 128), (256, 8, 128), (4100, 8, 96), (1048576, 4, 256), (0, 2, 32)]:
                    g = {1: 16, 2: G, 3: 0, 4: 16}[fmt]
                    assert kvq.kvq_storage_bytes(fmt, kind, g, T, H, D) == O.storage_bytes(fmt, kind, g, T, H, D)
    assert kvq.kvq_storage_bytes(1, 0, 16, 1, 1, 128) == 76
    assert kvq.kvq_storage_bytes(1, 0, 16, 1, 1, 100) == 0
    assert kvq.kvq_storage_bytes(9, 0, 16, 1, 1, 128) == 0


def test_status_strings(kvq_lib_path):
    import quantized_kv_cache_nvfp4_gb300 as kvq

    assert [kvq.kvq_status_string(i) for i in range(6)] == [
        "KVQ_OK", "KVQ_ERR_INVALID_ARG", "KVQ_ERR_UNSUPPORTED", "KVQ_ERR_MISALIGNED",
        "KVQ_ERR_NOT_DEVICE_PTR", "KVQ_ERR_CUDA"]


def test_host_checks_fail_before_any_cuda_call(kvq_lib_path):
    from quantized_kv_cache_nvfp4_gb300 import _abi

    lib = _abi.load()
    pool = _abi.Pool(_abi.Plane(), _abi.Plane(), 64, 16, 2, 100, 1)
    x = _abi.Bf16In(None, 256, 128)
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 1
    assert b"multiple of 16" in lib.kvq_last_error()
    pool.head_dim = 1024
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 2
    pool.head_dim = 128
    pool.num_slots = 65
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 1
    assert lib.kvq_quant_scatter(None, None, 4, None, ctypes.byref(pool), None, None) == 1
    pk = _abi.Packed(2, 0, 48, 4, 2, 128, None, None, None, None)
    assert lib.kvq_pack(ctypes.byref(x), ctypes.byref(pk), None) == 2
    pk = _abi.Packed(7, 0, 64, 4, 2, 128, None, None, None, None)
    assert lib.kvq_unpack(ctypes.byref(pk), None, None) == 1
    pool.head_dim, pool.fmt = 128, 2  # INT4 is not a pool format
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 1
    assert b"pool fmt" in lib.kvq_last_error()
    pool.fmt, pool.v_fmt = 1, 2  # nor is it a V-plane format
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 1
    assert b"v_fmt" in lib.kvq_last_error()
    pool.v_fmt, pool.num_slots = 3, 64  # FP8 V beside NVFP4 K is accepted ...
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 4, None, ctypes.byref(pool), None, None) == 1
    assert b"slot_ids is NULL" in lib.kvq_last_error()  # ... and the call stops at the slot ids
    pool.v_fmt = 0
    # zero-sized work is a no-op that needs no pointers
    assert lib.kvq_quant_scatter(ctypes.byref(x), None, 0, None, ctypes.byref(pool), None, None) == 0
    pk = _abi.Packed(2, 0, 64, 0, 2, 128, None, None, None, None)
    assert lib.kvq_pack(ctypes.byref(x), ctypes.byref(pk), None) == 0


def test_decode_attention_host_checks(kvq_lib_path):
    from quantized_kv_cache_nvfp4_gb300 import _abi

    lib = _abi.load()
    assert lib.kvq_decode_attention_workspace(0, 8, 32, 128, 8192) == 0
    assert lib.kvq_decode_attention_workspace(32, 8, 32, 128, 0) == 0
    pool = _abi.Pool(_abi.Plane(), _abi.Plane(), 64, 16, 2, 96, 1)
    q = _abi.Bf16In(None, 8 * 96, 96)
    o = _abi.Bf16Out(None, 8 * 96, 96)
    call = lambda hq: lib.kvq_decode_attention(ctypes.byref(pool), None, 1, 4, None, 64, ctypes.byref(q), hq,
                                               0.1, ctypes.byref(o), None, 0, None, None)
    assert call(8) == 2 and b"head_dim" in lib.kvq_last_error()  # 96 is not 64/128/256
    pool.head_dim = 128
    assert call(3) == 1 and b"multiple of num_heads" in lib.kvq_last_error()
    assert call(34) == 2 and b"16 query heads" in lib.kvq_last_error()
    assert call(8) == 1 and b"NULL" in lib.kvq_last_error()  # q's pointer
    for bad_scale in (0.0, -0.1, float("inf"), float("nan")):
        assert lib.kvq_decode_attention(ctypes.byref(pool), None, 1, 4, None, 64, ctypes.byref(q), 8, bad_scale,
                                        ctypes.byref(o), None, 0, None, None) == 1
        assert b"scale" in lib.kvq_last_error()
    assert lib.kvq_decode_attention(None, None, 1, 4, None, 64, ctypes.byref(q), 8, 0.1, ctypes.byref(o), None,
                                    0, None, None) == 1


def test_noalloc_entry_point_checks_arguments_like_the_workspace_one(kvq_lib_path):
    """The no-allocation attention entry point runs the same argument checks, in the
    same order, as the workspace one, before it looks at its own scratch limit: a
    bad num_q_heads on a shape that would need split partials gets the same status
    and reason from both."""
    from quantized_kv_cache_nvfp4_gb300 import _abi

    lib = _abi.load()
    pool = _abi.Pool(_abi.Plane(), _abi.Plane(), 16384 * 16, 16, 8, 128, 1)
    q = _abi.Bf16In(None, 32 * 128, 128)
    o = _abi.Bf16Out(None, 32 * 128, 128)
    for hq, want in ((4095, 1), (0, 1), (8 * 17, 2), (32, 1)):  # 32: the NULL q pointer
        a = lib.kvq_decode_attention(ctypes.byref(pool), None, 32, 512, None, 8192, ctypes.byref(q), hq, 0.1,
                                     ctypes.byref(o), None, 0, None, None)
        ea = lib.kvq_last_error()
        b = lib.kvq_decode_attention_noalloc(ctypes.byref(pool), None, 32, 512, None, 8192, ctypes.byref(q), hq,
                                             0.1, ctypes.byref(o), None, None)
        eb = lib.kvq_last_error()
        assert a == b == want, (hq, a, b, ea, eb)
        assert ea == eb


def test_noalloc_scratch_covers_every_split_workspace(kvq_lib_path):
    """The built-in 48 MiB scratch of kvq_decode_attention_noalloc holds the split
    partials of every supported shape (the workspace query is host-only)."""
    from quantized_kv_cache_nvfp4_gb300 import _abi

    lib = _abi.load()
    worst = 0
    for S in (1, 2, 3, 7, 32, 75, 151, 300, 455, 456, 1000):
        for H in (1, 2, 8):
            for group in (1, 4, 16):
                for D in (64, 128, 256):
                    for T in (1, 255, 256, 4096, 1 << 20):
                        worst = max(worst, lib.kvq_decode_attention_workspace(S, H, H * group, D, T))
    assert 0 < worst <= 48 << 20


def test_binding_constants_match_the_header():
    """Every status code, format, kind and device-status bit the header defines has
    the same value under the same name in the binding (KVQ_ prefix dropped, status
    codes by name), and the binding names none the header lacks."""
    from quantized_kv_cache_nvfp4_gb300 import _abi

    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    header = {m[0]: int(m[1]) for m in re.findall(r"\b(KVQ_(?:FMT|KIND|DEV)_\w+)\s*(?:=\s*|\s+)(\d+)u?\b", text)}
    status = {m[0]: int(m[1]) for m in re.findall(r"\b(KVQ_(?:OK|ERR_\w+))\s*=\s*(\d+)", text)}
    assert len(header) >= 11 and len(status) == 6
    for name, value in header.items():
        assert getattr(_abi, name[len("KVQ_"):]) == value, name
    bound = {n for n in dir(_abi) if re.fullmatch(r"(FMT|KIND|DEV)_[A-Z0-9_]+", n)}
    assert bound == {n[len("KVQ_"):] for n in header}
    assert _abi.STATUS_NAMES == {v: k for k, v in status.items()}
