"""Plain scalar CPU oracle for the KV-cache codec (ctypes front end).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this module; the product package never does.
The arithmetic lives in ``kvq_oracle.c`` (scalar C, one IEEE binary32 operation at
a time, built with ``-ffp-contract=off`` and no fast-math).  This file only
marshals numpy arrays; bf16 and fp16 values travel as uint16 bit patterns.

Pinning: ``tests/test_oracle_pins.py`` checks every function against facts that
the pages or the mathematics fix.  Parity with vLLM's ``ref_nvfp4_quant`` and
FlashLoop's ``packing.py`` is unpinned (their source is not available).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

FMT_NVFP4 = 1
FMT_INT4 = 2
FMT_FP8 = 3
FMT_NVFP4_TENSOR = 4
KIND_KEY = 0
KIND_VALUE = 1

BAD_SLOT = 1
BAD_BLOCK = 2
BAD_POS = 4
BAD_SEQLEN = 8

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (plain gcc, a second or so)."""
    stale = not os.path.exists(LIB) or os.path.getmtime(LIB) < max(
        os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "kvq_oracle.h"))
    )
    if force or stale:
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        _declare(L)
        if L.orc_subnormals_kept() != 1:
            raise RuntimeError("the host flushes subnormals (FTZ/DAZ): the oracle's binary32 "
                               "definitions do not hold in this process")
        _lib = L
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_U32 = ctypes.c_uint32


def _declare(L: ctypes.CDLL) -> None:
    sig = {
        "orc_subnormals_kept": (_I, []),
        "orc_f32_to_bf16_n": (None, [_P, _I64, _P]),
        "orc_f32_to_f16_n": (None, [_P, _I64, _P]),
        "orc_e2m1_encode_n": (None, [_P, _I64, _P]),
        "orc_e4m3_encode_n": (None, [_P, _I64, _P]),
        "orc_e2m1_value": (ctypes.c_float, [ctypes.c_uint8]),
        "orc_e4m3_value": (ctypes.c_float, [ctypes.c_uint8]),
        "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_nvfp4_encode_rows": (None, [_P, _I64, _I, _P, _P, _P]),
        "orc_nvfp4_decode_rows": (None, [_P, _P, _P, _I64, _I, _P]),
        "orc_nvfp4_scatter": (_U32, [_P, _I64, _I64, _I, _I, _I, _P, _I64, _P, _P, _P]),
        "orc_nvfp4_restore": (_U32, [_P, _P, _P, _I64, _I, _I, _I, _P, _I, _I, _P, _I, _P]),
        "orc_int4_pack": (None, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
        "orc_int4_unpack": (None, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
        "orc_residual_encode": (_U32, [_P, _P, _I, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
        "orc_residual_decode": (_U32, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _I, _I, _I, _P]),
        "orc_storage_bytes": (_I64, [_I, _I, _I, _I64, _I, _I]),
        "orc_nvfp4t_pack": (None, [_P, _I, _I, _I, _I, _P, _P, _P]),
        "orc_nvfp4t_unpack": (None, [_P, _P, _P, _I, _I, _I, _I, _P]),
        "orc_decode_attention": (_U32, [_P, _P, _P, _I, _P, _P, _P, _I, _I64, _I, _I, _I, _P, _I, _I,
                                        _P, _P, _I, ctypes.c_double, _P]),
        "orc_fp8_encode_rows": (None, [_P, _I64, _I, _P, _P]),
        "orc_fp8_decode_rows": (None, [_P, _P, _I64, _I, _P]),
        "orc_fp8_scatter": (_U32, [_P, _I64, _I64, _I, _I, _I, _P, _I64, _P, _P]),
        "orc_fp8_restore": (_U32, [_P, _P, _I64, _I, _I, _I, _P, _I, _I, _P, _I, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar primitives (array forms)
# --------------------------------------------------------------------------
def f32_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_n(_ptr(x), x.size, _ptr(y))
    return y


def bf16_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_f16(x) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16_n(_ptr(x), x.size, _ptr(y))
    return y


def f16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    return np.array([lib().orc_f16_to_f32(int(v)) for v in h.ravel()], np.float32).reshape(h.shape)


def e2m1_encode(q) -> np.ndarray:
    q = _c(q, np.float32)
    y = np.empty(q.shape, np.uint8)
    lib().orc_e2m1_encode_n(_ptr(q), q.size, _ptr(y))
    return y


def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1_value(int(code)))


def e4m3_encode(t) -> np.ndarray:
    t = _c(t, np.float32)
    y = np.empty(t.shape, np.uint8)
    lib().orc_e4m3_encode_n(_ptr(t), t.size, _ptr(y))
    return y


def e4m3_value(code: int) -> float:
    return float(lib().orc_e4m3_value(int(code)))


# --------------------------------------------------------------------------
# NVFP4 row codec
# --------------------------------------------------------------------------
def nvfp4_encode_rows(x_bf16: np.ndarray):
    """x [..., D] uint16 (bf16 bits) -> codes [..., D/2], bscale [..., D/16], rscale [...]."""
    x = _c(x_bf16, np.uint16)
    D = x.shape[-1]
    assert D % 16 == 0
    lead = x.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    codes = np.zeros(lead + (D // 2,), np.uint8)
    bscale = np.zeros(lead + (D // 16,), np.uint8)
    rscale = np.zeros(lead, np.float32)
    lib().orc_nvfp4_encode_rows(_ptr(x), n, D, _ptr(codes), _ptr(bscale), _ptr(rscale))
    return codes, bscale, rscale


def nvfp4_decode_rows(codes, bscale, rscale) -> np.ndarray:
    codes = _c(codes, np.uint8)
    bscale = _c(bscale, np.uint8)
    rscale = _c(rscale, np.float32)
    D = codes.shape[-1] * 2
    lead = codes.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    y = np.empty(lead + (D,), np.uint16)
    lib().orc_nvfp4_decode_rows(_ptr(codes), _ptr(bscale), _ptr(rscale), n, D, _ptr(y))
    return y


def new_pool(num_slots: int, H: int, D: int):
    """Zero-filled NVFP4 planes for one tensor: codes, bscale, rscale."""
    return (
        np.zeros((num_slots, H, D // 2), np.uint8),
        np.zeros((num_slots, H, D // 16), np.uint8),
        np.zeros((num_slots, H), np.float32),
    )


def nvfp4_scatter(x_flat, row_pitch, head_pitch, T, H, D, slot_ids, pool) -> int:
    """Encode x[t*row_pitch + h*head_pitch + d] into pool planes at slot_ids[t] (in place)."""
    x = _c(x_flat, np.uint16).ravel()
    if T > 0:
        need = (T - 1) * row_pitch + (H - 1) * head_pitch + D
        assert x.size >= need
    slot_ids = _c(slot_ids, np.int64)
    codes, bscale, rscale = pool
    return int(
        lib().orc_nvfp4_scatter(
            _ptr(x), row_pitch, head_pitch, T, H, D, _ptr(slot_ids), codes.shape[0],
            _ptr(codes), _ptr(bscale), _ptr(rscale),
        )
    )


def nvfp4_restore(pool, block_size, block_table, seq_lens, Tmax, out=None):
    """Gather pool rows through block_table into out [S][Tmax][H][D] (bf16 bits)."""
    codes, bscale, rscale = pool
    num_slots, H, half = codes.shape
    D = half * 2
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    S, max_blocks = block_table.shape
    if out is None:
        out = np.zeros((S, Tmax, H, D), np.uint16)
    st = lib().orc_nvfp4_restore(
        _ptr(codes), _ptr(bscale), _ptr(rscale), num_slots, H, D, block_size,
        _ptr(block_table), S, max_blocks, _ptr(seq_lens), Tmax, _ptr(out),
    )
    return out, int(st)


# --------------------------------------------------------------------------
# FP8 E4M3 row codec
# --------------------------------------------------------------------------
def fp8_encode_rows(x_bf16: np.ndarray):
    """x [..., D] uint16 (bf16 bits) -> codes [..., D] (E4M3 bytes), rscale [...]."""
    x = _c(x_bf16, np.uint16)
    D = x.shape[-1]
    lead = x.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    codes = np.zeros(lead + (D,), np.uint8)
    rscale = np.zeros(lead, np.float32)
    lib().orc_fp8_encode_rows(_ptr(x), n, D, _ptr(codes), _ptr(rscale))
    return codes, rscale


def fp8_decode_rows(codes, rscale) -> np.ndarray:
    codes = _c(codes, np.uint8)
    rscale = _c(rscale, np.float32)
    D = codes.shape[-1]
    lead = codes.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    y = np.empty(lead + (D,), np.uint16)
    lib().orc_fp8_decode_rows(_ptr(codes), _ptr(rscale), n, D, _ptr(y))
    return y


def new_fp8_pool(num_slots: int, H: int, D: int):
    """Zero-filled FP8 planes for one tensor: codes, rscale."""
    return np.zeros((num_slots, H, D), np.uint8), np.zeros((num_slots, H), np.float32)


def fp8_scatter(x_flat, row_pitch, head_pitch, T, H, D, slot_ids, pool) -> int:
    x = _c(x_flat, np.uint16).ravel()
    slot_ids = _c(slot_ids, np.int64)
    codes, rscale = pool
    return int(lib().orc_fp8_scatter(_ptr(x), row_pitch, head_pitch, T, H, D, _ptr(slot_ids),
                                     codes.shape[0], _ptr(codes), _ptr(rscale)))


def fp8_restore(pool, block_size, block_table, seq_lens, Tmax, out=None):
    codes, rscale = pool
    num_slots, H, D = codes.shape
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    S, max_blocks = block_table.shape
    if out is None:
        out = np.zeros((S, Tmax, H, D), np.uint16)
    st = lib().orc_fp8_restore(_ptr(codes), _ptr(rscale), num_slots, H, D, block_size,
                               _ptr(block_table), S, max_blocks, _ptr(seq_lens), Tmax, _ptr(out))
    return out, int(st)


# --------------------------------------------------------------------------
# INT4 affine codec
# --------------------------------------------------------------------------
def int4_meta_shape(kind, T, H, D, G):
    if kind == KIND_KEY:
        return (-(-T // G), H, D)
    return (T, H, -(-D // G))


def int4_pack(x_bf16, kind: int, G: int = 64):
    x = _c(x_bf16, np.uint16)
    T, H, D = x.shape
    assert D % 2 == 0
    codes = np.zeros((T, H, D // 2), np.uint8)
    ms = int4_meta_shape(kind, T, H, D, G)
    mn = np.zeros(ms, np.uint16)
    sc = np.zeros(ms, np.uint16)
    lib().orc_int4_pack(_ptr(x), T, H, D, kind, G, _ptr(codes), _ptr(mn), _ptr(sc))
    return codes, mn, sc


def int4_unpack(codes, mn, sc, kind: int, G: int = 64):
    codes = _c(codes, np.uint8)
    mn = _c(mn, np.uint16)
    sc = _c(sc, np.uint16)
    T, H, half = codes.shape
    D = half * 2
    y = np.empty((T, H, D), np.uint16)
    lib().orc_int4_unpack(_ptr(codes), _ptr(mn), _ptr(sc), T, H, D, kind, G, _ptr(y))
    return y


# --------------------------------------------------------------------------
# residual encode / decode
# --------------------------------------------------------------------------
def _payload_buffers(fmt, kind, P, H, D, G):
    if fmt == FMT_FP8:
        return np.zeros((P, H, D), np.uint8), None, None, np.zeros((P, H), np.float32)
    codes = np.zeros((P, H, D // 2), np.uint8)
    if fmt == FMT_NVFP4:
        return codes, np.zeros((P, H, D // 16), np.uint8), None, np.zeros((P, H), np.float32)
    ms = int4_meta_shape(kind, P, H, D, G)
    return codes, np.zeros(ms, np.uint16), np.zeros(ms, np.uint16), None


_DUMMY_I32 = np.zeros(1, np.int32)


def _pos_ptr(pos):
    """NULL means dense to the C side, so an empty position map gets a real pointer."""
    if pos is None:
        return None
    return _ptr(pos) if pos.size else _ptr(_DUMMY_I32)


def residual_encode(cur, prev, pos, fmt: int, kind: int, G: int = 64):
    """Returns (payload dict, status).  pos=None is the dense case."""
    cur = _c(cur, np.uint16)
    prev = _c(prev, np.uint16)
    T, H, D = cur.shape
    posa = None if pos is None else _c(pos, np.int32).ravel()
    P = T if posa is None else posa.size
    codes, ma, mb, rs = _payload_buffers(fmt, kind, P, H, D, G)
    pos_out = None if posa is None else np.zeros(P, np.int32)
    st = lib().orc_residual_encode(
        _ptr(cur), _ptr(prev), T, H, D, _pos_ptr(posa), P, fmt, kind, G,
        _ptr(codes), _ptr(ma), _ptr(mb), _ptr(rs), _pos_ptr(pos_out),
    )
    payload = dict(fmt=fmt, kind=kind, G=G, codes=codes, meta_a=ma, meta_b=mb, rscale=rs,
                   pos=pos_out)
    return payload, int(st)


def residual_decode(payload, prev, out=None):
    """out = prev with the payload's rows added at their positions (out may be prev)."""
    prev = _c(prev, np.uint16)
    T, H, D = prev.shape
    pos = payload["pos"]
    P = T if pos is None else pos.size
    if out is None:
        out = np.empty_like(prev)
    st = lib().orc_residual_decode(
        _ptr(payload["codes"]), _ptr(payload["meta_a"]), _ptr(payload["meta_b"]),
        _ptr(payload["rscale"]), payload["fmt"], payload["kind"], payload["G"],
        _pos_ptr(pos), P, _ptr(prev), T, H, D, _ptr(out),
    )
    return out, int(st)


# --------------------------------------------------------------------------
# NVFP4 with one FP32 scale per tensor, G16 blocks along the kind's axis
# --------------------------------------------------------------------------
def nvfp4t_bscale_shape(kind, T, H, D):
    return (-(-T // 16), H, D) if kind == KIND_KEY else (T, H, D // 16)


def nvfp4t_pack(x_bf16, kind: int):
    """x [T][H][D] bf16 bits -> codes [T][H][D/2], bscale (by kind), rscale [1]."""
    x = _c(x_bf16, np.uint16)
    T, H, D = x.shape
    codes = np.zeros((T, H, D // 2), np.uint8)
    bscale = np.zeros(nvfp4t_bscale_shape(kind, T, H, D), np.uint8)
    rscale = np.zeros(1, np.float32)
    lib().orc_nvfp4t_pack(_ptr(x), T, H, D, kind, _ptr(codes), _ptr(bscale), _ptr(rscale))
    return codes, bscale, rscale


def nvfp4t_unpack(codes, bscale, rscale, kind: int):
    codes = _c(codes, np.uint8)
    bscale = _c(bscale, np.uint8)
    rscale = _c(rscale, np.float32)
    T, H, half = codes.shape
    y = np.empty((T, H, 2 * half), np.uint16)
    lib().orc_nvfp4t_unpack(_ptr(codes), _ptr(bscale), _ptr(rscale), T, H, 2 * half, kind, _ptr(y))
    return y


# --------------------------------------------------------------------------
# paged decode attention over a quantised pool (fp64)
# --------------------------------------------------------------------------
def _plane(plane, fmt):
    """(codes, bscale or None, rscale) numpy planes -> C-contiguous arrays."""
    codes, bscale, rscale = plane
    return (_c(codes, np.uint8), None if fmt == FMT_FP8 else _c(bscale, np.uint8), _c(rscale, np.float32))


def decode_attention(k_plane, v_plane, fmt_k, fmt_v, block_size, block_table, seq_lens, q_bf16,
                     scale, out=None):
    """o[s][qh] = softmax over the sequence's tokens of scale * q . k, applied to v, with
    k / v the exact decoded pool rows.  Planes: (codes, bscale, rscale) as the pool holds
    them ([slots][H][...]); q: bf16 bits [S][Hq][D].  Returns (out float64, status)."""
    kc, kb, kr = _plane(k_plane, fmt_k)
    vc, vb, vr = _plane(v_plane, fmt_v)
    num_slots, H = kr.shape
    q = _c(q_bf16, np.uint16)
    S, Hq, D = q.shape
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    if out is None:
        out = np.zeros((S, Hq, D), np.float64)
    st = lib().orc_decode_attention(
        _ptr(kc), _ptr(kb), _ptr(kr), fmt_k, _ptr(vc), _ptr(vb), _ptr(vr), fmt_v, num_slots, H, D,
        block_size, _ptr(block_table), S, block_table.shape[1], _ptr(seq_lens), _ptr(q), Hq,
        float(scale), _ptr(out))
    return out, int(st)


def storage_bytes(fmt: int, kind: int, G: int, T: int, H: int, D: int) -> int:
    return int(lib().orc_storage_bytes(fmt, kind, G, T, H, D))
