"""ctypes mirror of include/kvq.h (structs, enums and function signatures)."""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")

KVQ_OK = 0
STATUS_NAMES = {
    0: "KVQ_OK",
    1: "KVQ_ERR_INVALID_ARG",
    2: "KVQ_ERR_UNSUPPORTED",
    3: "KVQ_ERR_MISALIGNED",
    4: "KVQ_ERR_NOT_DEVICE_PTR",
    5: "KVQ_ERR_CUDA",
}

FMT_NVFP4 = 1
FMT_INT4 = 2
FMT_FP8 = 3
FMT_NVFP4_TENSOR = 4
KIND_KEY = 0
KIND_VALUE = 1

DEV_BAD_SLOT = 1
DEV_BAD_BLOCK = 2
DEV_BAD_POS = 4
DEV_BAD_SEQLEN = 8
DEV_TIMEOUT = 16


class Bf16In(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("row_pitch", ctypes.c_int64), ("head_pitch", ctypes.c_int64)]


class Bf16Out(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("row_pitch", ctypes.c_int64), ("head_pitch", ctypes.c_int64)]


class Plane(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("bscale", ctypes.c_void_p), ("rscale", ctypes.c_void_p)]


class Pool(ctypes.Structure):
    _fields_ = [
        ("k", Plane),
        ("v", Plane),
        ("num_slots", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("fmt", ctypes.c_int32),
        ("v_fmt", ctypes.c_int32),
    ]


class Packed(ctypes.Structure):
    _fields_ = [
        ("fmt", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("rows", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("dim", ctypes.c_int32),
        ("codes", ctypes.c_void_p),
        ("meta0", ctypes.c_void_p),
        ("meta1", ctypes.c_void_p),
        ("rscale", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_ST = ctypes.c_int

SIGNATURES = {
    "kvq_quant_scatter": (_ST, [ctypes.POINTER(Bf16In), ctypes.POINTER(Bf16In), _I32, _P,
                                ctypes.POINTER(Pool), _P, _P]),
    "kvq_restore": (_ST, [ctypes.POINTER(Pool), _P, _I32, _I32, _P, _I32,
                          ctypes.POINTER(Bf16Out), ctypes.POINTER(Bf16Out), _P, _P]),
    "kvq_pack": (_ST, [ctypes.POINTER(Bf16In), ctypes.POINTER(Packed), _P]),
    "kvq_unpack": (_ST, [ctypes.POINTER(Packed), ctypes.POINTER(Bf16Out), _P]),
    "kvq_encode_residual": (_ST, [ctypes.POINTER(Bf16In), ctypes.POINTER(Bf16In), _I32, _P, _I32,
                                  ctypes.POINTER(Packed), _P, _P, _P]),
    "kvq_decode_residual": (_ST, [ctypes.POINTER(Packed), _P, _I32, ctypes.POINTER(Bf16In), _I32,
                                  ctypes.POINTER(Bf16Out), _P, _P]),
    "kvq_decode_attention": (_ST, [ctypes.POINTER(Pool), _P, _I32, _I32, _P, _I32, ctypes.POINTER(Bf16In),
                                   _I32, ctypes.c_float, ctypes.POINTER(Bf16Out), _P, ctypes.c_size_t,
                                   _P, _P]),
    "kvq_decode_attention_workspace": (ctypes.c_size_t, [_I32, _I32, _I32, _I32, _I32]),
    "kvq_decode_attention_noalloc": (_ST, [ctypes.POINTER(Pool), _P, _I32, _I32, _P, _I32, ctypes.POINTER(Bf16In),
                                           _I32, ctypes.c_float, ctypes.POINTER(Bf16Out), _P, _P]),
    "kvq_storage_bytes": (ctypes.c_size_t, [_ST, _ST, _I32, _I64, _I32, _I32]),
    "kvq_status_string": (ctypes.c_char_p, [_ST]),
    "kvq_last_error": (ctypes.c_char_p, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so once; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libkvq.so is missing ({path}); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`"
            )
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
