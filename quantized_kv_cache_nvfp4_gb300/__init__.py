"""GB300-native KV-cache quantisation codec: Python binding of libkvq.so.

The functions here carry the names of the C entry points in include/kvq.h and only
marshal arguments: torch tensors become pointers and pitches, the current CUDA
stream becomes the launch stream, and a non-OK status becomes ``KvqError``.  Every
step of the codec runs in the library's sm_103a kernels; there is no CPU path, and
a missing library raises.

Allocation helpers (``Nvfp4Pool``, ``Packed``) use torch for device memory only.
"""

from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import _abi
from ._abi import (DEV_BAD_BLOCK, DEV_BAD_POS, DEV_BAD_SEQLEN, DEV_BAD_SLOT, DEV_TIMEOUT, FMT_FP8, FMT_INT4,
                   FMT_NVFP4_TENSOR,
                   FMT_NVFP4, KIND_KEY, KIND_VALUE)

__all__ = [
    "KvqError", "KvPool", "Nvfp4Pool", "Packed", "kvq_quant_scatter", "kvq_restore", "kvq_pack",
    "kvq_unpack", "kvq_encode_residual", "kvq_decode_residual", "kvq_decode_attention",
    "kvq_decode_attention_workspace", "kvq_decode_attention_noalloc", "kvq_storage_bytes",
    "kvq_status_string", "kvq_last_error", "library_path", "FMT_NVFP4", "FMT_INT4", "FMT_FP8", "FMT_NVFP4_TENSOR", "KIND_KEY",
    "KIND_VALUE", "DEV_BAD_SLOT", "DEV_BAD_BLOCK", "DEV_BAD_POS", "DEV_BAD_SEQLEN", "DEV_TIMEOUT",
]


class KvqError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_abi.STATUS_NAMES.get(status, status)}: {detail}")


def library_path() -> str:
    return _abi.LIB_PATH


def _lib():
    return _abi.load()


def _check(status: int) -> None:
    if status != _abi.KVQ_OK:
        raise KvqError(status, _lib().kvq_last_error().decode())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> ctypes.c_void_p:
    """The launch stream: the given torch stream, else the current stream of the
    current device (its raw handle, without building a Stream object)."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _view3(t: torch.Tensor, name: str):
    """(ptr, row_pitch, head_pitch) of a bf16 [rows, heads, dim] tensor, inner stride 1."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    st = t.stride()
    if len(st) != 3 or (st[2] != 1 and t.size(2) > 1):
        raise ValueError(f"{name} must be [rows, heads, dim] with inner stride 1")
    return t.data_ptr(), st[0], st[1]


def _bf16_in(t: torch.Tensor, name: str):
    p, r, h = _view3(t, name)
    return _abi.Bf16In(p, r, h)


def _bf16_out(t: torch.Tensor, name: str):
    p, r, h = _view3(t, name)
    return _abi.Bf16Out(p, r, h)


# ---------------------------------------------------------------------------
# device memory holders
# ---------------------------------------------------------------------------
@dataclass
class KvPool:
    """Paged K/V planes, slot-major (slot = block * block_size + offset); each plane in
    its own format (fmt for K, v_fmt for V; v_fmt None = the same as fmt).

    NVFP4: codes [slots, H, D/2] u8, bscale [slots, H, D/16] u8 (E4M3), rscale [slots, H] f32.
    FP8:   codes [slots, H, D] u8 (E4M3), rscale [slots, H] f32 (no block scales)."""

    k_codes: torch.Tensor
    k_bscale: Optional[torch.Tensor]
    k_rscale: torch.Tensor
    v_codes: torch.Tensor
    v_bscale: Optional[torch.Tensor]
    v_rscale: torch.Tensor
    block_size: int
    fmt: int = FMT_NVFP4
    v_fmt: Optional[int] = None

    @classmethod
    def empty(cls, num_slots: int, num_heads: int, head_dim: int, block_size: int = 16,
              device="cuda", fill: Optional[int] = None, fmt: int = FMT_NVFP4,
              v_fmt: Optional[int] = None) -> "KvPool":
        def u8(*shape):
            t = torch.empty(shape, dtype=torch.uint8, device=device)
            return t.fill_(fill) if fill is not None else t

        def f32(*shape):
            t = torch.empty(shape, dtype=torch.float32, device=device)
            if fill is not None:
                t.view(torch.uint8).fill_(fill)
            return t

        def plane(f):
            if f == FMT_FP8:
                return u8(num_slots, num_heads, head_dim), None, f32(num_slots, num_heads)
            return (u8(num_slots, num_heads, head_dim // 2), u8(num_slots, num_heads, head_dim // 16),
                    f32(num_slots, num_heads))

        return cls(*plane(fmt), *plane(fmt if v_fmt is None else v_fmt), block_size, fmt, v_fmt)

    @property
    def num_slots(self) -> int:
        return self.k_codes.size(0)

    @property
    def num_heads(self) -> int:
        return self.k_codes.size(1)

    @property
    def head_dim(self) -> int:
        return self.k_codes.size(2) * (1 if self.fmt == FMT_FP8 else 2)

    def _planes(self):
        return [t for t in (self.k_codes, self.k_bscale, self.k_rscale, self.v_codes, self.v_bscale,
                            self.v_rscale) if t is not None]

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self._planes())

    def _struct(self) -> _abi.Pool:
        """The C struct of the pool, built once and kept while its planes are the same
        tensors (a plane replaced by another tensor rebuilds it)."""
        planes = (self.k_codes, self.k_bscale, self.k_rscale, self.v_codes, self.v_bscale, self.v_rscale)
        key = tuple(None if t is None else (id(t), t.data_ptr()) for t in planes) + (
            self.block_size, self.fmt, self.v_fmt)
        cached = self.__dict__.get("_c_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        for t in self._planes():
            if not t.is_contiguous():
                raise ValueError("pool planes must be contiguous")
        bs = lambda t: None if t is None else t.data_ptr()
        st = _abi.Pool(
            _abi.Plane(self.k_codes.data_ptr(), bs(self.k_bscale), self.k_rscale.data_ptr()),
            _abi.Plane(self.v_codes.data_ptr(), bs(self.v_bscale), self.v_rscale.data_ptr()),
            self.num_slots, self.block_size, self.num_heads, self.head_dim, self.fmt,
            0 if self.v_fmt is None else self.v_fmt)
        self.__dict__["_c_struct"] = (key, st)
        return st


Nvfp4Pool = KvPool  # the NVFP4 pool is the default format of KvPool


@dataclass
class Packed:
    """A logical packed tensor [rows, heads, dim] (see kvq_packed in include/kvq.h)."""

    fmt: int
    kind: int
    group_size: int
    rows: int
    heads: int
    dim: int
    codes: torch.Tensor
    meta0: Optional[torch.Tensor]
    meta1: Optional[torch.Tensor] = None
    rscale: Optional[torch.Tensor] = None

    @classmethod
    def empty(cls, fmt: int, kind: int, rows: int, heads: int, dim: int, group_size: int = 64,
              device="cuda") -> "Packed":
        if fmt == FMT_NVFP4_TENSOR:
            bs = (math.ceil(rows / 16), heads, dim) if kind == KIND_KEY else (rows, heads, dim // 16)
            return cls(fmt, kind, 16, rows, heads, dim,
                       torch.empty((rows, heads, dim // 2), dtype=torch.uint8, device=device),
                       torch.empty(bs, dtype=torch.uint8, device=device), None,
                       torch.empty((1,), dtype=torch.float32, device=device))
        if fmt == FMT_FP8:
            return cls(fmt, kind, 0, rows, heads, dim,
                       torch.empty((rows, heads, dim), dtype=torch.uint8, device=device), None, None,
                       torch.empty((rows, heads), dtype=torch.float32, device=device))
        codes = torch.empty((rows, heads, dim // 2), dtype=torch.uint8, device=device)
        if fmt == FMT_NVFP4:
            return cls(fmt, kind, 16, rows, heads, dim, codes,
                       torch.empty((rows, heads, dim // 16), dtype=torch.uint8, device=device),
                       None, torch.empty((rows, heads), dtype=torch.float32, device=device))
        if kind == KIND_KEY:
            ms = (math.ceil(rows / group_size), heads, dim)
        else:
            ms = (rows, heads, math.ceil(dim / group_size))
        return cls(fmt, kind, group_size, rows, heads, dim, codes,
                   torch.empty(ms, dtype=torch.float16, device=device),
                   torch.empty(ms, dtype=torch.float16, device=device), None)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.codes, self.meta0, self.meta1, self.rscale)
                   if t is not None)

    def _struct(self) -> _abi.Packed:
        """The C struct, built once and kept while the buffers and sizes are the same."""
        bufs = (self.codes, self.meta0, self.meta1, self.rscale)
        key = tuple(None if t is None else (id(t), t.data_ptr()) for t in bufs) + (
            self.fmt, self.kind, self.group_size, self.rows, self.heads, self.dim)
        cached = self.__dict__.get("_c_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        for t in bufs:
            if t is not None and not t.is_contiguous():
                raise ValueError("packed buffers must be contiguous")
        st = _abi.Packed(self.fmt, self.kind, self.group_size, self.rows, self.heads, self.dim,
                         self.codes.data_ptr(), None if self.meta0 is None else self.meta0.data_ptr(),
                         None if self.meta1 is None else self.meta1.data_ptr(),
                         None if self.rscale is None else self.rscale.data_ptr())
        self.__dict__["_c_struct"] = (key, st)
        return st


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def kvq_quant_scatter(k: Optional[torch.Tensor], v: Optional[torch.Tensor], slot_ids: torch.Tensor,
                      pool: KvPool, dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantise + scatter of K/V [T, H, D] bf16 into pool slots slot_ids[T] (int64), in the
    pool's format (NVFP4 or FP8)."""
    src = k if k is not None else v
    if src is None:
        raise ValueError("k and v are both None")
    if slot_ids.dtype != torch.int64:
        raise TypeError("slot_ids must be int64")
    T = src.size(0)
    kin = _bf16_in(k, "k") if k is not None else None
    vin = _bf16_in(v, "v") if v is not None else None
    ps = pool._struct()
    _check(_lib().kvq_quant_scatter(
        ctypes.byref(kin) if kin is not None else None, ctypes.byref(vin) if vin is not None else None,
        T, _ptr(slot_ids), ctypes.byref(ps), _ptr(dev_status), _stream(stream)))


def _seq_view(t: torch.Tensor, S: int, Tmax: int, name: str):
    """[S, Tmax, H, D] (or [S*Tmax, H, D]) bf16 -> Bf16Out over S*Tmax rows."""
    if t.dim() == 4:
        if t.size(0) != S or t.size(1) != Tmax or (S > 1 and t.stride(0) != Tmax * t.stride(1)):
            raise ValueError(f"{name} must be [S, Tmax, H, D] with sequence stride Tmax*token stride")
        t = t.flatten(0, 1)
    return _bf16_out(t, name)


def kvq_restore(pool: KvPool, block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                k_out: Optional[torch.Tensor], v_out: Optional[torch.Tensor],
                dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Paged restore into k_out / v_out [S, max_seq_len, H, D] bf16."""
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous [S, max_blocks]")
    S, max_blocks = block_table.shape
    ko = _seq_view(k_out, S, max_seq_len, "k_out") if k_out is not None else None
    vo = _seq_view(v_out, S, max_seq_len, "v_out") if v_out is not None else None
    ps = pool._struct()
    _check(_lib().kvq_restore(
        ctypes.byref(ps), _ptr(block_table), S, max_blocks, _ptr(seq_lens), max_seq_len,
        ctypes.byref(ko) if ko is not None else None, ctypes.byref(vo) if vo is not None else None,
        _ptr(dev_status), _stream(stream)))


def kvq_pack(x: torch.Tensor, out: Packed, stream=None) -> Packed:
    xin = _bf16_in(x, "x")
    ps = out._struct()
    _check(_lib().kvq_pack(ctypes.byref(xin), ctypes.byref(ps), _stream(stream)))
    return out


def kvq_unpack(packed: Packed, y: torch.Tensor, stream=None) -> torch.Tensor:
    yo = _bf16_out(y, "y")
    ps = packed._struct()
    _check(_lib().kvq_unpack(ctypes.byref(ps), ctypes.byref(yo), _stream(stream)))
    return y


def kvq_encode_residual(cur: torch.Tensor, prev: torch.Tensor, pos: Optional[torch.Tensor],
                        payload: Packed, pos_out: Optional[torch.Tensor] = None,
                        dev_status: Optional[torch.Tensor] = None, stream=None) -> Packed:
    if pos is not None and pos.dtype != torch.int32:
        raise TypeError("pos must be int32")
    ci, pi = _bf16_in(cur, "cur"), _bf16_in(prev, "prev")
    n = cur.size(0) if pos is None else pos.numel()
    ps = payload._struct()
    pos_ptr = _ptr(pos)
    if pos is not None and pos.numel() == 0:
        pos_ptr = ctypes.c_void_p(prev.data_ptr())  # non-NULL marks "sparse, nothing kept"
    _check(_lib().kvq_encode_residual(
        ctypes.byref(ci), ctypes.byref(pi), cur.size(0), pos_ptr, n, ctypes.byref(ps),
        _ptr(pos_out), _ptr(dev_status), _stream(stream)))
    return payload


def kvq_decode_residual(payload: Packed, pos: Optional[torch.Tensor], prev: torch.Tensor,
                        out: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    if pos is not None and pos.dtype != torch.int32:
        raise TypeError("pos must be int32")
    pi, oo = _bf16_in(prev, "prev"), _bf16_out(out, "out")
    n = prev.size(0) if pos is None else pos.numel()
    ps = payload._struct()
    pos_ptr = _ptr(pos)
    if pos is not None and pos.numel() == 0:
        pos_ptr = ctypes.c_void_p(prev.data_ptr())  # non-NULL marks "sparse, nothing kept"
    _check(_lib().kvq_decode_residual(
        ctypes.byref(ps), pos_ptr, n, ctypes.byref(pi), prev.size(0), ctypes.byref(oo),
        _ptr(dev_status), _stream(stream)))
    return out


def kvq_decode_attention_workspace(num_seqs: int, num_heads: int, num_q_heads: int, head_dim: int,
                                   max_seq_len: int) -> int:
    return int(_lib().kvq_decode_attention_workspace(num_seqs, num_heads, num_q_heads, head_dim, max_seq_len))


def kvq_decode_attention(pool: KvPool, block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                         q: torch.Tensor, scale: float, out: torch.Tensor,
                         workspace: Optional[torch.Tensor] = None,
                         dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention of q [S, Hq, D] bf16 over the pool's K/V (decoded in registers)
    into out [S, Hq, D] bf16.  A workspace tensor is allocated when none is given."""
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous [S, max_blocks]")
    S, max_blocks = block_table.shape
    qi, oo = _bf16_in(q, "q"), _bf16_out(out, "out")
    Hq = q.size(1)
    need = kvq_decode_attention_workspace(S, pool.num_heads, Hq, pool.head_dim, max_seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ps = pool._struct()
    _check(_lib().kvq_decode_attention(
        ctypes.byref(ps), _ptr(block_table), S, max_blocks, _ptr(seq_lens), max_seq_len, ctypes.byref(qi), Hq,
        float(scale), ctypes.byref(oo), _ptr(workspace), nbytes, _ptr(dev_status), _stream(stream)))
    return out


def kvq_decode_attention_noalloc(pool: KvPool, block_table: torch.Tensor, seq_lens: torch.Tensor,
                                 max_seq_len: int, q: torch.Tensor, scale: float, out: torch.Tensor,
                                 dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kvq_decode_attention with the library's built-in split scratch: no workspace and no
    allocation (calls must not overlap on one device)."""
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous [S, max_blocks]")
    S, max_blocks = block_table.shape
    qi, oo = _bf16_in(q, "q"), _bf16_out(out, "out")
    ps = pool._struct()
    _check(_lib().kvq_decode_attention_noalloc(
        ctypes.byref(ps), _ptr(block_table), S, max_blocks, _ptr(seq_lens), max_seq_len, ctypes.byref(qi),
        q.size(1), float(scale), ctypes.byref(oo), _ptr(dev_status), _stream(stream)))
    return out


def kvq_storage_bytes(fmt: int, kind: int, group_size: int, rows: int, heads: int, dim: int) -> int:
    return int(_lib().kvq_storage_bytes(fmt, kind, group_size, rows, heads, dim))


def kvq_status_string(status: int) -> str:
    return _lib().kvq_status_string(status).decode()


def kvq_last_error() -> str:
    return _lib().kvq_last_error().decode()
