"""Helpers shared by the GPU parity tests: tensor <-> numpy bit views and oracle
calls on the same inputs.  No codec arithmetic lives here."""

import numpy as np
import torch

import oracle as O
from quantized_kv_cache_nvfp4_gb300 import synth

DEV = "cuda"
POISON = 0xA5  # fill byte for outputs, so that an unwritten byte is visible


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f32bits(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def f16bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def poison_bf16(shape, device=DEV) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    t.view(torch.uint8).fill_(POISON)
    return t


def status_word(device=DEV) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def assert_rows_equal(got_codes, got_bs, got_rs, want_codes, want_bs, want_rs, what=""):
    np.testing.assert_array_equal(got_codes, want_codes, err_msg=f"{what} codes")
    np.testing.assert_array_equal(got_bs, want_bs, err_msg=f"{what} block scales")
    np.testing.assert_array_equal(f32bits(got_rs), f32bits(want_rs), err_msg=f"{what} row scales")


def oracle_rows(x: torch.Tensor):
    """Oracle NVFP4 encode of every (token, head) row of a [T, H, D] bf16 tensor."""
    return O.nvfp4_encode_rows(bits(x.contiguous()))


def oracle_on_all_cores(fn, *arrays, threads=None):
    """Apply a row-wise oracle function to every row of `arrays` (split along axis 0)
    on every host core.  Each thread runs the unchanged oracle on its own contiguous
    chunk; the C oracle keeps no global state and ctypes releases the interpreter
    lock, so the chunks run in parallel.  Returns what fn returns, with the chunks'
    results concatenated along axis 0."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    n = arrays[0].shape[0]
    threads = threads or os.cpu_count() or 1
    edges = np.linspace(0, n, 4 * threads + 1).astype(np.int64)
    spans = [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda ab: fn(*[np.ascontiguousarray(x[ab[0]:ab[1]]) for x in arrays]), spans))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[j] for p in parts]) for j in range(len(parts[0])))
    return np.concatenate(parts)
