"""ctypes front end of oracle.c -- TEST INFRASTRUCTURE.

``apply`` is the oracle of one projection's LoRA delta over a batch; the
arithmetic lives in oracle.c (fp64 loops, every weight element fetched
through the page table).  This module only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

F16, BF16 = 0, 1
_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        L.oracle_lora_apply.restype = ctypes.c_int
        L.oracle_lora_apply.argtypes = [
            P, P, ctypes.c_int32, ctypes.c_int32,          # pool, page_slot, H, dtype
            P, P, P, ctypes.c_int32,                       # page_table, pt_off, rank, num_adapters
            ctypes.c_int32, P, P, ctypes.c_int32,          # num_proj, proj_in, proj_out, p
            P, ctypes.c_int32, P, ctypes.c_int32,          # token_adapter, T, tokens, n_tokens
            P, ctypes.c_int64, P, ctypes.c_int64,          # x, ldx, y_in, ldy
            ctypes.c_double, P,                            # s, adapter_scale (fp64 per adapter id, or NULL)
            P, P, P, ctypes.c_int64,                       # y_out, y_exact, v_out, v_ld
            ctypes.c_int32]                                # num_threads
        L.oracle_decode_array.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32]
        L.oracle_encode_array.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32]
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def dtype_code(dtype: str) -> int:
    return F16 if dtype == "f16" else BF16


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of 16-bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_decode_array(_ptr(b), _ptr(out), b.size, dtype_code(dtype))
    return out


def encode(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round-to-nearest-even of fp64 values into 16-bit patterns."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_encode_array(_ptr(v), _ptr(out), v.size, dtype_code(dtype))
    return out


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def apply(store, pool, p: int, token_adapter: np.ndarray, x: np.ndarray, y_in: np.ndarray,
          s: float, dtype: str, tokens: Optional[Sequence[int]] = None, want_exact: bool = False,
          want_v: bool = False, num_threads: int = 1, adapter_scale: Optional[np.ndarray] = None,
          on_bad: str = "raise"):
    """Oracle of y_out = round(y_in + s s_a (x A) B) for projection p.

    adapter_scale: s_a per adapter id (float64, max_adapters entries), or None
    for s_a = 1 everywhere.

    store: oracle.pool.OracleStore with the touched adapters' pages written.
    pool:  oracle.pool.OraclePool whose page tables address those pages.
    Returns (y_out, y_exact or None, v or None); rows of tokens not listed in
    ``tokens`` are left as zeros in every output.

    on_bad: what a token naming an id other than -1 outside [0, max_adapters)
    or a non-resident adapter does: "raise" (ValueError) or "keep" (its row
    is returned unchanged, like a base-only token's).
    """
    T = int(token_adapter.shape[0])
    dims = pool.proj
    pt, pt_off = pool.flat_tables()
    ta = np.ascontiguousarray(token_adapter, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    y_in = np.ascontiguousarray(y_in, dtype=np.uint16)
    h_in, h_out = dims[p].h_in, dims[p].h_out
    assert x.shape == (T, h_in) and y_in.shape == (T, h_out)
    y_out = np.zeros((T, h_out), dtype=np.uint16)
    y_exact = np.zeros((T, h_out), dtype=np.float64) if want_exact else None
    v_ld = max(1, pool.max_rank)
    v = np.zeros((T, v_ld), dtype=np.float64) if want_v else None
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    proj_in = np.asarray([d.h_in for d in dims], dtype=np.int32)
    proj_out = np.asarray([d.h_out for d in dims], dtype=np.int32)
    rank = np.ascontiguousarray(pool.rank, dtype=np.int32)
    sc = None
    if adapter_scale is not None:
        sc = np.ascontiguousarray(adapter_scale, dtype=np.float64)
        assert sc.shape == (pool.max_adapters,)
    rc = lib().oracle_lora_apply(
        _ptr(store.data), _ptr(store.page_slot), pool.H, dtype_code(dtype),
        _ptr(pt), _ptr(pt_off), _ptr(rank), pool.max_adapters,
        len(dims), _ptr(proj_in), _ptr(proj_out), p,
        _ptr(ta), T, _ptr(tok), 0 if tok is None else tok.shape[0],
        _ptr(x), h_in, _ptr(y_in), h_out,
        float(s), _ptr(sc), _ptr(y_out), _ptr(y_exact), _ptr(v), v_ld, int(num_threads))
    if rc != 0 and on_bad == "raise":
        raise ValueError("oracle: a token names an adapter that is not resident or an id out of range")
    return y_out, y_exact, v


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
