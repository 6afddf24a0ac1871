"""Shared test helpers: library conversions of 16-bit patterns and oracle set-up.

The conversions here use numpy / torch (library routines), never the oracle's
own decoder, so that tests comparing the two pin the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import pool as opool


def lib_values(bits: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values of 16-bit patterns via numpy (fp16) or torch (bf16)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def lib_bits(values: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns of fp32 values (torch round-to-nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    t = t.to(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def oracle_pool_for(wl, max_adapters=None, max_rank=None):
    """Replay the workload's pool call sequence on the oracle allocator."""
    pool = opool.OraclePool(
        wl.pool_pages, wl.H, [(p.h_in, p.h_out) for p in wl.projections],
        max_adapters or wl.spec.num_adapters,
        max_rank or int(max(wl.spec.rank_set + tuple(wl.ranks.tolist()))))
    pool.replay(wl.pool_ops, wl.ranks)
    return pool


def oracle_store_for(wl, pool, adapters):
    """Write the listed adapters' rows into the oracle's own pool copy."""
    store = opool.OracleStore(wl.pool_pages, wl.H)
    for a in sorted(set(int(a) for a in adapters)):
        store.write_adapter(pool, a, wl.adapter(a))
    return store


def touched(token_adapter) -> list:
    return sorted(set(int(a) for a in np.asarray(token_adapter) if a >= 0))


def dense_weights(wl, adapters, p):
    """Dense fp64 (A [H_in, r], B [r, H_out]) per adapter, straight from the generator."""
    out = {}
    for a in adapters:
        A_rows, B_rows = wl.adapter(a)[p]
        out[a] = (lib_values(A_rows, wl.spec.dtype).T.copy(), lib_values(B_rows, wl.spec.dtype))
    return out


def within_tol(got: np.ndarray, want: np.ndarray, atol=5e-3, rtol=1e-2) -> np.ndarray:
    """The elementwise bar |got - want| <= atol + rtol * |want|."""
    return np.abs(got - want) <= atol + rtol * np.abs(want)
