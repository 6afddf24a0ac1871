"""Set-up shared by the GPU tests: a device pool for a workload, its inputs on
the device, and the oracle's answer for the same seeded inputs.

Inputs come only from lora_adapters_gb300.workloads; expected values only
from oracle/.  Nothing here computes any part of the method itself.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

from lora_adapters_gb300 import slora, workloads
from oracle import lora as olora
from oracle import pool as opool
from tests import helpers as H


@dataclasses.dataclass
class GpuCase:
    wl: workloads.Workload
    pool: slora.Pool
    ta_dev: torch.Tensor
    xs: List[torch.Tensor]
    ys: List[torch.Tensor]
    oracle_pool: opool.OraclePool
    touched: List[int]

    def fresh_y(self):
        for p, y in enumerate(self.ys):
            y.copy_(torch.from_numpy(self.wl.y_in(p).view(np.int16)).view(y.dtype).to(y.device))


def _tdtype(dtype):
    return torch.float16 if dtype == "f16" else torch.bfloat16


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(_tdtype(dtype)).to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def build_case(wl: workloads.Workload, weights: str = "all", max_tokens: Optional[int] = None,
               max_rank: Optional[int] = None, max_adapters: Optional[int] = None) -> GpuCase:
    """weights: "all" loads every adapter's drawn weights; "touched" draws weights
    only for adapters the batch uses and loads zeros for the rest (their pages
    are still allocated, in the same order, so the page layout is unchanged)."""
    sp = wl.spec
    dims = [(p.h_in, p.h_out) for p in sp.projections]
    touched = H.touched(wl.token_adapter)
    mr = max_rank or int(max(sp.rank_set + tuple(wl.ranks.tolist())))
    ma = max_adapters or sp.num_adapters
    pool = slora.Pool(wl.pool_pages, wl.H, sp.dtype, dims, ma, mr, max_tokens or max(wl.T, 1), device="cuda")
    zeros = {}

    def weights_of(a):
        if weights == "all" or a in touched_set:
            return wl.adapter(a)
        r = int(wl.ranks[a])
        if r not in zeros:
            zeros[r] = [(np.zeros((r, i), np.uint16), np.zeros((r, o), np.uint16)) for i, o in dims]
        return zeros[r]

    touched_set = set(touched)
    pool.replay(wl.pool_ops, wl.ranks, weights_of)
    torch.cuda.synchronize()
    ta = torch.from_numpy(wl.token_adapter.copy()).to("cuda")
    xs = [to_dev(wl.x(p), sp.dtype) for p in range(len(dims))]
    ys = [to_dev(wl.y_in(p), sp.dtype) for p in range(len(dims))]
    opool_ = H.oracle_pool_for(wl, max_adapters=ma, max_rank=mr)
    return GpuCase(wl, pool, ta, xs, ys, opool_, touched)


def oracle_outputs(case: GpuCase, tokens=None, threads=None, adapter_scale=None) -> Dict[int, np.ndarray]:
    """Oracle y_out (16-bit patterns) per projection, for `tokens` (all if None);
    adapter_scale: s_a per adapter id (float64) or None."""
    wl = case.wl
    store = H.oracle_store_for(wl, case.oracle_pool, case.touched)
    out = {}
    for p in range(len(wl.projections)):
        y_out, _, _ = olora.apply(store, case.oracle_pool, p, wl.token_adapter, wl.x(p), wl.y_in(p),
                                  wl.spec.s, wl.spec.dtype, tokens=tokens,
                                  num_threads=threads or olora.default_threads(), adapter_scale=adapter_scale)
        out[p] = y_out
    return out


def compare(got_bits: np.ndarray, want_bits: np.ndarray, dtype: str, rows=None):
    """Elementwise |gpu - oracle| <= 5e-3 + 1e-2 |oracle|; returns (ok, max_abs_err, n_bad)."""
    g = H.lib_values(got_bits if rows is None else got_bits[rows], dtype)
    w = H.lib_values(want_bits if rows is None else want_bits[rows], dtype)
    ok = H.within_tol(g, w)
    return bool(ok.all()), float(np.abs(g - w).max(initial=0.0)), int((~ok).sum())


class _DevArray:
    """Describes library-owned device memory so torch can alias it (no copy)."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def read_i32(ptr: int, n: int) -> np.ndarray:
    """Copy n int32 values at a device address owned by the library to the host."""
    if n == 0:
        return np.zeros(0, dtype=np.int32)
    torch.cuda.synchronize()
    return torch.as_tensor(_DevArray(ptr, n, "<i4"), device="cuda").cpu().numpy().copy()


def seg_arrays(seg):
    """(perm, seg_start, seg_adapter, counts) of a segment handle, on the host."""
    counts = read_i32(seg.counts, 16)
    S, n = int(counts[0]), int(counts[1])
    return read_i32(seg.perm, n), read_i32(seg.seg_start, S + 1), read_i32(seg.seg_adapter, S), counts
