"""Run in a process of its own with SLORA_DEBUG=1 (tests/test_gpu_debug.py):
the SLORA_DEBUG build of the library on the GPU.

* A batch computes as the release build does (every row against the oracle),
  and the device status stays OK.
* A page index planted in the device page table (past the pool's last page,
  then negative), for an A row and a B row of an adapter the batch uses, is
  caught by the kernels' bounds checks: the device status reports
  SLORA_ERR_DEVICE_ASSERT, in DECODE (CUDA-core kernel) and PREFILL
  (tensor-core kernels) mode; the checked index is replaced by page 0, so
  nothing is read outside the pool.
* With the old index put back, the batch is right again.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lora_adapters_gb300 import slora, workloads  # noqa: E402
from tests import gpu_setup as G  # noqa: E402


def _apply(case, mode):
    wl = case.wl
    case.fresh_y()
    seg = case.pool.build_segments(case.ta_dev)
    case.pool.apply_multi(seg, list(range(len(wl.projections))), case.xs, case.ys, wl.spec.s, mode)
    torch.cuda.synchronize()
    return case.pool.status()


def _check_rows(case, want, mode):
    assert _apply(case, mode) == slora.OK
    for p in range(len(case.wl.projections)):
        ok, err, bad = G.compare(G.to_bits(case.ys[p]), want[p], case.wl.spec.dtype)
        assert ok, f"mode {mode} projection {p}: {bad} elements out of tolerance, max |err| {err}"


def main() -> int:
    assert slora.DEBUG and slora.LIB_PATH.endswith("libslora_debug.so"), slora.LIB_PATH
    torch.cuda.set_device(0)
    wl = workloads.make("tiny")
    case = G.build_case(wl)
    want = G.oracle_outputs(case)
    for mode in (slora.MODE_DECODE, slora.MODE_PREFILL):
        _check_rows(case, want, mode)
    op = case.oracle_pool
    stride = op.max_rank * op.chunks_per_rank()
    a = case.touched[0]
    num_pages = wl.pool_pages
    for which in ("A", "B"):
        entry = a * stride + op.entry_of(a, 0, which, 0, 0)
        for bad in (num_pages + 7, -3):
            old = slora.slora_debug_poke_page_table(case.pool.handle, entry, bad)
            for mode in (slora.MODE_DECODE, slora.MODE_PREFILL):
                st = _apply(case, mode)
                assert st == slora.ERR_DEVICE_ASSERT, (which, bad, mode, st)
            assert slora.slora_debug_poke_page_table(case.pool.handle, entry, old) == bad
    for mode in (slora.MODE_DECODE, slora.MODE_PREFILL):
        _check_rows(case, want, mode)
    case.pool.close()
    print("debug build OK")
    return 0


if __name__ == "__main__":
    sys.exit(main())
