"""Error paths on the GPU, made on the host or by a wait limit -- no fault,
trap or hang of the GPU itself.

* A copy enqueue of an adapter load that fails (injected on the host with
  slora_debug_set_fault) rolls the load back: the allocator state is byte for
  byte as before, and the adapter loads and computes correctly afterwards.
* A wait of the apply kernel given a limit of one poll gives up: the kernel
  records SLORA_ERR_TIMEOUT, drains its own copies and returns; the device
  status reports it, and the next call with the normal limit is correct.
"""
import numpy as np
import pytest
import torch

from lora_adapters_gb300 import slora, workloads
from tests import gpu_setup as G
from tests.test_abi_host import _snapshot_bytes
from tests.test_gpu_parity import SMALL, _run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lora_adapters_gb300 import build

    build.build()
    slora.lib()


def test_failed_copy_enqueue_rolls_the_load_back():
    wl = workloads.make(SMALL["mlp_ragged_bf16"])
    case = G.build_case(wl)
    pool = case.pool
    want = G.oracle_outputs(case)
    a = case.touched[0]
    r = int(wl.ranks[a])
    slora.slora_adapter_evict(pool.handle, a)
    # a load enqueues the page-table copy, one copy per contiguous run of
    # host weight blocks, the scatter kernel, the scale kernel and the rank
    # copy: fail each in turn until the load gets past all of them
    failed = 0
    for nth in range(1, 64):
        before = _snapshot_bytes(slora, pool.handle)
        slora.slora_debug_set_fault(pool.handle, slora.FAULT_COPY, nth)
        try:
            pool.load(a, r, wl.adapter(a))
        except slora.SloraError as e:
            assert e.code == slora.ERR_CUDA and "injected" in str(e)
            assert np.array_equal(_snapshot_bytes(slora, pool.handle), before), nth
            pool.sync_loads()
            failed += 1
            continue
        break                       # the fault lay past the load's last enqueue
    assert failed >= 5
    slora.slora_debug_set_fault(pool.handle, slora.FAULT_NONE, 0)
    pool.sync_loads()
    _run_and_check(case, slora.MODE_DECODE, want)
    pool.close()


def test_apply_wait_limit_gives_up_and_reports_timeout():
    wl = workloads.make("llama7b_decode")
    case = G.build_case(wl, weights="touched")
    pool = case.pool
    slora.slora_debug_set_wait_limit(pool.handle, 1)
    case.fresh_y()
    seg = pool.build_segments(case.ta_dev)
    pool.apply_multi(seg, list(range(len(wl.projections))), case.xs, case.ys, wl.spec.s, slora.MODE_DECODE)
    torch.cuda.synchronize()
    assert pool.status() == slora.ERR_TIMEOUT
    assert pool.status() == slora.OK                      # reading clears it
    slora.slora_debug_set_wait_limit(pool.handle, 0)      # the built-in limit again
    _run_and_check(case, slora.MODE_DECODE)
    pool.close()
