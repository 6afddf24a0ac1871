"""GPU test of the serving-trace driver: one traced step checked by the oracle.

The pool state at the probed step is rebuilt by replaying the driver's log of
pool calls on the oracle's own allocator; the adapters resident then get their
weights from the seeded host store; the step's ids, x and y_in were drawn on
the host.  The GPU's y for that step must match the oracle element by element.
"""
import numpy as np
import pytest
import torch

from lora_adapters_gb300 import trace
from oracle import lora as olora
from oracle import pool as opool
from tests import gpu_setup as G
from tests.test_trace import small_spec

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("probe_step", [5, 37])
def test_traced_step_matches_oracle(probe_step):
    sp = small_spec(steps=40)
    tr = trace.Trace(sp, device=torch.device("cuda", 0), probe_step=probe_step)
    res = tr.run()
    pr = tr.probe
    assert pr is not None and pr["ids"].shape[0] > 0
    assert res.loads > 0 and res.gpu_ms > 0
    op = opool.OraclePool(sp.pool_pages, sp.H, [(p.h_in, p.h_out) for p in sp.projections], sp.num_adapters,
                          max(sp.rank_set))
    op.replay(res.ops[:pr["ops"]], res.ranks)
    store = opool.OracleStore(sp.pool_pages, sp.H)
    for a in sorted(op.tables):
        store.write_adapter(op, a, tr.store.weights(a))
    for p in range(len(sp.projections)):
        want, _, _ = olora.apply(store, op, p, pr["ids"], pr["x"][p], pr["y_in"][p], sp.s, sp.dtype,
                                 num_threads=olora.default_threads())
        ok, err, bad = G.compare(pr["y"][p], want, sp.dtype)
        assert ok, f"projection {p}: {bad} elements out of tolerance, max |err| {err}"
    tr.close()
