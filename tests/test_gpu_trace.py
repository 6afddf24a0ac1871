"""GPU test of the serving-trace driver: one traced step checked by the oracle.

The pool state at the probed step is rebuilt by replaying the driver's log of
pool calls on the oracle's own allocator; the adapters resident then get their
weights from the seeded host store; the step's ids, x and y_in were drawn on
the host.  The GPU's y for that step must match the oracle element by element.
"""
import dataclasses

import numpy as np
import pytest
import torch

from lora_adapters_gb300 import trace
from oracle import lora as olora
from oracle import pool as opool
from tests import gpu_setup as G
from tests.test_trace import small_spec

pytestmark = pytest.mark.gpu


def _check_probe(tr, res, sp):
    """The probed layer's y against the oracle: the pool state at the probe
    rebuilt by the oracle allocator from the logged calls, the rows of the
    batch's adapters for that layer written from the host store."""
    pr = tr.probe
    assert pr is not None and pr["ids"].shape[0] > 0
    op = opool.OraclePool(sp.pool_pages, sp.H, [(p.h_in, p.h_out) for p in sp.projections], sp.num_adapters,
                          max(sp.rank_set))
    op.replay(res.ops[:pr["ops"]], res.ranks)
    n = len(sp.layer_projections)
    layer_projs = list(range(pr["layer"] * n, (pr["layer"] + 1) * n))
    store = opool.OracleStore(sp.pool_pages, sp.H)
    for a in sorted(set(int(a) for a in pr["ids"])):
        store.write_adapter(op, a, tr.store.weights(a), only=set(layer_projs))
    for i, p in enumerate(layer_projs):
        want, _, _ = olora.apply(store, op, p, pr["ids"], pr["x"][i], pr["y_in"][i], sp.s, sp.dtype,
                                 num_threads=olora.default_threads())
        ok, err, bad = G.compare(pr["y"][i], want, sp.dtype)
        assert ok, f"projection {p}: {bad} elements out of tolerance, max |err| {err}"


@pytest.mark.parametrize("probe_step,layer", [(5, 1), (37, 0)])
def test_traced_step_matches_oracle(probe_step, layer):
    sp = small_spec(steps=40)
    tr = trace.Trace(sp, device=torch.device("cuda", 0), probe_step=probe_step, probe_layer=layer)
    res = tr.run()
    assert res.loads > 0 and res.gpu_ms > 0
    _check_probe(tr, res, sp)
    tr.close()


def test_traced_step_after_evictions_matches_oracle():
    """The small trace with its pool under pressure: a step probed after LRU
    evictions (pages of evicted adapters reused by later loads and KV)."""
    sp = small_spec(steps=200)
    tr = trace.Trace(sp, device=torch.device("cuda", 0), probe_step=60, probe_layer=1, probe_after_eviction=True)
    res = tr.run()
    assert res.evictions > 0 and tr.probe["evictions_before"] > 0
    _check_probe(tr, res, sp)
    tr.close()


@pytest.mark.slow
def test_full_size_trace_step_after_evictions_matches_oracle():
    """The full-size trace: 32 layers of q, k, v, o, 2000 adapters, 80 GB
    pool shared with 64 KV pages per token.  Run until adapters have been
    evicted for room, probe the last layer of the next step, check it."""
    sp = dataclasses.replace(trace.TraceSpec(), steps=700)
    tr = trace.Trace(sp, device=torch.device("cuda", 0), probe_step=300, probe_after_eviction=True)
    res = tr.run()
    assert res.evictions > 0 and tr.probe is not None and tr.probe["evictions_before"] > 0
    assert res.load_bytes > 0 and res.tokens > 0
    _check_probe(tr, res, sp)
    tr.close()
