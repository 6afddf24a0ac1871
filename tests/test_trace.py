"""CPU tests of the serving-trace driver on a planning pool (no GPU work).

The driver's log of pool calls is replayed by the oracle's own allocator:
page ownership, ranks and page tables must match the library's pool bit for
bit after hundreds of steps of KV growth, request completions, adapter loads
and least-recently-used evictions.
"""
import dataclasses

import numpy as np

from lora_adapters_gb300 import slora, trace, workloads
from oracle import pool as opool


def small_spec(**kw):
    # two layers of q, k, v, o; K and V of both layers per token
    base = dict(H=256, layer_projections=workloads._qkvo(256), layers=2, kv_pages_per_token=4,
                num_adapters=60, pool_bytes=256 * 2 * 6000, token_budget=128, max_running=24,
                arrivals_per_step=1.5, prompt_len=(4, 60), output_len=(4, 40), steps=300, max_loads_per_step=4)
    base.update(kw)
    return dataclasses.replace(trace.TraceSpec(), **base)


def test_spec_lists_every_layers_projections():
    sp = small_spec(layers=3)
    assert len(sp.projections) == 12
    assert [p.name for p in sp.projections[4:8]] == ["L1.q", "L1.k", "L1.v", "L1.o"]
    full = trace.TraceSpec()
    assert len(full.projections) == 128 and full.kv_pages_per_token == 2 * full.layers


def test_trace_pool_state_replays_on_the_oracle_allocator():
    sp = small_spec()
    tr = trace.Trace(sp)
    res = tr.run()
    assert res.loads > 0 and res.evictions > 0 and res.finished > 0      # the trace exercised all of it
    op = opool.OraclePool(sp.pool_pages, sp.H, [(p.h_in, p.h_out) for p in sp.projections], sp.num_adapters,
                          max(sp.rank_set))
    op.replay(res.ops, res.ranks)
    snap = slora.slora_pool_snapshot(tr.pool.handle)
    assert np.array_equal(snap["owner"], op.owner)
    assert np.array_equal(snap["rank"], op.rank)
    assert snap["free_pages"] == op.free_count
    for a, tab in op.tables.items():
        assert np.array_equal(snap["page_table"][a, :tab.shape[0]], tab)
    # every running request's adapter is resident; its KV pages match its tokens
    for rq in tr.running:
        assert op.rank[rq.adapter] > 0
        kv = sum(tr.kv[h].shape[0] for h in rq.kv_handles)
        assert kv == (rq.prompt + rq.output) * sp.kv_pages_per_token
    # pages: free + KV + adapters = all
    kv_pages = sum(p.shape[0] for p in tr.kv.values())
    ad_pages = sum(int(op.rank[a]) * op.chunks_per_rank() for a in op.tables)
    assert op.free_count + kv_pages + ad_pages == sp.pool_pages
    tr.close()


def test_trace_is_deterministic():
    a = trace.Trace(small_spec(steps=120)).run()
    b = trace.Trace(small_spec(steps=120)).run()
    assert len(a.ops) == len(b.ops)
    for x, y in zip(a.ops, b.ops):
        assert x[0] == y[0] and x[1] == y[1]
        if x[0] == "kv_free":
            assert np.array_equal(x[2], y[2])
        elif x[0] == "kv_alloc":
            assert x[2] == y[2]
    assert a.tokens == b.tokens and a.finished == b.finished


def test_trace_accounts_for_every_request_and_the_load_stall():
    sp = small_spec(steps=250)
    tr = trace.Trace(sp)
    res = tr.run()
    # every arrival is admitted or still waiting; every admitted request is
    # running or finished
    assert res.arrivals == res.admitted + len(tr.waiting)
    assert res.admitted == res.finished + len(tr.running)
    assert 0 < res.arrival_misses < res.arrivals
    # a miss waits at least one step for its load (an adapter loaded in step
    # k serves from step k + 1); queueing adds to both kinds of wait
    assert res.wait_steps_miss >= 1.0
    assert res.wait_steps_hit >= 0.0
    s = res.summary()
    assert s["adapter_hit_rate"] == 1.0 - res.arrival_misses / res.arrivals
    tr.close()



def test_full_size_trace_replays_on_the_oracle_allocator():
    """The full-size trace's bookkeeping (32 layers, 2000 adapters, 80 GB
    pool, 9.8 M pages) for 600 steps: evictions happen, and the pool state
    after them replays bit for bit on the oracle's allocator."""
    sp = dataclasses.replace(trace.TraceSpec(), steps=600)
    tr = trace.Trace(sp)
    res = tr.run()
    assert res.evictions > 0 and res.loads > res.evictions
    op = opool.OraclePool(sp.pool_pages, sp.H, [(p.h_in, p.h_out) for p in sp.projections], sp.num_adapters,
                          max(sp.rank_set))
    op.replay(res.ops, res.ranks)
    snap = slora.slora_pool_snapshot(tr.pool.handle)
    assert snap["free_pages"] == op.free_count
    assert np.array_equal(snap["owner"], op.owner)
    assert np.array_equal(snap["rank"], op.rank)
    tr.close()
