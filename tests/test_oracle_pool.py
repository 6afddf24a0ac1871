"""Pins of the allocator / page-table / segment oracle (CPU only).

Checked against the hand-derived fixtures in tests/golden and against the
properties the policy fixes: allocated and free pages partition the pool, no
page has two owners, an adapter of rank r owns exactly
r * sum_q (ceil(h_in_q/H) + ceil(h_out_q/H)) pages, an allocation returns the
n smallest pages that were free before it, and a failed call changes nothing.
"""
import json
import os

import numpy as np
import pytest

from lora_adapters_gb300 import workloads
from oracle import pool as opool
from tests import helpers as H


def _check_partition(pool: opool.OraclePool):
    free = set(pool._free.tolist())
    assert len(free) == pool._free.shape[0]
    assert free == set(np.flatnonzero(pool.owner == opool.FREE).tolist())
    for a, tab in pool.tables.items():
        assert (pool.owner[tab] == a).all()
        assert tab.shape[0] == pool.adapter_pages(pool.rank[a])
        assert np.unique(tab).shape[0] == tab.shape[0]
    owned = np.concatenate([t for t in pool.tables.values()]) if pool.tables else np.zeros(0, int)
    assert (pool.owner >= 0).sum() == owned.shape[0]


def test_random_call_sequences_keep_the_invariants():
    rng = np.random.default_rng(4)
    pool = opool.OraclePool(300, 16, [(16, 16), (16, 40)], max_adapters=12, max_rank=8)
    kv = []
    for step in range(600):
        op = rng.integers(0, 4)
        before_free = pool._free.copy()
        before_owner = pool.owner.copy()
        try:
            if op == 0:
                n = int(rng.integers(0, 40))
                got = pool.kv_alloc(n)
                assert got.tolist() == before_free[:n].tolist()   # n smallest free pages
                kv.extend(got.tolist())
            elif op == 1 and kv:
                idx = rng.choice(len(kv), size=int(rng.integers(1, min(len(kv), 30) + 1)), replace=False)
                pages = [kv[i] for i in idx]
                pool.kv_free(pages)
                kv = [p for i, p in enumerate(kv) if i not in set(idx.tolist())]
            elif op == 2:
                a = int(rng.integers(0, 12))
                r = int(rng.integers(1, 9))
                got = pool.load(a, r)
                assert got.tolist() == before_free[:pool.adapter_pages(r)].tolist()
            else:
                a = int(rng.integers(0, 12))
                pool.evict(a)
        except (opool.OracleOOM, opool.OracleInvalid):
            assert np.array_equal(pool._free, before_free)      # failed call: nothing changed
            assert np.array_equal(pool.owner, before_owner)
        _check_partition(pool)


def test_invalid_calls_are_rejected_without_change():
    pool = opool.OraclePool(64, 8, [(8, 8)], max_adapters=4, max_rank=4)
    kv = pool.kv_alloc(10)
    snap = (pool._free.copy(), pool.owner.copy())
    for bad in (lambda: pool.load(4, 2), lambda: pool.load(0, 5), lambda: pool.load(0, 0),
                lambda: pool.evict(1), lambda: pool.kv_free([kv[0], kv[0]]),
                lambda: pool.kv_free([64]), lambda: pool.kv_free([20]), lambda: pool.kv_alloc(-1),
                lambda: pool.kv_alloc(55)):
        with pytest.raises((opool.OracleOOM, opool.OracleInvalid)):
            bad()
        assert np.array_equal(pool._free, snap[0]) and np.array_equal(pool.owner, snap[1])
    pool.load(0, 2)
    with pytest.raises(opool.OracleInvalid):
        pool.load(0, 2)                                          # already resident
    with pytest.raises(opool.OracleInvalid):
        pool.kv_free([int(pool.tables[0][0])])                   # an adapter page is not KV


def test_adapter_page_count_matches_generator_count():
    for name in ("tiny", "llama7b_decode", "llama13b_mlp_decode"):
        sp = workloads.SPECS[name]
        pool = opool.OraclePool(10, sp.H, [(p.h_in, p.h_out) for p in sp.projections], 1, 128)
        for r in (1, 8, 64):
            assert pool.adapter_pages(r) == workloads.adapter_page_count(r, sp.projections, sp.H)
    # 13824 / 5120 -> 3 pages per row: gate, up (1 + 3 each) and down (3 + 1): 12 per rank
    sp = workloads.SPECS["llama13b_mlp_decode"]
    assert workloads.adapter_page_count(1, sp.projections, sp.H) == 12


def test_workload_replay_scatters_adapter_pages():
    wl = workloads.make("tiny")
    pool = H.oracle_pool_for(wl)
    _check_partition(pool)
    pages = np.concatenate([pool.tables[a] for a in range(4)])
    assert (np.diff(np.sort(pages)) > 1).any()                   # not one contiguous run
    assert pool.free_count == 128 - pages.shape[0]


def test_golden_segments(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "segments_hand.json")))
    seg = opool.build_segments(np.asarray(g["token_adapter"]), np.asarray(g["rank"]))
    assert seg.perm.tolist() == g["expected_perm"]
    assert seg.seg_start.tolist() == g["expected_seg_start"]
    assert seg.seg_adapter.tolist() == g["expected_seg_adapter"]
    assert seg.bad_tokens == g["expected_bad_tokens"]


def test_segments_out_of_range_ids_by_hand():
    """Only -1 means "no adapter": ids below it and past the last adapter are
    left out and counted, like an adapter that is not resident."""
    seg = opool.build_segments(np.asarray([1, -2, 0, -1, 5, 1, 2, 0]), np.asarray([4, 8, 0]))
    assert seg.perm.tolist() == [2, 7, 0, 5]
    assert seg.seg_start.tolist() == [0, 2, 4]
    assert seg.seg_adapter.tolist() == [0, 1]
    assert seg.bad_tokens == 3          # -2, 5 (out of range), 2 (rank 0)


@pytest.mark.parametrize("T,N,frac_none", [(0, 5, 0.0), (1, 5, 0.0), (300, 7, 0.2), (5000, 1000, 0.05),
                                           (64, 3, 1.0)])
def test_segment_properties(T, N, frac_none):
    rng = np.random.default_rng(T + N)
    ta = rng.integers(0, N, T).astype(np.int32)
    ta[rng.random(T) < frac_none] = -1
    rank = rng.integers(1, 5, N).astype(np.int32)
    seg = opool.build_segments(ta, rank)
    kept = np.flatnonzero(ta >= 0)
    assert sorted(seg.perm.tolist()) == kept.tolist()            # a permutation of kept tokens
    counts = np.bincount(ta[kept], minlength=N)
    assert seg.seg_adapter.tolist() == np.flatnonzero(counts).tolist()   # ascending ids
    assert np.diff(seg.seg_start).tolist() == counts[counts > 0].tolist()
    for s in range(seg.num_segs):
        part = seg.perm[seg.seg_start[s]:seg.seg_start[s + 1]]
        assert (ta[part] == seg.seg_adapter[s]).all()
        assert (np.diff(part) > 0).all()                         # stable: original order kept
