"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Integer / index work (device page contents, perm, seg_start, seg_adapter,
counts) must be bit-exact; y must satisfy |gpu - oracle| <= 5e-3 + 1e-2 |oracle|
elementwise (fp16/bf16 storage, fp32 accumulation, one rounding).
"""
import dataclasses

import numpy as np
import pytest
import torch

from lora_adapters_gb300 import slora, workloads
from oracle import pool as opool
from tests import gpu_setup as G
from tests import helpers as H

pytestmark = pytest.mark.gpu

MODES = [slora.MODE_DECODE, slora.MODE_AUTO, slora.MODE_PREFILL]

# Small cases that still span several token tiles, rank chunks, column tiles
# and page chunks, with ragged tails everywhere.
SMALL = {
    "tiny": workloads.spec("tiny"),
    "tiny_bf16": workloads.spec("tiny", dtype="bf16", seed=3),
    "mlp_ragged_bf16": workloads.WorkloadSpec(
        name="mlp_ragged", H=256, dtype="bf16",
        projections=(workloads.Projection("gate", 256, 1384), workloads.Projection("up", 256, 1384),
                     workloads.Projection("down", 1384, 256)),
        num_adapters=37, rank_set=(1, 7, 16, 33, 64), kind="decode", tokens=203, popularity="zipf",
        zipf_alpha=1.2, pool_factor=1.4, s=0.5, seed=21),
    "prefill_ragged_f16": workloads.WorkloadSpec(
        name="prefill_ragged", H=512, dtype="f16", projections=workloads._qkvo(512),
        num_adapters=11, rank_set=(8, 16, 128), kind="prefill", requests=9, prompt_len=(1, 300),
        pool_factor=1.3, s=-1.25, seed=5),
    # ranks above 128 take the whole B area of the tensor-core expand kernel
    "prefill_bigrank_f16": workloads.WorkloadSpec(
        name="prefill_bigrank", H=256, dtype="f16", projections=workloads._qkvo(256),
        num_adapters=5, rank_set=(129, 200, 256, 64), kind="prefill", requests=7, prompt_len=(1, 260),
        pool_factor=1.2, s=0.75, seed=8),
    # one K block in the first projection (no K split in tc_shrink, x columns
    # past h_in zero-filled), ranks on both sides of 128, runs longer than a
    # 256-token tile
    "short_k_f16": workloads.WorkloadSpec(
        name="short_k", H=64, dtype="f16",
        projections=(workloads.Projection("a", 48, 200), workloads.Projection("b", 200, 48)),
        num_adapters=6, rank_set=(3, 40, 130, 17), kind="prefill", requests=6, prompt_len=(1, 600),
        pool_factor=1.3, s=0.9, seed=14),
    "many_tokens_f16": workloads.WorkloadSpec(
        name="many_tokens", H=128, dtype="f16", projections=(workloads.Projection("q", 128, 136),),
        num_adapters=300, rank_set=(2, 8, 24), kind="decode", tokens=3001, popularity="uniform",
        pool_factor=1.2, s=1.0, seed=8),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lora_adapters_gb300 import build

    build.build()
    slora.lib()


def _run_and_check(case: G.GpuCase, mode: int, want=None, rows=None, multi=True):
    wl = case.wl
    case.fresh_y()
    seg = case.pool.build_segments(case.ta_dev)
    n = len(wl.projections)
    if multi:
        case.pool.apply_multi(seg, list(range(n)), case.xs, case.ys, wl.spec.s, mode)
    else:
        for p in range(n):
            case.pool.apply(seg, p, case.xs[p], case.ys[p], wl.spec.s, mode)
    torch.cuda.synchronize()
    assert case.pool.status() == slora.OK
    want = want if want is not None else G.oracle_outputs(case, tokens=rows)
    for p in range(n):
        got = G.to_bits(case.ys[p])
        ok, err, bad = G.compare(got, want[p], wl.spec.dtype, rows=rows)
        assert ok, f"projection {p} mode {mode}: {bad} elements out of tolerance, max |err| {err}"
    return seg, want


def _check_segments(case: G.GpuCase, seg):
    want = opool.build_segments(case.wl.token_adapter, case.oracle_pool.rank)
    perm, start, adapter, counts = G.seg_arrays(seg)
    assert counts[0] == want.num_segs and counts[1] == want.perm.shape[0] and counts[2] == want.bad_tokens
    assert np.array_equal(perm, want.perm)
    assert np.array_equal(start, want.seg_start)
    assert np.array_equal(adapter, want.seg_adapter)


def _check_pages(case: G.GpuCase, adapters):
    """Device page contents of the given adapters equal the oracle's own load, bit for bit."""
    store = H.oracle_store_for(case.wl, case.oracle_pool, adapters)
    buf = case.pool.buffer
    for a in adapters:
        tab = case.oracle_pool.tables[a].astype(np.int64)
        got = G.to_bits(buf[torch.from_numpy(tab).to(buf.device)])
        want = store.data[store.page_slot[tab]]
        assert np.array_equal(got, want), f"adapter {a} pages differ"


@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases_all_modes(name):
    wl = workloads.make(SMALL[name])
    case = G.build_case(wl)
    snap = case.pool.snapshot()
    assert np.array_equal(snap["owner"], case.oracle_pool.owner)
    _check_pages(case, case.touched)
    want = None
    for mode in MODES:
        seg, want = _run_and_check(case, mode, want)
        _check_segments(case, seg)
    _run_and_check(case, slora.MODE_AUTO, want, multi=False)
    # AUTO's split at any batch size: every segment on the tensor-core
    # kernels, then short segments on the CUDA cores and long ones on the
    # tensor cores
    slora.slora_set_tc_min_batch(case.pool.handle, 0)
    for thr in (0, 3):
        slora.slora_set_tc_threshold(case.pool.handle, thr)
        seg, _ = _run_and_check(case, slora.MODE_AUTO, want)
        _check_segments(case, seg)
    case.pool.close()


# Segment lengths on both sides of every tile size of both kernel families
# (the CUDA-core kernel's 4-token tiles; the tensor-core kernels' 32-token
# combine groups and 128- and 256-token tiles), each on an adapter of its own
# so that each run is exactly one segment, over ranks from 1 to 256 (one and
# two M blocks), with base-only runs between some of them.  The projections
# have ragged K (320 = one page and a quarter) and ragged N (320 columns).
EDGE_LENS = (1, 3, 4, 5, 31, 32, 33, 127, 128, 129, 255, 256, 257, 300)
EDGE_RANKS = (1, 4, 9, 16, 64, 128, 129, 256, 8, 33, 100, 200, 2, 64)


def _edge_workload(dtype: str, seed: int, token_adapter: np.ndarray) -> workloads.Workload:
    sp = workloads.WorkloadSpec(
        name="tile_edges", H=256, dtype=dtype,
        projections=(workloads.Projection("a", 256, 320), workloads.Projection("b", 320, 256)),
        num_adapters=len(EDGE_RANKS), rank_set=(1,), fixed_ranks=EDGE_RANKS, kind="decode", tokens=1,
        pool_factor=1.3, s=0.7, seed=seed)
    wl = workloads.make(sp)
    return dataclasses.replace(wl, token_adapter=np.ascontiguousarray(token_adapter, dtype=np.int32),
                               request_lens=None)


def _edge_tokens() -> np.ndarray:
    runs = []
    for i, n in enumerate(EDGE_LENS):
        runs.append(np.full(n, i, np.int32))
        if i % 4 == 1:
            runs.append(np.full(5, -1, np.int32))
    return np.concatenate(runs)


@pytest.mark.parametrize("dtype,seed", [("f16", 31), ("bf16", 32)])
def test_tile_edges_all_modes(dtype, seed):
    """Every row, in every mode and at AUTO splits on both sides of the tile
    sizes, for segments whose lengths sit on every tile edge."""
    wl = _edge_workload(dtype, seed, _edge_tokens())
    case = G.build_case(wl)
    want = None
    for mode in MODES:
        seg, want = _run_and_check(case, mode, want)
        _check_segments(case, seg)
    slora.slora_set_tc_min_batch(case.pool.handle, 0)
    for thr in (0, 4, 33, 129, 257):
        slora.slora_set_tc_threshold(case.pool.handle, thr)
        _run_and_check(case, slora.MODE_AUTO, want)
    case.pool.close()


@pytest.mark.parametrize("adapter", [0, 7])
def test_one_token_batch_all_modes(adapter):
    """A batch of a single token (rank 1, or rank 256 with two M blocks):
    every kernel path with one partial tile of one row."""
    wl = _edge_workload("f16", 33, np.array([adapter], np.int32))
    case = G.build_case(wl)
    want = None
    for mode in MODES:
        seg, want = _run_and_check(case, mode, want)
        _check_segments(case, seg)
    slora.slora_set_tc_min_batch(case.pool.handle, 0)
    slora.slora_set_tc_threshold(case.pool.handle, 1)
    _run_and_check(case, slora.MODE_AUTO, want)
    case.pool.close()


@pytest.mark.parametrize("mode,split", [(slora.MODE_DECODE, None), (slora.MODE_PREFILL, None),
                                        (slora.MODE_AUTO, 33)])
def test_cuda_graph_capture_replays_the_step(mode, split):
    """The segment build and the multi-projection apply, captured in a CUDA
    graph on the pool's compute stream (not the legacy default stream) and
    replayed: every replay equals the eager call bit for bit and the oracle
    within tolerance, in every mode (AUTO split between both kernel
    families)."""
    wl = _edge_workload("f16", 34, _edge_tokens())
    sp = wl.spec
    dims = [(p.h_in, p.h_out) for p in sp.projections]
    cs = torch.cuda.Stream()
    pool = slora.Pool(wl.pool_pages, wl.H, sp.dtype, dims, sp.num_adapters, max(EDGE_RANKS), wl.T,
                      device="cuda", compute_stream=cs)
    pool.replay(wl.pool_ops, wl.ranks, wl.adapter)
    if split is not None:
        slora.slora_set_tc_min_batch(pool.handle, 0)
        slora.slora_set_tc_threshold(pool.handle, split)
    torch.cuda.synchronize()
    ta = torch.from_numpy(wl.token_adapter.copy()).cuda()
    xs = [G.to_dev(wl.x(p), sp.dtype) for p in range(len(dims))]
    y0 = [G.to_dev(wl.y_in(p), sp.dtype) for p in range(len(dims))]
    ys = [y.clone() for y in y0]
    projs = list(range(len(dims)))
    with torch.cuda.stream(cs):
        seg = pool.build_segments(ta)
        pool.apply_multi(seg, projs, xs, ys, sp.s, mode)
    torch.cuda.synchronize()
    eager = [G.to_bits(y) for y in ys]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        seg = pool.build_segments(ta)
        pool.apply_multi(seg, projs, xs, ys, sp.s, mode)
    opool_ = H.oracle_pool_for(wl, max_adapters=sp.num_adapters, max_rank=max(EDGE_RANKS))
    case = G.GpuCase(wl, pool, ta, xs, ys, opool_, H.touched(wl.token_adapter))
    want = G.oracle_outputs(case)
    for _ in range(3):
        for y, y_ in zip(ys, y0):
            y.copy_(y_)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for p in projs:
            got = G.to_bits(ys[p])
            assert np.array_equal(got, eager[p]), f"projection {p}: replay differs from the eager call"
            ok, err, bad = G.compare(got, want[p], sp.dtype)
            assert ok, f"projection {p}: {bad} elements out of tolerance, max |err| {err}"
    assert pool.status() == slora.OK
    pool.close()


def test_full_size_llama7b_decode():
    """The benchmark workload: H=4096, q/k/v/o, 256 tokens, 1000 adapters, Zipf 1."""
    wl = workloads.make("llama7b_decode")
    case = G.build_case(wl, weights="all")
    seg, want = _run_and_check(case, slora.MODE_DECODE)
    _check_segments(case, seg)
    _check_pages(case, case.touched[:8])
    _run_and_check(case, slora.MODE_AUTO, want)
    case.pool.close()


def test_full_size_llama7b_prefill_every_row():
    """The prefill batch (8,561 tokens, 29 segments): every row of every
    projection against the oracle, in every mode and with every segment on
    the tensor cores as well as with the AUTO split."""
    wl = workloads.make("llama7b_prefill")
    case = G.build_case(wl, weights="touched")
    want = G.oracle_outputs(case)
    for mode in (slora.MODE_DECODE, slora.MODE_AUTO, slora.MODE_PREFILL):
        seg, _ = _run_and_check(case, mode, want)
    _check_segments(case, seg)
    for thr in (0, 200):
        slora.slora_set_tc_threshold(case.pool.handle, thr)
        _run_and_check(case, slora.MODE_AUTO, want)
    case.pool.close()


def test_full_size_llama13b_mlp_decode():
    """120 GB pool filled by 2000 adapters and KV slots, bf16, gate/up/down."""
    wl = workloads.make("llama13b_mlp_decode")
    case = G.build_case(wl, weights="touched")
    assert case.pool.snapshot()["free_pages"] == 0
    seg, _ = _run_and_check(case, slora.MODE_DECODE)
    _check_segments(case, seg)
    case.pool.close()


def test_edge_cases():
    wl = workloads.make("tiny")
    case = G.build_case(wl)
    pool = case.pool
    # empty batch
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    seg = pool.build_segments(empty)
    pool.apply(seg, 0, case.xs[0], case.ys[0], 1.0)
    torch.cuda.synchronize()
    assert G.seg_arrays(seg)[3][0] == 0
    # every token base-only: y unchanged, no segments
    case.fresh_y()
    ta = torch.full((wl.T,), -1, dtype=torch.int32, device="cuda")
    seg = pool.build_segments(ta)
    pool.apply(seg, 0, case.xs[0], case.ys[0], 1.0)
    torch.cuda.synchronize()
    assert np.array_equal(G.to_bits(case.ys[0]), wl.y_in(0))
    # s = 0 and a stale segment handle
    case.fresh_y()
    seg = pool.build_segments(case.ta_dev)
    pool.apply(seg, 0, case.xs[0], case.ys[0], 0.0)
    torch.cuda.synchronize()
    assert np.array_equal(G.to_bits(case.ys[0]), wl.y_in(0))
    pool.build_segments(case.ta_dev)
    with pytest.raises(slora.SloraError):
        pool.apply(seg, 0, case.xs[0], case.ys[0], 1.0)
    # a token naming an adapter that is not resident is left out and reported
    case.fresh_y()
    ta = case.ta_dev.clone()
    ta[0] = 3
    slora.slora_adapter_evict(pool.handle, 3)
    seg = pool.build_segments(ta)
    pool.apply(seg, 0, case.xs[0], case.ys[0], 1.0)
    torch.cuda.synchronize()
    assert pool.status() == slora.ERR_NOT_RESIDENT
    assert np.array_equal(G.to_bits(case.ys[0])[0], wl.y_in(0)[0])
    assert pool.status() == slora.OK                  # reading clears it
    pool.close()


def test_segment_build_token_orders():
    """The segment kernel on token orders of every kind, bit for bit: long runs
    of one adapter (placed run by run), short runs and random orders (placed
    tile by tile), the boundary between the two, a single tile plus one
    token, invalid and non-resident ids."""
    wl = workloads.make("tiny")
    case = G.build_case(wl, max_tokens=20000)
    pool = case.pool
    slora.slora_adapter_evict(pool.handle, 3)
    rank = case.oracle_pool.rank.copy()
    rank[3] = 0
    rng = np.random.default_rng(5)

    def runs(n, lo, hi, ids, cap=20000):
        keys = rng.choice(ids, n)
        return np.repeat(keys, rng.integers(lo, hi + 1, n)).astype(np.int32)[:cap]

    orders = {
        "prefill runs": (runs(40, 50, 400, [0, 1, 2, -1]), False),
        "runs of 8": (np.repeat(np.arange(400) % 3, 8).astype(np.int32), False),
        "runs of 7": (np.repeat(np.arange(400) % 3, 7).astype(np.int32), False),
        "short runs": (runs(2000, 1, 6, [0, 1, 2, -1]), False),
        "random": (rng.choice([0, 1, 2, -1], 5000).astype(np.int32), False),
        "one tile + 1": (runs(8, 200, 300, [0, 1, 2])[:1025], False),
        "20000 tokens": (runs(80, 200, 500, [0, 1, 2]), False),
        "bad ids in runs": (runs(30, 50, 300, [0, 1, 2, 3, 7, -1, -3]), True),
        "bad ids scattered": (rng.choice([0, 1, 2, 3, 9, -1], 3000).astype(np.int32), True),
    }
    for name, (ta, bad) in orders.items():
        seg = pool.build_segments(torch.from_numpy(ta).to("cuda"))
        torch.cuda.synchronize()
        want = opool.build_segments(ta, rank)
        perm, start, adapter, counts = G.seg_arrays(seg)
        assert counts[0] == want.num_segs and counts[1] == want.perm.shape[0], name
        assert counts[2] == want.bad_tokens, name
        assert np.array_equal(perm, want.perm), name
        assert np.array_equal(start, want.seg_start), name
        assert np.array_equal(adapter, want.seg_adapter), name
        status = pool.status()   # reading clears it
        assert (status != slora.OK) == bad, (name, status)
    pool.close()


def test_segment_build_small_batches():
    """Batches of up to 1024 tokens take the one-token-per-thread segment
    kernel: checked bit for bit at warp and block edges, with every token on
    its own adapter (as many segments as threads), one adapter for every
    token, base-only tokens, and invalid and non-resident ids."""
    wl = workloads.make(SMALL["many_tokens_f16"])
    case = G.build_case(wl, max_tokens=1024)
    pool = case.pool
    slora.slora_adapter_evict(pool.handle, 7)
    rank = case.oracle_pool.rank.copy()
    rank[7] = 0
    N = wl.spec.num_adapters
    rng = np.random.default_rng(11)
    orders = {}
    for T in (1, 2, 31, 32, 33, 63, 64, 65, 255, 256, 300):
        ids = rng.permutation(np.setdiff1d(np.arange(N), [7]))[:T]   # every token its own adapter
        orders[f"distinct {T}"] = (ids.astype(np.int32), False)
    orders["one adapter x 1024"] = (np.full(1024, 5, np.int32), False)
    orders["random 512"] = (rng.integers(-1, N, 512).astype(np.int32), True)   # includes adapter 7
    orders["random 1024"] = (rng.choice(np.arange(40), 1024).astype(np.int32), True)
    orders["bad ids 1000"] = (rng.choice([0, 1, 2, 7, -1, -2, N, N + 5], 1000).astype(np.int32), True)
    orders["base only 77"] = (np.full(77, -1, np.int32), False)
    for name, (ta, bad) in orders.items():
        seg = pool.build_segments(torch.from_numpy(ta).to("cuda"))
        torch.cuda.synchronize()
        want = opool.build_segments(ta, rank)
        perm, start, adapter, counts = G.seg_arrays(seg)
        assert counts[0] == want.num_segs and counts[1] == want.perm.shape[0], name
        assert counts[2] == want.bad_tokens, name
        assert np.array_equal(perm, want.perm), name
        assert np.array_equal(start, want.seg_start), name
        assert np.array_equal(adapter, want.seg_adapter), name
        status = pool.status()
        assert (status != slora.OK) == (want.bad_tokens > 0), (name, status)
        assert bad or want.bad_tokens == 0, name
    pool.close()


def test_evict_and_reload_into_other_pages_gives_identical_y():
    wl = workloads.make("tiny")
    case = G.build_case(wl)
    seg, want = _run_and_check(case, slora.MODE_DECODE)
    first = [G.to_bits(y) for y in case.ys]
    old = {a: slora.slora_adapter_pages(case.pool.handle, a) for a in range(4)}
    hold = slora.slora_pages_alloc(case.pool.handle, 5)
    for a in range(4):
        slora.slora_adapter_evict(case.pool.handle, a)
    for a in (3, 1, 0, 2):
        case.pool.load(a, int(wl.ranks[a]), wl.adapter(a))
    case.pool.sync_loads()
    assert any(not np.array_equal(old[a], slora.slora_adapter_pages(case.pool.handle, a)) for a in range(4))
    case.fresh_y()
    seg = case.pool.build_segments(case.ta_dev)
    case.pool.apply(seg, 0, case.xs[0], case.ys[0], wl.spec.s, slora.MODE_DECODE)
    torch.cuda.synchronize()
    assert np.array_equal(G.to_bits(case.ys[0]), first[0])
    del hold
    case.pool.close()


@pytest.mark.parametrize("name", ["tiny", "mlp_ragged_bf16", "prefill_ragged_f16"])
def test_per_adapter_scale(name):
    """y += s s_a (x A_a) B_a with a scale per adapter, on both kernel paths;
    a reload starts from s_a = 1 again."""
    wl = workloads.make(SMALL[name])
    case = G.build_case(wl)
    rng = np.random.default_rng(17)
    scale = np.ones(case.oracle_pool.max_adapters)
    for a in case.touched:
        scale[a] = float(np.float32(rng.uniform(-1.5, 2.5)))
        case.pool.set_scale(a, scale[a])
    scale[case.touched[0]] = 0.0
    case.pool.set_scale(case.touched[0], 0.0)
    want = G.oracle_outputs(case, adapter_scale=scale)
    for mode in MODES:
        _run_and_check(case, mode, want)
    slora.slora_set_tc_threshold(case.pool.handle, 0)
    slora.slora_set_tc_min_batch(case.pool.handle, 0)
    _run_and_check(case, slora.MODE_AUTO, want)
    # evict + reload: the adapter's scale is 1 again (page placement does not
    # change the result)
    a = case.touched[-1]
    slora.slora_adapter_evict(case.pool.handle, a)
    case.pool.load(a, int(wl.ranks[a]), wl.adapter(a))
    case.pool.sync_loads()
    scale[a] = 1.0
    _run_and_check(case, slora.MODE_DECODE, G.oracle_outputs(case, adapter_scale=scale))
    # errors: not resident, not finite
    with pytest.raises(slora.SloraError) as e:
        case.pool.set_scale(-1, 1.0)
    assert e.value.code == slora.ERR_NOT_RESIDENT
    with pytest.raises(slora.SloraError) as e:
        case.pool.set_scale(case.touched[0], float("nan"))
    assert e.value.code == slora.ERR_INVALID
    case.pool.close()


def test_timing_hooks_count_launches():
    wl = workloads.make("tiny")
    case = G.build_case(wl)
    slora.slora_timing_enable(case.pool.handle, True)
    seg = case.pool.build_segments(case.ta_dev)
    case.pool.apply(seg, 0, case.xs[0], case.ys[0], 1.0, slora.MODE_DECODE)
    t = slora.slora_timing_read(case.pool.handle)
    assert t["build_segments"][1] == 1 and t["apply_cc"][1] == 1
    assert all(ms >= 0 for ms, _ in t.values())
    case.pool.close()


def test_auto_mode_split_follows_the_batch_size():
    """AUTO runs a batch below tc_min_batch tokens wholly on the CUDA-core
    kernel, and a batch at or above it with long segments on the tensor
    cores; both give the oracle's answer."""
    wl = workloads.make(SMALL["prefill_ragged_f16"])
    case = G.build_case(wl)
    pool = case.pool
    slora.slora_set_tc_threshold(pool.handle, 16)
    want = G.oracle_outputs(case)
    for min_batch, tc in ((wl.T + 1, False), (wl.T, True)):
        slora.slora_set_tc_min_batch(pool.handle, min_batch)
        slora.slora_timing_enable(pool.handle, True)
        slora.slora_timing_read(pool.handle)
        _run_and_check(case, slora.MODE_AUTO, want)
        t = slora.slora_timing_read(pool.handle)
        slora.slora_timing_enable(pool.handle, False)
        assert t["apply_cc"][1] == 1
        assert (t["shrink_tc"][1] > 0) == tc and (t["expand_tc"][1] > 0) == tc, (min_batch, t)
    with pytest.raises(slora.SloraError):
        slora.slora_set_tc_min_batch(pool.handle, -1)
    pool.close()
