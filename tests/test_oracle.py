"""Pins of the CPU oracle against things other than itself (CPU only).

* 16-bit conversions: numpy's fp16 and torch's bf16 conversions (library
  routines), exhaustive where the input space is small, and closed-form
  ties-to-even cases.
* The paged LoRA delta: a hand-derived worked example (tests/golden), the
  dense brute force (numpy fp64 matmul on weights taken straight from the
  generator, never through pages), and the invariants the definition fixes:
  zero B or zero A or s = 0 leave y unchanged, tokens permute with their
  outputs, the delta is linear in s, one adapter for every token equals a
  dense GEMM chain, and evict + reload into other pages changes nothing.
"""
import json
import os

import numpy as np
import pytest
import torch

from lora_adapters_gb300 import workloads
from oracle import lora as olora
from oracle import pool as opool
from oracle import ref
from tests import helpers as H

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- conversions
def test_f16_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = olora.decode(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    got = olora.decode(bits, "bf16")
    want = H.lib_values(bits, "bf16")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _f16_grid():
    rng = np.random.default_rng(1)
    mags = np.concatenate([
        rng.standard_normal(20000),
        rng.standard_normal(5000) * 1e-6,      # subnormal range
        rng.standard_normal(2000) * 7e4,       # overflow range
        rng.uniform(-65520, 65520, 2000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14, 2.0 ** -14 - 2.0 ** -25]),
    ])
    # exact midpoints between neighbouring fp16 values: ties must go to even
    b = rng.integers(0, 0x7bff, 5000).astype(np.uint16)
    lo = b.view(np.float16).astype(np.float64)
    hi = (b + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    return np.concatenate([mags, (lo + hi) / 2, -(lo + hi) / 2])


def test_f16_encode_vs_numpy():
    v = _f16_grid()
    got = olora.encode(v, "f16")
    want = v.astype(np.float16).view(np.uint16)   # numpy: direct fp64 -> fp16, RNE
    assert np.array_equal(got, want)


def test_bf16_encode_vs_torch_on_f32_values():
    # Values exactly representable in fp32, so torch's fp32 -> bf16 conversion
    # rounds once, the same single rounding the oracle performs from fp64.
    rng = np.random.default_rng(2)
    v32 = np.concatenate([
        rng.standard_normal(50000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),   # subnormal
        (rng.standard_normal(5000) * 3e38).astype(np.float32),    # near overflow
        rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    v32 = v32[np.isfinite(v32)]
    got = olora.encode(v32.astype(np.float64), "bf16")
    want = H.lib_bits(v32, "bf16")
    assert np.array_equal(got, want)


def test_bf16_ties_to_even_closed_form():
    # Midpoint between bf16 patterns b and b+1 must round to the even one.
    rng = np.random.default_rng(3)
    b = rng.integers(0x0080, 0x7f7e, 4000).astype(np.uint16)
    lo = H.lib_values(b, "bf16")
    hi = H.lib_values((b + 1).astype(np.uint16), "bf16")
    mid = (lo + hi) / 2
    got = olora.encode(mid, "bf16")
    want = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(got, want)
    # just above / below the midpoint go up / down
    assert np.array_equal(olora.encode(np.nextafter(mid, np.inf), "bf16"), (b + 1).astype(np.uint16))
    assert np.array_equal(olora.encode(np.nextafter(mid, -np.inf), "bf16"), b)
    # overflow threshold (2 - 2^-8) * 2^127 rounds to infinity, just below stays finite
    thr = (2 - 2.0 ** -8) * 2.0 ** 127
    assert olora.encode(np.array([thr]), "bf16")[0] == 0x7f80
    assert olora.encode(np.array([np.nextafter(thr, 0)]), "bf16")[0] == 0x7f7f


# ------------------------------------------------------------ golden example
def _golden_state(g):
    dims = [tuple(d) for d in g["projections"]]
    pool = opool.OraclePool(g["num_pages"], g["H"], dims, g["max_adapters"], g["max_rank"])
    ops = [tuple(o) for o in g["ops"]]
    pool.replay(ops, np.asarray(g["ranks"], dtype=np.int32))
    store = opool.OracleStore(g["num_pages"], g["H"])
    for a in (0, 1):
        A = np.asarray(g["A_columns"][str(a)], dtype=np.float32)   # rows = columns of A
        B = np.asarray(g["B_rows"][str(a)], dtype=np.float32)
        store.write_adapter(pool, a, [(H.lib_bits(A, "f16"), H.lib_bits(B, "f16"))])
    return pool, store


def test_golden_hand_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "hand_tiny.json")))
    pool, store = _golden_state(g)
    for a, tab in g["expected_page_tables"].items():
        assert pool.tables[int(a)].tolist() == tab
    assert pool.owner.tolist() == g["expected_owner"]
    assert pool._free.tolist() == g["expected_free_after_loads"]
    ta = np.asarray(g["token_adapter"], dtype=np.int32)
    x = H.lib_bits(np.asarray(g["x"], dtype=np.float32), "f16")
    y = H.lib_bits(np.asarray(g["y_in"], dtype=np.float32), "f16")
    y_out, y_exact, v = olora.apply(store, pool, 0, ta, x, y, g["s"], "f16", want_exact=True, want_v=True)
    assert np.array_equal(y_exact, np.asarray(g["expected_y"], dtype=np.float64))
    assert np.array_equal(H.lib_values(y_out, "f16"), np.asarray(g["expected_y"]))
    for i, ev in enumerate(g["expected_v"]):
        if ev is not None:
            assert v[i, :len(ev)].tolist() == ev
    with pytest.raises(opool.OracleOOM):
        pool.kv_alloc(1)
    pool.evict(0)
    got = pool.kv_alloc(2)
    assert got.tolist() == g["after_evict_0_then_kv_alloc_2"]["returned"]
    assert pool._free.tolist() == g["after_evict_0_then_kv_alloc_2"]["free"]


# --------------------------------------------------------------- brute force
SMALL_SPECS = [
    workloads.spec("tiny"),
    workloads.spec("tiny", dtype="bf16", seed=5),
    # multi-page rows with a ragged tail (h = 160 over pages of 64), three projections
    workloads.WorkloadSpec(
        name="mlp_small", H=64, dtype="bf16",
        projections=(workloads.Projection("gate", 64, 160), workloads.Projection("up", 64, 160),
                     workloads.Projection("down", 160, 64)),
        num_adapters=9, rank_set=(1, 3, 16), kind="decode", tokens=40, popularity="zipf",
        zipf_alpha=1.2, pool_factor=1.5, s=0.75, seed=11),
    workloads.WorkloadSpec(
        name="prefill_small", H=32, dtype="f16", projections=workloads._qkvo(32),
        num_adapters=5, rank_set=(8, 16, 32), kind="prefill", requests=6, prompt_len=(1, 20),
        pool_factor=2.0, s=-1.5, seed=7),
]


@pytest.mark.parametrize("sp", SMALL_SPECS, ids=lambda s: f"{s.name}-{s.dtype}")
def test_paged_oracle_equals_dense_brute_force(sp):
    wl = workloads.make(sp)
    pool = H.oracle_pool_for(wl)
    adapters = H.touched(wl.token_adapter)
    store = H.oracle_store_for(wl, pool, adapters)
    for p in range(len(wl.projections)):
        x, y = wl.x(p), wl.y_in(p)
        y_out, y_exact, _ = olora.apply(store, pool, p, wl.token_adapter, x, y, sp.s, sp.dtype,
                                        want_exact=True)
        want = ref.brute_force(wl.token_adapter, H.lib_values(x, sp.dtype), H.lib_values(y, sp.dtype),
                               H.dense_weights(wl, adapters, p), sp.s)
        assert np.allclose(y_exact, want, rtol=1e-12, atol=1e-12)
        # the rounded output is the library's RNE rounding of the exact value
        if sp.dtype == "f16":
            assert np.array_equal(y_out, y_exact.astype(np.float16).view(np.uint16))


def _tiny_state(**kw):
    wl = workloads.make("tiny", **kw)
    pool = H.oracle_pool_for(wl)
    return wl, pool


def test_zero_B_or_zero_A_or_zero_s_leaves_y_unchanged():
    wl, pool = _tiny_state()
    x, y = wl.x(0), wl.y_in(0)
    for which in ("A", "B"):
        store = opool.OracleStore(wl.pool_pages, wl.H)
        for a in range(4):
            A, B = wl.adapter(a)[0]
            if which == "A":
                A = np.zeros_like(A)
            else:
                B = np.zeros_like(B)
            store.write_adapter(pool, a, [(A, B)])
        y_out, _, _ = olora.apply(store, pool, 0, wl.token_adapter, x, y, 1.0, "f16")
        assert np.array_equal(y_out, y)
    store = H.oracle_store_for(wl, pool, range(4))
    y_out, _, _ = olora.apply(store, pool, 0, wl.token_adapter, x, y, 0.0, "f16")
    assert np.array_equal(y_out, y)


def test_tokens_permute_with_outputs():
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    x, y = wl.x(0), wl.y_in(0)
    perm = np.random.default_rng(9).permutation(wl.T)
    _, e1, _ = olora.apply(store, pool, 0, wl.token_adapter, x, y, 1.0, "f16", want_exact=True)
    _, e2, _ = olora.apply(store, pool, 0, wl.token_adapter[perm], x[perm], y[perm], 1.0, "f16",
                           want_exact=True)
    assert np.array_equal(e1[perm], e2)


def test_linear_in_s():
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    x, y = wl.x(0), wl.y_in(0)
    y0 = H.lib_values(y, "f16")

    def delta(s):
        return olora.apply(store, pool, 0, wl.token_adapter, x, y, s, "f16", want_exact=True)[1] - y0

    d1, d2, d3 = delta(1.0), delta(2.0), delta(-0.75)
    assert np.allclose(d2, 2 * d1, rtol=1e-12, atol=1e-12)
    assert np.allclose(delta(0.25) + d3, delta(0.25 - 0.75), rtol=1e-12, atol=1e-12)
    assert np.abs(d1).max() > 0.1


def test_per_adapter_scale_against_dense_brute_force():
    """y = y_in + s s_a (x A_a) B_a: each adapter's tokens against numpy's
    dense product with that adapter's own factor; s_a = 1 everywhere gives
    exactly the unscaled result, s_a = 0 leaves the adapter's tokens alone."""
    sp = SMALL_SPECS[1]
    wl = workloads.make(sp)
    pool = H.oracle_pool_for(wl)
    adapters = H.touched(wl.token_adapter)
    store = H.oracle_store_for(wl, pool, adapters)
    scale = np.ones(pool.max_adapters)
    rng = np.random.default_rng(4)
    scale[adapters] = rng.uniform(-2.0, 2.0, len(adapters))
    scale[adapters[0]] = 0.0
    for p in range(len(wl.projections)):
        x, y = wl.x(p), wl.y_in(p)
        X, Y = H.lib_values(x, sp.dtype), H.lib_values(y, sp.dtype)
        dense = H.dense_weights(wl, adapters, p)
        y_out, e, _ = olora.apply(store, pool, p, wl.token_adapter, x, y, sp.s, sp.dtype, want_exact=True,
                                  adapter_scale=scale)
        for a in adapters:
            only_a = np.where(wl.token_adapter == a, a, -1).astype(np.int32)
            want = ref.brute_force(only_a, X, Y, {a: dense[a]}, sp.s * scale[a])
            rows = wl.token_adapter == a
            assert np.allclose(e[rows], want[rows], rtol=1e-12, atol=1e-12)
        rows0 = wl.token_adapter == adapters[0]
        assert np.array_equal(y_out[rows0], y[rows0])
        ones = olora.apply(store, pool, p, wl.token_adapter, x, y, sp.s, sp.dtype, want_exact=True,
                           adapter_scale=np.ones(pool.max_adapters))[1]
        plain = olora.apply(store, pool, p, wl.token_adapter, x, y, sp.s, sp.dtype, want_exact=True)[1]
        assert np.array_equal(ones, plain)


def test_base_only_tokens_unchanged():
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    ta = wl.token_adapter.copy()
    ta[::3] = -1
    x, y = wl.x(0), wl.y_in(0)
    y_out, _, _ = olora.apply(store, pool, 0, ta, x, y, 1.0, "f16")
    assert np.array_equal(y_out[::3], y[::3])
    assert not np.array_equal(y_out[1::3], y[1::3])


def test_out_of_range_ids_are_errors_and_left_unchanged():
    """Only -1 means "no adapter": -2, an id past the last adapter and an
    evicted adapter are errors (ValueError by default); with on_bad="keep"
    their rows come back unchanged and every other row is what it is when
    those tokens carry no adapter at all."""
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    x, y = wl.x(0), wl.y_in(0)
    pool.evict(2)
    for bad_id in (-2, -7, 4, 1000, 2):
        ta = wl.token_adapter.copy()
        ta[ta == 2] = 1                     # no token on the evicted adapter except the planted ones
        ta[[1, 6]] = bad_id
        with pytest.raises(ValueError):
            olora.apply(store, pool, 0, ta, x, y, 1.0, "f16")
        got, _, _ = olora.apply(store, pool, 0, ta, x, y, 1.0, "f16", on_bad="keep")
        base = ta.copy()
        base[[1, 6]] = -1
        want, _, _ = olora.apply(store, pool, 0, base, x, y, 1.0, "f16")
        assert np.array_equal(got, want), bad_id
        assert np.array_equal(got[[1, 6]], y[[1, 6]]), bad_id


def test_single_adapter_batch_equals_dense_gemm_chain():
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    x, y = wl.x(0), wl.y_in(0)
    ta = np.full(wl.T, 3, dtype=np.int32)
    _, e, _ = olora.apply(store, pool, 0, ta, x, y, 1.0, "f16", want_exact=True)
    A, B = H.dense_weights(wl, [3], 0)[3]
    X = H.lib_values(x, "f16")
    want = H.lib_values(y, "f16") + (X @ A) @ B            # one GEMM chain for the whole batch
    assert np.allclose(e, want, rtol=1e-12, atol=1e-12)


def test_evict_and_reload_into_other_pages_is_identical():
    wl, pool = _tiny_state()
    store = H.oracle_store_for(wl, pool, range(4))
    x, y = wl.x(0), wl.y_in(0)
    y1, _, _ = olora.apply(store, pool, 0, wl.token_adapter, x, y, 1.0, "f16")
    old = {a: pool.tables[a].copy() for a in range(4)}
    hold = pool.kv_alloc(5)                 # occupy the lowest free pages first
    for a in range(4):
        pool.evict(a)
    for a in (3, 1, 0, 2):                  # reload in another order
        pool.load(a, int(wl.ranks[a]))
    assert any(not np.array_equal(old[a], pool.tables[a]) for a in range(4))
    del hold
    store2 = H.oracle_store_for(wl, pool, range(4))
    y2, _, _ = olora.apply(store2, pool, 0, wl.token_adapter, x, y, 1.0, "f16")
    assert np.array_equal(y1, y2)


def test_planted_index_mistake_is_caught():
    """A transposed page-table walk (B chunks read in A's order) must fail the brute force."""
    sp = SMALL_SPECS[2]
    wl = workloads.make(sp)
    pool = H.oracle_pool_for(wl)
    adapters = H.touched(wl.token_adapter)
    store = H.oracle_store_for(wl, pool, adapters)
    # plant the mistake in the oracle's inputs: swap two pages of one adapter's B rows
    a = adapters[0]
    tab = pool.tables[a]
    e0 = pool.entry_of(a, 0, "B", 0, 0)
    e1 = pool.entry_of(a, 0, "B", 0, 1)
    tab[e0], tab[e1] = tab[e1], tab[e0]
    x, y = wl.x(0), wl.y_in(0)
    _, y_exact, _ = olora.apply(store, pool, 0, wl.token_adapter, x, y, sp.s, sp.dtype, want_exact=True)
    want = ref.brute_force(wl.token_adapter, H.lib_values(x, sp.dtype), H.lib_values(y, sp.dtype),
                           H.dense_weights(wl, adapters, 0), sp.s)
    assert not np.allclose(y_exact, want, rtol=1e-9, atol=1e-9)
