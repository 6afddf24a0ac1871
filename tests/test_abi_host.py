"""CPU tests of the C-ABI library: it loads, exports every declared symbol, and
its host allocator / page tables replay bit-exactly against the oracle
allocator on planning pools (no device buffer, so no CUDA call is made).
"""
import os
import re

import numpy as np
import pytest

from lora_adapters_gb300 import workloads
from oracle import pool as opool
from tests import helpers as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def S():
    from lora_adapters_gb300 import build, slora

    build.build()
    slora.lib()
    return slora


def _declared_symbols():
    out = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            out |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(slora_\w+)\s*\(", text, re.M))
    return out


def test_library_exports_every_declared_symbol(S):
    declared = _declared_symbols()
    assert "slora_lora_apply" in declared and "slora_build_segments" in declared
    lib = S.lib()
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(S.EXPORTED) | {n for n in declared if hasattr(lib, n)}


def test_debug_library_builds_and_exports_every_declared_symbol():
    """The SLORA_DEBUG build (bounds checks in every kernel) compiles and
    exports the same calls; it is loaded here without any GPU work."""
    import ctypes

    from lora_adapters_gb300 import build

    path = build.build(debug=True)
    assert path.endswith("libslora_debug.so")
    lib = ctypes.CDLL(path)
    for name in sorted(_declared_symbols()):
        assert hasattr(lib, name), name


def _planning_pool(S, wl, max_adapters=None, max_rank=None):
    sp = wl.spec
    return S.Pool(wl.pool_pages, wl.H, sp.dtype, [(p.h_in, p.h_out) for p in sp.projections],
                  max_adapters or sp.num_adapters,
                  max_rank or int(max(sp.rank_set + tuple(wl.ranks.tolist()))), max_tokens=wl.T)


def _compare(snap, pool: opool.OraclePool):
    assert snap["free_pages"] == pool.free_count
    assert np.array_equal(snap["owner"], pool.owner)
    assert np.array_equal(snap["rank"], pool.rank)
    pt, _ = pool.flat_tables(stride=snap["page_table"].shape[1])
    assert np.array_equal(snap["page_table"].reshape(-1), pt)


@pytest.mark.parametrize("name", ["tiny", "llama7b_decode", "llama7b_prefill"])
def test_workload_replay_matches_oracle_allocator(S, name):
    wl = workloads.make(name)
    pool = _planning_pool(S, wl)
    pool.replay(wl.pool_ops, wl.ranks)
    _compare(pool.snapshot(), H.oracle_pool_for(wl))
    pool.close()


def test_full_size_mlp_pool_replay_matches_oracle():
    from lora_adapters_gb300 import build, slora as S

    build.build()
    wl = workloads.make("llama13b_mlp_decode")
    assert wl.pool_pages == 11_718_750
    pool = _planning_pool(S, wl)
    pool.replay(wl.pool_ops, wl.ranks)
    snap = pool.snapshot()
    assert snap["free_pages"] == 0                  # adapters + KV fill the pool
    _compare(snap, H.oracle_pool_for(wl))
    pool.close()


def test_random_call_sequence_matches_oracle(S):
    rng = np.random.default_rng(12)
    dims = [(16, 16), (16, 40)]
    pool = S.Pool(300, 16, "f16", dims, max_adapters=12, max_rank=8, max_tokens=8)
    ref = opool.OraclePool(300, 16, dims, max_adapters=12, max_rank=8)
    kv = []
    for step in range(800):
        op = int(rng.integers(0, 4))
        if op == 0:
            n = int(rng.integers(0, 40))
            try:
                want = ref.kv_alloc(n)
            except opool.OracleOOM:
                with pytest.raises(S.SloraError) as e:
                    S.slora_pages_alloc(pool.handle, n)
                assert e.value.code == S.ERR_OOM
            else:
                got = S.slora_pages_alloc(pool.handle, n)
                assert got.tolist() == want.tolist()
                kv.extend(got.tolist())
        elif op == 1 and kv:
            idx = rng.choice(len(kv), size=int(rng.integers(1, min(len(kv), 30) + 1)), replace=False)
            pages = [kv[i] for i in idx]
            if rng.random() < 0.1:
                pages.append(pages[0])                     # duplicate: must be rejected
                with pytest.raises(opool.OracleInvalid):
                    ref.kv_free(pages)
                with pytest.raises(S.SloraError) as e:
                    S.slora_pages_free(pool.handle, pages)
                assert e.value.code == S.ERR_INVALID
            else:
                ref.kv_free(pages)
                S.slora_pages_free(pool.handle, pages)
                drop = set(idx.tolist())
                kv = [p for i, p in enumerate(kv) if i not in drop]
        elif op == 2:
            a, r = int(rng.integers(0, 12)), int(rng.integers(1, 9))
            try:
                ref.load(a, r)
            except (opool.OracleOOM, opool.OracleInvalid) as ex:
                with pytest.raises(S.SloraError) as e:
                    pool.load(a, r)
                want = S.ERR_OOM if isinstance(ex, opool.OracleOOM) else S.ERR_EXISTS
                assert e.value.code == want
            else:
                pool.load(a, r)
                assert S.slora_adapter_pages(pool.handle, a).tolist() == ref.tables[a].tolist()
        else:
            a = int(rng.integers(0, 12))
            try:
                ref.evict(a)
            except opool.OracleInvalid:
                with pytest.raises(S.SloraError) as e:
                    S.slora_adapter_evict(pool.handle, a)
                assert e.value.code == S.ERR_NOT_RESIDENT
            else:
                S.slora_adapter_evict(pool.handle, a)
        if step % 50 == 0:
            _compare(pool.snapshot(), ref)
    _compare(pool.snapshot(), ref)
    pool.close()


def test_argument_validation(S):
    with pytest.raises(S.SloraError) as e:
        S.slora_pool_create(0, 0, 256, S.F16, 4, 16, 16, [256], [256])
    assert e.value.code == S.ERR_INVALID
    with pytest.raises(S.SloraError):
        S.slora_pool_create(0, 10, 100, S.F16, 4, 16, 16, [256], [256])      # H not a multiple of 8
    with pytest.raises(S.SloraError):
        S.slora_pool_create(0, 10, 256, S.F16, 4, 1000, 16, [256], [256])    # rank above the limit
    with pytest.raises(S.SloraError):
        S.slora_pool_create(0, 10, 256, S.F16, 4, 16, 16, [250], [256])      # dim not a multiple of 8
    h = S.slora_pool_create(0, 64, 256, S.F16, 4, 16, 16, [256], [256])
    with pytest.raises(S.SloraError) as e:
        S.slora_build_segments(h, 0, 0)                                      # planning pool: no GPU work
    assert e.value.code == S.ERR_INVALID
    seg = S.slora_segments()
    with pytest.raises(S.SloraError) as e:
        S.slora_lora_apply_bmm(h, seg, 0, 0, 256, 0, 256, 1.0)             # the comparator: GPU only
    assert e.value.code == S.ERR_INVALID
    assert S.slora_bmm_scratch_bytes(h) == 0
    with pytest.raises(S.SloraError) as e:
        S.slora_adapter_load(h, 4, 2, None, None)
    assert e.value.code == S.ERR_INVALID
    with pytest.raises(S.SloraError) as e:
        S.slora_adapter_load(h, 0, 17, None, None)
    assert e.value.code == S.ERR_INVALID
    S.slora_adapter_load(h, 0, 16, None, None)                               # 32 of 64 pages
    S.slora_adapter_load(h, 1, 15, None, None)                               # 30 more
    with pytest.raises(S.SloraError) as e:
        S.slora_adapter_load(h, 2, 2, None, None)                            # 4 > 2 free
    assert e.value.code == S.ERR_OOM
    with pytest.raises(S.SloraError) as e:
        S.slora_adapter_load(h, 1, 1, None, None)
    assert e.value.code == S.ERR_EXISTS
    assert S.slora_pool_info(h)["free_pages"] == 2
    S.slora_pool_destroy(h)


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with the shared library absent every call raises."""
    from lora_adapters_gb300 import slora

    monkeypatch.setattr(slora, "_lib", None)
    monkeypatch.setattr(slora, "LIB_PATH", str(tmp_path / "libslora.so"))
    with pytest.raises(ImportError):
        slora.slora_pool_create(0, 64, 256, slora.F16, 4, 16, 16, [256], [256])


def _snapshot_bytes(S, h):
    import ctypes

    n = ctypes.c_size_t()
    S.lib().slora_pool_snapshot(h, None, ctypes.byref(n))
    buf = np.zeros(n.value, np.uint8)
    assert S.lib().slora_pool_snapshot(h, buf.ctypes.data, ctypes.byref(n)) == S.OK
    return buf


def test_injected_page_allocation_failure_changes_nothing(S):
    """SLORA_FAULT_PAGE_ALLOC: the nth page-taking call fails with OOM as if
    the pool were full, the allocator state stays byte for byte as before, and
    the fault fires once."""
    h = S.slora_pool_create(0, 200, 64, S.F16, 8, 8, 16, [64, 128], [128, 64])
    S.slora_adapter_load(h, 0, 4, None, None)
    S.slora_debug_set_fault(h, S.FAULT_PAGE_ALLOC, 3)
    S.slora_pages_alloc(h, 5)                                   # event 1
    S.slora_adapter_load(h, 1, 2, None, None)                   # event 2
    before = _snapshot_bytes(S, h)
    with pytest.raises(S.SloraError) as e:                      # event 3: fails
        S.slora_adapter_load(h, 2, 3, None, None)
    assert e.value.code == S.ERR_OOM and "injected" in str(e.value)
    assert np.array_equal(_snapshot_bytes(S, h), before)
    S.slora_adapter_load(h, 2, 3, None, None)                   # disarmed: the same call succeeds
    S.slora_debug_set_fault(h, S.FAULT_PAGE_ALLOC, 1)
    before = _snapshot_bytes(S, h)
    with pytest.raises(S.SloraError) as e:
        S.slora_pages_alloc(h, 1)
    assert e.value.code == S.ERR_OOM
    assert np.array_equal(_snapshot_bytes(S, h), before)
    S.slora_debug_set_fault(h, S.FAULT_PAGE_ALLOC, 1)
    S.slora_debug_set_fault(h, S.FAULT_NONE, 0)                 # disarmed before it fires
    S.slora_pages_alloc(h, 1)
    for kind, nth in ((3, 1), (-1, 1), (S.FAULT_COPY, -2)):
        with pytest.raises(S.SloraError) as e:
            S.slora_debug_set_fault(h, kind, nth)
        assert e.value.code == S.ERR_INVALID
    S.slora_pool_destroy(h)


def test_fault_armed_from_the_environment():
    """SLORA_FAULT=alloc:2 arms the fault in every pool the process creates."""
    import subprocess
    import sys

    code = ("from lora_adapters_gb300 import slora as S\n"
            "h = S.slora_pool_create(0, 64, 64, S.F16, 4, 4, 4, [64], [64])\n"
            "S.slora_pages_alloc(h, 1)\n"
            "try:\n    S.slora_pages_alloc(h, 1)\nexcept S.SloraError as e:\n    print('code', e.code)\n")
    env = dict(os.environ, SLORA_FAULT="alloc:2")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert "code -2" in out.stdout
