"""The allocation-free entry point, slora_lora_apply_noalloc.

It serves callers that cannot call cudaMalloc where they compute the LoRA
delta: a serving runtime whose own arena already holds all GPU memory (page
pool, KV cache, activations) and may not grow, or code that must not allocate
while it serves.  Every buffer is the caller's; the scratch lives in one
static device array that all calls share.  Its output is checked against the
CPU oracle on calls made back to back (the second call reuses the scratch the
first left behind), and its documented treatment of bad input -- ranks it
cannot use count as "not resident", such tokens and base-only tokens keep
their rows bit for bit, the call's status names the error -- is checked too.

This file is named so that pytest collects it last.
"""
import copy

import numpy as np
import pytest
import torch

from lora_adapters_gb300 import workloads
from oracle import lora as olora
from tests import helpers as H


def _lib():
    from lora_adapters_gb300 import build, slora

    build.build()
    slora.lib()
    return slora


def test_noalloc_rejects_batches_above_its_scratch():
    S = _lib()
    with pytest.raises(S.SloraError) as e:
        S.slora_lora_apply_noalloc(16, 256, S.F16, 16, 64, 16, 4, [256], [256], 0, 16,
                                   S.NOALLOC_MAX_TOKENS + 1, 16, 256, 16, 256, 1.0)
    assert e.value.code == S.ERR_INVALID


CASES = {
    "tiny_f16": workloads.spec("tiny"),
    "mlp_multi_page_bf16": workloads.WorkloadSpec(
        name="mlp_multi_page", H=256, dtype="bf16",
        projections=(workloads.Projection("gate", 256, 1384), workloads.Projection("down", 1384, 256)),
        num_adapters=23, rank_set=(3, 16, 64), kind="decode", tokens=1500, popularity="zipf",
        zipf_alpha=1.1, pool_factor=1.3, s=0.75, seed=4),
}


class _Caller:
    """A caller that owns every buffer: the pool's pages, its page table and
    ranks (copied out of a pool that laid the adapters out), x, y, status."""

    def __init__(self, S, wl):
        from tests import gpu_setup as G

        self.S, self.G, self.wl = S, G, wl
        self.case = G.build_case(wl)
        snap = self.case.pool.snapshot()
        self.pt = torch.from_numpy(np.ascontiguousarray(snap["page_table"])).cuda()
        self.rank_host = np.ascontiguousarray(snap["rank"]).copy()
        self.stride = int(snap["page_table"].shape[1])
        self.dt = S.F16 if wl.spec.dtype == "f16" else S.BF16
        self.store = H.oracle_store_for(wl, self.case.oracle_pool, self.case.touched)

    def apply(self, p, ta_host, rank_host=None, status=None):
        """One call of the entry point on projection p; returns y (16-bit patterns)."""
        wl, G = self.wl, self.G
        rank = torch.from_numpy(self.rank_host if rank_host is None else rank_host).cuda()
        ta = torch.from_numpy(np.ascontiguousarray(ta_host, dtype=np.int32)).cuda()
        y = G.to_dev(wl.y_in(p), wl.spec.dtype)
        x = self.case.xs[p]
        self.S.slora_lora_apply_noalloc(
            self.case.pool.buffer.data_ptr(), wl.H, self.dt, self.pt.data_ptr(), self.stride,
            rank.data_ptr(), wl.spec.num_adapters, [q.h_in for q in wl.projections],
            [q.h_out for q in wl.projections], p, ta.data_ptr(), int(ta.numel()), x.data_ptr(), x.stride(0),
            y.data_ptr(), y.stride(0), wl.spec.s, torch.cuda.current_stream().cuda_stream,
            0 if status is None else status.data_ptr())
        torch.cuda.synchronize()
        return G.to_bits(y)

    def oracle(self, p, ta_host, rank_host=None):
        """The oracle's y for the same call; `rank_host` as the entry point
        reads it (ranks it cannot use given as 0)."""
        wl = self.wl
        pool = self.case.oracle_pool
        if rank_host is not None:
            pool = copy.copy(pool)
            pool.rank = np.asarray(rank_host, dtype=np.int32)
        y, _, _ = olora.apply(self.store, pool, p, np.asarray(ta_host, dtype=np.int32), wl.x(p), wl.y_in(p),
                              wl.spec.s, wl.spec.dtype, num_threads=olora.default_threads(), on_bad="keep")
        return y


def _assert_close(got, want, dtype, what):
    ok = H.within_tol(H.lib_values(got, dtype), H.lib_values(want, dtype))
    assert ok.all(), f"{what}: {(~ok).sum()} elements out of tolerance"


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_on_two_calls_in_a_row(name):
    S = _lib()
    wl = workloads.make(CASES[name])
    c = _Caller(S, wl)
    rng = np.random.default_rng(1)
    # the second batch is a shuffled copy of the first (the scratch the first
    # call left behind must not leak into it); status in device memory for the
    # first call, pinned host memory for the second
    batches = [wl.token_adapter, wl.token_adapter[rng.permutation(wl.T)]]
    statuses = [torch.full((1,), 12345, dtype=torch.int32, device="cuda"),
                torch.full((1,), 12345, dtype=torch.int32).pin_memory()]
    for call, (ta, st) in enumerate(zip(batches, statuses)):
        for p in range(len(wl.projections)):
            st.fill_(12345)
            got = c.apply(p, ta, status=st)
            assert int(st.cpu()[0]) == S.OK, f"call {call}, projection {p}: status {int(st.cpu()[0])}"
            want = c.oracle(p, ta)
            _assert_close(got, want, wl.spec.dtype, f"call {call}, projection {p}")
            assert not np.array_equal(got, wl.y_in(p))          # the delta was applied
    c.case.pool.close()


@pytest.mark.gpu
def test_noalloc_bad_ranks_and_ids_leave_rows_unchanged():
    """Ranks 0, -3, one past what the page-table stride holds, and 300 count
    as "not resident"; tokens on those adapters, base-only tokens (-1) and an
    id past the last adapter keep their rows bit for bit; the other rows match
    the oracle; the status names the error (NOT_RESIDENT for the ranks,
    INVALID for the id)."""
    S = _lib()
    wl = workloads.make(CASES["mlp_multi_page_bf16"])
    c = _Caller(S, wl)
    touched = c.case.touched
    assert len(touched) >= 5
    rmax = c.stride // c.case.oracle_pool.chunks_per_rank()
    bad_rank = c.rank_host.copy()
    for a, r in zip(touched[:4], (0, -3, rmax + 1, 300)):
        bad_rank[a] = r
    eff_rank = bad_rank.copy()
    eff_rank[(eff_rank < 1) | (eff_rank > rmax)] = 0          # as the entry point reads them
    ta = wl.token_adapter.copy()
    ta[::7] = -1
    dt = wl.spec.dtype
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for p in range(len(wl.projections)):
        y0 = wl.y_in(p)
        # ranks it cannot use
        got = c.apply(p, ta, rank_host=bad_rank, status=status)
        assert int(status.cpu()[0]) == S.ERR_NOT_RESIDENT
        keep = (ta == -1) | np.isin(ta, touched[:4])
        assert keep.sum() > 0 and (~keep).sum() > 0
        assert np.array_equal(got[keep], y0[keep])
        want = c.oracle(p, ta, rank_host=eff_rank)
        _assert_close(got[~keep], want[~keep], dt, f"projection {p}, bad ranks")
        # an id past the last adapter
        ta2 = ta.copy()
        ta2[3] = wl.spec.num_adapters
        got = c.apply(p, ta2, status=status)
        assert int(status.cpu()[0]) == S.ERR_INVALID
        keep2 = (ta2 == -1) | (np.arange(wl.T) == 3)
        assert np.array_equal(got[keep2], y0[keep2])
        want = c.oracle(p, ta2)
        _assert_close(got[~keep2], want[~keep2], dt, f"projection {p}, bad id")
    # an empty batch reports OK and touches nothing
    status.fill_(12345)
    c.apply(0, np.zeros(0, dtype=np.int32), status=status)
    assert int(status.cpu()[0]) == S.OK
    c.case.pool.close()
