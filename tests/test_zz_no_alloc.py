"""The allocation-free entry point, slora_lora_apply_noalloc.

It serves callers that cannot call cudaMalloc where they compute the LoRA
delta (a runtime whose arena already holds all GPU memory, code that must not
allocate while serving): every buffer is theirs, and the scratch lives in one
static device array.  Its output must match the pool entry point's output on
the same batch, within the parity tolerance, on calls made back to back (the
second call reuses the scratch the first one left behind).

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from lora_adapters_gb300 import workloads
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


def _device_tables(pool):
    snap = pool.snapshot()
    pt = torch.from_numpy(np.ascontiguousarray(snap["page_table"])).cuda()
    rank = torch.from_numpy(np.ascontiguousarray(snap["rank"])).cuda()
    return pt, rank, int(snap["page_table"].shape[1])


CASES = {
    "tiny_f16": workloads.spec("tiny"),
    "mlp_multi_page_bf16": workloads.WorkloadSpec(
        name="mlp_multi_page", H=256, dtype="bf16",
        projections=(workloads.Projection("gate", 256, 1384), workloads.Projection("down", 1384, 256)),
        num_adapters=23, rank_set=(3, 16, 64), kind="decode", tokens=1500, popularity="zipf",
        zipf_alpha=1.1, pool_factor=1.3, s=0.75, seed=4),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_pool_entry_point_twice(name):
    S = _lib()
    from tests import gpu_setup as G

    wl = workloads.make(CASES[name])
    case = G.build_case(wl)
    pool = case.pool
    pt, rank, stride = _device_tables(pool)
    proj_in = [p.h_in for p in wl.projections]
    proj_out = [p.h_out for p in wl.projections]
    dt = S.F16 if wl.spec.dtype == "f16" else S.BF16
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(1)
    # two calls back to back; the second batch is a shuffled copy of the first
    batches = [wl.token_adapter, wl.token_adapter[rng.permutation(wl.T)]]
    for call, ta_host in enumerate(batches):
        ta = torch.from_numpy(np.ascontiguousarray(ta_host)).cuda()
        for p in range(len(wl.projections)):
            y0 = G.to_dev(wl.y_in(p), wl.spec.dtype)
            # existing entry point
            y_ref = y0.clone()
            seg = pool.build_segments(ta)
            pool.apply(seg, p, case.xs[p], y_ref, wl.spec.s, S.MODE_DECODE)
            # allocation-free entry point
            y_na = y0.clone()
            S.slora_lora_apply_noalloc(pool.buffer.data_ptr(), wl.H, dt, pt.data_ptr(), stride,
                                       rank.data_ptr(), wl.spec.num_adapters, proj_in, proj_out, p,
                                       ta.data_ptr(), wl.T, case.xs[p].data_ptr(), case.xs[p].stride(0),
                                       y_na.data_ptr(), y_na.stride(0), wl.spec.s, stream)
            torch.cuda.synchronize()
            got, want = G.to_bits(y_na), G.to_bits(y_ref)
            ok = H.within_tol(H.lib_values(got, wl.spec.dtype), H.lib_values(want, wl.spec.dtype))
            assert ok.all(), f"call {call}, projection {p}: {(~ok).sum()} elements differ"
            assert not np.array_equal(got, G.to_bits(y0))        # the delta was applied
    pool.close()
