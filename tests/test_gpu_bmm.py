"""GPU parity of the padded batched-matmul comparator (slora_lora_apply_bmm).

The comparator computes the same delta as the paged kernels, by the
"traditional batched matmul" variant the pages compare S-LoRA with: every
token's adapter rows gathered into dense tensors padded to one rank, then
batched GEMMs.  It must meet the same bar against the oracle:
|gpu - oracle| <= 5e-3 + 1e-2 |oracle| elementwise.
"""
import numpy as np
import pytest
import torch

from lora_adapters_gb300 import slora, workloads
from tests import gpu_setup as G
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from lora_adapters_gb300 import build

    build.build()


def _run_bmm(case, rows=None, want=None, scale=None):
    wl = case.wl
    seg = case.pool.build_segments(case.ta_dev)
    for p in range(len(wl.projections)):
        case.pool.apply_bmm(seg, p, case.xs[p], case.ys[p], wl.spec.s)
    torch.cuda.synchronize()
    assert case.pool.status() == slora.OK
    want = want if want is not None else G.oracle_outputs(case, tokens=rows, adapter_scale=scale)
    for p in range(len(wl.projections)):
        ok, err, bad = G.compare(G.to_bits(case.ys[p]), want[p], wl.spec.dtype, rows=rows)
        assert ok, f"projection {p}: {bad} elements out of tolerance, max |err| {err}"


@pytest.mark.parametrize("name", ["tiny", "tiny_bf16", "mlp_ragged_bf16", "prefill_ragged_f16", "short_k_f16",
                                  "prefill_bigrank_f16"])
def test_bmm_comparator_small_cases(name):
    wl = workloads.make(SMALL[name])
    case = G.build_case(wl)
    _run_bmm(case)
    assert slora.slora_bmm_scratch_bytes(case.pool.handle) > 0
    case.pool.close()


def test_bmm_comparator_per_adapter_scale():
    wl = workloads.make(SMALL["mlp_ragged_bf16"])
    case = G.build_case(wl)
    rng = np.random.default_rng(29)
    scale = np.ones(case.oracle_pool.max_adapters)
    for a in case.touched:
        scale[a] = float(np.float32(rng.uniform(-1.0, 2.0)))
        case.pool.set_scale(a, scale[a])
    _run_bmm(case, scale=scale)
    case.pool.close()


def test_bmm_comparator_full_size_llama7b_decode_every_row():
    """The 7B decode batch (H=4096, q/k/v/o, 256 tokens, 1000 adapters): every row."""
    wl = workloads.make("llama7b_decode")
    case = G.build_case(wl, weights="touched")
    _run_bmm(case)
    case.pool.close()
