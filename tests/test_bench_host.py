"""Host-side arithmetic of the benchmark: the roofline numerator.

The algorithmic bytes of a step are x and the adapter's A rows read once per
projection and segment, y read and written once and the B rows read once;
these tests check the split by kernel against closed forms for batches whose
answer is obvious, not against the same loop written again.
"""
import dataclasses
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from lora_adapters_gb300 import workloads  # noqa: E402


@dataclasses.dataclass
class _Wl:
    token_adapter: np.ndarray
    ranks: np.ndarray
    projections: tuple


P = workloads.Projection


def test_one_adapter_is_one_gemm_chain():
    # T tokens on one adapter of rank r, one projection H_in -> H_out, 16-bit:
    # x (T H_in) + A (r H_in) + y in and out (2 T H_out) + B (r H_out)
    T, r, hi, ho = 300, 24, 1000, 1384
    wl = _Wl(np.zeros(T, np.int32), np.array([r]), (P("q", hi, ho),))
    ab = bench.algorithmic_bytes(wl)
    assert ab["shrink_cc"] == 2 * (T * hi + r * hi)
    assert ab["expand_cc"] == 2 * (2 * T * ho + r * ho)
    assert ab["step"] == ab["apply_cc"] == ab["shrink_cc"] + ab["expand_cc"]
    assert ab["distinct_adapters"] == 1 and ab["tokens"] == T


def test_base_only_tokens_cost_nothing_and_threshold_splits_paths():
    # adapter 0: 100 tokens (tensor cores at threshold 64), adapter 1: 10
    # tokens (CUDA cores), 7 base-model-only tokens (no bytes at all)
    ta = np.array([0] * 100 + [1] * 10 + [-1] * 7, np.int32)
    wl = _Wl(ta, np.array([8, 16]), (P("a", 64, 128), P("b", 128, 64)))
    ab = bench.algorithmic_bytes(wl, tc_threshold=64)
    per = lambda n, r: sum(2 * (n + r) * p.h_in + 2 * (2 * n + r) * p.h_out for p in wl.projections)  # noqa: E731
    assert ab["shrink_tc"] + ab["expand_tc"] == per(100, 8)
    assert ab["shrink_cc"] + ab["expand_cc"] == per(10, 16)
    assert ab["step"] == per(100, 8) + per(10, 16)
    assert ab["tokens"] == 110
    # with every segment on the CUDA cores the total is the same
    assert bench.algorithmic_bytes(wl)["step"] == ab["step"]


def test_decode_workload_bytes_are_dominated_by_adapter_rows():
    # the benchmark workload: 256 tokens over about 130 distinct adapters;
    # x and y are 3 x 256 x 4096 x 2 bytes per projection, the rest is rows
    wl = workloads.make("llama7b_decode")
    ab = bench.algorithmic_bytes(wl)
    xy = 4 * 3 * 256 * 4096 * 2
    rows = ab["step"] - xy
    assert 0 < xy < rows
    distinct_ranks = sum(int(wl.ranks[a]) for a in np.unique(wl.token_adapter[wl.token_adapter >= 0]))
    assert rows == 4 * 2 * 4096 * 2 * distinct_ranks


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    d = tmp_path / "lora_adapters_gb300" / "csrc"
    d.mkdir(parents=True)
    for f in ("kernels.cu", "tc_kernels.cu", "internal.h"):
        (d / f).write_text("int a = 1;  // one\n/* block\n comment */ int b;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._kernel_source_hash()
    (d / "kernels.cu").write_text("int a = 1;  // a different comment\nint b;\n")
    assert bench._kernel_source_hash() == h0
    (d / "kernels.cu").write_text("int a = 2;\nint b;\n")
    assert bench._kernel_source_hash() != h0


def test_staging_layout_aligns_and_separates_the_pieces():
    sizes = [4 * 301, 2 * 256 * 5120, 2 * 512 * 13824, 2, 0, 2 * 7 * 33]
    offs, total = bench.staging_layout(sizes)
    assert offs[0] == 0 and all(o % 256 == 0 for o in offs)
    ends = [o + n for o, n in zip(offs, sizes)]
    assert all(e <= o2 for e, o2 in zip(ends, offs[1:]))        # no overlap, in order
    assert total >= ends[-1] and total - ends[-1] < 256 and total % 256 == 0


@pytest.mark.parametrize("n,chunk", [(0, 32), (1, 32), (32, 32), (33, 32), (58198016, 32 << 20), (100, 7)])
def test_copy_spans_cover_every_byte_once(n, chunk):
    spans = bench.copy_spans(n, chunk)
    assert all(0 < m <= chunk for _, m in spans)
    assert [c for c, _ in spans] == list(range(0, n, chunk))
    assert sum(m for _, m in spans) == n
    assert len(spans) == -(-n // chunk)
