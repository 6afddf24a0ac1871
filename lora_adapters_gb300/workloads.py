"""Seeded synthetic workloads for the heterogeneous-batch LoRA delta.

This module only DRAWS inputs: token-to-adapter assignments, adapter ranks,
activations, adapter weights and the page-pool call sequence that scatters
adapter rows across the pool.  It holds none of the method's arithmetic (no
LoRA product, no page-table layout, no allocation policy), so both the CPU
oracle and the CUDA path can take their inputs from here without sharing any
of the computation they are checked on.

Shapes follow the S-LoRA workloads: a Llama-7B-shaped attention layer (q, k,
v, o projections, H = 4096) for decode and prefill, and a Llama-13B-shaped MLP
(gate/up 5120 -> 13824, down 13824 -> 5120) for decode
("S-LoRA: Serving Thousands of Concurrent LoRA Adapters", abstract: thousands
of adapters with different ranks served from one GPU; the rank mix r = 8, 16,
64 is the one the cmlonder.com newsletter names under "Iddia ve Gerceklik").

Value distributions: x ~ N(0, 1), y_in ~ N(0, 1) (stands in for the base
projection's output), A ~ N(0, 1/H_in), B ~ N(0, 1/r), each rounded once to
the storage type (fp16 or bf16) by torch's round-to-nearest-even conversion.
16-bit values are carried as uint16 bit patterns because numpy has no bf16.

Every stream is derived from ``numpy.random.SeedSequence(seed)`` with a fixed
spawn key, so a draw never depends on which other draws were made before it:
  (0,)      token -> adapter assignment       (1,)      adapter ranks
  (2, p)    x of projection p                 (3, p)    y_in of projection p
  (4, a)    A rows of adapter a (all proj.)   (5, a)    B rows of adapter a
  (6,)      pool fragmentation churn          (7,)      reserved (traces)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

F16 = "f16"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class Projection:
    name: str
    h_in: int
    h_out: int


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and structure of one synthetic batch (see the module docstring)."""

    name: str
    H: int                                  # hidden size = page size in elements
    dtype: str                              # F16 or BF16
    projections: Tuple[Projection, ...]
    num_adapters: int                       # adapters resident in the pool
    rank_set: Tuple[int, ...]               # ranks drawn uniformly from this set
    # token -> adapter structure
    kind: str                               # "decode" (1 token / request) or "prefill"
    tokens: int = 0                         # decode: tokens in the batch
    requests: int = 0                       # prefill: requests in the batch
    prompt_len: Tuple[int, int] = (8, 512)  # prefill: uniform prompt length range
    popularity: str = "uniform"             # "uniform" or "zipf"
    zipf_alpha: float = 1.0
    fixed_ranks: Optional[Tuple[int, ...]] = None   # overrides rank_set if given
    # pool sizing
    pool_pages: Optional[int] = None        # exact page count, or
    pool_factor: float = 1.25               # pages = factor * adapter pages
    pool_bytes: Optional[int] = None        # or pages = bytes // (H * 2)
    free_fraction_left: float = 0.5         # of non-adapter pages left free after churn
    s: float = 1.0
    seed: int = 0


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _qkvo(h: int) -> Tuple[Projection, ...]:
    return tuple(Projection(n, h, h) for n in ("q", "k", "v", "o"))


# The five workloads.  The first four are batches of one layer; the mixed
# serving trace is built from the 7B decode/prefill shapes by the trace driver.
SPECS: Dict[str, WorkloadSpec] = {
    "tiny": WorkloadSpec(
        name="tiny", H=256, dtype=F16,
        projections=(Projection("q", 256, 256),),
        num_adapters=4, rank_set=(4, 8, 16), fixed_ranks=(4, 8, 8, 16),
        kind="decode", tokens=16, popularity="uniform",
        pool_pages=256, s=1.0),
    "llama7b_decode": WorkloadSpec(
        name="llama7b_decode", H=4096, dtype=F16, projections=_qkvo(4096),
        num_adapters=1000, rank_set=(8, 16, 32, 64),
        kind="decode", tokens=256, popularity="zipf", zipf_alpha=1.0,
        pool_factor=1.25),
    "llama7b_prefill": WorkloadSpec(
        name="llama7b_prefill", H=4096, dtype=F16, projections=_qkvo(4096),
        num_adapters=200, rank_set=(8, 16, 32, 64, 128),
        kind="prefill", requests=32, prompt_len=(8, 512), popularity="uniform",
        pool_factor=1.25),
    "llama13b_mlp_decode": WorkloadSpec(
        name="llama13b_mlp_decode", H=5120, dtype=BF16,
        projections=(Projection("gate", 5120, 13824), Projection("up", 5120, 13824),
                     Projection("down", 13824, 5120)),
        num_adapters=2000, rank_set=(16, 32, 64),
        kind="decode", tokens=512, popularity="zipf", zipf_alpha=1.2,
        pool_bytes=120_000_000_000, free_fraction_left=0.0),
}


def spec(name: str, **overrides) -> WorkloadSpec:
    """A named workload, optionally with fields replaced (smaller test cases)."""
    return dataclasses.replace(SPECS[name], **overrides)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=tuple(key)))


def _to_bits(values_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 draws to the storage type; return the uint16 bit patterns."""
    import torch  # conversion only (round-to-nearest-even), no method arithmetic

    t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32))
    t = t.to(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def pages_per_row(length: int, H: int) -> int:
    """Pages one weight row of ``length`` elements spans (the tail is padding)."""
    return _ceil_div(length, H)


@dataclasses.dataclass
class Workload:
    """One seeded batch: assignments, ranks, pool call sequence, and lazy values."""

    spec: WorkloadSpec
    ranks: np.ndarray                 # int32[num_adapters]
    token_adapter: np.ndarray         # int32[T]; -1 = base model only
    request_lens: Optional[np.ndarray]
    pool_pages: int
    pool_ops: List[tuple]             # replayed by every allocator under test

    @property
    def T(self) -> int:
        return int(self.token_adapter.shape[0])

    @property
    def H(self) -> int:
        return self.spec.H

    @property
    def projections(self) -> Tuple[Projection, ...]:
        return self.spec.projections

    def x(self, p: int) -> np.ndarray:
        """uint16[T, h_in] bit patterns of x for projection p, N(0, 1)."""
        pr = self.projections[p]
        v = _rng(self.spec.seed, 2, p).standard_normal((self.T, pr.h_in), dtype=np.float32)
        return _to_bits(v, self.spec.dtype)

    def y_in(self, p: int) -> np.ndarray:
        """uint16[T, h_out] bit patterns of the base output y for projection p."""
        pr = self.projections[p]
        v = _rng(self.spec.seed, 3, p).standard_normal((self.T, pr.h_out), dtype=np.float32)
        return _to_bits(v, self.spec.dtype)

    def adapter(self, a: int) -> List[Tuple[np.ndarray, np.ndarray]]:
        """Per projection: (A rows uint16[r, h_in], B rows uint16[r, h_out]).

        Row k of the A block is column k of the H_in x r matrix A (one row per
        rank index, contiguous along the hidden dimension); row k of the B
        block is row k of the r x H_out matrix B.
        """
        r = int(self.ranks[a])
        ga = _rng(self.spec.seed, 4, a)
        gb = _rng(self.spec.seed, 5, a)
        out = []
        for pr in self.projections:
            A = ga.standard_normal((r, pr.h_in), dtype=np.float32) * np.float32(1.0 / math.sqrt(pr.h_in))
            B = gb.standard_normal((r, pr.h_out), dtype=np.float32) * np.float32(1.0 / math.sqrt(r))
            out.append((_to_bits(A, self.spec.dtype), _to_bits(B, self.spec.dtype)))
        return out


def adapter_page_count(rank: int, projections: Sequence[Projection], H: int) -> int:
    """Pages an adapter of this rank occupies: r rows of A and r rows of B per projection."""
    return sum(rank * (pages_per_row(p.h_in, H) + pages_per_row(p.h_out, H)) for p in projections)


def make(name_or_spec, **overrides) -> Workload:
    """Draw the workload named ``name_or_spec`` (or given as a spec)."""
    sp = name_or_spec if isinstance(name_or_spec, WorkloadSpec) else spec(name_or_spec, **overrides)
    if isinstance(name_or_spec, WorkloadSpec) and overrides:
        sp = dataclasses.replace(sp, **overrides)
    N = sp.num_adapters

    # adapter ranks (stream 1)
    if sp.fixed_ranks is not None:
        ranks = np.asarray(sp.fixed_ranks, dtype=np.int32)
        assert ranks.shape[0] == N
    else:
        ranks = _rng(sp.seed, 1).choice(np.asarray(sp.rank_set, dtype=np.int32), size=N)
        ranks = ranks.astype(np.int32)

    # token -> adapter (stream 0)
    g = _rng(sp.seed, 0)
    request_lens = None
    if sp.kind == "decode":
        if sp.popularity == "zipf":
            k = np.arange(1, N + 1, dtype=np.float64)
            prob = k ** (-sp.zipf_alpha)
            prob /= prob.sum()
            ta = g.choice(N, size=sp.tokens, p=prob)
        else:
            ta = g.integers(0, N, size=sp.tokens)
    elif sp.kind == "prefill":
        lo, hi = sp.prompt_len
        request_lens = g.integers(lo, hi + 1, size=sp.requests)
        req_adapter = g.integers(0, N, size=sp.requests)
        ta = np.repeat(req_adapter, request_lens)
    else:
        raise ValueError(sp.kind)
    token_adapter = np.ascontiguousarray(ta, dtype=np.int32)

    # pool size and fragmentation churn (stream 6)
    total = sum(adapter_page_count(int(r), sp.projections, sp.H) for r in ranks)
    if sp.pool_pages is not None:
        pool_pages = int(sp.pool_pages)
    elif sp.pool_bytes is not None:
        pool_pages = int(sp.pool_bytes // (sp.H * 2))
    else:
        pool_pages = int(math.ceil(sp.pool_factor * total))
    if pool_pages < total:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {total} adapter pages")
    gf = _rng(sp.seed, 6)
    if sp.name == "tiny":
        n_free = pool_pages // 2
    else:
        n_free = total + int(sp.free_fraction_left * (pool_pages - total))
    # Fill the whole pool with KV slots, then release a random subset: the
    # adapters loaded next land on scattered pages between live KV slots.
    # Positions index into the list the allocation returned, so the sequence
    # does not depend on which page numbers an allocator hands out.
    free_pos = np.sort(gf.choice(pool_pages, size=n_free, replace=False)).astype(np.int64)
    ops: List[tuple] = [("kv_alloc", "kv0", pool_pages), ("kv_free", "kv0", free_pos)]
    ops += [("load", a) for a in range(N)]
    return Workload(sp, ranks, token_adapter, request_lens, pool_pages, ops)


def zipf_probabilities(N: int, alpha: float) -> np.ndarray:
    k = np.arange(1, N + 1, dtype=np.float64)
    p = k ** (-alpha)
    return p / p.sum()
