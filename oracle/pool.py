"""Oracle of the unified page pool, adapter page tables and token segments.

TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's CPU leg
use this module.

Unified Paging ("S-LoRA: Serving Thousands of Concurrent LoRA Adapters",
nubint.ai review, abstract and method list; dongaigc.com summary, section 1
"unified paging"): one pool of fixed-size pages holds both the weights of
adapters of different ranks and the KV-cache slots of requests of different
lengths.  A page holds H elements, the size of one token's K (or V) vector
for one layer, so one adapter weight row of a hidden-size projection fills
exactly one page.  KV pages are taken when needed and returned when a request
ends (the PagedAttention description on the fatihsoysal.com page, section
"vLLM'in PagedAttention Mekanizmasi").

The pages fix no allocation policy; the reading used everywhere here is:
  * allocation always takes the n LOWEST-numbered free pages, in ascending
    order, all or nothing (too few free pages: nothing changes);
  * an adapter of rank r takes r * sum_q (ceil(h_in_q/H) + ceil(h_out_q/H))
    pages at load, listed in its page table in this order: for each
    projection q, the A rows k = 0..r-1 (each split into ceil(h_in_q/H)
    chunks), then the B rows k = 0..r-1 (ceil(h_out_q/H) chunks each); the
    i-th lowest page goes to the i-th entry;
  * evicting an adapter or freeing KV pages returns those pages at once.

Segments ("SGMV", segmented gather matrix-vector, in the cmlonder.com
newsletter, section "Iddia ve Gerceklik"): the tokens of one batch are grouped
by adapter so that each adapter's pages are read once.  Reading: a stable
sort of token indices by adapter id, ascending; tokens with id -1 carry no
adapter and are left out; one segment per distinct adapter id.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

FREE = -1
KV = -2


class OracleOOM(Exception):
    pass


class OracleInvalid(Exception):
    pass


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclasses.dataclass
class ProjDims:
    h_in: int
    h_out: int


class OraclePool:
    """Page allocator + page tables, replayable call by call."""

    def __init__(self, num_pages: int, H: int, projections: Sequence[Tuple[int, int]],
                 max_adapters: int, max_rank: int):
        self.num_pages = int(num_pages)
        self.H = int(H)
        self.proj = [ProjDims(int(i), int(o)) for i, o in projections]
        self.max_adapters = int(max_adapters)
        self.max_rank = int(max_rank)
        self.owner = np.full(self.num_pages, FREE, dtype=np.int32)
        self._free = np.arange(self.num_pages, dtype=np.int64)   # sorted ascending
        self.rank = np.zeros(self.max_adapters, dtype=np.int32)
        self.tables: Dict[int, np.ndarray] = {}
        self.kv_handles: Dict[str, np.ndarray] = {}

    # -- sizes ---------------------------------------------------------------
    def chunks_per_rank(self) -> int:
        """Page-table entries per unit of rank (all projections, A and B)."""
        return sum(_ceil_div(p.h_in, self.H) + _ceil_div(p.h_out, self.H) for p in self.proj)

    def adapter_pages(self, rank: int) -> int:
        return int(rank) * self.chunks_per_rank()

    @property
    def free_count(self) -> int:
        return int(self._free.shape[0])

    # -- allocation ----------------------------------------------------------
    def _take(self, n: int, owner: int) -> np.ndarray:
        if n > self._free.shape[0]:
            raise OracleOOM(f"need {n} pages, {self._free.shape[0]} free")
        pages = self._free[:n].copy()
        self._free = self._free[n:]
        self.owner[pages] = owner
        return pages

    def _give_back(self, pages: np.ndarray) -> None:
        # the freed pages are not in the free list: their union, kept sorted,
        # is the merge of two sorted runs (a stable sort finds and merges runs)
        self.owner[pages] = FREE
        self._free = np.sort(np.concatenate([self._free, np.sort(pages.astype(np.int64))]), kind="stable")

    def kv_alloc(self, n: int) -> np.ndarray:
        if n < 0:
            raise OracleInvalid("negative count")
        return self._take(int(n), KV)

    def kv_free(self, pages) -> None:
        pages = np.asarray(pages, dtype=np.int64)
        if pages.size == 0:
            return
        if (pages < 0).any() or (pages >= self.num_pages).any():
            raise OracleInvalid("page out of range")
        if np.unique(pages).size != pages.size:
            raise OracleInvalid("page listed twice")
        if (self.owner[pages] != KV).any():
            raise OracleInvalid("page is not a KV page")
        self._give_back(pages)

    def load(self, a: int, rank: int) -> np.ndarray:
        if not (0 <= a < self.max_adapters):
            raise OracleInvalid("adapter id out of range")
        if not (1 <= rank <= self.max_rank):
            raise OracleInvalid("rank out of range")
        if self.rank[a] != 0:
            raise OracleInvalid("adapter already resident")
        pages = self._take(self.adapter_pages(rank), a)
        self.rank[a] = rank
        self.tables[a] = pages.astype(np.int32)
        return self.tables[a]

    def evict(self, a: int) -> None:
        if not (0 <= a < self.max_adapters) or self.rank[a] == 0:
            raise OracleInvalid("adapter not resident")
        self._give_back(self.tables.pop(a).astype(np.int64))
        self.rank[a] = 0

    # -- replay of a workload's call sequence --------------------------------
    def replay(self, ops, ranks) -> None:
        for op in ops:
            if op[0] == "kv_alloc":
                self.kv_handles[op[1]] = self.kv_alloc(op[2])
            elif op[0] == "kv_free":
                h = self.kv_handles[op[1]]
                self.kv_free(h[np.asarray(op[2], dtype=np.int64)])
            elif op[0] == "load":
                self.load(op[1], int(ranks[op[1]]))
            elif op[0] == "evict":
                self.evict(op[1])
            else:
                raise ValueError(op)

    # -- page-table views ------------------------------------------------------
    def entry_of(self, a: int, p: int, which: str, k: int, c: int) -> int:
        """Index into adapter a's page table of chunk c of row k of A or B of projection p."""
        r = int(self.rank[a])
        before = sum(_ceil_div(q.h_in, self.H) + _ceil_div(q.h_out, self.H) for q in self.proj[:p])
        ppi = _ceil_div(self.proj[p].h_in, self.H)
        ppo = _ceil_div(self.proj[p].h_out, self.H)
        base = r * before
        if which == "A":
            return base + k * ppi + c
        return base + r * ppi + k * ppo + c

    def flat_tables(self, stride: Optional[int] = None):
        """(page_table int32[], pt_off int64[max_adapters]) with adapter a at a*stride.

        stride defaults to max_rank * chunks_per_rank(), a fixed region per
        adapter id; unused entries are -1.
        """
        stride = stride if stride is not None else self.max_rank * self.chunks_per_rank()
        pt = np.full(self.max_adapters * stride, -1, dtype=np.int32)
        for a, tab in self.tables.items():
            pt[a * stride: a * stride + tab.shape[0]] = tab
        pt_off = np.arange(self.max_adapters, dtype=np.int64) * stride
        return pt, pt_off


class OracleStore:
    """The oracle's own copy of pool contents, kept only for pages that hold adapter rows.

    ``page_slot[page]`` is the row of ``data`` that holds that page's H
    elements (-1: no contents kept).  Writing an adapter places each weight
    row chunk on the page its page-table entry names (the "load" step: the
    adapter rows copied from host memory into their pool pages).
    """

    def __init__(self, num_pages: int, H: int):
        self.H = int(H)
        self.page_slot = np.full(int(num_pages), -1, dtype=np.int64)
        self._chunks: List[np.ndarray] = []
        self._n = 0
        self._data: Optional[np.ndarray] = None

    def write_adapter(self, pool: OraclePool, a: int, weights, only=None) -> None:
        """Place adapter a's rows on its pages.  ``only``: the projections to
        write (all if None); the others' pages keep no contents, so a check
        of one layer of a many-layer pool stores only that layer's rows."""
        r = int(pool.rank[a])
        H = self.H
        table = pool.tables[a].astype(np.int64)
        entry = 0
        for p, (A, B) in enumerate(weights):
            for M, dim in ((A, pool.proj[p].h_in), (B, pool.proj[p].h_out)):
                pp = _ceil_div(dim, H)
                if only is None or p in only:
                    assert M.shape == (r, dim), (M.shape, r, dim)
                    padded = np.zeros((r, pp * H), dtype=np.uint16)   # tail of the last page: zeros
                    padded[:, :dim] = M
                    chunks = padded.reshape(r * pp, H)
                    self.page_slot[table[entry:entry + r * pp]] = np.arange(self._n, self._n + r * pp)
                    self._chunks.append(chunks)
                    self._n += r * pp
                entry += r * pp
        assert entry == table.shape[0]
        self._data = None

    @property
    def data(self) -> np.ndarray:
        if self._data is None:
            self._data = (np.concatenate(self._chunks, axis=0) if self._chunks
                          else np.zeros((1, self.H), dtype=np.uint16))
        return self._data

    def page(self, page: int) -> np.ndarray:
        s = self.page_slot[page]
        assert s >= 0
        return self.data[s]


@dataclasses.dataclass
class Segments:
    perm: np.ndarray          # int32[n_sorted]: token indices, stably sorted by adapter
    seg_start: np.ndarray     # int32[num_segs + 1]
    seg_adapter: np.ndarray   # int32[num_segs]
    bad_tokens: int           # tokens naming an adapter that is not resident

    @property
    def num_segs(self) -> int:
        return int(self.seg_adapter.shape[0])


def build_segments(token_adapter, rank) -> Segments:
    """Group the batch's tokens by adapter (stable, ascending id; see module doc).

    Tokens with id -1 are skipped.  Tokens naming an id that is out of range
    (below -1 or past the last adapter) or not resident (rank 0) are skipped
    too and counted in ``bad_tokens``.
    """
    ta = [int(v) for v in np.asarray(token_adapter)]
    rank = np.asarray(rank)
    keep, bad = [], 0
    for i, a in enumerate(ta):
        if a == -1:
            continue
        if a < 0 or a >= rank.shape[0] or rank[a] <= 0:
            bad += 1
            continue
        keep.append(i)
    perm = sorted(keep, key=lambda i: ta[i])           # Python's sort is stable
    seg_start, seg_adapter = [], []
    for j, i in enumerate(perm):
        if j == 0 or ta[i] != ta[perm[j - 1]]:
            seg_start.append(j)
            seg_adapter.append(ta[i])
    seg_start.append(len(perm))
    return Segments(np.asarray(perm, dtype=np.int32), np.asarray(seg_start, dtype=np.int32),
                    np.asarray(seg_adapter, dtype=np.int32), bad)
