"""Serving-trace driver: continuous batching over the unified page pool.

The pages describe S-LoRA as a serving system in which adapter weights and
KV-cache tensors share one paged memory pool, adapters live in host memory and
are fetched on demand when a request needs one, and every step batches the
tokens of many requests on many adapters ("S-LoRA: Serving Thousands of
Concurrent LoRA Adapters": the nubint.ai review's method list -- unified
paging, host-memory adapter store, on-demand loading; the dongaigc.com
summary, section 1 "unified paging"; the scheduler loop of the continuous-
batching page, "vLLM Zamanlayicisi").  This module drives the library through
such a trace for one decoder layer's share of memory and compute:

* requests arrive (Poisson per step), each with a prompt length, an output
  length and an adapter drawn Zipf-like from a large host store;
* every step has a token budget: one decode token for each running request
  first, then prompt chunks of requests in prefill;
* KV pages (``kv_pages_per_token`` per token, for the request's whole length,
  taken when it is admitted) and adapter pages come from the same pool; when
  the adapter of one of the first ``prefetch_window`` waiting requests is not
  resident it is loaded asynchronously, evicting least-recently-used adapters
  that no running request holds; a request joins the batch once its adapter
  was loaded in an earlier step;
* each step runs the segment kernel and the apply for the layer's
  projections on the step's tokens (AUTO mode: long prompt chunks on the
  tensor cores).

Every pool call is logged (``TraceResult.ops``) in the form the oracle's
allocator replays, so a test can rebuild the pool state independently and
check a step's outputs.  With ``device=None`` the trace runs on a planning
pool (host bookkeeping only, no GPU work), which the CPU tests use.
"""
from __future__ import annotations

import collections
import dataclasses
import time
from typing import Dict, List, Optional, Tuple

import numpy as np

from . import slora, workloads


@dataclasses.dataclass(frozen=True)
class TraceSpec:
    name: str = "serve_trace_7b"
    H: int = 4096
    dtype: str = "f16"
    projections: Tuple[workloads.Projection, ...] = workloads._qkvo(4096)
    num_adapters: int = 2000
    rank_set: Tuple[int, ...] = (8, 16, 32, 64)
    zipf_alpha: float = 1.0
    pool_bytes: int = 120 * 10**9 // 32      # one layer's share of a 120 GB pool
    kv_pages_per_token: int = 2              # this layer's K and V vectors
    token_budget: int = 1024
    max_running: int = 256                   # requests in the batch at once
    arrivals_per_step: float = 4.0
    prompt_len: Tuple[int, int] = (8, 512)
    output_len: Tuple[int, int] = (8, 128)   # with the 256-request cap, the 1024-token budget fills
    max_loads_per_step: int = 32
    prefetch_window: int = 64                # misses loaded only for the first waiting requests
    steps: int = 1000
    s: float = 0.01                          # y accumulates one delta per step
    seed: int = 0

    @property
    def pool_pages(self) -> int:
        return self.pool_bytes // (self.H * 2)


@dataclasses.dataclass
class Request:
    rid: int
    adapter: int
    prompt: int
    output: int
    prefilled: int = 0
    generated: int = 0
    kv_handles: List[str] = dataclasses.field(default_factory=list)
    admitted_step: int = -1
    arrived_step: int = 0
    missed: bool = False         # its adapter was not resident (or still loading) when it arrived


@dataclasses.dataclass
class TraceResult:
    steps: int
    tokens: int
    decode_tokens: int
    prefill_tokens: int
    gpu_ms: float                # kernel time of the path (segments + apply), from the pool's timing hooks
    step_event_ms: float         # the steps bracketed by events; includes the GPU's waits for the host
    load_kernel_ms: float        # the adapter loads' scatter kernels (copy stream, overlapping the steps)
    loads: int
    load_bytes: int
    evictions: int
    admitted: int                # requests admitted into the batch
    arrival_misses: int          # arrivals whose adapter was not resident yet
    arrivals: int
    wait_steps_hit: float        # mean steps from arrival to admission, adapter resident on arrival
    wait_steps_miss: float       # the same for arrivals that had to wait for a load (the stall)
    finished: int
    mean_running: float
    peak_kv_pages: int
    ops: List[tuple]
    ranks: np.ndarray
    wall_s: float

    def summary(self) -> dict:
        d = {k: v for k, v in dataclasses.asdict(self).items() if k not in ("ops", "ranks")}
        d["tokens_per_s_per_layer"] = self.tokens / (self.gpu_ms * 1e-3) if self.gpu_ms > 0 else None
        d["load_gbs_over_gpu_time"] = self.load_bytes / (self.gpu_ms * 1e-3) / 1e9 if self.gpu_ms > 0 else None
        d["adapter_hit_rate"] = 1.0 - self.arrival_misses / max(1, self.arrivals)
        return d


class HostStore:
    """Every adapter's rows in one pinned host buffer (A rows then B rows per projection)."""

    def __init__(self, spec: TraceSpec, ranks: np.ndarray, device):
        import torch

        self.spec = spec
        row = sum(p.h_in + p.h_out for p in spec.projections)
        self.off = np.zeros(spec.num_adapters + 1, dtype=np.int64)
        self.off[1:] = np.cumsum(ranks.astype(np.int64) * row)
        total = int(self.off[-1])
        self.buf = torch.empty(total, dtype=torch.int16).pin_memory()
        self.bits = self.buf.numpy().view(np.uint16)
        # seeded host draws, N(0, 1/64), rounded once to the storage type
        rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=(22,)))
        piece = 1 << 24
        for s in range(0, total, piece):
            n = min(piece, total - s)
            self.bits[s:s + n] = workloads._to_bits(rng.standard_normal(n, dtype=np.float32) * 0.125, spec.dtype)
        self.ranks = ranks

    def addresses(self, a: int):
        """Host addresses of adapter a's A and B rows per projection."""
        base = self.buf.data_ptr()
        r = int(self.ranks[a])
        o = int(self.off[a])
        hA, hB = [], []
        for p in self.spec.projections:
            hA.append(base + 2 * o)
            o += r * p.h_in
            hB.append(base + 2 * o)
            o += r * p.h_out
        return hA, hB

    def weights(self, a: int):
        """Adapter a's rows per projection as uint16 arrays (A rows [r, h_in], B rows [r, h_out])."""
        r = int(self.ranks[a])
        o = int(self.off[a])
        out = []
        for p in self.spec.projections:
            A = self.bits[o:o + r * p.h_in].reshape(r, p.h_in)
            o += r * p.h_in
            B = self.bits[o:o + r * p.h_out].reshape(r, p.h_out)
            o += r * p.h_out
            out.append((A, B))
        return out


def _zipf_probs(n: int, alpha: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** -alpha
    return p / p.sum()


class Trace:
    def __init__(self, spec: TraceSpec, device=None, probe_step: Optional[int] = None):
        self.spec = spec
        self.device = device
        rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=(20,)))
        self.ranks = rng.choice(np.asarray(spec.rank_set), size=spec.num_adapters).astype(np.int32)
        self.rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=(21,)))
        self.zipf = _zipf_probs(spec.num_adapters, spec.zipf_alpha)
        dims = [(p.h_in, p.h_out) for p in spec.projections]
        self.pool = slora.Pool(spec.pool_pages, spec.H, spec.dtype, dims, spec.num_adapters,
                               max(spec.rank_set), spec.token_budget, device=device)
        self.pages_per_rank = sum(-(-p.h_in // spec.H) - (-p.h_out // spec.H) for p in spec.projections)
        self.store = HostStore(spec, self.ranks, device) if device is not None else None
        self.resident: "collections.OrderedDict[int, int]" = collections.OrderedDict()  # adapter -> load step
        self.refs: Dict[int, int] = collections.defaultdict(int)
        self.kv: Dict[str, np.ndarray] = {}
        self.ops: List[tuple] = []
        self.waiting: "collections.deque[Request]" = collections.deque()
        self.running: List[Request] = []
        self.next_rid = 0
        self.next_kv = 0
        # at the first step from probe_step on that has tokens, the batch gets
        # fresh seeded host inputs, and the step's ids, x, y_in and (after the
        # apply) y are kept in self.probe
        self.probe_step = probe_step
        self.probe = None
        if device is not None:
            import torch

            T, n = spec.token_budget, len(spec.projections)
            tdt = self.pool.tdtype
            self.xs = [torch.empty((T, p.h_in), dtype=tdt, device=device) for p in spec.projections]
            self.ys = [torch.empty((T, p.h_out), dtype=tdt, device=device) for p in spec.projections]
            rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=(23,)))
            for x in self.xs + self.ys:
                bits = workloads._to_bits(rng.standard_normal(tuple(x.shape), dtype=np.float32), spec.dtype)
                x.copy_(torch.from_numpy(bits.view(np.int16)).view(tdt))
            self.ta_dev = torch.empty(T, dtype=torch.int32, device=device)
            self.n = n

    # ------------------------------------------------------------------ pool calls
    def _kv_alloc(self, n: int) -> Optional[str]:
        if n == 0:
            return None
        if slora.slora_pool_info(self.pool.handle)["free_pages"] < n and not self._evict_for(n):
            return None
        h = f"kv{self.next_kv}"
        self.next_kv += 1
        self.kv[h] = slora.slora_pages_alloc(self.pool.handle, n)
        self.ops.append(("kv_alloc", h, n))
        return h

    def _kv_free(self, h: str) -> None:
        pages = self.kv.pop(h)
        slora.slora_pages_free(self.pool.handle, pages)
        self.ops.append(("kv_free", h, np.arange(pages.shape[0])))

    def _evict_for(self, need: int) -> bool:
        """Evict least-recently-used adapters no running request holds until `need` pages are free."""
        free = slora.slora_pool_info(self.pool.handle)["free_pages"]
        for a in list(self.resident.keys()):
            if free >= need:
                break
            if self.refs[a] == 0:
                slora.slora_adapter_evict(self.pool.handle, a)
                self.ops.append(("evict", a))
                del self.resident[a]
                free += int(self.ranks[a]) * self.pages_per_rank
                self.evictions += 1
        return free >= need

    def _load(self, a: int, step: int) -> bool:
        need = int(self.ranks[a]) * self.pages_per_rank
        if slora.slora_pool_info(self.pool.handle)["free_pages"] < need and not self._evict_for(need):
            return False
        if self.store is not None:
            hA, hB = self.store.addresses(a)
            slora.slora_adapter_load(self.pool.handle, a, int(self.ranks[a]), hA, hB)
            self.load_bytes += need * self.spec.H * 2
        else:
            slora.slora_adapter_load(self.pool.handle, a, int(self.ranks[a]), None, None)
        self.ops.append(("load", a))
        self.resident[a] = step
        self.loads += 1
        return True

    # ------------------------------------------------------------------ the trace
    def run(self, steps: Optional[int] = None) -> TraceResult:
        sp = self.spec
        steps = sp.steps if steps is None else steps
        self.loads = self.load_bytes = self.evictions = 0
        finished = 0
        waits_hit: List[int] = []
        waits_miss: List[int] = []
        arrivals = arrival_misses = 0
        tokens = dec_tokens = pre_tokens = 0
        running_sum = 0
        peak_kv = 0
        gpu_ms = step_ms = load_ms = 0.0
        events = []
        if self.device is not None:
            # per-kernel events around every launch: the GPU time of the path
            # itself, which the step events overstate whenever the GPU waits
            # for the host between launches
            slora.slora_timing_enable(self.pool.handle, True)
            slora.slora_timing_read(self.pool.handle)   # (reading also resets the counters)
        t0 = time.perf_counter()
        for step in range(steps):
            # arrivals
            for _ in range(self.rng.poisson(sp.arrivals_per_step)):
                a = int(self.rng.choice(sp.num_adapters, p=self.zipf))
                rq = Request(self.next_rid, a, int(self.rng.integers(sp.prompt_len[0], sp.prompt_len[1] + 1)),
                             int(self.rng.integers(sp.output_len[0], sp.output_len[1] + 1)))
                rq.arrived_step = step
                rq.missed = not (a in self.resident and self.resident[a] < step)
                arrivals += 1
                arrival_misses += rq.missed
                self.waiting.append(rq)
                self.next_rid += 1
            # admission: adapters loaded in an earlier step; start loads for misses
            loads_now = 0
            still = collections.deque()
            pos = 0
            while self.waiting:
                rq = self.waiting.popleft()
                pos += 1
                if rq.adapter in self.resident:
                    if self.resident[rq.adapter] < step and len(self.running) < sp.max_running:
                        # the request's KV pages for its whole length come with
                        # admission, so running requests never stall on memory
                        self.refs[rq.adapter] += 1          # its adapter must stay while we make room
                        h = self._kv_alloc((rq.prompt + rq.output) * sp.kv_pages_per_token)
                        if h is not None:
                            self.resident.move_to_end(rq.adapter)
                            rq.kv_handles.append(h)
                            rq.admitted_step = step
                            self.running.append(rq)
                            (waits_miss if rq.missed else waits_hit).append(step - rq.arrived_step)
                            continue
                        self.refs[rq.adapter] -= 1
                elif (pos <= sp.prefetch_window and loads_now < sp.max_loads_per_step
                      and self._load(rq.adapter, step)):
                    loads_now += 1
                still.append(rq)
            self.waiting = still
            # the step's batch: decode tokens first, then prompt chunks
            budget = sp.token_budget
            ids: List[int] = []
            plan = []
            for rq in self.running:
                if budget == 0:
                    break
                if rq.prefilled == rq.prompt:
                    ids.append(rq.adapter)
                    plan.append((rq, 1, "decode"))
                    budget -= 1
            for rq in self.running:
                if budget == 0:
                    break
                if rq.prefilled < rq.prompt:
                    n = min(rq.prompt - rq.prefilled, budget)
                    ids += [rq.adapter] * n
                    plan.append((rq, n, "prefill"))
                    budget -= n
            T = len(ids)
            if T and self.device is not None:
                import torch

                st = self.pool.compute_stream
                with torch.cuda.stream(st):
                    # from pageable memory: staged before the call returns, so
                    # the next step may build its ids while this copy is queued
                    self.ta_dev[:T].copy_(torch.from_numpy(np.asarray(ids, dtype=np.int32)), non_blocking=True)
                    probe = self.probe is None and self.probe_step is not None and step >= self.probe_step
                    if probe:
                        rng = np.random.default_rng(np.random.SeedSequence(sp.seed, spawn_key=(24, step)))
                        xb = [workloads._to_bits(rng.standard_normal((T, p.h_in), dtype=np.float32), sp.dtype)
                              for p in sp.projections]
                        yb = [workloads._to_bits(rng.standard_normal((T, p.h_out), dtype=np.float32), sp.dtype)
                              for p in sp.projections]
                        for d_, h_ in zip(self.xs + self.ys, xb + yb):
                            d_[:T].copy_(torch.from_numpy(h_.view(np.int16)).view(self.pool.tdtype))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    seg = self.pool.build_segments(self.ta_dev[:T])
                    self.pool.apply_multi(seg, list(range(self.n)), [x[:T] for x in self.xs],
                                          [y[:T] for y in self.ys], sp.s, slora.MODE_AUTO)
                    e1.record(st)
                    events.append((e0, e1))
                    if probe:
                        torch.cuda.synchronize()
                        self.probe = {"step": step, "ids": np.asarray(ids, dtype=np.int32), "x": xb, "y_in": yb,
                                      "y": [y[:T].cpu().view(torch.int16).numpy().view(np.uint16).copy()
                                            for y in self.ys],
                                      "ops": len(self.ops)}
            # progress, completions
            for rq, n, kind in plan:
                if kind == "decode":
                    rq.generated += 1
                    dec_tokens += 1
                else:
                    rq.prefilled += n
                    pre_tokens += n
            tokens += T
            done = [rq for rq in self.running if rq.generated >= rq.output]
            for rq in done:
                for h in rq.kv_handles:
                    self._kv_free(h)
                self.refs[rq.adapter] -= 1
                finished += 1
            self.running = [rq for rq in self.running if rq.generated < rq.output]
            running_sum += len(self.running)
            kv_now = sum(p.shape[0] for p in self.kv.values())
            peak_kv = max(peak_kv, kv_now)
        if events:
            import torch

            torch.cuda.synchronize()
            step_ms = sum(a.elapsed_time(b) for a, b in events)
            tm = slora.slora_timing_read(self.pool.handle)
            slora.slora_timing_enable(self.pool.handle, False)
            gpu_ms = sum(ms for k, (ms, _) in tm.items() if k != "scatter")
            load_ms = tm.get("scatter", (0.0, 0))[0]
            st = self.pool.status()
            if st != slora.OK:
                raise RuntimeError(f"device status {st} after the trace")
        return TraceResult(steps, tokens, dec_tokens, pre_tokens, gpu_ms, step_ms, load_ms, self.loads, self.load_bytes,
                           self.evictions, len(waits_hit) + len(waits_miss), arrival_misses, arrivals,
                           float(np.mean(waits_hit)) if waits_hit else 0.0,
                           float(np.mean(waits_miss)) if waits_miss else 0.0,
                           finished, running_sum / max(1, steps), peak_kv,
                           list(self.ops), self.ranks.copy(), time.perf_counter() - t0)

    def close(self):
        self.pool.close()


def main():
    import argparse
    import json

    import torch

    ap = argparse.ArgumentParser(description="serving-trace driver (one layer of a 7B model)")
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--arrivals", type=float, default=4.0)
    args = ap.parse_args()
    from . import build

    build.build()
    spec = dataclasses.replace(TraceSpec(), steps=args.steps, arrivals_per_step=args.arrivals)
    tr = Trace(spec, device=torch.device("cuda", 0))
    res = tr.run()
    out = res.summary()
    out["workload"] = spec.name
    print(json.dumps(out))
    tr.close()


if __name__ == "__main__":
    main()
