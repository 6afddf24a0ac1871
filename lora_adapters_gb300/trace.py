"""Serving-trace driver: continuous batching over the unified page pool.

The pages describe S-LoRA as a serving system in which adapter weights and
KV-cache tensors share one paged memory pool, adapters live in host memory and
are fetched on demand when a request needs one, and every step batches the
tokens of many requests on many adapters ("S-LoRA: Serving Thousands of
Concurrent LoRA Adapters": the nubint.ai review's method list -- unified
paging, host-memory adapter store, on-demand loading; the dongaigc.com
summary, section 1 "unified paging"; the scheduler loop of the continuous-
batching page, "vLLM Zamanlayicisi").  When the adapters requests need do not
all fit beside the KV cache, adapters travel back and forth over the bus
(cmlonder.com newsletter, section "Iddia ve Gerceklik": thrashing when the
active adapters exceed the GPU's share).  This module drives the library
through such a trace for a whole decoder of ``layers`` layers:

* one pool holds every layer's adapter rows (an adapter carries q, k, v, o of
  every layer: ``layers`` x 4 projections) and every layer's KV slots (K and
  V of one token in one layer are two pages);
* requests arrive (Poisson per step), each with a prompt length, an output
  length and an adapter drawn Zipf-like from a large host store;
* every step has a token budget: one decode token for each running request
  first, then prompt chunks of requests in prefill;
* a request's KV pages for its whole length are taken when it is admitted;
  when the adapter of one of the first ``prefetch_window`` waiting requests
  is not resident it is loaded asynchronously, evicting least-recently-used
  adapters that no running request holds; a request joins the batch once its
  adapter was loaded in an earlier step;
* each step groups its tokens by adapter once and applies the LoRA delta of
  every layer's q, k, v, o (one multi-projection apply per layer, AUTO mode).

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
    name: str = "serve_trace_7b_32l"
    H: int = 4096
    dtype: str = "f16"
    layers: int = 32
    layer_projections: Tuple[workloads.Projection, ...] = workloads._qkvo(4096)
    num_adapters: int = 2000
    rank_set: Tuple[int, ...] = (8, 16, 32, 64)
    zipf_alpha: float = 1.0
    # 80 GB of the GPU's memory for the pool: the adapters this trace's
    # requests use (about 70 GB of rows for the 32 layers) plus the running
    # requests' KV (about 45 GB) do not fit, so least-recently-used adapters
    # are evicted and loaded again
    pool_bytes: int = 80 * 10**9
    kv_pages_per_token: int = 64             # K and V of every layer
    token_budget: int = 1024
    max_running: int = 256                   # requests in the batch at once
    arrivals_per_step: float = 4.0
    prompt_len: Tuple[int, int] = (8, 512)
    output_len: Tuple[int, int] = (8, 128)   # with the 256-request cap, the 1024-token budget fills
    max_loads_per_step: int = 16
    prefetch_window: int = 64                # misses loaded only for the first waiting requests
    steps: int = 1000
    s: float = 0.01                          # y accumulates one delta per layer and step
    seed: int = 0

    @property
    def pool_pages(self) -> int:
        return self.pool_bytes // (self.H * 2)

    @property
    def projections(self) -> Tuple[workloads.Projection, ...]:
        """Every layer's projections, layer by layer: the pool's projection list."""
        return tuple(workloads.Projection(f"L{l}.{p.name}", p.h_in, p.h_out)
                     for l in range(self.layers) for p in self.layer_projections)


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
    load_stall_ms: float         # time the compute stream waited for adapter copies still in flight
    load_copy_ms: float          # copy-stream time of the loads (host copies + scatter)
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
    layers: int = 1

    def summary(self) -> dict:
        d = {k: v for k, v in dataclasses.asdict(self).items() if k not in ("ops", "ranks")}
        # every token passes through every layer: layer-token products per
        # second of the path's kernel time
        d["tokens_per_s_per_layer"] = (self.tokens * self.layers / (self.gpu_ms * 1e-3)
                                       if self.gpu_ms > 0 else None)
        d["load_gbs_over_copy_time"] = (self.load_bytes / (self.load_copy_ms * 1e-3) / 1e9
                                        if self.load_copy_ms > 0 else None)
        d["load_stall_us_per_step"] = 1e3 * self.load_stall_ms / max(1, self.steps)
        d["adapter_hit_rate"] = 1.0 - self.arrival_misses / max(1, self.arrivals)
        return d


class HostStore:
    """Every adapter's rows in one pinned host buffer (A rows then B rows per
    projection of one layer).

    Every layer of an adapter gets the same rows: a load still copies the
    whole adapter, every layer's rows, over the bus into its own pages, but the
    host holds one layer's worth (4 GB for 2000 adapters instead of 123 GB).
    """

    def __init__(self, spec: TraceSpec, ranks: np.ndarray, device):
        import torch

        self.spec = spec
        row = sum(p.h_in + p.h_out for p in spec.layer_projections)
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
        """Host addresses of adapter a's A and B rows for every projection of the pool."""
        base = self.buf.data_ptr()
        r = int(self.ranks[a])
        o = int(self.off[a])
        hA, hB = [], []
        for p in self.spec.layer_projections:
            hA.append(base + 2 * o)
            o += r * p.h_in
            hB.append(base + 2 * o)
            o += r * p.h_out
        return hA * self.spec.layers, hB * self.spec.layers

    def weights(self, a: int):
        """Adapter a's rows for every projection of the pool as uint16 arrays
        (A rows [r, h_in], B rows [r, h_out]); views, not copies."""
        r = int(self.ranks[a])
        o = int(self.off[a])
        out = []
        for p in self.spec.layer_projections:
            A = self.bits[o:o + r * p.h_in].reshape(r, p.h_in)
            o += r * p.h_in
            B = self.bits[o:o + r * p.h_out].reshape(r, p.h_out)
            o += r * p.h_out
            out.append((A, B))
        return out * self.spec.layers


def _zipf_probs(n: int, alpha: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** -alpha
    return p / p.sum()


class Trace:
    def __init__(self, spec: TraceSpec, device=None, probe_step: Optional[int] = None,
                 probe_layer: Optional[int] = None, probe_after_eviction: bool = False):
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
        # At the first step from probe_step on that has tokens (and, with
        # probe_after_eviction, comes after an eviction), layer probe_layer
        # gets fresh seeded host inputs, and its ids, x, y_in and (after the
        # apply) y are kept in self.probe.
        self.probe_step = probe_step
        self.probe_layer = spec.layers - 1 if probe_layer is None else probe_layer
        self.probe_after_eviction = probe_after_eviction
        self.probe = None
        self.evictions = 0
        if device is not None:
            import torch

            # x and y of one layer's projections, used by every layer in turn
            T, n = spec.token_budget, len(spec.layer_projections)
            tdt = self.pool.tdtype
            self.xs = [torch.empty((T, p.h_in), dtype=tdt, device=device) for p in spec.layer_projections]
            self.ys = [torch.empty((T, p.h_out), dtype=tdt, device=device) for p in spec.layer_projections]
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
            self.load_bytes += int(self.ranks[a]) * sum(p.h_in + p.h_out for p in self.spec.projections) * 2
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
        if self.device is not None:
            import torch
        finished = 0
        waits_hit: List[int] = []
        waits_miss: List[int] = []
        arrivals = arrival_misses = 0
        tokens = dec_tokens = pre_tokens = 0
        running_sum = 0
        peak_kv = 0
        gpu_ms = step_ms = load_ms = stall_ms = copy_ms = 0.0
        events = []
        copy_pairs = []      # copy-stream events around each step's loads
        if self.device is not None:
            import torch
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
            # admission: requests whose adapter was loaded in an earlier step
            # and whose copies have finished
            still = collections.deque()
            while self.waiting:
                rq = self.waiting.popleft()
                if rq.adapter in self.resident:
                    if (self.resident[rq.adapter] < step and len(self.running) < sp.max_running
                            and slora.slora_adapter_ready(self.pool.handle, rq.adapter)):
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
                st = self.pool.compute_stream
                with torch.cuda.stream(st):
                    # from pageable memory: staged before the call returns, so
                    # the next step may build its ids while this copy is queued
                    self.ta_dev[:T].copy_(torch.from_numpy(np.asarray(ids, dtype=np.int32)), non_blocking=True)
                    probe = (self.probe is None and self.probe_step is not None and step >= self.probe_step
                             and (self.evictions > 0 or not self.probe_after_eviction))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    # the segment build makes the compute stream wait for the
                    # batch's adapters' loads still in flight (none, with
                    # admission on finished loads); one grouping serves every layer
                    seg = slora.slora_build_segments_for(self.pool.handle, self.ta_dev.data_ptr(), T,
                                                         np.asarray(ids, dtype=np.int32))
                    npl = self.n
                    for layer in range(sp.layers):
                        if probe and layer == self.probe_layer:
                            rng = np.random.default_rng(np.random.SeedSequence(sp.seed, spawn_key=(24, step)))
                            xb = [workloads._to_bits(rng.standard_normal((T, p.h_in), dtype=np.float32), sp.dtype)
                                  for p in sp.layer_projections]
                            yb = [workloads._to_bits(rng.standard_normal((T, p.h_out), dtype=np.float32), sp.dtype)
                                  for p in sp.layer_projections]
                            for d_, h_ in zip(self.xs + self.ys, xb + yb):
                                d_[:T].copy_(torch.from_numpy(h_.view(np.int16)).view(self.pool.tdtype))
                        self.pool.apply_multi(seg, list(range(layer * npl, (layer + 1) * npl)),
                                              [x[:T] for x in self.xs], [y[:T] for y in self.ys], sp.s,
                                              slora.MODE_AUTO)
                        if probe and layer == self.probe_layer:
                            torch.cuda.synchronize()
                            self.probe = {"step": step, "layer": layer, "ids": np.asarray(ids, dtype=np.int32),
                                          "x": xb, "y_in": yb,
                                          "y": [y[:T].cpu().view(torch.int16).numpy().view(np.uint16).copy()
                                                for y in self.ys],
                                          "ops": len(self.ops), "evictions_before": self.evictions}
                    e1.record(st)
                    events.append((e0, e1))
            # loads for the adapters of the first waiting requests that miss
            # (queued after the step's kernels; the requests join a later step)
            if self.device is not None:
                # the copy stream starts this step's loads once the step's
                # kernels are done (as every load does): c0 marks that point
                done_ev = torch.cuda.Event()
                done_ev.record(self.pool.compute_stream)
                self.pool.copy_stream.wait_event(done_ev)
                c0 = torch.cuda.Event(enable_timing=True)
                c0.record(self.pool.copy_stream)
            loads_now = 0
            for pos, rq in enumerate(self.waiting):
                if pos >= sp.prefetch_window or loads_now >= sp.max_loads_per_step:
                    break
                if rq.adapter not in self.resident and self._load(rq.adapter, step):
                    loads_now += 1
            if self.device is not None and loads_now:
                c1 = torch.cuda.Event(enable_timing=True)
                c1.record(self.pool.copy_stream)
                copy_pairs.append((c0, c1))
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
            torch.cuda.synchronize()
            step_ms = sum(a.elapsed_time(b) for a, b in events)
            copy_ms = sum(a.elapsed_time(b) for a, b in copy_pairs)
            tm = slora.slora_timing_read(self.pool.handle)
            slora.slora_timing_enable(self.pool.handle, False)
            gpu_ms = sum(ms for k, (ms, _) in tm.items() if k not in ("scatter", "load_wait"))
            load_ms = tm.get("scatter", (0.0, 0))[0]
            stall_ms = tm.get("load_wait", (0.0, 0))[0]   # the compute stream's waits for copies
            st = self.pool.status()
            if st != slora.OK:
                raise RuntimeError(f"device status {st} after the trace")
        return TraceResult(steps, tokens, dec_tokens, pre_tokens, gpu_ms, step_ms, load_ms, stall_ms, copy_ms,
                           self.loads, self.load_bytes,
                           self.evictions, len(waits_hit) + len(waits_miss), arrival_misses, arrivals,
                           float(np.mean(waits_hit)) if waits_hit else 0.0,
                           float(np.mean(waits_miss)) if waits_miss else 0.0,
                           finished, running_sum / max(1, steps), peak_kv,
                           list(self.ops), self.ranks.copy(), time.perf_counter() - t0, sp.layers)

    def close(self):
        self.pool.close()


def main():
    """One bench-style JSON line for the serving trace (rank 0, one GPU)."""
    import argparse
    import json

    import torch

    ap = argparse.ArgumentParser(description="serving trace over the unified pool (Llama-7B shape)")
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--arrivals", type=float, default=4.0)
    ap.add_argument("--pool-gb", type=float, default=80.0)
    args = ap.parse_args()
    from . import build

    build.build()
    spec = dataclasses.replace(TraceSpec(), steps=args.steps, layers=args.layers, arrivals_per_step=args.arrivals,
                               pool_bytes=int(args.pool_gb * 1e9), kv_pages_per_token=2 * args.layers)
    tr = Trace(spec, device=torch.device("cuda", 0))
    res = tr.run()
    s = res.summary()
    line = {"metric": "lora_delta_tokens_per_s_per_layer", "value": s["tokens_per_s_per_layer"], "unit": "tokens/s",
            "n_gpus": 1, "steps": res.steps, "higher_is_better": True, "dtype": spec.dtype, "data": "synthetic",
            "config": {"workload": spec.name, "H": spec.H, "layers": spec.layers,
                       "projections_per_layer": [p.name for p in spec.layer_projections],
                       "adapters": spec.num_adapters, "ranks": list(spec.rank_set),
                       "popularity": f"zipf(alpha={spec.zipf_alpha:g})", "pool_gb": spec.pool_bytes / 1e9,
                       "kv_pages_per_token": spec.kv_pages_per_token, "token_budget": spec.token_budget,
                       "arrivals_per_step": spec.arrivals_per_step, "mode": "auto"},
            "trace": s}
    print(json.dumps(line))
    tr.close()


if __name__ == "__main__":
    main()
