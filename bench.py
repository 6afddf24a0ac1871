"""Benchmark of the heterogeneous-batch paged LoRA delta, one layer per step.

One step = the whole hot path over one batch: group the batch's tokens by
adapter (build_segments), then y += s (x A_a) B_a for every projection of the
layer (one multi-projection apply).  The default run measures three
workloads, each a line of its own inside one printed JSON object:

* the headline, the largest single-GPU configuration: a Llama-13B-shaped
  MLP decode batch -- H = 5120, gate/up 5120 -> 13824 and down 13824 -> 5120,
  512 tokens (one per request), 2000 adapters of ranks {16, 32, 64} resident
  in a 120 GB pool filled up with KV slots, token -> adapter Zipf(1.2), bf16;
* the first entry of the line's ``configs`` list: the Llama-7B-shaped decode batch -- q/k/v/o 4096 -> 4096,
  256 tokens, 1000 adapters of ranks {8, 16, 32, 64}, Zipf(1), fp16;
* the second entry: the Llama-7B-shaped prefill batch -- 32 requests of
  U{8..512} tokens, 200 adapters of ranks {8..128}, fp16, long segments on
  the tensor cores.

L2 is flushed before every timed step (a 256 MiB device write, then a 256 MiB
device read, so that the write's dirty lines leave L2 before the step starts),
so adapter pages, x and y come from HBM; only the steps themselves are timed,
with CUDA events on the compute stream.  ``--workload NAME`` measures one
workload alone (one line).  ``--impl reference`` times the CPU oracle on a
bounded sample of the headline workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "lora_delta_tokens_per_s_per_layer"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
TC_THRESHOLD = 8           # the library's AUTO defaults: segments of >= 8 tokens on the tensor cores,
TC_MIN_BATCH = 2048        # in batches of >= 2048 tokens
HEADLINE = "llama13b_mlp_decode"
EXTRA = ("llama7b_decode", "llama7b_prefill")
DEFAULT_MODE = {"llama13b_mlp_decode": "decode", "llama7b_decode": "decode", "llama7b_prefill": "prefill",
                "tiny": "decode"}

# ncu DRAM counters of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum, per launch) on each workload, with the hash of the
# kernel source they were taken from; reported as null once the source has
# changed.  The 13B MLP batch was captured in a compact pool holding only the
# batch's adapters (--compact-pool: the same kernel work on the same rows).
NCU_TRAFFIC = {
    # apply_cc, 13B MLP decode (compact pool, same work): 793.70 MB read + 25.25 MB written (mean of 2 launches)
    ("apply_cc", "llama13b_mlp_decode"): (818947584, "79ef4a8af322f883"),
    # apply_cc, 7B decode: 277.73 MB read + 1.05 MB written (mean of 2 launches)
    ("apply_cc", "llama7b_decode"): (278776192, "79ef4a8af322f883"),
    # tc_expand, 7B prefill: 360.35 MB read + 217.89 MB written (mean of 2 launches)
    ("expand_tc", "llama7b_prefill"): (578235392, "79ef4a8af322f883"),
}
# ncu sm__pipe_tensor_cycles_active (% of active cycles) of the tensor-core
# kernels on the prefill batch, with the kernel-source hash.
NCU_TENSOR_PIPE = {
    "llama7b_prefill": ({"expand_tc": 10.91, "shrink_tc": 23.79}, "79ef4a8af322f883"),
}


def _kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and whitespace do not count."""
    h = hashlib.sha256()
    for f in ("kernels.cu", "tc_kernels.cu", "internal.h", "ptx.cuh"):
        p = os.path.join(ROOT, "lora_adapters_gb300", "csrc", f)
        if os.path.exists(p):
            src = open(p).read()
            src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
            src = re.sub(r"//[^\n]*", " ", src)
            h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense 16-bit tensor peak (TFLOP/s): fp16 and bf16 run at the same rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops"]), "measured (bf16 burst; fp16 has the same dense rate)"
    return 1900.0, "fallback"


# ---------------------------------------------------------------- workload
def algorithmic_bytes(wl, tc_threshold=None, elt=2):
    """Algorithmic bytes of one step, split by kernel.

    Per projection and segment of T_s tokens on adapter a (rank r_a):
    shrink reads x (T_s * H_in) and A_a once (r_a * H_in); expand reads and
    writes y (2 * T_s * H_out) and reads B_a once (r_a * H_out).  Segments of
    at least `tc_threshold` tokens go to the tensor-core kernels (None: all
    on the CUDA-core kernels).  Page tables, segments and the shrink
    scratch are metadata and not counted.
    """
    ta = wl.token_adapter
    ids, counts = np.unique(ta[ta >= 0], return_counts=True)
    out = {"shrink_cc": 0, "expand_cc": 0, "shrink_tc": 0, "expand_tc": 0}
    for a, n in zip(ids, counts):
        r, n = int(wl.ranks[a]), int(n)
        path = "tc" if tc_threshold is not None and n >= tc_threshold else "cc"
        out["shrink_" + path] += sum((n + r) * p.h_in * elt for p in wl.projections)
        out["expand_" + path] += sum((2 * n + r) * p.h_out * elt for p in wl.projections)
    out["apply_cc"] = out["shrink_cc"] + out["expand_cc"]     # one launch does both phases
    out["step"] = out["shrink_cc"] + out["expand_cc"] + out["shrink_tc"] + out["expand_tc"]
    out["distinct_adapters"] = int(ids.shape[0])
    out["tokens"] = int(counts.sum())
    return out


def algorithmic_flops(wl, tc_threshold=None):
    """Multiply-add flops of one step (2 per product), split like the bytes:
    shrink 2 T_s r_a H_in and expand 2 T_s r_a H_out per segment and projection."""
    ta = wl.token_adapter
    ids, counts = np.unique(ta[ta >= 0], return_counts=True)
    out = {"shrink_cc": 0, "expand_cc": 0, "shrink_tc": 0, "expand_tc": 0}
    for a, n in zip(ids, counts):
        r, n = int(wl.ranks[a]), int(n)
        path = "tc" if tc_threshold is not None and n >= tc_threshold else "cc"
        out["shrink_" + path] += sum(2 * n * r * p.h_in for p in wl.projections)
        out["expand_" + path] += sum(2 * n * r * p.h_out for p in wl.projections)
    out["step"] = sum(out[k] for k in ("shrink_cc", "expand_cc", "shrink_tc", "expand_tc"))
    return out


def compact_pool(wl):
    """The same batch in a pool that holds only the adapters the batch uses
    (pre-fragmented the same way: the pool filled with KV slots, a seeded half
    released, then the adapters loaded), for profilers that save and restore
    device memory: every kernel does the same work on the same rows as on the
    full pool, whose other adapters and KV slots this batch never reads."""
    import dataclasses

    used = sorted(set(int(a) for a in wl.token_adapter if a >= 0))
    per_rank = sum(-(-p.h_in // wl.H) + -(-p.h_out // wl.H) for p in wl.projections)
    need = sum(int(wl.ranks[a]) * per_rank for a in used)
    pages = 2 * need
    free = np.sort(np.random.default_rng(np.random.SeedSequence(wl.spec.seed, spawn_key=(6,))).choice(
        pages, size=need + need // 2, replace=False)).astype(np.int64)
    ops = [("kv_alloc", "kv0", pages), ("kv_free", "kv0", free)] + [("load", a) for a in used]
    return dataclasses.replace(wl, pool_pages=pages, pool_ops=ops)


def setup_device(wl, device):
    """A device pool holding the workload's adapters, and its inputs.

    Adapters that the batch uses get their drawn weights; the others (whose
    pages are allocated in the same order but never read by this batch) get
    zeros, so that the 2000-adapter pools load in seconds."""
    import torch

    from lora_adapters_gb300 import slora

    sp = wl.spec
    dims = [(p.h_in, p.h_out) for p in sp.projections]
    pool = slora.Pool(wl.pool_pages, wl.H, sp.dtype, dims, sp.num_adapters, max(sp.rank_set),
                      max(wl.T, 1), device=device)
    used = set(int(a) for a in wl.token_adapter if a >= 0)
    zeros = {}

    def weights_of(a):
        if a in used:
            return wl.adapter(a)
        r = int(wl.ranks[a])
        if r not in zeros:
            zeros[r] = [(np.zeros((r, i), np.uint16), np.zeros((r, o), np.uint16)) for i, o in dims]
        return zeros[r]

    pool.replay(wl.pool_ops, wl.ranks, weights_of)
    tdt = pool.tdtype

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).to(device)

    xs = [dev(wl.x(p)) for p in range(len(dims))]
    y0 = [dev(wl.y_in(p)) for p in range(len(dims))]
    ys = [y.clone() for y in y0]
    ta = torch.from_numpy(wl.token_adapter.copy()).to(device)
    torch.cuda.synchronize()
    return pool, ta, xs, ys, y0


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not runnable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        lines = [l.strip() for l in open(self.out.name) if l.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"unavailable": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _gpu_id(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[0] if vis else str(torch.cuda.current_device())


# ---------------------------------------------------------------- CPU oracle
class OracleSample:
    """The CPU oracle set up once for the batch (untimed); ``run`` times it on a token sample."""

    def __init__(self, wl):
        from oracle import pool as opool

        self.wl = wl
        sp = wl.spec
        self.pool = opool.OraclePool(wl.pool_pages, wl.H, [(p.h_in, p.h_out) for p in sp.projections],
                                     sp.num_adapters, max(sp.rank_set))
        self.pool.replay(wl.pool_ops, wl.ranks)
        self.store = opool.OracleStore(wl.pool_pages, wl.H)
        for a in sorted(set(int(a) for a in wl.token_adapter if a >= 0)):
            self.store.write_adapter(self.pool, a, wl.adapter(a))
        self.inputs = [(wl.x(p), wl.y_in(p)) for p in range(len(sp.projections))]

    def run(self, n_tokens: int, threads: int, seed: int = 0):
        from oracle import lora as olora

        wl, sp = self.wl, self.wl.spec
        rng = np.random.default_rng(seed)
        rows = np.sort(rng.choice(wl.T, size=min(n_tokens, wl.T), replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        for p, (x, y) in enumerate(self.inputs):
            olora.apply(self.store, self.pool, p, wl.token_adapter, x, y, sp.s, sp.dtype, tokens=rows,
                        num_threads=threads)
        return time.perf_counter() - t0, len(rows)


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def workload_config(wl, mode, gpus):
    sp = wl.spec
    return {"workload": sp.name, "H": sp.H, "tokens_per_step": wl.T,
            "projections": [f"{p.name}:{p.h_in}->{p.h_out}" for p in sp.projections],
            "adapters_resident": sp.num_adapters, "ranks": list(sp.rank_set),
            "popularity": f"{sp.popularity}{'(alpha=%g)' % sp.zipf_alpha if sp.popularity == 'zipf' else ''}",
            "pool_pages": wl.pool_pages, "page_bytes": sp.H * 2, "pool_gb": wl.pool_pages * sp.H * 2 / 1e9,
            "mode": mode,
            "l2": "flushed before every timed step: 256 MiB device write, then 256 MiB device read",
            "parallelism": f"replicas x{gpus}"}


def oracle_baseline(wl, seconds: float):
    """The CPU oracle on a bounded token sample, at all host threads and at one."""
    orc = OracleSample(wl)
    out = {}
    for threads in (cpu_threads(), 1):
        t1, n1 = orc.run(2, threads)
        n_tok = int(max(2, min(wl.T, seconds / 4 / max(t1 / n1, 1e-6))))
        t, nn, reps = 0.0, 0, 0
        while t < seconds and reps < 200:
            dt, dn = orc.run(n_tok, threads, seed=1 + reps)
            t, nn, reps = t + dt, nn + dn, reps + 1
        out[threads] = (nn / t, f"{reps} x {n_tok} of the {wl.T} tokens, all {len(wl.projections)} projections, "
                                f"fp64 C loops, {t:.1f} s of oracle time")
    threads = cpu_threads()
    return {"value": out[threads][0], "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": out[threads][1], "value_1_thread": out[1][0], "sample_1_thread": out[1][1]}


def run_reference(args, wl, cfg):
    """The reference arm: the CPU oracle, as it stands, on host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = cpu_threads()
    orc = OracleSample(wl)
    wt, wn = 0.0, 0
    for _ in range(args.warmup):
        t, n = orc.run(max(1, args.ref_tokens // 4), threads)
        wt, wn = wt + t, wn + n
    # tokens per step: at most --ref-tokens, fewer when K steps of that size
    # would take more than about a minute of CPU time
    sample = int(max(1, min(args.ref_tokens, 60.0 / max(args.steps * wt / max(wn, 1), 1e-9))))
    total_t, total_n = 0.0, 0
    for k in range(args.steps):
        t, n = orc.run(sample, threads, seed=k)
        total_t += t
        total_n += n
    value = total_n / total_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{sample} tokens of the batch per step, all {len(wl.projections)} "
                                       f"projections"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- replicas
class Replicas:
    """N independent replicas of the path, one process per GPU (the path has
    no exchange step, so no collective touches the data): rank and world from
    the launcher's environment, a barrier around each timed region, the
    maximum over ranks of a time, and the whole-job rate (units of all ranks
    divided by that time)."""

    def __init__(self, backend: str, device=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.device = device
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist

            if backend == "nccl":
                dist.init_process_group("nccl", device_id=device)
            else:
                dist.init_process_group(backend)
            self.dist = dist

    def barrier(self) -> None:
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.dist is None:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def rate(self, units_per_rank: float, seconds: float) -> float:
        return self.world * units_per_rank / seconds

    def close(self) -> None:
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


# ---------------------------------------------------------------- GPU arm
def staging_layout(nbytes, align: int = 256):
    """Offsets of pieces of the given sizes laid end to end, each starting on
    an `align`-byte boundary, and the total size."""
    offs, total = [], 0
    for n in nbytes:
        offs.append(total)
        total += (n + align - 1) // align * align
    return offs, total


def copy_spans(n: int, chunk: int):
    """(start, length) of the copies that move n bytes, at most `chunk` each."""
    return [(c, min(chunk, n - c)) for c in range(0, n, chunk)]


def _link_gbs(torch, device, h2d: int, d2h: int):
    """A plain pinned-memory copy of one step's bytes each way, alone: the
    link-bound floor of the end-to-end step."""
    out = {}
    for name, nbytes, up in (("h2d", h2d, True), ("d2h", d2h, False)):
        host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
        s = torch.cuda.Stream(device=device)
        best = None
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                (dev.copy_(host, non_blocking=True) if up else host.copy_(dev, non_blocking=True))
                b.record(s)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name + "_gbs"] = nbytes / (best * 1e-3) / 1e9
        out[name + "_ms"] = best
        del host, dev
    return out


def measure(name, mode_name, args, rep, device, rank, world):
    """Every number of one workload's line (rank 0 prints it)."""
    import torch

    from lora_adapters_gb300 import slora, workloads

    wl = workloads.make(name, seed=rank)      # each replica draws its own batch
    if args.compact_pool:
        wl = compact_pool(wl)
    sp = wl.spec
    cfg = workload_config(wl, mode_name, args.gpus)
    if args.compact_pool:
        cfg["pool"] = "compact: only the batch's adapters (profiling)"
    mode = {"auto": slora.MODE_AUTO, "decode": slora.MODE_DECODE, "prefill": slora.MODE_PREFILL}[mode_name]

    pool, ta, xs, ys, y0 = setup_device(wl, device)
    tc_threshold = TC_THRESHOLD
    if args.tc_threshold is not None:
        tc_threshold = args.tc_threshold
        slora.slora_set_tc_threshold(pool.handle, tc_threshold)
        cfg["tc_threshold"] = tc_threshold
    n = len(sp.projections)
    projs = list(range(n))
    stream = pool.compute_stream
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=device)

    def flush(k):
        # evict L2: write a buffer larger than L2, then read another one so
        # that the written lines are back in HBM before the timed step
        flush_w.fill_(k & 0xff)
        flush_r.sum()

    def step():
        seg = pool.build_segments(ta)
        if args.impl == "bmm":
            for p_ in projs:
                pool.apply_bmm(seg, p_, xs[p_], ys[p_], sp.s)
        else:
            pool.apply_multi(seg, projs, xs, ys, sp.s, mode)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-timed steps (inputs resident in HBM; per-kernel hooks off)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    rep.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(_gpu_id(torch))
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush(k)
            starts[k].record(stream)
            step()
            ends[k].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    rep.barrier()
    if pool.status() != slora.OK:
        raise RuntimeError(f"{name}: a kernel reported an error during the timed steps")
    ms = sum(s_.elapsed_time(e) for s_, e in zip(starts, ends))
    ms_step = rep.max(ms / args.steps)
    value = rep.rate(wl.T, ms_step * 1e-3)
    hbm_peak, peak_kind = _peaks()

    if args.impl == "bmm":
        # the comparator: step time and the same algorithmic bytes only
        ab = algorithmic_bytes(wl, None)
        line = {"impl": "bmm", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": sp.dtype, "data": "synthetic", "config": cfg,
                "comparator": "every token's rows gathered and padded to the pool's max rank, two cuBLAS "
                              "strided-batched GEMMs, one rounding",
                "scratch_bytes": slora.slora_bmm_scratch_bytes(pool.handle),
                "step_algorithmic_bytes": ab["step"],
                "step_frac_of_hbm": ab["step"] / (ms_step * 1e-3) / 1e9 / hbm_peak,
                "clocks": clk, "gpu_launches": (1 + 3 * n) * args.steps}
        pool.close()
        return line

    # ---- per-kernel durations: the same steps again, each kernel bracketed by
    # events on the compute stream (this serialises the launches a little, so
    # the step time above is taken without it)
    slora.slora_timing_enable(pool.handle, True)
    slora.slora_timing_read(pool.handle)                  # reset the totals
    hook_steps = min(args.steps, 500)
    with torch.cuda.stream(stream):
        for k in range(hook_steps):
            flush(k)
            step()
    kern = slora.slora_timing_read(pool.handle)
    slora.slora_timing_enable(pool.handle, False)

    # ---- roofline of the dominant kernel
    thr = {"decode": None, "auto": tc_threshold if wl.T >= TC_MIN_BATCH else None, "prefill": 0}[mode_name]
    ab = algorithmic_bytes(wl, thr)
    fl = algorithmic_flops(wl, thr)
    per_kernel = {}
    for kname, (tms, cnt) in kern.items():
        if cnt:
            per_kernel[kname] = {"avg_us": 1e3 * tms / cnt, "launches": int(cnt),
                                 "us_per_step": 1e3 * tms / hook_steps}
            if kname in ab:
                per_launch = ab[kname] * hook_steps / cnt
                per_kernel[kname]["bytes_per_launch"] = per_launch
                per_kernel[kname]["gbs"] = per_launch / (per_kernel[kname]["avg_us"] * 1e-6) / 1e9
                per_kernel[kname]["frac_of_hbm"] = per_kernel[kname]["gbs"] / hbm_peak
    # the dominant kernel: the one with the most device time per step among
    # those that move the path's algorithmic bytes
    movers = [k for k in per_kernel if "gbs" in per_kernel[k]]
    dom = max(movers, key=lambda k: per_kernel[k]["us_per_step"])
    achieved = per_kernel[dom]["gbs"]
    src_hash = _kernel_source_hash()
    tr = NCU_TRAFFIC.get((dom, sp.name))
    traffic = tr[0] if tr and tr[1] == src_hash else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": peak_kind, "traffic": traffic,
                "traffic_over_algorithmic": (traffic / per_kernel[dom]["bytes_per_launch"]) if traffic else None,
                "algorithmic_bytes_per_launch": per_kernel[dom]["bytes_per_launch"],
                "avg_launch_us": per_kernel[dom]["avg_us"],
                "step_algorithmic_bytes": ab["step"],
                "step_achieved_gbs": ab["step"] / (ms_step * 1e-3) / 1e9,
                "step_frac": ab["step"] / (ms_step * 1e-3) / 1e9 / hbm_peak,
                "kernels": per_kernel, "source_hash": src_hash}
    tc_us = sum(per_kernel.get(k, {}).get("us_per_step", 0.0) for k in ("shrink_tc", "expand_tc"))
    if tc_us > 0:
        # the tensor-core kernels against the dense 16-bit tensor peak (their
        # arithmetic intensity is below the ridge: HBM stays the bound)
        tpk, tkind = _tensor_peak()
        tflops = (fl["shrink_tc"] + fl["expand_tc"]) / (tc_us * 1e-6) / 1e12
        tensor = {"achieved_tflops": tflops, "peak_tflops": tpk, "frac": tflops / tpk, "peak_source": tkind,
                  "algorithmic_flops_per_step": fl["shrink_tc"] + fl["expand_tc"]}
        for k in ("shrink_tc", "expand_tc"):
            if k in per_kernel:
                per_kernel[k]["tflops"] = fl[k] / (per_kernel[k]["us_per_step"] * 1e-6) / 1e12
        pipe = NCU_TENSOR_PIPE.get(sp.name)
        if pipe and pipe[1] == src_hash:
            tensor["ncu_tensor_pipe_active_pct"] = pipe[0]
        roofline["tensor"] = tensor
    # kernels behind each timing hook: the shrink_tc hook covers tc_shrink and
    # the tc_combine launch that adds its K parts
    per_hook = {"shrink_tc": 2}
    launches = int(round(sum(c * per_hook.get(k, 1) for k, (_, c) in kern.items() if k != "load_wait")
                         / hook_steps)) * args.steps

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its token ids, x and y in from pinned host memory and its y back out, as
    # a serving loop would: inputs of later steps go in on one copy stream and
    # results of earlier steps come out on another while a step computes.
    # With small copies (decode batches) three sets of device buffers let a
    # step's inputs go in without waiting for the result of the step two
    # before it; with large ones (the prefill batch: 840 MB per step) two sets
    # measured faster, since more copies in flight at once share the link.
    # No L2 flush here: x and y arrive from the host every step and the
    # adapter rows a step reads exceed L2 on the decode batches.
    # A step's inputs are staged in one contiguous pinned buffer -- the token
    # ids, every projection's x, then every y, each piece 256-byte aligned --
    # and the device buffer of a set has the same layout.  Copies move up to
    # kCopyChunk bytes each: few enough that issuing them (about 10 us of host
    # time a copy) does not bound a small step, large enough that the two
    # directions, sharing the link, interleave.  Measured: the 7B decode step
    # (one copy each way) 104 us against 135 us with a copy per tensor; the
    # 13B step (two each way) 340 us against 373 us with a copy per tensor
    # and 339-391 us, depending on the box, with one each way.
    pieces = [ta] + list(xs) + list(y0)
    nbytes = [t.numel() * t.element_size() for t in pieces]
    offs, total = staging_layout(nbytes)
    y_lo, y_hi = offs[1 + len(xs)], offs[-1] + nbytes[-1]
    pin_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(pieces, offs, nbytes):
        pin_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())

    def views(buf):
        v = [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(pieces, offs, nbytes)]
        return v[0], v[1:1 + len(xs)], v[1 + len(xs):]

    n_sets = 3 if total + (y_hi - y_lo) <= (256 << 20) else 2
    sets = []
    for _ in range(n_sets):
        buf = torch.empty(total, dtype=torch.uint8, device=device)
        sets.append((buf,) + views(buf))
    out_y = [torch.zeros(y_hi - y_lo, dtype=torch.uint8).pin_memory() for _ in sets]   # padding stays 0
    h2d = total
    d2h = y_hi - y_lo
    kCopyChunk = 32 << 20

    def copy_chunks(dst, dst_off, src, src_off, n):
        for c, m in copy_spans(n, kCopyChunk):
            dst[dst_off + c:dst_off + c + m].copy_(src[src_off + c:src_off + c + m], non_blocking=True)
    s_in = torch.cuda.Stream(device=device)
    s_out = torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_comp = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]
    for e in ev_out:
        e.record(s_out)

    def e2e_step(k):
        b = k % len(sets)
        buf, d_ta, d_xs, d_ys = sets[b]
        s_in.wait_event(ev_out[b])          # the result of the set's previous step has left it
        with torch.cuda.stream(s_in):
            copy_chunks(buf, 0, pin_in, 0, total)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        with torch.cuda.stream(stream):
            seg = pool.build_segments(d_ta)
            pool.apply_multi(seg, projs, d_xs, d_ys, sp.s, mode)
            ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            copy_chunks(out_y[b], 0, buf, y_lo, y_hi - y_lo)
            ev_out[b].record(s_out)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize()
    rep.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    s_in.wait_event(t_start)
    for k in range(args.steps):
        e2e_step(k)
    for e in ev_out:
        stream.wait_event(e)
    t_end.record(stream)
    t_end.synchronize()
    e_ms = t_start.elapsed_time(t_end) / args.steps
    # every buffer set computed the same batch from the same inputs: their
    # results must agree bit for bit (a copy racing a kernel would show here)
    if args.steps >= len(sets):
        for other in out_y[1:]:
            if not torch.equal(out_y[0], other):
                raise RuntimeError("pipelined end-to-end steps disagree")
    rep.barrier()
    e_ms = rep.max(e_ms)
    link = _link_gbs(torch, device, h2d, d2h)
    e2e = {"value": rep.rate(wl.T, e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms,
           "pipelining": f"{n_sets} buffer sets: later steps' inputs in and earlier steps' y out while a step "
                         f"computes; contiguous pinned staging, copies of at most {kCopyChunk >> 20} MB",
           "l2": "not flushed",
           "link": dict(link, note="one plain pinned copy of the step's input bytes (h2d) and of its output "
                                   "bytes (d2h), each alone: the end-to-end step cannot beat the larger "
                                   "of the two"),
           "link_bound_ms": max(link["h2d_ms"], link["d2h_ms"])}
    pool.close()
    del step, e2e_step, pool, xs, ys, y0, sets, out_y, pin_in, pieces, flush_w, flush_r, ta
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on a bounded sample, rank 0 at N = 1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(wl, args.cpu_seconds if name == HEADLINE else args.cpu_seconds / 2)

    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": sp.dtype, "data": "synthetic", "config": cfg,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches, "wall_s_timed_region": wall}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference", "bmm"],
                    help="bmm: the padded batched-matmul comparator through slora_lora_apply_bmm")
    ap.add_argument("--workload", default="all",
                    help="all: the headline workload plus the two 7B batches; else one workload")
    ap.add_argument("--mode", default=None, choices=["auto", "decode", "prefill"],
                    help="default: decode for decode batches, prefill for the prefill batch")
    ap.add_argument("--tc-threshold", type=int, default=None,
                    help="AUTO mode: segments of at least this many tokens on the tensor cores (library default 64)")
    ap.add_argument("--ref-tokens", type=int, default=24)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time per thread count (headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compact-pool", action="store_true",
                    help="profiling: a pool holding only the batch's adapters (same kernel work, small footprint)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from lora_adapters_gb300 import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    names = [HEADLINE, *EXTRA] if args.workload == "all" else [args.workload]
    if args.impl == "reference":
        wl = workloads.make(names[0], seed=rank)
        run_reference(args, wl, workload_config(wl, args.mode or DEFAULT_MODE.get(names[0], "decode"), args.gpus))
        return

    import torch

    from lora_adapters_gb300 import build

    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    rep = Replicas("nccl", device)
    lines = [measure(nm, args.mode or DEFAULT_MODE.get(nm, "decode"), args, rep, device, rank, world)
             for nm in names]
    rep.close()
    if rank == 0:
        line = dict(lines[0])
        if len(lines) > 1:
            line["configs"] = lines[1:]
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
