"""Thin ctypes binding of libslora.so (include/slora.h).

Every ``slora_*`` function here has the C function's name and arguments and
only marshals them; all work happens in the library.  ``Pool`` is a small
convenience wrapper over the same calls for torch tensors.

The library is loaded from this package directory (built by
``lora_adapters_gb300.build``).  If it is missing the import of the binding
fails loudly: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
# SLORA_DEBUG=1 in the environment selects the build with bounds checks in
# every kernel (libslora_debug.so); either way the library must exist.
DEBUG = os.environ.get("SLORA_DEBUG", "") == "1"
LIB_PATH = os.path.join(HERE, "libslora_debug.so" if DEBUG else "libslora.so")

OK = 0
ERR_INVALID = -1
ERR_OOM = -2
ERR_EXISTS = -3
ERR_NOT_RESIDENT = -4
ERR_BUSY = -5
ERR_CUDA = -6
ERR_DEVICE = -7
ERR_TIMEOUT = -8
ERR_DEVICE_ASSERT = -9
F16, BF16 = 0, 1
MODE_AUTO, MODE_DECODE, MODE_PREFILL = 0, 1, 2

EXPORTED = (
    "slora_pool_create", "slora_pool_destroy", "slora_pages_alloc", "slora_pages_free",
    "slora_pool_info", "slora_adapter_load", "slora_adapter_evict", "slora_adapter_pages",
    "slora_build_segments", "slora_lora_apply", "slora_lora_apply_multi", "slora_device_status",
    "slora_pool_snapshot", "slora_timing_enable", "slora_timing_read", "slora_set_tc_threshold",
    "slora_last_error_string", "slora_lora_apply_noalloc", "slora_adapter_set_scale",
    "slora_lora_apply_bmm", "slora_bmm_scratch_bytes", "slora_set_tc_min_batch", "slora_debug_set_fault",
    "slora_debug_set_wait_limit", "slora_adapter_ready", "slora_build_segments_for",
    "slora_debug_poke_page_table",
)
FAULT_NONE, FAULT_PAGE_ALLOC, FAULT_COPY = 0, 1, 2


class SloraError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {code}: {msg}")
        self.code = code


class slora_segments(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("max_segs", ctypes.c_int32),
                ("perm", ctypes.c_void_p), ("seg_start", ctypes.c_void_p),
                ("seg_adapter", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("generation", ctypes.c_uint64)]


_lib = None
P = ctypes.c_void_p
I32, I64 = ctypes.c_int32, ctypes.c_int64
_SIGS = {
    "slora_pool_create": [ctypes.POINTER(P), P, I64, I32, I32, I32, I32, I32, I32, P, P, P, P],
    "slora_pool_destroy": [P],
    "slora_pages_alloc": [P, I64, P],
    "slora_pages_free": [P, I64, P],
    "slora_pool_info": [P, P, P, P, P],
    "slora_adapter_load": [P, I32, I32, P, P, ctypes.POINTER(P)],
    "slora_adapter_evict": [P, I32],
    "slora_adapter_set_scale": [P, I32, ctypes.c_float],
    "slora_adapter_ready": [P, I32, P],
    "slora_adapter_pages": [P, I32, P, I64, P],
    "slora_build_segments": [P, P, I32, ctypes.POINTER(slora_segments)],
    "slora_build_segments_for": [P, P, I32, P, ctypes.POINTER(slora_segments)],
    "slora_lora_apply": [P, ctypes.POINTER(slora_segments), I32, P, I64, P, I64, ctypes.c_float, I32],
    "slora_lora_apply_multi": [P, ctypes.POINTER(slora_segments), I32, P, P, P, P, P, ctypes.c_float, I32],
    "slora_lora_apply_bmm": [P, ctypes.POINTER(slora_segments), I32, P, I64, P, I64, ctypes.c_float],
    "slora_bmm_scratch_bytes": [P, ctypes.POINTER(ctypes.c_size_t)],
    "slora_device_status": [P, P],
    "slora_pool_snapshot": [P, P, ctypes.POINTER(ctypes.c_size_t)],
    "slora_timing_enable": [P, I32],
    "slora_timing_read": [P, I32, P, P, P, P],
    "slora_set_tc_threshold": [P, I32],
    "slora_set_tc_min_batch": [P, I32],
    "slora_debug_set_fault": [P, I32, I64],
    "slora_debug_set_wait_limit": [P, ctypes.c_uint32],
    "slora_debug_poke_page_table": [P, I64, I32, P],
    "slora_lora_apply_noalloc": [P, I32, I32, P, I64, P, I32, I32, P, P, I32, P, I32, P, I64, P, I64,
                                 ctypes.c_float, P, P],
}


def lib() -> ctypes.CDLL:
    """Load libslora.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{os.path.basename(LIB_PATH)} not built at {LIB_PATH}: "
                              "run lora_adapters_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.slora_last_error_string.argtypes = []
        L.slora_last_error_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(rc: int, fn: str) -> int:
    if rc != OK:
        raise SloraError(rc, fn, slora_last_error_string())
    return rc


def _arr(values, ctype):
    return (ctype * len(values))(*values)


# ---- the C functions under their own names ------------------------------------
def slora_last_error_string() -> str:
    s = lib().slora_last_error_string()
    return s.decode() if s else ""


def slora_pool_create(d_pool: int, num_pages: int, page_elems: int, dtype: int, max_adapters: int,
                      max_rank: int, max_tokens: int, proj_in: Sequence[int], proj_out: Sequence[int],
                      compute_stream: int = 0, copy_stream: int = 0) -> int:
    out = P()
    _check(lib().slora_pool_create(ctypes.byref(out), d_pool or None, num_pages, page_elems, dtype,
                                   max_adapters, max_rank, max_tokens, len(proj_in),
                                   _arr(proj_in, I32), _arr(proj_out, I32),
                                   compute_stream or None, copy_stream or None), "slora_pool_create")
    return out.value


def slora_pool_destroy(pool: int) -> None:
    _check(lib().slora_pool_destroy(pool), "slora_pool_destroy")


def slora_pages_alloc(pool: int, n: int) -> np.ndarray:
    out = np.empty(max(n, 0), dtype=np.int32)
    _check(lib().slora_pages_alloc(pool, n, out.ctypes.data), "slora_pages_alloc")
    return out


def slora_pages_free(pool: int, pages) -> None:
    pages = np.ascontiguousarray(pages, dtype=np.int32)
    _check(lib().slora_pages_free(pool, pages.shape[0], pages.ctypes.data), "slora_pages_free")


def slora_pool_info(pool: int):
    free, num, ppr = I64(), I64(), I64()
    H = I32()
    _check(lib().slora_pool_info(pool, ctypes.byref(free), ctypes.byref(num), ctypes.byref(H),
                                 ctypes.byref(ppr)), "slora_pool_info")
    return {"free_pages": free.value, "num_pages": num.value, "page_elems": H.value,
            "pages_per_rank": ppr.value}


def slora_adapter_load(pool: int, adapter_id: int, rank: int, h_A: Optional[Sequence[int]],
                       h_B: Optional[Sequence[int]]) -> int:
    """h_A / h_B: host addresses per projection (or None on a planning pool). Returns the event."""
    ev = P()
    A = _arr(h_A, P) if h_A is not None else None
    B = _arr(h_B, P) if h_B is not None else None
    _check(lib().slora_adapter_load(pool, adapter_id, rank, A, B, ctypes.byref(ev)), "slora_adapter_load")
    return ev.value or 0


def slora_adapter_evict(pool: int, adapter_id: int) -> None:
    _check(lib().slora_adapter_evict(pool, adapter_id), "slora_adapter_evict")


def slora_adapter_ready(pool: int, adapter_id: int) -> bool:
    r = I32()
    _check(lib().slora_adapter_ready(pool, adapter_id, ctypes.byref(r)), "slora_adapter_ready")
    return bool(r.value)


def slora_adapter_set_scale(pool: int, adapter_id: int, scale: float) -> None:
    _check(lib().slora_adapter_set_scale(pool, adapter_id, float(scale)), "slora_adapter_set_scale")


def slora_adapter_pages(pool: int, adapter_id: int) -> np.ndarray:
    n = I64()
    _check(lib().slora_adapter_pages(pool, adapter_id, None, 0, ctypes.byref(n)), "slora_adapter_pages")
    out = np.empty(n.value, dtype=np.int32)
    _check(lib().slora_adapter_pages(pool, adapter_id, out.ctypes.data, n.value, ctypes.byref(n)),
           "slora_adapter_pages")
    return out


def slora_build_segments(pool: int, d_token_adapter: int, T: int) -> slora_segments:
    seg = slora_segments()
    _check(lib().slora_build_segments(pool, d_token_adapter or None, T, ctypes.byref(seg)),
           "slora_build_segments")
    return seg


def slora_build_segments_for(pool: int, d_token_adapter: int, T: int, h_token_adapter) -> slora_segments:
    """h_token_adapter: host int32 array of the same ids (or None)."""
    seg = slora_segments()
    h = None
    if h_token_adapter is not None:
        h_token_adapter = np.ascontiguousarray(h_token_adapter, dtype=np.int32)
        h = h_token_adapter.ctypes.data
    _check(lib().slora_build_segments_for(pool, d_token_adapter or None, T, h, ctypes.byref(seg)),
           "slora_build_segments_for")
    return seg


def slora_lora_apply(pool: int, seg: slora_segments, proj: int, d_x: int, ldx: int, d_y: int, ldy: int,
                     s: float, mode: int = MODE_AUTO) -> None:
    _check(lib().slora_lora_apply(pool, ctypes.byref(seg), proj, d_x, ldx, d_y, ldy, s, mode),
           "slora_lora_apply")


def slora_lora_apply_bmm(pool: int, seg: slora_segments, proj: int, d_x: int, ldx: int, d_y: int, ldy: int,
                         s: float) -> None:
    _check(lib().slora_lora_apply_bmm(pool, ctypes.byref(seg), proj, d_x, ldx, d_y, ldy, s), "slora_lora_apply_bmm")


def slora_bmm_scratch_bytes(pool: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().slora_bmm_scratch_bytes(pool, ctypes.byref(n)), "slora_bmm_scratch_bytes")
    return n.value


def slora_lora_apply_multi(pool: int, seg: slora_segments, projs: Sequence[int], d_x: Sequence[int],
                           ldx: Sequence[int], d_y: Sequence[int], ldy: Sequence[int], s: float,
                           mode: int = MODE_AUTO) -> None:
    n = len(projs)
    _check(lib().slora_lora_apply_multi(pool, ctypes.byref(seg), n, _arr(projs, I32), _arr(d_x, P),
                                        _arr(ldx, I64), _arr(d_y, P), _arr(ldy, I64), s, mode),
           "slora_lora_apply_multi")


def slora_device_status(pool: int) -> int:
    st = I32()
    _check(lib().slora_device_status(pool, ctypes.byref(st)), "slora_device_status")
    return st.value


def slora_pool_snapshot(pool: int) -> dict:
    n = ctypes.c_size_t()
    _check(lib().slora_pool_snapshot(pool, None, ctypes.byref(n)), "slora_pool_snapshot")
    buf = np.empty(n.value, dtype=np.uint8)
    _check(lib().slora_pool_snapshot(pool, buf.ctypes.data, ctypes.byref(n)), "slora_pool_snapshot")
    num_pages, free_pages = buf[:16].view(np.int64)
    max_adapters, stride = buf[16:24].view(np.int32)
    body = buf[24:].view(np.int32)
    owner = body[:num_pages]
    rank = body[num_pages:num_pages + max_adapters]
    pt = body[num_pages + max_adapters:].reshape(max_adapters, stride)
    return {"num_pages": int(num_pages), "free_pages": int(free_pages), "owner": owner, "rank": rank,
            "page_table": pt}


def slora_timing_enable(pool: int, enable: bool) -> None:
    _check(lib().slora_timing_enable(pool, 1 if enable else 0), "slora_timing_enable")


def slora_timing_read(pool: int) -> dict:
    cap = 16
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    launches = (ctypes.c_int64 * cap)()
    n = I32()
    _check(lib().slora_timing_read(pool, cap, names, ms, launches, ctypes.byref(n)), "slora_timing_read")
    return {names[i].decode(): (ms[i], launches[i]) for i in range(n.value)}


def slora_set_tc_threshold(pool: int, min_tokens: int) -> None:
    _check(lib().slora_set_tc_threshold(pool, min_tokens), "slora_set_tc_threshold")


def slora_set_tc_min_batch(pool: int, min_tokens: int) -> None:
    _check(lib().slora_set_tc_min_batch(pool, min_tokens), "slora_set_tc_min_batch")


def slora_debug_set_fault(pool: int, kind: int, nth: int) -> None:
    _check(lib().slora_debug_set_fault(pool, kind, nth), "slora_debug_set_fault")


def slora_debug_set_wait_limit(pool: int, polls: int) -> None:
    _check(lib().slora_debug_set_wait_limit(pool, polls), "slora_debug_set_wait_limit")


def slora_debug_poke_page_table(pool: int, entry: int, value: int) -> int:
    """Writes one device page-table entry (SLORA_DEBUG build only); returns the old value."""
    old = ctypes.c_int32(0)
    _check(lib().slora_debug_poke_page_table(pool, entry, value, ctypes.byref(old)), "slora_debug_poke_page_table")
    return old.value


NOALLOC_MAX_TOKENS = 2048


def slora_lora_apply_noalloc(d_pool: int, page_elems: int, dtype: int, d_page_table: int, pt_stride: int,
                             d_rank: int, max_adapters: int, proj_in: Sequence[int], proj_out: Sequence[int],
                             proj: int, d_token_adapter: int, T: int, d_x: int, ldx: int, d_y: int, ldy: int,
                             s: float, stream: int = 0, status: int = 0) -> None:
    """The allocation-free apply (every buffer caller-owned; see slora.h).

    status: address of one int32 (device or pinned host memory) that receives
    the call's device status on the stream, or 0 for none."""
    _check(lib().slora_lora_apply_noalloc(d_pool, page_elems, dtype, d_page_table, pt_stride, d_rank,
                                          max_adapters, len(proj_in), _arr(proj_in, I32), _arr(proj_out, I32),
                                          proj, d_token_adapter or None, T, d_x or None, ldx, d_y or None, ldy, s,
                                          stream or None, status or None), "slora_lora_apply_noalloc")


# ---- convenience wrapper for torch tensors -----------------------------------------
class Pool:
    """A pool over a torch device buffer (or a planning pool when device=None)."""

    def __init__(self, num_pages: int, H: int, dtype: str, projections, max_adapters: int, max_rank: int,
                 max_tokens: int, device=None, compute_stream=None, copy_stream=None):
        import torch

        self.H, self.dtype = int(H), dtype
        self.projections = [(int(i), int(o)) for i, o in projections]
        self.tdtype = torch.float16 if dtype == "f16" else torch.bfloat16
        self.buffer = None
        d_pool, cs, ps = 0, 0, 0
        if device is not None:
            self.buffer = torch.empty((int(num_pages), int(H)), dtype=self.tdtype, device=device)
            d_pool = self.buffer.data_ptr()
            self.compute_stream = compute_stream or torch.cuda.current_stream(device)
            self.copy_stream = copy_stream or torch.cuda.Stream(device)
            cs, ps = self.compute_stream.cuda_stream, self.copy_stream.cuda_stream
        self.handle = slora_pool_create(d_pool, num_pages, H, F16 if dtype == "f16" else BF16, max_adapters,
                                        max_rank, max_tokens, [i for i, _ in self.projections],
                                        [o for _, o in self.projections], cs, ps)
        self._arena = None
        self._arena_t = None
        self._arena_off = 0

    def close(self):
        if self.handle:
            slora_pool_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load(self, adapter_id: int, rank: int, weights=None) -> int:
        """weights: per projection (A rows [r, h_in], B rows [r, h_out]) uint16 arrays, or None.

        The arrays are copied into a pinned host arena that the asynchronous
        copies read from; the arena is reused only after the copy stream has
        drained (``sync_loads``), so callers may drop their arrays at once.
        """
        if weights is None:
            return slora_adapter_load(self.handle, adapter_id, rank, None, None)
        arrays = []
        for A, B in weights:
            arrays += [np.ascontiguousarray(A, dtype=np.uint16), np.ascontiguousarray(B, dtype=np.uint16)]
        need = sum(a.nbytes + 16 for a in arrays)
        if self._arena is None or self._arena_off + need > self._arena.nbytes:
            self.sync_loads()
            if self._arena is None or need > self._arena.nbytes:
                import torch

                size = max(need, 256 << 20)
                self._arena_t = torch.empty(size, dtype=torch.uint8).pin_memory()
                self._arena = self._arena_t.numpy()
        addrs = []
        base = self._arena.ctypes.data
        for a in arrays:
            off = (self._arena_off + 15) & ~15
            self._arena[off:off + a.nbytes] = a.view(np.uint8).reshape(-1)
            addrs.append(base + off)
            self._arena_off = off + a.nbytes
        return slora_adapter_load(self.handle, adapter_id, rank, addrs[0::2], addrs[1::2])

    def set_scale(self, adapter_id: int, scale: float) -> None:
        slora_adapter_set_scale(self.handle, adapter_id, scale)

    def sync_loads(self):
        if self.buffer is not None:
            self.copy_stream.synchronize()
        self._arena_off = 0

    def replay(self, ops, ranks, weights_of=None) -> dict:
        """Replay a workload's pool call sequence; returns the KV handles' page lists."""
        handles = {}
        for op in ops:
            if op[0] == "kv_alloc":
                handles[op[1]] = slora_pages_alloc(self.handle, op[2])
            elif op[0] == "kv_free":
                slora_pages_free(self.handle, handles[op[1]][np.asarray(op[2], dtype=np.int64)])
            elif op[0] == "load":
                a = op[1]
                w = weights_of(a) if weights_of is not None else None
                self.load(a, int(ranks[a]), w)
            elif op[0] == "evict":
                slora_adapter_evict(self.handle, op[1])
            else:
                raise ValueError(op)
        self.sync_loads()
        return handles

    def build_segments(self, token_adapter_dev) -> slora_segments:
        return slora_build_segments(self.handle, token_adapter_dev.data_ptr() if token_adapter_dev.numel() else 0,
                                    int(token_adapter_dev.numel()))

    def apply(self, seg, proj: int, x, y, s: float, mode: int = MODE_AUTO) -> None:
        slora_lora_apply(self.handle, seg, proj, x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), s, mode)

    def apply_bmm(self, seg, proj: int, x, y, s: float) -> None:
        """The padded batched-matmul comparator (slora_lora_apply_bmm)."""
        slora_lora_apply_bmm(self.handle, seg, proj, x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), s)

    def apply_multi(self, seg, projs, xs, ys, s: float, mode: int = MODE_AUTO) -> None:
        slora_lora_apply_multi(self.handle, seg, list(projs), [x.data_ptr() for x in xs],
                               [x.stride(0) for x in xs], [y.data_ptr() for y in ys],
                               [y.stride(0) for y in ys], s, mode)

    def snapshot(self) -> dict:
        return slora_pool_snapshot(self.handle)

    def status(self) -> int:
        return slora_device_status(self.handle)
