"""Python binding of libpps.so: paged, prefix-shared, mixed-batch attention
for GB300 (sm_103a).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  The
binding raises ``PPSError`` when the library is missing or a call fails; there
is no fallback.

    plan = attn_plan(q_indptr, kv_len, page_indptr, page_indices, Hq, Hkv, d, P, num_pages)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    kv_append(pool_k, pool_v, k_new, v_new, q_indptr_d, cached_len_d, page_indptr_d, page_indices_d)
    attn_run(plan, q, pool_k, pool_v, out, ws)
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

__all__ = [
    "PPSError", "Plan", "lib", "build", "kv_append", "attn_plan", "attn_run", "plan_destroy",
    "attn_step_host", "attn_step", "StepCall", "event_array",
    "get_device_error", "set_stream_error_word", "get_stream_error", "launch_count", "status_string", "version", "LIB_PATH",
    "PLAN_NO_GROUPS", "PLAN_CUDA_CORES_ONLY", "PLAN_SMALL_ROWS_CUDA_CORES", "PLAN_FUSED_APPEND", "KERNEL_BANDWIDTH", "KERNEL_TENSOR", "KERNEL_MERGE",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpps.so")

PLAN_NO_GROUPS = 1
PLAN_CUDA_CORES_ONLY = 2
PLAN_SMALL_ROWS_CUDA_CORES = 4
PLAN_FUSED_APPEND = 8
KERNEL_BANDWIDTH, KERNEL_TENSOR, KERNEL_MERGE = 0, 1, 2
NUM_KERNEL_CLASSES = 3
TASK_INTS = 8
NO_CAUSAL = 0x3FFFFFFF
ARRAYS = {"bw_tasks": 0, "mma_tasks": 1, "rows": 2, "pages": 3, "merge_tokens": 4,
          "merge_indptr": 5, "merge_pids": 6, "tree_mask": 7, "tt_cta": 8}
TREE_MAX_TOKENS = 64


class PPSError(RuntimeError):
    pass


class _Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


class _PlanOptions(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("bw_chunk_tokens", ctypes.c_int32),
                ("mma_chunk_tokens", ctypes.c_int32), ("flags", ctypes.c_int32)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_requests", "num_tokens", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "num_groups")] + [(n, ctypes.c_int64) for n in (
            "num_bw_tasks", "num_mma_tasks", "num_partials", "num_merge_tokens", "table_bytes",
            "workspace_bytes", "kv_bytes_unique", "kv_bytes_read")] + [
        ("flops_mma", ctypes.c_double), ("flops_total", ctypes.c_double),
        ("kv_bytes_bw", ctypes.c_int64), ("flops_mma_issued", ctypes.c_double),
        ("num_tree_requests", ctypes.c_int32), ("small_rows_on_tensor", ctypes.c_int32)]


class _CacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_pages", "page_size", "free_pages",
                                              "active_requests")] + [
        (n, ctypes.c_int64) for n in ("tree_nodes", "evictions", "reused_tokens", "begun_tokens",
                                      "tick")]


_lib = None
_I32P = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile libpps.so in place (nvcc, sm_103a)."""
    from .builder import build as _build
    return _build(force=force)


def lib():
    """The loaded library (raises PPSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise PPSError(f"{LIB_PATH} is missing: build it with paged_prefix_shared_gb300.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    L.pps_kv_append.argtypes = [ctypes.POINTER(_Pool), vp, vp, vp, vp, vp, vp, i32, i32, vp]
    # host int32 arrays by address (see _host_addr)
    L.pps_attn_plan.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                ctypes.c_float, ctypes.POINTER(_PlanOptions),
                                ctypes.POINTER(vp), ctypes.POINTER(sz)]
    L.pps_attn_plan_tree.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                     i32, i32, ctypes.c_float, ctypes.POINTER(_PlanOptions),
                                     ctypes.POINTER(vp), ctypes.POINTER(sz)]
    L.pps_attn_run.argtypes = [vp, vp, ctypes.POINTER(_Pool), vp, vp, sz, vp]
    L.pps_copy_slots.argtypes = [ctypes.POINTER(_Pool), vp, vp, vp, i32, vp]
    L.pps_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    L.pps_partition.argtypes = [_I32P, _I32P, _I32P, _I32P, i32, i32, i32, _I32P,
                                ctypes.POINTER(ctypes.c_int64)]
    L.pps_partition.restype = i32
    L.pps_gemm_bf16.restype = i32
    L.pps_cache_create.argtypes = [i32, i32, i32, ctypes.POINTER(vp)]
    L.pps_cache_destroy.argtypes = [vp]
    L.pps_cache_begin.argtypes = [vp, _I32P, i32, _I32P, _I32P, _I32P]
    L.pps_cache_extend.argtypes = [vp, i32, _I32P, i32, _I32P]
    L.pps_cache_finish.argtypes = [vp, i32, i32]
    L.pps_cache_request_pages.argtypes = [vp, i32, ctypes.POINTER(_I32P), _I32P, _I32P]
    L.pps_cache_get_stats.argtypes = [vp, ctypes.POINTER(_CacheStats)]
    L.pps_cache_dump.argtypes = [vp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                                 ctypes.POINTER(ctypes.c_int64)]
    L.pps_cache_extend_batch.argtypes = [vp, _I32P, _I32P, _I32P, i32, _I32P, _I32P]
    L.pps_cache_tables.argtypes = [vp, _I32P, i32, _I32P, _I32P, _I32P, ctypes.c_int64]
    for f in (L.pps_cache_extend_batch, L.pps_cache_tables):
        f.restype = i32
    L.pps_engine_create.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
    L.pps_engine_destroy.argtypes = [vp]
    L.pps_engine_parts.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp)]
    L.pps_engine_add.argtypes = [vp, _I32P, i32, i32, _I32P, _I32P, _I32P]
    L.pps_engine_finish.argtypes = [vp, i32, i32]
    L.pps_engine_schedule.argtypes = [vp, _I32P, _I32P, _I32P, i32, _I32P]
    L.pps_engine_commit.argtypes = [vp, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P,
                                    ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), _I32P]
    for f in (L.pps_engine_create, L.pps_engine_destroy, L.pps_engine_parts, L.pps_engine_add,
              L.pps_engine_finish, L.pps_engine_schedule, L.pps_engine_commit):
        f.restype = i32
    L.pps_sched_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
    L.pps_sched_destroy.argtypes = [vp]
    L.pps_sched_add.argtypes = [vp, i32, i32, i32]
    L.pps_sched_remove.argtypes = [vp, i32]
    L.pps_sched_set_gen_tokens.argtypes = [vp, i32, i32]
    L.pps_sched_step.argtypes = [vp, _I32P, _I32P, _I32P, i32, _I32P]
    L.pps_sched_counts.argtypes = [vp, _I32P, ctypes.POINTER(ctypes.c_int64), _I32P]
    for f in (L.pps_sched_create, L.pps_sched_destroy, L.pps_sched_add, L.pps_sched_remove,
              L.pps_sched_set_gen_tokens, L.pps_sched_step, L.pps_sched_counts):
        f.restype = i32
    for f in (L.pps_copy_slots, L.pps_cache_create, L.pps_cache_destroy, L.pps_cache_begin,
              L.pps_cache_extend, L.pps_cache_finish, L.pps_cache_request_pages,
              L.pps_cache_get_stats, L.pps_cache_dump):
        f.restype = i32
    L.pps_attn_run_events.argtypes = [vp, vp, ctypes.POINTER(_Pool), vp, vp, sz, vp,
                                      ctypes.POINTER(vp)]
    L.pps_attn_step_host.argtypes = [ctypes.POINTER(_Pool), vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                     i32, ctypes.c_float, ctypes.POINTER(_PlanOptions), vp, vp,
                                     sz, ctypes.POINTER(sz), vp]
    L.pps_attn_step_host.restype = i32
    L.pps_attn_step.argtypes = [ctypes.POINTER(_Pool), vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                ctypes.c_float, ctypes.POINTER(_PlanOptions), vp, vp, sz,
                                ctypes.POINTER(sz), vp, vp]
    L.pps_attn_step.restype = i32
    L.pps_set_stream_error_word.argtypes = [vp, vp]
    L.pps_set_stream_error_word.restype = i32
    L.pps_get_stream_error.argtypes = [vp, ctypes.POINTER(i32), i32]
    L.pps_get_stream_error.restype = i32
    L.pps_attn_run_noalloc.argtypes = [vp, vp, ctypes.POINTER(_Pool), vp, vp]
    L.pps_attn_run_noalloc.restype = i32
    L.pps_plan_destroy.argtypes = [vp]
    L.pps_plan_get_info.argtypes = [vp, ctypes.POINTER(_PlanInfo)]
    L.pps_plan_get_array.argtypes = [vp, i32, ctypes.POINTER(_I32P), ctypes.POINTER(ctypes.c_int64)]
    L.pps_get_device_error.argtypes = [_I32P, i32]
    L.pps_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    L.pps_selftest_wait_timeout.restype = i32
    L.pps_launch_count.restype = ctypes.c_uint64
    L.pps_status_string.restype = ctypes.c_char_p
    L.pps_status_string.argtypes = [i32]
    L.pps_version.restype = i32
    for f in (L.pps_kv_append, L.pps_attn_plan, L.pps_attn_plan_tree, L.pps_attn_run,
              L.pps_attn_run_events,
              L.pps_plan_destroy, L.pps_plan_get_info, L.pps_plan_get_array,
              L.pps_get_device_error):
        f.restype = i32
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().pps_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != 0:
        raise PPSError(f"{what}: {status_string(code)} ({code})")


def version() -> int:
    return int(lib().pps_version())


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().pps_launch_count())


def _host_i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(_I32P)


def _host_addr(a):
    """(contiguous int32 array, its address as an int): for the per-step calls,
    where building a ctypes pointer object costs more than the call itself."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.__array_interface__["data"][0]


def _dev(t, dtype=None):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise PPSError("tensors must be contiguous CUDA tensors")
    if dtype is not None and t.dtype != dtype:
        raise PPSError(f"expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    # the current stream's handle without building a Stream object (a few
    # microseconds per call, paid on every launch of a serving loop)
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return ctypes.c_void_p(raw(torch._C._cuda_getDevice()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _pool(pool_k, pool_v):
    import torch
    if pool_k.shape != pool_v.shape or pool_k.dim() != 4:
        raise PPSError("pool_k / pool_v must both be [num_pages, Hkv, page_size, head_dim]")
    n, h, p, d = pool_k.shape
    return _Pool(_dev(pool_k, torch.bfloat16), _dev(pool_v, torch.bfloat16), n, h, p, d)


def kv_append(pool_k, pool_v, k_new, v_new, q_indptr, cached_len, page_indptr, page_indices,
              stream=None):
    """pps_kv_append: all arguments are CUDA tensors (int32 tables, bf16 rows)."""
    import torch
    pool = _pool(pool_k, pool_v)
    R = int(cached_len.shape[0])
    T = int(k_new.shape[0])
    _check(lib().pps_kv_append(ctypes.byref(pool), _dev(k_new, torch.bfloat16),
                               _dev(v_new, torch.bfloat16), _dev(q_indptr, torch.int32),
                               _dev(cached_len, torch.int32), _dev(page_indptr, torch.int32),
                               _dev(page_indices, torch.int32), R, T, _stream(stream)),
           "pps_kv_append")


class Plan:
    """Owner of a pps_plan (host memory); freed by destroy() or garbage collection."""

    def __init__(self, handle, workspace_bytes):
        self._h = handle
        self.workspace_bytes = int(workspace_bytes)

    @property
    def handle(self):
        if self._h is None:
            raise PPSError("plan already destroyed")
        return self._h

    def info(self) -> dict:
        inf = _PlanInfo()
        _check(lib().pps_plan_get_info(self.handle, ctypes.byref(inf)), "pps_plan_get_info")
        return {n: getattr(inf, n) for n, _ in _PlanInfo._fields_}

    def array(self, name) -> np.ndarray:
        ptr = _I32P()
        cnt = ctypes.c_int64()
        _check(lib().pps_plan_get_array(self.handle, ARRAYS[name], ctypes.byref(ptr),
                                        ctypes.byref(cnt)), "pps_plan_get_array")
        if cnt.value == 0:
            a = np.zeros(0, dtype=np.int32)
        else:
            a = np.ctypeslib.as_array(ptr, shape=(cnt.value,)).copy()
        return a.reshape(-1, TASK_INTS) if name.endswith("tasks") else a

    def destroy(self):
        if self._h is not None:
            lib().pps_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def attn_plan(q_indptr, kv_len, page_indptr, page_indices, num_q_heads, num_kv_heads, head_dim,
              page_size, num_pages, sm_scale=None, num_sms=0, bw_chunk_tokens=0,
              mma_chunk_tokens=0, flags=0, tree_parent=None) -> Plan:
    """pps_attn_plan on host int32 arrays (numpy or lists); with ``tree_parent``
    (one parent index per new token, -1 = off the cached context) it calls
    pps_attn_plan_tree."""
    qi, qi_p = _host_addr(q_indptr)
    kl, kl_p = _host_addr(kv_len)
    pi, pi_p = _host_addr(page_indptr)
    px, px_p = _host_addr(page_indices if len(page_indices) else np.zeros(1, np.int32))
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    opts = _PlanOptions(int(num_sms), int(bw_chunk_tokens), int(mma_chunk_tokens), int(flags))
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    if tree_parent is None:
        _check(lib().pps_attn_plan(qi_p, kl_p, pi_p, px_p, len(kl), int(num_q_heads),
                                   int(num_kv_heads), int(head_dim), int(page_size),
                                   int(num_pages), float(sm_scale), ctypes.byref(opts),
                                   ctypes.byref(h), ctypes.byref(ws)), "pps_attn_plan")
    else:
        tp, tp_p = _host_addr(tree_parent if len(tree_parent) else np.zeros(1, np.int32))
        _check(lib().pps_attn_plan_tree(qi_p, kl_p, pi_p, px_p, tp_p, len(kl), int(num_q_heads),
                                        int(num_kv_heads), int(head_dim), int(page_size),
                                        int(num_pages), float(sm_scale), ctypes.byref(opts),
                                        ctypes.byref(h), ctypes.byref(ws)), "pps_attn_plan_tree")
    return Plan(h, ws.value)


def plan_destroy(plan: Plan):
    plan.destroy()


def attn_run(plan: Plan, q, pool_k, pool_v, out, workspace, stream=None, events=None):
    """pps_attn_run (or pps_attn_run_events when `events` is a list of
    2 * NUM_KERNEL_CLASSES torch.cuda.Event objects / None)."""
    import torch
    pool = _pool(pool_k, pool_v)
    ws = _dev(workspace)
    nbytes = workspace.numel() * workspace.element_size()
    if events is None:
        code = lib().pps_attn_run(plan.handle, _dev(q, torch.bfloat16), ctypes.byref(pool),
                                  _dev(out, torch.bfloat16), ws, nbytes, _stream(stream))
    else:
        handles = []
        for e in events:
            if e is not None and not e.cuda_event:
                e.record()          # torch creates the CUDA event on first record
            handles.append(ctypes.c_void_p(e.cuda_event) if e is not None else None)
        arr = (ctypes.c_void_p * (2 * NUM_KERNEL_CLASSES))(*handles)
        code = lib().pps_attn_run_events(plan.handle, _dev(q, torch.bfloat16), ctypes.byref(pool),
                                         _dev(out, torch.bfloat16), ws, nbytes, _stream(stream),
                                         arr)
    _check(code, "pps_attn_run")


def get_device_error(clear: bool = True) -> int:
    code = ctypes.c_int32()
    _check(lib().pps_get_device_error(ctypes.byref(code), int(bool(clear))), "pps_get_device_error")
    return int(code.value)


def set_stream_error_word(word, stream=None):
    """pps_set_stream_error_word: device errors of later calls on `stream`
    (default: the current stream) go to `word`, a one-element int32 CUDA
    tensor the caller zeroes and keeps alive; None removes the registration."""
    import torch
    if word is not None and (not word.is_cuda or word.dtype != torch.int32 or word.numel() < 1):
        raise PPSError("word must be an int32 CUDA tensor")
    _check(lib().pps_set_stream_error_word(_stream(stream),
                                           None if word is None else ctypes.c_void_p(word.data_ptr())),
           "pps_set_stream_error_word")


def get_stream_error(stream=None, clear: bool = True) -> int:
    """pps_get_stream_error: the error word of `stream` (waits for the stream)."""
    code = ctypes.c_int32()
    _check(lib().pps_get_stream_error(_stream(stream), ctypes.byref(code), int(bool(clear))),
           "pps_get_stream_error")
    return int(code.value)


def selftest_wait_timeout(limit_ns: int = 10_000_000, stream=None):
    """Launch the bounded-wait diagnostic kernel (see pps_selftest_wait_timeout)."""
    _check(lib().pps_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "pps_selftest_wait_timeout")


NOALLOC_SCRATCH_BYTES = 32 << 20


def attn_run_noalloc(plan: Plan, q, pool_k, pool_v, out, stream=None):
    """pps_attn_run_noalloc: pps_attn_run without a caller workspace, for callers
    that cannot allocate device memory.  Uses the library's fixed
    NOALLOC_SCRATCH_BYTES device array; plans that need more are rejected
    (PPSError).  Calls that overlap on the GPU race on that one array."""
    import torch
    pool = _pool(pool_k, pool_v)
    _check(lib().pps_attn_run_noalloc(plan.handle, _dev(q, torch.bfloat16), ctypes.byref(pool),
                                      _dev(out, torch.bfloat16), _stream(stream)),
           "pps_attn_run_noalloc")


# ---- copy-on-write and the host prefix cache ------------------------------------------

def copy_slots(pool_k, pool_v, src_pages, dst_pages, num_slots, stream=None):
    """pps_copy_slots: int32 CUDA tensors [count] of source pages, destination
    pages and slot counts."""
    import torch
    pool = _pool(pool_k, pool_v)
    n = int(src_pages.shape[0])
    _check(lib().pps_copy_slots(ctypes.byref(pool), _dev(src_pages, torch.int32),
                                _dev(dst_pages, torch.int32), _dev(num_slots, torch.int32), n,
                                _stream(stream)), "pps_copy_slots")


class CacheFull(PPSError):
    """pps_cache_*: no free page and nothing evictable."""


CACHE_LRU, CACHE_LFU = 0, 1


class Cache:
    """Owner of a pps_cache (host radix-tree prefix cache + page allocator)."""

    def __init__(self, num_pages, page_size, policy=CACHE_LRU):
        h = ctypes.c_void_p()
        _check(lib().pps_cache_create(int(num_pages), int(page_size), int(policy),
                                      ctypes.byref(h)), "pps_cache_create")
        self._h = h
        self.page_size = int(page_size)

    def _status(self, code, what):
        if code == -8:
            raise CacheFull(f"{what}: {status_string(code)}")
        _check(code, what)

    def begin(self, tokens):
        """Returns (request id, cached_len, copy or None); copy = (src, dst, slots)."""
        t, tp = _host_i32(tokens)
        rid, cached = ctypes.c_int32(), ctypes.c_int32()
        cp = (ctypes.c_int32 * 3)()
        self._status(lib().pps_cache_begin(self._h, tp, len(t), ctypes.byref(rid),
                                           ctypes.byref(cached), cp), "pps_cache_begin")
        copy = (cp[0], cp[1], cp[2]) if cp[2] > 0 else None
        return rid.value, cached.value, copy

    def extend(self, request, tokens):
        """Appends tokens; returns their first position."""
        t, tp = _host_i32(tokens if len(tokens) else np.zeros(1, np.int32))
        first = ctypes.c_int32()
        self._status(lib().pps_cache_extend(self._h, int(request), tp, len(tokens),
                                            ctypes.byref(first)), "pps_cache_extend")
        return first.value

    def extend_batch(self, requests, token_indptr, tokens):
        """pps_cache_extend_batch; returns the first new position of each request.
        On CacheFull the requests before the failing one stay extended."""
        r, rp = _host_i32(requests)
        ti, tip = _host_i32(token_indptr)
        t, tp = _host_i32(tokens if len(tokens) else np.zeros(1, np.int32))
        first = np.zeros(max(len(r), 1), np.int32)
        done = ctypes.c_int32()
        self._status(lib().pps_cache_extend_batch(self._h, rp, tip, tp, len(r),
                                                  first.ctypes.data_as(_I32P),
                                                  ctypes.byref(done)), "pps_cache_extend_batch")
        return first[:len(r)]

    def tables(self, requests):
        """(kv_len, page_indptr, page_indices) of the given requests, in order."""
        r, rp = _host_i32(requests)
        n = len(r)
        kv = np.zeros(max(n, 1), np.int32)
        ip = np.zeros(n + 1, np.int32)
        if getattr(self, "_px", None) is None:
            self._px = np.zeros(1 << 16, np.int32)
        while True:
            code = lib().pps_cache_tables(self._h, rp, n, kv.ctypes.data_as(_I32P),
                                          ip.ctypes.data_as(_I32P),
                                          self._px.ctypes.data_as(_I32P), len(self._px))
            if code == 0:
                break
            need = sum(len(self.pages(x)) for x in r)              # raises on an unknown id
            if need <= len(self._px):
                _check(code, "pps_cache_tables")
            self._px = np.zeros(2 * need, np.int32)
        return kv[:n], ip, self._px[:ip[-1]].copy()

    def finish(self, request, insert=True):
        self._status(lib().pps_cache_finish(self._h, int(request), int(bool(insert))),
                     "pps_cache_finish")

    def pages(self, request):
        ptr, n, nt = _I32P(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pps_cache_request_pages(self._h, int(request), ctypes.byref(ptr),
                                             ctypes.byref(n), ctypes.byref(nt)),
               "pps_cache_request_pages")
        return np.ctypeslib.as_array(ptr, shape=(n.value,)).copy() if n.value else \
            np.zeros(0, np.int32)

    def stats(self) -> dict:
        st = _CacheStats()
        _check(lib().pps_cache_get_stats(self._h, ctypes.byref(st)), "pps_cache_get_stats")
        return {n: getattr(st, n) for n, _ in _CacheStats._fields_}

    def dump(self):
        """List of (page, parent page, chunk tuple, last use, hits)."""
        need = ctypes.c_int64()
        _check(lib().pps_cache_dump(self._h, None, 0, ctypes.byref(need)), "pps_cache_dump")
        buf = np.zeros(max(need.value, 1), np.int64)
        _check(lib().pps_cache_dump(self._h, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                    need.value, ctypes.byref(need)), "pps_cache_dump")
        rec = 5 + self.page_size
        out = []
        for k in range(need.value // rec):
            r = buf[k * rec:(k + 1) * rec]
            out.append((int(r[0]), int(r[1]), tuple(int(x) for x in r[5:5 + int(r[2])]),
                        int(r[3]), int(r[4])))
        return out

    def destroy(self):
        if self._h is not None:
            lib().pps_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class Scheduler:
    """Owner of a pps_sched (token-wise budget scheduler)."""

    def __init__(self, budget, reserved=0):
        h = ctypes.c_void_p()
        _check(lib().pps_sched_create(int(budget), int(reserved), ctypes.byref(h)),
               "pps_sched_create")
        self._h = h
        self._cap = 1024
        self._buf = [np.zeros(self._cap, np.int32) for _ in range(3)]

    def add(self, request, prompt_tokens, gen_tokens=1):
        _check(lib().pps_sched_add(self._h, int(request), int(prompt_tokens), int(gen_tokens)),
               "pps_sched_add")

    def remove(self, request):
        _check(lib().pps_sched_remove(self._h, int(request)), "pps_sched_remove")

    def set_gen_tokens(self, request, gen_tokens):
        _check(lib().pps_sched_set_gen_tokens(self._h, int(request), int(gen_tokens)),
               "pps_sched_set_gen_tokens")

    def counts(self):
        a, b, c = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
        _check(lib().pps_sched_counts(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "pps_sched_counts")
        return a.value, b.value, c.value

    def step(self):
        """(requests, tokens, is_prefill) int32 arrays of the next batch."""
        n = ctypes.c_int32()
        while True:
            r, t, p = self._buf
            code = lib().pps_sched_step(self._h, r.ctypes.data_as(_I32P), t.ctypes.data_as(_I32P),
                                        p.ctypes.data_as(_I32P), self._cap, ctypes.byref(n))
            if code == 0:
                break
            pr, _, gr = self.counts()
            if pr + gr <= self._cap:
                _check(code, "pps_sched_step")
            self._cap = 2 * (pr + gr)
            self._buf = [np.zeros(self._cap, np.int32) for _ in range(3)]
        k = n.value
        return self._buf[0][:k].copy(), self._buf[1][:k].copy(), self._buf[2][:k].copy()

    def destroy(self):
        if self._h is not None:
            lib().pps_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class Engine:
    """Owner of a pps_engine: a prefix cache and a token-wise scheduler driven
    by two calls per serving step (schedule, then commit)."""

    def __init__(self, num_pages, page_size, budget, reserved=0, policy=CACHE_LRU):
        h = ctypes.c_void_p()
        _check(lib().pps_engine_create(int(num_pages), int(page_size), int(policy), int(budget),
                                       int(reserved), ctypes.byref(h)), "pps_engine_create")
        self._h = h
        self.page_size = int(page_size)
        c, s = ctypes.c_void_p(), ctypes.c_void_p()
        _check(lib().pps_engine_parts(h, ctypes.byref(c), ctypes.byref(s)), "pps_engine_parts")
        self._cache, self._sched = c, s
        self._cap = 1024
        self._sb = [np.zeros(self._cap, np.int32) for _ in range(3)]
        self._tb = [np.zeros(self._cap + 1, np.int32) for _ in range(5)]
        self._px = np.zeros(1 << 16, np.int32)

    def add(self, tokens, gen_tokens=1):
        """Admits a prompt; returns (request id, cached_len, copy or None) as Cache.begin."""
        t, tp = _host_i32(tokens)
        rid, cached = ctypes.c_int32(), ctypes.c_int32()
        cp = (ctypes.c_int32 * 3)()
        code = lib().pps_engine_add(self._h, tp, len(t), int(gen_tokens), ctypes.byref(rid),
                                    ctypes.byref(cached), cp)
        if code == -8:
            raise CacheFull(f"pps_engine_add: {status_string(code)}")
        _check(code, "pps_engine_add")
        return rid.value, cached.value, ((cp[0], cp[1], cp[2]) if cp[2] > 0 else None)

    def finish(self, request, insert=True):
        _check(lib().pps_engine_finish(self._h, int(request), int(bool(insert))),
               "pps_engine_finish")

    def counts(self):
        a, b, c = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
        _check(lib().pps_sched_counts(self._sched, ctypes.byref(a), ctypes.byref(b),
                                      ctypes.byref(c)), "pps_sched_counts")
        return a.value, b.value, c.value

    def stats(self) -> dict:
        st = _CacheStats()
        _check(lib().pps_cache_get_stats(self._cache, ctypes.byref(st)), "pps_cache_get_stats")
        return {n: getattr(st, n) for n, _ in _CacheStats._fields_}

    def pages(self, request):
        ptr, n, nt = _I32P(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pps_cache_request_pages(self._cache, int(request), ctypes.byref(ptr),
                                             ctypes.byref(n), ctypes.byref(nt)),
               "pps_cache_request_pages")
        return np.ctypeslib.as_array(ptr, shape=(n.value,)).copy() if n.value else \
            np.zeros(0, np.int32)

    def schedule(self):
        """(requests, tokens, is_prefill) of the next batch (views, valid until
        the next call)."""
        n = ctypes.c_int32()
        while True:
            r, t, p = self._sb
            code = lib().pps_engine_schedule(self._h, r.ctypes.data_as(_I32P),
                                             t.ctypes.data_as(_I32P), p.ctypes.data_as(_I32P),
                                             self._cap, ctypes.byref(n))
            if code == 0:
                break
            pr, _, gr = self.counts()
            if pr + gr <= self._cap:
                _check(code, "pps_engine_schedule")
            self._cap = 2 * (pr + gr)
            self._sb = [np.zeros(self._cap, np.int32) for _ in range(3)]
            self._tb = [np.zeros(self._cap + 1, np.int32) for _ in range(5)]
        k = n.value
        return self._sb[0][:k], self._sb[1][:k], self._sb[2][:k]

    def commit(self, gen_tokens):
        """Appends the batch's generated tokens (int32, generation entries'
        tokens concatenated in batch order) and returns the tables of the
        entries kept: (requests, q_indptr, cached_len, kv_len, page_indptr,
        page_indices), views valid until the next call."""
        g, gp = _host_i32(gen_tokens if len(gen_tokens) else np.zeros(1, np.int32))
        need, n = ctypes.c_int64(), ctypes.c_int32()
        while True:
            rq, qi, cl, kl, pi = self._tb
            code = lib().pps_engine_commit(self._h, gp, rq.ctypes.data_as(_I32P),
                                           qi.ctypes.data_as(_I32P), cl.ctypes.data_as(_I32P),
                                           kl.ctypes.data_as(_I32P), pi.ctypes.data_as(_I32P),
                                           self._px.ctypes.data_as(_I32P), len(self._px),
                                           ctypes.byref(need), ctypes.byref(n))
            if code == 0:
                break
            if code != -1 or need.value <= len(self._px):
                _check(code, "pps_engine_commit")
            self._px = np.zeros(2 * need.value, np.int32)
        k = n.value
        rq, qi, cl, kl, pi = self._tb
        return rq[:k], qi[:k + 1], cl[:k], kl[:k], pi[:k + 1], self._px[:pi[k]]

    def destroy(self):
        if self._h is not None:
            lib().pps_engine_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


_step_scratch = {}


def _host_ptr(t, dtype):
    """Address of a contiguous CPU tensor (torch, page-locked for asynchronous copies)."""
    if t.is_cuda or not t.is_contiguous() or t.dtype != dtype:
        raise PPSError(f"expected a contiguous host tensor of {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def attn_step_host(pool_k, pool_v, q, k_new, v_new, q_indptr, kv_len, page_indptr, page_indices,
                   out, tree_parent=None, sm_scale=None, num_sms=0, bw_chunk_tokens=0,
                   mma_chunk_tokens=0, flags=0, scratch=None, stream=None):
    """pps_attn_step_host: q, k_new, v_new, out are bf16 CPU tensors (page-locked
    for asynchronous copies), the tables host int32 arrays; the pool is on the
    device.  Device scratch is the given uint8 CUDA tensor, or one this module
    keeps per device and grows.  `out` is complete once the stream reaches the
    end of the step (synchronize before reading it)."""
    import torch
    pool = _pool(pool_k, pool_v)
    qi, qi_p = _host_addr(q_indptr)
    kl, kl_p = _host_addr(kv_len)
    pi, pi_p = _host_addr(page_indptr)
    px, px_p = _host_addr(page_indices if len(page_indices) else np.zeros(1, np.int32))
    tp, tp_p = (None, None) if tree_parent is None else \
        _host_addr(tree_parent if len(tree_parent) else np.zeros(1, np.int32))
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(pool_k.shape[3])
    opts = _PlanOptions(int(num_sms), int(bw_chunk_tokens), int(mma_chunk_tokens), int(flags))
    bf = torch.bfloat16
    args = [ctypes.byref(pool), _host_ptr(q, bf), _host_ptr(k_new, bf), _host_ptr(v_new, bf),
            qi_p, kl_p, pi_p, px_p, tp_p, len(kl), int(q.shape[1]), float(sm_scale),
            ctypes.byref(opts), _host_ptr(out, bf)]
    need = ctypes.c_size_t()
    dev = pool_k.device
    for _ in range(2):
        sc = scratch if scratch is not None else _step_scratch.get(dev)
        ptr = _dev(sc) if sc is not None else None
        n = sc.numel() if sc is not None else 0
        code = lib().pps_attn_step_host(*args, ptr, n, ctypes.byref(need), _stream(stream))
        if code != -4 or scratch is not None:
            break
        _step_scratch[dev] = torch.empty(int(need.value * 1.25) + 256, dtype=torch.uint8, device=dev)
    _check(code, "pps_attn_step_host")


def attn_step(pool_k, pool_v, q, k_new, v_new, q_indptr, kv_len, page_indptr, page_indices, out,
              tree_parent=None, sm_scale=None, num_sms=0, bw_chunk_tokens=0, mma_chunk_tokens=0,
              flags=0, scratch=None, stream=None, events=None):
    """pps_attn_step: q, k_new, v_new, out are bf16 CUDA tensors, the tables host
    int32 arrays.  Scratch as attn_step_host; `events` as attn_run."""
    import torch
    pool = _pool(pool_k, pool_v)
    qi, qi_p = _host_addr(q_indptr)
    kl, kl_p = _host_addr(kv_len)
    pi, pi_p = _host_addr(page_indptr)
    px, px_p = _host_addr(page_indices if len(page_indices) else np.zeros(1, np.int32))
    tp, tp_p = (None, None) if tree_parent is None else \
        _host_addr(tree_parent if len(tree_parent) else np.zeros(1, np.int32))
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(pool_k.shape[3])
    opts = _PlanOptions(int(num_sms), int(bw_chunk_tokens), int(mma_chunk_tokens), int(flags))
    bf = torch.bfloat16
    ev = None
    if events is not None:
        handles = []
        for e in events:
            if e is not None and not e.cuda_event:
                e.record()          # torch creates the CUDA event on first record
            handles.append(ctypes.c_void_p(e.cuda_event) if e is not None else None)
        ev = (ctypes.c_void_p * (2 * NUM_KERNEL_CLASSES))(*handles)
    args = [ctypes.byref(pool), _dev(q, bf), _dev(k_new, bf), _dev(v_new, bf), qi_p, kl_p, pi_p,
            px_p, tp_p, len(kl), int(q.shape[1]), float(sm_scale), ctypes.byref(opts),
            _dev(out, bf)]
    need = ctypes.c_size_t()
    dev = pool_k.device
    for _ in range(2):
        sc = scratch if scratch is not None else _step_scratch.get(dev)
        ptr = _dev(sc) if sc is not None else None
        n = sc.numel() if sc is not None else 0
        code = lib().pps_attn_step(*args, ptr, n, ctypes.byref(need), _stream(stream), ev)
        if code != -4 or scratch is not None:
            break
        _step_scratch[dev] = torch.empty(int(need.value * 1.25) + 256, dtype=torch.uint8, device=dev)
    _check(code, "pps_attn_step")


class StepCall:
    """One step of the attention path as a reusable native call:
    pps_attn_step (device rows) or pps_attn_step_host (``host=True``: rows in
    page-locked CPU tensors), with every argument marshalled once.  Each call
    still uploads the tables, appends the rows, plans the batch on the host
    and runs the attention: only the Python-side conversions are done up
    front, for a loop that repeats one batch shape (a benchmark, or a caller
    that rewrites the same host tables in place between steps).  The tensors
    and arrays given here must stay alive and keep their addresses."""

    def __init__(self, pool_k, pool_v, q, k_new, v_new, q_indptr, kv_len, page_indptr,
                 page_indices, out, tree_parent=None, host=False, sm_scale=None, num_sms=0,
                 bw_chunk_tokens=0, mma_chunk_tokens=0, flags=0, stream=None):
        import torch
        self._keep = [pool_k, pool_v, q, k_new, v_new, out]
        self._pool = _pool(pool_k, pool_v)
        tabs = [_host_addr(a) for a in (q_indptr, kv_len, page_indptr,
                                        page_indices if len(page_indices) else np.zeros(1, np.int32))]
        tp = None if tree_parent is None else \
            _host_addr(tree_parent if len(tree_parent) else np.zeros(1, np.int32))
        self._keep += [a for a, _ in tabs] + ([tp[0]] if tp else [])
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(pool_k.shape[3])
        self._opts = _PlanOptions(int(num_sms), int(bw_chunk_tokens), int(mma_chunk_tokens),
                                  int(flags))
        bf = torch.bfloat16
        rows = (lambda t: _host_ptr(t, bf)) if host else (lambda t: _dev(t, bf))
        self._host = host
        self._fn = lib().pps_attn_step_host if host else lib().pps_attn_step
        self._args = [ctypes.byref(self._pool), rows(q), rows(k_new), rows(v_new),
                      *[a for _, a in tabs], tp[1] if tp else None, len(tabs[1][0]),
                      int(q.shape[1]), float(sm_scale), ctypes.byref(self._opts), rows(out)]
        need = ctypes.c_size_t()
        extra = [] if host else [None]
        code = self._fn(*self._args, None, 0, ctypes.byref(need), _stream(stream), *extra)
        if code != -4:
            _check(code, "pps_attn_step" + ("_host" if host else ""))
        self.scratch = torch.empty(max(int(need.value), 256), dtype=torch.uint8,
                                   device=pool_k.device)
        self._tail = [_dev(self.scratch), self.scratch.numel(), None, _stream(stream)]

    def __call__(self, events=None):
        """One step.  ``events``: None, or an ``event_array`` (device rows only)."""
        if self._host:
            code = self._fn(*self._args, *self._tail)
        else:
            code = self._fn(*self._args, *self._tail, events)
        _check(code, "pps_attn_step" + ("_host" if self._host else ""))


def event_array(events):
    """2 * NUM_KERNEL_CLASSES torch.cuda.Event objects (or None) as the C array
    of cudaEvent_t that pps_attn_run_events / pps_attn_step take."""
    handles = []
    for e in events:
        if e is not None and not e.cuda_event:
            e.record()          # torch creates the CUDA event on first record
        handles.append(ctypes.c_void_p(e.cuda_event) if e is not None else None)
    return (ctypes.c_void_p * (2 * NUM_KERNEL_CLASSES))(*handles)


def gemm_bf16(a, w, c, stream=None):
    """pps_gemm_bf16: c[M, N] = a[M, K] @ w[N, K]^T (bf16 CUDA tensors)."""
    import torch
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(c.shape) != (M, N):
        raise PPSError("shapes: a [M, K], w [N, K], c [M, N]")
    _check(lib().pps_gemm_bf16(_dev(a, torch.bfloat16), _dev(w, torch.bfloat16),
                               _dev(c, torch.bfloat16), int(M), int(N), int(K), _stream(stream)),
           "pps_gemm_bf16")


def partition(q_indptr, kv_len, page_indptr, page_indices, page_size, num_parts):
    """pps_partition: (part of each request, work of each part)."""
    qi, qi_p = _host_i32(q_indptr)
    kl, kl_p = _host_i32(kv_len)
    pi, pi_p = _host_i32(page_indptr)
    px, px_p = _host_i32(page_indices if len(page_indices) else np.zeros(1, np.int32))
    part = np.zeros(max(len(kl), 1), np.int32)
    load = np.zeros(int(num_parts), np.int64)
    _check(lib().pps_partition(qi_p, kl_p, pi_p, px_p, len(kl), int(page_size), int(num_parts),
                               part.ctypes.data_as(_I32P),
                               load.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))),
           "pps_partition")
    return part[:len(kl)], load
