"""ctypes binding of libpa.so (include/pa.h).

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity, and their raw device pointers are handed to the C ABI together with
the current CUDA stream.  Every step of the computation runs in libpa's CUDA
kernels; there is no fallback of any kind, and a missing or unloadable library
raises immediately.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpa.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "pa.h")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_PLAN_MISMATCH = -3
PA_ERR_CUDA = -4
PA_ERR_OOM = -5

BF16, FP16, FP8_E4M3 = 0, 1, 2
_DTYPES = {"bf16": BF16, "fp16": FP16, "fp8": FP8_E4M3}
PROPORTIONAL, UNIFORM = 0, 1
K_ROWS, K_GROUPED = 0, 1  # K cache layouts: [nb, Hkv, bs, D] / [nb, Hkv, D/16, bs, 16]

DEVERR_STALE_PLAN = 0x1
DEVERR_BAD_PAGE = 0x2
DEVERR_PLAN_OVERFLOW = 0x4
DEVERR_TIMEOUT = 0x8

TILE_TOKENS = 256

_lib = None


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Loads libpa.so (built in-tree by ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.pa_plan_build.argtypes = [ctypes.POINTER(P), i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                  i32]
    lib.pa_plan_refresh.argtypes = [P, P, P, P]
    lib.pa_decode.argtypes = [P, P, i32, i32, i32, i32, P, P, i32, f32, f32, i32, i32, i32, P,
                              i32, P, P, i32, f32, P, P]
    lib.pa_decode_ex.argtypes = [P, P, i32, i32, i32, i32, P, P, i32, f32, f32, i32, i32, i32, P,
                                 i32, P, P, i32, f32, P, i32, P, P]
    lib.pa_plan_set_window.argtypes = [P, i32]
    lib.pa_plan_set_kv_dtype.argtypes = [P, i32]
    lib.pa_plan_set_wait_limit.argtypes = [P, ctypes.c_longlong]
    lib.pa_plan_set_fused_merge.argtypes = [P, i32]
    lib.pa_plan_get_fused_merge.argtypes = [P, ctypes.POINTER(i32)]
    lib.pa_plan_skip_stage_for_test.argtypes = [P, i32]
    lib.pa_plan_info.argtypes = [P, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_longlong)]
    lib.pa_plan_download.argtypes = [P, P, P, ctypes.POINTER(i32), P]
    lib.pa_plan_read_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), i32, P]
    lib.pa_plan_set_split_events.argtypes = [P, P, P]
    lib.pa_plan_set_call_events.argtypes = [P, P, P]
    lib.pa_plan_destroy.argtypes = [P]
    lib.pa_sparse_select.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, i32, P, i32, P, P, P]
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    for name in ("pa_plan_build", "pa_plan_refresh", "pa_decode", "pa_decode_ex",
                 "pa_plan_set_window", "pa_plan_set_kv_dtype", "pa_plan_info",
                 "pa_plan_set_wait_limit", "pa_plan_skip_stage_for_test",
                 "pa_plan_set_fused_merge", "pa_plan_get_fused_merge",
                 "pa_plan_download", "pa_plan_read_errors", "pa_plan_set_split_events",
                 "pa_plan_set_call_events", "pa_sparse_select",
                 "pa_plan_destroy"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def declared_symbols() -> list[str]:
    """Names of the functions include/pa.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PaError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, device: torch.device, dtypes=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")


def kv_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    raise ValueError(f"unsupported KV cache dtype {t.dtype}")


class Plan:
    """A work plan plus its scratch, bound to one device (pa_plan_build)."""

    def __init__(self, num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 max_query_len: int = 1, max_tokens: Optional[int] = None,
                 max_partitions: int = 0, budget: int = 0, kind: int = PROPORTIONAL,
                 device=None):
        lib = load()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self.num_seqs, self.num_q_heads, self.num_kv_heads = num_seqs, num_q_heads, num_kv_heads
        self.head_dim, self.max_query_len = head_dim, max_query_len
        self.max_tokens = max_tokens if max_tokens is not None else num_seqs * max_query_len
        h = ctypes.c_void_p()
        _check(lib.pa_plan_build(ctypes.byref(h), self.device.index, num_seqs, num_kv_heads,
                                 num_q_heads, head_dim, max_query_len, self.max_tokens,
                                 max_partitions, budget, kind), "pa_plan_build")
        self._h = h
        self.with_cu = None

    # -- facts
    def info(self) -> dict:
        v = [ctypes.c_int() for _ in range(6)]
        b = ctypes.c_longlong()
        _check(load().pa_plan_info(self._h, *[ctypes.byref(x) for x in v], ctypes.byref(b)),
               "pa_plan_info")
        keys = ("capacity", "num_seqs", "budget", "max_partitions", "kind", "device")
        d = {k: x.value for k, x in zip(keys, v)}
        d["device_bytes"] = b.value
        return d

    @property
    def capacity(self) -> int:
        return self.info()["capacity"]

    # -- plan
    def refresh(self, context_lens: torch.Tensor, cu_query_lens: Optional[torch.Tensor] = None,
                stream=None):
        _need(context_lens, "context_lens", self.device, (torch.int32,))
        if cu_query_lens is not None:
            _need(cu_query_lens, "cu_query_lens", self.device, (torch.int32,))
        _check(load().pa_plan_refresh(self._h, _ptr(context_lens), _ptr(cu_query_lens),
                                      _stream(self.device, stream)), "pa_plan_refresh")

    def download(self, stream=None):
        """(work_info [C,4], reduce_info [n,2]) as int32 CPU tensors (synchronises)."""
        C = self.capacity
        work = torch.empty((C, 4), dtype=torch.int32)
        red = torch.empty((self.num_seqs, 2), dtype=torch.int32)
        cap = ctypes.c_int(-1)
        _check(load().pa_plan_download(self._h, _ptr(work), _ptr(red), ctypes.byref(cap),
                                       _stream(self.device, stream)), "pa_plan_download")
        assert cap.value == C
        return work, red

    def read_errors(self, clear: bool = True, stream=None) -> int:
        e = ctypes.c_uint32()
        _check(load().pa_plan_read_errors(self._h, ctypes.byref(e), int(clear),
                                          _stream(self.device, stream)), "pa_plan_read_errors")
        return e.value

    def set_split_events(self, start=None, stop=None):
        a = None if start is None else ctypes.c_void_p(start.cuda_event)
        b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
        _check(load().pa_plan_set_split_events(self._h, a, b), "pa_plan_set_split_events")

    def set_call_events(self, start=None, stop=None):
        a = None if start is None else ctypes.c_void_p(start.cuda_event)
        b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
        _check(load().pa_plan_set_call_events(self._h, a, b), "pa_plan_set_call_events")

    # -- decode
    def decode(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               block_tables: torch.Tensor, context_lens: torch.Tensor,
               cu_query_lens: Optional[torch.Tensor] = None, scale: Optional[float] = None,
               k_scale: float = 1.0, v_scale: float = 1.0, out: Optional[torch.Tensor] = None,
               stream=None, sinks: Optional[torch.Tensor] = None) -> torch.Tensor:
        dev = self.device
        if sinks is not None:
            _need(sinks, "sinks", dev, (torch.float32,))
            if sinks.shape != (q.shape[1],):
                raise ValueError("sinks must be [num_q_heads] float32")
        _need(q, "q", dev, (torch.bfloat16, torch.float16))
        _need(k_cache, "k_cache", dev)
        _need(v_cache, "v_cache", dev, (k_cache.dtype,))
        # K as [nb, Hkv, bs, D], or grouped as [nb, Hkv, D/16, bs, 16] (5-D)
        grouped = k_cache.dim() == 5
        _need(block_tables, "block_tables", dev, (torch.int32,))
        _need(context_lens, "context_lens", dev, (torch.int32,))
        if cu_query_lens is not None:
            _need(cu_query_lens, "cu_query_lens", dev, (torch.int32,))
        if grouped:
            nb_, hk_, g_, bs_, x_ = k_cache.shape
            if x_ != 16 or v_cache.dim() != 4 or tuple(v_cache.shape) != (nb_, hk_, bs_, 16 * g_):
                raise ValueError("grouped K must be [num_blocks, Hkv, D/16, bs, 16] with V "
                                 "[num_blocks, Hkv, bs, D]")
        if q.dim() != 3 or v_cache.dim() != 4 or (not grouped and v_cache.shape != k_cache.shape):
            raise ValueError("q must be [T, Hq, D]; k/v caches [num_blocks, Hkv, bs, D]")
        if block_tables.dim() != 2:
            raise ValueError("block_tables must be [num_seqs, max_blocks]")
        if out is None:
            out = torch.empty_like(q)
        else:
            _need(out, "out", dev, (q.dtype,))
            if out.shape != q.shape:
                raise ValueError("out must have q's shape")
        T, Hq, D = q.shape
        nb, Hkv, bs, Dk = v_cache.shape
        if Dk != D:
            raise ValueError("cache head_dim differs from q's")
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        qcode = FP16 if q.dtype == torch.float16 else BF16
        _check(load().pa_decode_ex(self._h, _ptr(q), qcode, T, Hq, D, _ptr(k_cache),
                                   _ptr(v_cache), kv_code(k_cache), float(k_scale),
                                   float(v_scale), nb, Hkv, bs, _ptr(block_tables),
                                   block_tables.shape[1], _ptr(context_lens), _ptr(cu_query_lens),
                                   context_lens.shape[0], float(scale), _ptr(sinks),
                                   K_GROUPED if grouped else K_ROWS, _ptr(out),
                                   _stream(dev, stream)), "pa_decode_ex")
        return out

    def set_window(self, sliding_window: int):
        """Sliding window for the next refresh on (0: none)."""
        _check(load().pa_plan_set_window(self._h, int(sliding_window)), "pa_plan_set_window")

    def set_kv_dtype(self, kv_dtype):
        """Cache element type the decode calls will read ("bf16", "fp16",
        "fp8" or a PA_* code), for the next refresh on."""
        code = _DTYPES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
        _check(load().pa_plan_set_kv_dtype(self._h, code), "pa_plan_set_kv_dtype")

    @property
    def fused_merge(self) -> bool:
        """True when pa_decode merges the partials inside the split kernel."""
        v = ctypes.c_int()
        _check(load().pa_plan_get_fused_merge(self._h, ctypes.byref(v)), "pa_plan_get_fused_merge")
        return bool(v.value)

    def set_fused_merge(self, enable: bool):
        """Merge in the split kernel (where the plan allows it) or in a separate
        merge kernel."""
        _check(load().pa_plan_set_fused_merge(self._h, int(bool(enable))),
               "pa_plan_set_fused_merge")

    def kernels_per_decode(self) -> int:
        return 1 if self.fused_merge else 2

    def set_wait_limit(self, wait_limit_ns: int):
        """Limit of the decode kernel's bounded waits (0: the default 4 s)."""
        _check(load().pa_plan_set_wait_limit(self._h, int(wait_limit_ns)),
               "pa_plan_set_wait_limit")

    def skip_stage_for_test(self, stage: int):
        """Test hook: every CTA leaves its pipeline stage `stage` un-issued, so
        its waits run out (-1: off)."""
        _check(load().pa_plan_skip_stage_for_test(self._h, int(stage)),
               "pa_plan_skip_stage_for_test")

    def close(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            _check(load().pa_plan_destroy(h), "pa_plan_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_for(w, kind: int = PROPORTIONAL, budget: Optional[int] = None,
             max_partitions: Optional[int] = None, device=None) -> Plan:
    """A plan sized for a Workload (see workloads.py)."""
    ql = 1
    if w.cu_query_lens is not None:
        cu = w.cu_query_lens.cpu()
        ql = max(1, int((cu[1:] - cu[:-1]).max()))
    plan = Plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, max_query_len=ql,
                max_tokens=w.num_tokens,
                max_partitions=w.max_partitions if max_partitions is None else max_partitions,
                budget=(w.budget or 0) if budget is None else budget, kind=kind, device=device)
    if getattr(w, "window", 0):
        plan.set_window(w.window)
    plan.set_kv_dtype(w.kv_dtype)
    return plan


def decode_workload(plan: Plan, w, out=None, stream=None, sinks=None) -> torch.Tensor:
    return plan.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                       w.cu_query_lens, w.scale, w.k_scale, w.v_scale, out=out, stream=stream,
                       sinks=sinks)


def sparse_select(block_scores: Optional[torch.Tensor], context_lens: torch.Tensor,
                  block_tables: torch.Tensor, block_size: int, top_k: int, init_blocks: int,
                  local_blocks: int, sel_block_tables: Optional[torch.Tensor] = None,
                  sel_context_lens: Optional[torch.Tensor] = None,
                  device_errors: Optional[torch.Tensor] = None, stream=None):
    """pa_sparse_select: the sparse block table [n, init + top_k + local] (or the
    width of sel_block_tables when given) and the selected lengths [n], both
    int32 on the device of context_lens."""
    dev = context_lens.device
    _need(context_lens, "context_lens", dev, (torch.int32,))
    _need(block_tables, "block_tables", dev, (torch.int32,))
    if block_tables.dim() != 2 or block_tables.shape[0] != context_lens.shape[0]:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    n, max_blocks = block_tables.shape
    stride = 0
    if block_scores is not None:
        _need(block_scores, "block_scores", dev, (torch.float32,))
        if block_scores.dim() != 2 or block_scores.shape[0] != n:
            raise ValueError("block_scores must be [num_seqs, >= max_blocks]")
        stride = block_scores.shape[1]
    if sel_block_tables is None:
        sel_block_tables = torch.empty((n, init_blocks + top_k + local_blocks), dtype=torch.int32,
                                       device=dev)
    _need(sel_block_tables, "sel_block_tables", dev, (torch.int32,))
    if sel_context_lens is None:
        sel_context_lens = torch.empty(n, dtype=torch.int32, device=dev)
    _need(sel_context_lens, "sel_context_lens", dev, (torch.int32,))
    if device_errors is not None:
        _need(device_errors, "device_errors", dev, (torch.int32,))
    with torch.cuda.device(dev):
        _check(load().pa_sparse_select(_ptr(block_scores), stride, _ptr(context_lens),
                                       _ptr(block_tables), max_blocks, n, int(block_size),
                                       int(top_k), int(init_blocks), int(local_blocks),
                                       _ptr(sel_block_tables), sel_block_tables.shape[1],
                                       _ptr(sel_context_lens), _ptr(device_errors),
                                       _stream(dev, stream)), "pa_sparse_select")
    return sel_block_tables, sel_context_lens
