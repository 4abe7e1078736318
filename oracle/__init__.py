"""fp64 CPU oracle for paged-KV GQA decode attention and its work plan.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers allowed.  The product
path (``paged_kv_decode_split_gb300``) never imports this package, and this
package never imports the product.  The arithmetic lives in ``pa_oracle.c``
(plain C, compiled here with gcc, no shared code with the CUDA library); this
module only marshals numpy arrays into it.

Inputs are raw element bits: bf16/fp16 tensors as ``uint16`` arrays, fp8 as
``uint8``.  Dtype codes: 0 = bf16, 1 = fp16, 2 = fp8 e4m3fn.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpa_oracle.so")

BF16, FP16, FP8_E4M3 = 0, 1, 2
PLAN_PROPORTIONAL, PLAN_UNIFORM = 0, 1
TILE = 256  # partition tile in tokens

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library (gcc, OpenMP, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = dbl
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = dbl
        lib.oracle_e4m3fn_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3fn_to_double.restype = dbl
        lib.oracle_plan_capacity.argtypes = [i32, i32, i32, i32]
        lib.oracle_plan_capacity.restype = i64
        lib.oracle_plan.argtypes = [i32, P, P, i32, i32, i32, i32, i32, P, i64, P]
        lib.oracle_plan.restype = i64
        lib.oracle_plan_window.argtypes = [i32, P, P, i32, i32, i32, i32, i32, i32, P, i64, P]
        lib.oracle_plan_window.restype = i64
        lib.oracle_sparse_select.argtypes = [P, i32, P, P, i32, i32, i32, i32, i32, i32, P,
                                             i32, P]
        lib.oracle_sparse_select.restype = i32
        lib.oracle_decode.argtypes = [P, i32, i32, i32, i32, P, P, i32, dbl, dbl, i32, i32,
                                      P, i32, P, P, i32, dbl, P]
        lib.oracle_decode.restype = None
        lib.oracle_decode_ext.argtypes = [P, i32, i32, i32, i32, P, P, i32, dbl, dbl, i32, i32,
                                          P, i32, P, P, i32, dbl, i32, P, i32, P]
        lib.oracle_decode_ext.restype = None
        lib.oracle_decode_planned.argtypes = [P, i32, i32, i32, i32, P, P, i32, dbl, dbl, i32,
                                              i32, P, i32, P, P, i32, dbl, P, P, i32, P]
        lib.oracle_decode_planned.restype = None
        lib.oracle_decode_planned_ext.argtypes = [P, i32, i32, i32, i32, P, P, i32, dbl, dbl,
                                                  i32, i32, P, i32, P, P, i32, dbl, P, P, i32,
                                                  i32, P, i32, P]
        lib.oracle_decode_planned_ext.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(bits)


def fp16_to_double(bits: int) -> float:
    return _load().oracle_fp16_to_double(bits)


def e4m3fn_to_double(byte: int) -> float:
    return _load().oracle_e4m3fn_to_double(byte)


def num_threads() -> int:
    return _load().oracle_num_threads()


def plan_capacity(n: int, num_kv_heads: int, max_partitions: int, budget: int) -> int:
    return int(_load().oracle_plan_capacity(n, num_kv_heads, max_partitions, budget))


def plan(context_lens, cu_query_lens, num_kv_heads: int, max_partitions: int, budget: int,
         kind: int = PLAN_PROPORTIONAL, tile: int = TILE, window: int = 0):
    """Work plan for the given lengths (and sliding window; 0 = none).  Returns
    (work_info [C,4], reduce_info [n,2])."""
    lens = _c(context_lens, np.int32)
    cu = _c(cu_query_lens, np.int32)
    n = lens.shape[0]
    C = plan_capacity(n, num_kv_heads, max_partitions, budget)
    work = np.zeros((C, 4), dtype=np.int32)
    red = np.zeros((n, 2), dtype=np.int32)
    if window:
        got = _load().oracle_plan_window(n, _ptr(lens), _ptr(cu), num_kv_heads, max_partitions,
                                         budget, tile, kind, window, _ptr(work), C, _ptr(red))
    else:
        got = _load().oracle_plan(n, _ptr(lens), _ptr(cu), num_kv_heads, max_partitions, budget,
                                  tile, kind, _ptr(work), C, _ptr(red))
    assert got == C
    return work, red


def _decode_args(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                 context_lens, cu_query_lens, scale):
    q = _c(q_bits, np.uint16)
    kd = np.uint8 if kv_dtype == FP8_E4M3 else np.uint16
    k = _c(k_cache, kd)
    v = _c(v_cache, kd)
    bt = _c(block_tables, np.int32)
    lens = _c(context_lens, np.int32)
    cu = _c(cu_query_lens, np.int32)
    T, Hq, D = q.shape
    _, Hkv, bs, Dv = v.shape
    # K: [nb, Hkv, bs, D], or the 5-D [nb, Hkv, D/16, bs, 16]
    assert k.shape == v.shape or k.shape == (v.shape[0], Hkv, D // 16, bs, 16)
    assert Dv == D and Hq % Hkv == 0
    out = np.zeros((T, Hq, D), dtype=np.float64)
    args = [_ptr(q), q_dtype, T, Hq, D, _ptr(k), _ptr(v), kv_dtype, float(k_scale),
            float(v_scale), Hkv, bs, _ptr(bt), bt.shape[1], _ptr(lens), _ptr(cu),
            lens.shape[0], float(scale)]
    keep = (q, k, v, bt, lens, cu)
    return args, out, keep


def decode(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
           context_lens, cu_query_lens, scale, window: int = 0, sinks=None):
    """Exact paged decode in fp64 (sliding window: 0 = none; sinks: [Hq] logits or
    None; K in either layout, told apart by its rank).  Returns out
    [num_tokens, Hq, D] float64."""
    args, out, _keep = _decode_args(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale,
                                    v_scale, block_tables, context_lens, cu_query_lens, scale)
    k_layout = 1 if np.ndim(k_cache) == 5 else 0
    if window or sinks is not None or k_layout:
        sk = _c(sinks, np.float64)
        _load().oracle_decode_ext(*args, int(window), _ptr(sk), k_layout, _ptr(out))
    else:
        _load().oracle_decode(*args, _ptr(out))
    return out


def sparse_select(scores, context_lens, block_tables, block_size: int, top_k: int,
                  init_blocks: int, local_blocks: int, sel_stride: int | None = None):
    """Sparse top-k block selection (the readings in pa_oracle.c).  scores
    [n, >= max_blocks] float32 (None when top_k == 0).  Returns (sel_tables
    [n, sel_stride] int32 -- physical blocks of the selected logical blocks in
    ascending order, then -1 -- and sel_lens [n] int32, the tokens they hold)."""
    bt = _c(block_tables, np.int32)
    lens = _c(context_lens, np.int32)
    n, max_blocks = bt.shape
    if sel_stride is None:
        sel_stride = init_blocks + top_k + local_blocks
    sc = None if scores is None else _c(scores, np.float32)
    stride = 0 if sc is None else sc.shape[1]
    if sc is None and top_k > 0:
        raise ValueError("scores are needed when top_k > 0")
    sel = np.empty((n, sel_stride), dtype=np.int32)
    sl = np.empty(n, dtype=np.int32)
    _load().oracle_sparse_select(_ptr(sc), stride, _ptr(lens), _ptr(bt), max_blocks, n,
                                 block_size, top_k, init_blocks, local_blocks, _ptr(sel),
                                 sel_stride, _ptr(sl))
    return sel, sl


def sparse_decode(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                  context_lens, scale, scores, block_size: int, top_k: int, init_blocks: int,
                  local_blocks: int):
    """Sparse top-k decode: one query token per request attends to the keys of
    its selected blocks (sparse_select), i.e. the exact decode over the sparse
    block table and the selected lengths."""
    sel, sl = sparse_select(scores, context_lens, block_tables, block_size, top_k, init_blocks,
                            local_blocks)
    return decode(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, sel, sl, None,
                  scale)


def decode_planned(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, block_tables,
                   context_lens, cu_query_lens, scale, work_info, reduce_info, tile: int = TILE,
                   window: int = 0, sinks=None):
    """The same result computed by partial softmaxes over the plan's tasks plus an
    LSE-weighted merge, in fp64."""
    args, out, _keep = _decode_args(q_bits, q_dtype, k_cache, v_cache, kv_dtype, k_scale,
                                    v_scale, block_tables, context_lens, cu_query_lens, scale)
    w = _c(work_info, np.int32)
    r = _c(reduce_info, np.int32)
    k_layout = 1 if np.ndim(k_cache) == 5 else 0
    if window or sinks is not None or k_layout:
        sk = _c(sinks, np.float64)
        _load().oracle_decode_planned_ext(*args, _ptr(w), _ptr(r), tile, int(window), _ptr(sk),
                                          k_layout, _ptr(out))
    else:
        _load().oracle_decode_planned(*args, _ptr(w), _ptr(r), tile, _ptr(out))
    return out
