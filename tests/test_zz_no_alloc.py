"""pa_decode_static: the decode entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc while decoding (an engine whose
caching allocator and KV pool own the HBM, or code inside a CUDA-graph
capture): its plan and partial results live in a static device array.  These
tests call it through the C ABI and compare it with the plan-based entry point
(pa_plan_build + pa_plan_refresh + pa_decode) on the same inputs, over two
calls in a row that share the static array."""
from __future__ import annotations

import ctypes

import pytest
import torch

from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp16": 1e-2, "fp8": 3e-2}


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    lib = binding.load()
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.pa_decode_static.argtypes = [P, i32, i32, i32, i32, P, P, i32, f32, f32, i32, i32, i32, P,
                                     i32, P, P, i32, i32, i32, i32, i32, f32, P, P, P]
    lib.pa_decode_static.restype = i32
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def static_decode(lib, w, out, max_query_len=1, budget=0, kind=binding.PROPORTIONAL,
                  errors=None):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q_code = binding.FP16 if w.q.dtype == torch.float16 else binding.BF16
    return lib.pa_decode_static(
        _p(w.q), q_code, w.num_tokens, w.num_q_heads, w.head_dim, _p(w.k_cache), _p(w.v_cache),
        binding.kv_code(w.k_cache), w.k_scale, w.v_scale, w.k_cache.shape[0], w.num_kv_heads,
        w.block_size, _p(w.block_tables), w.block_tables.shape[1], _p(w.context_lens),
        _p(w.cu_query_lens), w.num_seqs, max_query_len, w.max_partitions, budget, kind, w.scale,
        _p(out), _p(errors), stream)


def planned_decode(w, max_query_len=1, budget=0, kind=binding.PROPORTIONAL):
    plan = binding.Plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                        max_query_len=max_query_len, max_tokens=w.num_tokens,
                        max_partitions=w.max_partitions, budget=budget, kind=kind,
                        device=w.q.device)
    plan.refresh(w.context_lens, w.cu_query_lens)
    out = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    return out


def _max_diff(a, b):
    return float((a.float() - b.float()).abs().max())


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_two_calls_match_the_planned_path(lib, kv):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc", [4000, 17, 900, 12000, 256, 1], None, 32, 4, 128, 16, kv,
                      seed=3, kv_scale=0.05, device=dev, budget=296, spare_blocks=8)
    errors = torch.zeros(1, dtype=torch.int32, device=dev)
    for call in range(2):
        if call == 1:  # the second call sees other lengths (and so another plan)
            w.context_lens.copy_(torch.tensor([3990, 30, 20, 11999, 250, 16],
                                              dtype=torch.int32, device=dev))
        ref = planned_decode(w, budget=296)
        out = torch.full_like(w.q, float("nan"))  # every row must be written
        st = static_decode(lib, w, out, budget=296, errors=errors if call == 0 else None)
        assert st == binding.PA_OK, binding.status_string(st)
        torch.cuda.synchronize()
        assert int(errors.item()) == 0
        assert torch.isfinite(out.float()).all()
        assert _max_diff(out, ref) <= TOL[kv]


def test_verify_rows_two_calls(lib):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_verify", [3000, 40, 700], [3, 3, 3], 6, 1, 256, 64, "bf16",
                      seed=4, pad_tokens=4, device=dev)
    for _ in range(2):
        ref = planned_decode(w, max_query_len=3)
        out = torch.full_like(w.q, float("nan"))
        assert static_decode(lib, w, out, max_query_len=3) == binding.PA_OK
        torch.cuda.synchronize()
        assert _max_diff(out, ref) <= TOL["bf16"]
        assert torch.all(out[9:] == 0)


def test_too_large_a_batch_is_rejected(lib):
    dev = torch.device("cuda", 0)
    # 100-row prompts at Hq 12, D 256 need ~190 MB of partial rows: above the 32 MiB array
    w = wl.make_batch("no_alloc_big", [16384] * 7 + [100], [1] * 7 + [100], 12, 2, 256, 64,
                      "bf16", seed=5, device=dev)
    out = torch.zeros_like(w.q)
    assert static_decode(lib, w, out, max_query_len=100) == binding.PA_ERR_UNSUPPORTED
    assert torch.all(out == 0)


@pytest.mark.parametrize("D,kv", [(512, "bf16"), (1024, "fp8")])
def test_wide_heads_match_the_planned_path(lib, D, kv):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_wide", [3000, 17, 900, 5000], None, 16, 2, D, 16, kv, seed=6,
                      kv_scale=0.05, device=dev)
    ref = planned_decode(w)
    out = torch.full_like(w.q, float("nan"))
    assert static_decode(lib, w, out) == binding.PA_OK
    torch.cuda.synchronize()
    assert _max_diff(out, ref) <= TOL[kv]
