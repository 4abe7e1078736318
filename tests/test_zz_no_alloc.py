"""pa_decode_static: the decode entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc while decoding -- typically a
serving engine that gave nearly all HBM to its own KV-cache pool and caching
allocator, so a library allocation would fail or eat into memory promised to KV
pages.  Its plan and partial results live in a fixed-size static device array
that every call shares.  These tests call it through the C ABI and compare its
output element by element with the fp64 oracle (and with the plan-based entry
point pa_plan_build + pa_plan_refresh + pa_decode, within the same bounds),
over two calls in a row that reuse the static array; every call reports its
device error word, which must stay 0 except where a fault is planted.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
from __future__ import annotations

import ctypes

import pytest
import torch

from helpers import TOL, oracle_decode, parity
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu


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


def static_decode(lib, w, out, errors, max_query_len=1, budget=0, kind=binding.PROPORTIONAL):
    """One pa_decode_static call; `errors` (a device int32 the caller zeroes)
    receives the PA_DEVERR_* bits."""
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


def checked_call(lib, w, max_query_len=1, budget=0, kind=binding.PROPORTIONAL, what="",
                 absolute=True):
    """A static call into a NaN-filled output (every row must be written),
    its error word 0, its result against the oracle and the planned path.
    absolute=False holds it to the relative bounds only (sharp attention,
    outputs of order 1-4, where bf16 rounding alone exceeds 1e-2)."""
    errors = torch.zeros(1, dtype=torch.int32, device=w.q.device)
    out = torch.full_like(w.q, float("nan"))
    st = static_decode(lib, w, out, errors, max_query_len, budget, kind)
    assert st == binding.PA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0, what
    parity(out, oracle_decode(w.to("cpu")), w.kv_dtype if absolute else None, what=what)
    ref = planned_decode(w, max_query_len, budget, kind)
    if absolute:
        assert float((out.float() - ref.float()).abs().max()) <= TOL[w.kv_dtype], what
    else:
        parity(out, ref.float().cpu().numpy(), None, what=what + " vs planned path")
    return out


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_two_calls_match_the_oracle(lib, kv):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc", [4000, 17, 900, 12000, 256, 1], None, 32, 4, 128, 16, kv,
                      seed=3, kv_scale=0.05, device=dev, budget=296, spare_blocks=8)
    for call in range(2):
        if call == 1:  # the second call sees other lengths (and so another plan)
            w.context_lens.copy_(torch.tensor([3990, 30, 20, 11999, 250, 16],
                                              dtype=torch.int32, device=dev))
        checked_call(lib, w, budget=296, what=f"call {call}")


def test_sharp_long_request_as_pieces(lib):
    """One 40000-key request among short ones (one partition each, the long
    slot cut into pieces and merged), sharp queries: outputs of order 1, so a
    wrong piece or merge weight shows."""
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_sharp", [40000] + [300 + 37 * i for i in range(15)], None, 8, 2,
                      128, 16, "bf16", seed=12, device=dev, budget=32, q_std=6.0)
    for call in range(2):
        checked_call(lib, w, budget=32, what=f"call {call}", absolute=False)


def test_verify_rows_two_calls(lib):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_verify", [3000, 40, 700], [3, 3, 3], 6, 1, 256, 64, "bf16",
                      seed=4, pad_tokens=4, device=dev)
    for call in range(2):
        out = checked_call(lib, w, max_query_len=3, what=f"call {call}")
        assert torch.all(out[9:] == 0)


@pytest.mark.parametrize("D,kv", [(512, "bf16"), (1024, "fp8")])
def test_wide_heads_match_the_oracle(lib, D, kv):
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_wide", [3000, 17, 900, 5000], None, 16, 2, D, 16, kv, seed=6,
                      kv_scale=0.05, device=dev)
    checked_call(lib, w)


def test_bad_page_sets_the_error_word(lib):
    """An out-of-range block-table entry: the call reports PA_DEVERR_BAD_PAGE
    through the caller's error word, the page reads as zeros (no fault), the
    other request is still right, and the next call is clean."""
    dev = torch.device("cuda", 0)
    w = wl.make_batch("no_alloc_bad", [3000, 800], None, 8, 2, 128, 16, "bf16", seed=7,
                      device=dev)
    good = w.block_tables[0, 3].item()
    w.block_tables[0, 3] = w.k_cache.shape[0] + 5
    errors = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full_like(w.q, float("nan"))
    assert static_decode(lib, w, out, errors) == binding.PA_OK
    torch.cuda.synchronize()
    assert int(errors.item()) & binding.DEVERR_BAD_PAGE
    parity(out[[1]], oracle_decode(wl.subset(w, [1])), "bf16")
    w.block_tables[0, 3] = good
    checked_call(lib, w, what="after the bad page")


def test_too_large_a_batch_is_rejected(lib):
    dev = torch.device("cuda", 0)
    # 100-row prompts at Hq 12, D 256 need ~190 MB of partial rows: above the 32 MiB array
    w = wl.make_batch("no_alloc_big", [16384] * 7 + [100], [1] * 7 + [100], 12, 2, 256, 64,
                      "bf16", seed=5, device=dev)
    out = torch.zeros_like(w.q)
    errors = torch.zeros(1, dtype=torch.int32, device=dev)
    assert static_decode(lib, w, out, errors, max_query_len=100) == binding.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 0) and int(errors.item()) == 0
