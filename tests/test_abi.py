"""The C ABI without a GPU: the library loads, exports every function that
include/pa.h declares, and rejects bad arguments before touching CUDA."""
from __future__ import annotations

import ctypes

import pytest

from paged_kv_decode_split_gb300 import _build, binding


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = binding.declared_symbols()
    for must in ("pa_plan_build", "pa_plan_refresh", "pa_decode", "pa_plan_destroy",
                 "pa_plan_download", "pa_plan_read_errors", "pa_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in binding.declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code, name in ((0, "PA_OK"), (-1, "PA_ERR_INVALID_ARG"), (-2, "PA_ERR_UNSUPPORTED"),
                       (-3, "PA_ERR_PLAN_MISMATCH"), (-4, "PA_ERR_CUDA"), (-5, "PA_ERR_OOM")):
        assert binding.status_string(code) == name
    assert binding.status_string(17) == "PA_ERR_UNKNOWN"


def _build_status(lib, **kw):
    args = dict(device=0, n=4, hq=8, hkv=2, d=64, qlen=1, tokens=4, parts=0, budget=0, kind=0)
    args.update(kw)
    h = ctypes.c_void_p()
    st = lib.pa_plan_build(ctypes.byref(h), args["device"], args["n"], args["hkv"], args["hq"],
                           args["d"], args["qlen"], args["tokens"], args["parts"],
                           args["budget"], args["kind"])
    assert h.value is None  # nothing allocated on any rejected call
    return st


@pytest.mark.parametrize("kw,want", [
    (dict(n=0), binding.PA_ERR_INVALID_ARG),
    (dict(device=-1), binding.PA_ERR_INVALID_ARG),
    (dict(qlen=0), binding.PA_ERR_INVALID_ARG),
    (dict(kind=7), binding.PA_ERR_INVALID_ARG),
    (dict(n=4097), binding.PA_ERR_UNSUPPORTED),
    (dict(hq=6, hkv=4), binding.PA_ERR_UNSUPPORTED),
    (dict(hq=2, hkv=8), binding.PA_ERR_UNSUPPORTED),  # num_kv_heads comes before num_q_heads
    (dict(d=96), binding.PA_ERR_UNSUPPORTED),
    (dict(d=192), binding.PA_ERR_UNSUPPORTED),   # above 128: multiples of 128 only
    (dict(d=1152), binding.PA_ERR_UNSUPPORTED),  # above 1024
    (dict(parts=1 << 20), binding.PA_ERR_UNSUPPORTED),
])
def test_plan_build_rejects_bad_parameters_before_cuda(lib, kw, want):
    assert _build_status(lib, **kw) == want


def test_sparse_select_rejects_bad_arguments_before_cuda(lib):
    """Validation returns before any launch, so these need no GPU."""
    assert lib.pa_sparse_select(None, 0, None, None, 4, 2, 16, 0, 1, 1, None, 2, None, None,
                                None) == binding.PA_ERR_INVALID_ARG
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation
    # top_k > 0 without scores
    assert lib.pa_sparse_select(None, 4, p, p, 4, 2, 16, 2, 1, 1, p, 4, p, None,
                                None) == binding.PA_ERR_INVALID_ARG
    # rows narrower than init + top_k + local
    assert lib.pa_sparse_select(p, 4, p, p, 4, 2, 16, 2, 1, 1, p, 3, p, None,
                                None) == binding.PA_ERR_INVALID_ARG
    # score rows shorter than the block table
    assert lib.pa_sparse_select(p, 3, p, p, 4, 2, 16, 2, 1, 1, p, 4, p, None,
                                None) == binding.PA_ERR_INVALID_ARG
    # negative counts
    assert lib.pa_sparse_select(p, 4, p, p, 4, 2, 16, -1, 1, 1, p, 4, p, None,
                                None) == binding.PA_ERR_INVALID_ARG
    # more requests than the planner's domain
    assert lib.pa_sparse_select(p, 4, p, p, 4, 4097, 16, 2, 1, 1, p, 4, p, None,
                                None) == binding.PA_ERR_UNSUPPORTED


def test_null_handles(lib):
    assert lib.pa_plan_build(None, 0, 4, 2, 8, 64, 1, 4, 0, 0, 0) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_refresh(None, None, None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_destroy(None) == binding.PA_OK
    assert lib.pa_plan_info(None, None, None, None, None, None, None, None) == \
        binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_download(None, None, None, None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_split_events(None, None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_call_events(None, None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_window(None, 5) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_kv_dtype(None, binding.BF16) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_wait_limit(None, 0) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_set_fused_merge(None, 1) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_get_fused_merge(None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_plan_skip_stage_for_test(None, -1) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode_ex(None, None, 0, 1, 8, 64, None, None, 0, 1.0, 1.0, 1, 2, 16, None, 1,
                            None, None, 1, 1.0, None, binding.K_ROWS, None,
                            None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode(None, None, 0, 1, 8, 64, None, None, 0, 1.0, 1.0, 1, 2, 16, None, 1,
                         None, None, 1, 1.0, None, None) == binding.PA_ERR_INVALID_ARG
