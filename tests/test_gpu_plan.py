"""The on-device planner against the oracle's plan rule: bit-exact work_info and
reduce_info for every configuration, random batches and the edge cases."""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _gpu_plan(dev, lens, cu, Hq, Hkv, D=128, P=0, W=0, kind=binding.PROPORTIONAL, max_qlen=None,
              max_tokens=None, window=0):
    n = len(lens)
    if max_qlen is None:
        max_qlen = 1 if cu is None else max(1, int(np.max(np.diff(cu))))
    if max_tokens is None:
        max_tokens = n if cu is None else max(1, int(cu[-1]))
    plan = binding.Plan(n, Hq, Hkv, D, max_query_len=max_qlen, max_tokens=max_tokens,
                        max_partitions=P, budget=W, kind=kind, device=dev)
    plan.set_window(window)
    lt = torch.tensor(np.asarray(lens, np.int32), device=dev)
    ct = None if cu is None else torch.tensor(np.asarray(cu, np.int32), device=dev)
    plan.refresh(lt, ct)
    work, red = plan.download()
    return plan, work.numpy(), red.numpy()


def _oracle_plan(plan, lens, cu, Hkv, kind, window=0):
    info = plan.info()
    return oracle.plan(np.asarray(lens, np.int32), None if cu is None else np.asarray(cu, np.int32),
                       Hkv, info["max_partitions"], info["budget"], kind, window=window)


@pytest.mark.parametrize("name", list(wl.CONFIGS))
@pytest.mark.parametrize("kind", [binding.PROPORTIONAL, binding.UNIFORM])
def test_config_plans_bit_exact(dev, name, kind):
    w = wl.CONFIGS[name](0, dev) if name not in ("large_bf16", "large_fp8") else None
    if w is None:  # only the lengths matter: skip drawing 8 GB of cache values
        lens = wl.lognormal_lengths(512, 2048, 1.2, 16, 65536, 0)
        cu, Hq, Hkv, W, win = None, 64, 8, 0, 0
    else:
        lens = w.context_lens.tolist()
        cu = None if w.cu_query_lens is None else w.cu_query_lens.tolist()
        Hq, Hkv, W, win = w.num_q_heads, w.num_kv_heads, w.budget or 0, w.window
    plan, work, red = _gpu_plan(dev, lens, cu, Hq, Hkv, W=W, kind=kind, window=win)
    ow, orr = _oracle_plan(plan, lens, cu, Hkv, kind, window=win)
    assert np.array_equal(work, ow)
    assert np.array_equal(red, orr)
    assert plan.read_errors() == 0


def test_skewed_plan_sizes(dev):
    # 2 x 148 budget, Hkv 4 -> capacity 74
    for seed in range(3):
        w = wl.skewed(seed, "cpu")
        plan, work, red = _gpu_plan(dev, w.context_lens.tolist(), None, 32, 4, W=296)
        assert plan.capacity == 74
        assert 1 <= red[:, 1].sum() <= 74


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("kind", [binding.PROPORTIONAL, binding.UNIFORM])
def test_random_batches_bit_exact(dev, seed, kind):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.choice([1, 2, 7, 31, 300, 1024, 4095, 4096]))
    lens = np.clip(np.round(np.exp(rng.normal(np.log(3000), 1.7, n))), 1, 200000).astype(np.int32)
    lens[rng.random(n) < 0.15] = 0
    cu = None
    if seed % 2:
        ql = rng.integers(0, 5, n)
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    P = int(rng.choice([1, 3, 64, 256]))
    W = int(rng.choice([0, 17, 296, 1000]))
    plan, work, red = _gpu_plan(dev, lens, cu, 8 * Hkv, Hkv, P=P, W=W, kind=kind)
    ow, orr = _oracle_plan(plan, lens, cu, Hkv, kind)
    assert np.array_equal(work, ow) and np.array_equal(red, orr)


def test_refresh_in_place_follows_new_lengths(dev):
    lens = [5000, 300, 70000, 12]
    plan, _, _ = _gpu_plan(dev, lens, None, 32, 4, W=296)
    lt = torch.tensor(lens, dtype=torch.int32, device=dev)
    for step in range(5):
        lt += torch.tensor([1, 257, 0, 1000 * step], dtype=torch.int32, device=dev)
        plan.refresh(lt)
        work, red = plan.download()
        ow, orr = _oracle_plan(plan, lt.tolist(), None, 4, binding.PROPORTIONAL)
        assert np.array_equal(work.numpy(), ow) and np.array_equal(red.numpy(), orr)


def test_all_requests_empty(dev):
    plan, work, red = _gpu_plan(dev, [0, 0, 0], None, 8, 1)
    assert np.all(red[:, 1] == 0) and np.all(work[:, 0] == -1)


def test_query_rows_beyond_plan_limits_empty_the_plan(dev):
    cu = [0, 1, 9, 10]  # request 1 owns 8 rows
    plan, work, red = _gpu_plan(dev, [500, 500, 500], cu, 8, 1, max_qlen=4, max_tokens=16)
    assert np.all(red[:, 1] == 0)
    assert plan.read_errors() & binding.DEVERR_PLAN_OVERFLOW
    plan2, _, red2 = _gpu_plan(dev, [500, 500, 500], cu, 8, 1, max_qlen=8, max_tokens=9)
    assert np.all(red2[:, 1] == 0)
    assert plan2.read_errors() & binding.DEVERR_PLAN_OVERFLOW


@pytest.mark.parametrize("hkv,hq", [(2, 8), (4, 4), (1, 6)])
def test_plan_build_in_the_contract_order(dev, hkv, hq):
    """pa_plan_build(plan, device, num_seqs, num_kv_heads, num_q_heads, head_dim,
    ...) called through ctypes in that order: the capacity C = min(n P,
    max(n, ceil(W / Hkv))) that pa_plan_info and pa_plan_download report
    depends on which argument is the kv head count (with Hq != Hkv a swap gives
    another C), and the plan decodes a batch of those head counts."""
    lib = binding.load()
    n, W = 8, 64
    h = ctypes.c_void_p()
    st = lib.pa_plan_build(ctypes.byref(h), dev.index, n, hkv, hq, 128, 1, n, 0, W,
                           binding.PROPORTIONAL)
    assert st == binding.PA_OK, binding.status_string(st)
    try:
        cap = ctypes.c_int()
        seqs = ctypes.c_int()
        assert lib.pa_plan_info(h, ctypes.byref(cap), ctypes.byref(seqs), None, None, None, None,
                                None) == binding.PA_OK
        want = min(n * 256, max(n, math.ceil(W / hkv)))
        assert cap.value == want and seqs.value == n
        lens = torch.tensor([300, 17, 4000, 1, 900, 2600, 64, 5], dtype=torch.int32, device=dev)
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert lib.pa_plan_refresh(h, ctypes.c_void_p(lens.data_ptr()), None, s) == binding.PA_OK
        work = torch.empty((want, 4), dtype=torch.int32)
        red = torch.empty((n, 2), dtype=torch.int32)
        cap2 = ctypes.c_int(-1)
        assert lib.pa_plan_download(h, ctypes.c_void_p(work.data_ptr()),
                                    ctypes.c_void_p(red.data_ptr()), ctypes.byref(cap2),
                                    s) == binding.PA_OK
        assert cap2.value == want
        ow, orr = oracle.plan(lens.cpu().numpy(), None, hkv, 256, W)
        assert np.array_equal(work.numpy(), ow) and np.array_equal(red.numpy(), orr)
    finally:
        assert lib.pa_plan_destroy(h) == binding.PA_OK
