"""The CUDA decode path (planner + split-KV kernel + merge, through the C ABI)
against the fp64 oracle, element by element.

Tolerances (max |gpu - oracle| over every output element, outputs rounded to
bf16/fp16): 1e-2 with 16-bit caches, 3e-2 with fp8-e4m3 caches, the oracle
decoding the same fp8 bytes; and the relative bounds of helpers.parity over the
whole output and every row."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from helpers import TOL, oracle_plan, oracle_decode, parity
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def run(w, kind=binding.PROPORTIONAL, budget=None, max_partitions=None, out=None):
    plan = binding.plan_for(w, kind, budget, max_partitions)
    plan.refresh(w.context_lens, w.cu_query_lens)
    o = binding.decode_workload(plan, w, out=out)
    torch.cuda.synchronize()
    return o, plan


def max_diff(out: torch.Tensor, ref: np.ndarray) -> float:
    """max |gpu - oracle|, after checking the relative bounds (whole output and
    every row) and that the oracle's zero rows are exactly zero."""
    return parity(out, ref)["max_abs"]


def check(w, **kw):
    out, plan = run(w, **kw)
    ref = oracle_decode(w.to("cpu"))
    d = max_diff(out, ref)
    assert d <= TOL[w.kv_dtype], f"{w.name}: max|diff| {d}"
    assert plan.read_errors() == 0
    return out, ref, d


def batch(dev, lens, ql=None, H=(8, 2), D=128, bs=16, kv="bf16", q="bf16", pad=0, seed=0, **kw):
    return wl.make_batch("case", lens, ql, H[0], H[1], D, bs, kv, q, seed=seed, pad_tokens=pad,
                         kv_scale=0.05, device=dev, **kw)



# ---------------------------------------------------------------- small sweeps

def test_tiny(dev):
    for kind in (binding.PROPORTIONAL, binding.UNIFORM):
        check(wl.tiny(0, dev), kind=kind)


RAGGED = [1, 15, 17, 255, 256, 257, 700, 1500]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16"),
                                  ("fp8", "fp16")])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_dtype_shape_sweep(dev, D, kv, q, bs):
    check(batch(dev, RAGGED, H=(8, 2), D=D, bs=bs, kv=kv, q=q, seed=D + bs))


@pytest.mark.parametrize("H", [(4, 4), (6, 1), (12, 2), (16, 2), (32, 4), (64, 8)])
def test_gqa_group_sizes(dev, H):
    check(batch(dev, [33, 600, 1200], H=H, D=128, kv="bf16", seed=H[0]))


@pytest.mark.parametrize("P,W", [(1, 8), (2, 16), (4, 64), (16, 512), (256, 4096), (256, 296)])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_split_count_sweep(dev, P, W, kv):
    """The error must not grow with the number of partitions (the partials stay
    fp32 and are merged by their log-sum-exp)."""
    w = batch(dev, [9000, 40, 2600], H=(8, 1), D=128, kv=kv, seed=5, budget=W, max_partitions=P)
    _, _, d = check(w)
    assert d <= TOL[kv]


@pytest.mark.parametrize("kv,bs,D", [("bf16", 16, 128), ("fp8", 16, 128), ("fp8", 128, 128),
                                     ("bf16", 128, 64), ("fp16", 64, 64)])
def test_uneven_slots_run_as_pieces(dev, kv, bs, D):
    """A small budget leaves one slot per request, one of them 150x longer than
    the rest: the split kernel runs that slot as several pieces, and the merge
    combines them (the plan itself is unchanged).  CTAs take several pieces
    each, so the next piece's first stages are issued during the epilogue; with
    16-key pages both producer warps issue, with pages that hold a whole stage
    (fp8 at 128 keys, 64-dim bf16 at 128 keys) warp 0 issues K and V alone."""
    w = batch(dev, [40000] + [300 + 37 * i for i in range(15)], H=(8, 2), D=D, bs=bs, kv=kv,
              q="fp16" if kv == "fp16" else "bf16", seed=12, budget=32)
    out, plan = run(w)
    work, red = plan.download()
    assert bool((red[:, 1] == 1).all())  # one partition per request: pieces are not partitions
    ref = oracle_decode(w.to("cpu"))
    assert max_diff(out, ref) <= TOL[kv]
    assert plan.read_errors() == 0


@pytest.mark.parametrize("case", ["d128_48x8", "d1024_bf16", "d896_fp16", "d1024_fp8_plan_bf16",
                                  "d1024_bf16_plan_fp8"])
def test_more_ctas_than_one_wave(dev, case):
    """Plans whose CTAs (capacity x kv heads) outnumber those the GPU runs at
    once: the refresh cuts even slots into short pieces that the first wave
    shares, and CTAs past the resident count start by taking items from the
    work counter.  The plan (work_info, reduce_info) is the oracle's; the
    output matches the oracle.  A plan told another cache type than the decode
    reads is still correct (only the piece sizes differ)."""
    if case == "d128_48x8":  # C = n = 48, 384 CTAs; slots of 8 tiles
        w = batch(dev, [2048] * 40 + [1900, 2100, 1, 0, 700, 2048, 300, 2040], H=(64, 8), D=128,
                  seed=41)
    else:
        D = 896 if case.startswith("d896") else 1024
        kv = {"d1024_bf16": "bf16", "d896_fp16": "fp16", "d1024_fp8_plan_bf16": "fp8",
              "d1024_bf16_plan_fp8": "bf16"}[case]
        q = "fp16" if kv == "fp16" else "bf16"
        # C = min(4 x 16, 76) = 64: 256 CTAs, one per SM for 16-bit caches
        w = batch(dev, [12000, 9000, 15000, 20000], H=(32, 4), D=D, kv=kv, q=q, seed=D,
                  max_partitions=16)
    plan = binding.plan_for(w)
    if case.endswith("_plan_bf16"):
        plan.set_kv_dtype("bf16")
    elif case.endswith("_plan_fp8"):
        plan.set_kv_dtype(binding.FP8_E4M3)
    plan.refresh(w.context_lens, w.cu_query_lens)
    out = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    work, red = plan.download()
    ow, orr = oracle_plan(w, plan.info()["budget"])
    assert np.array_equal(work, ow) and np.array_equal(red, orr)
    assert plan.capacity * w.num_kv_heads > 152
    ref = oracle_decode(w.to("cpu"))
    assert max_diff(out, ref) <= TOL[w.kv_dtype]
    assert plan.read_errors() == 0


FUSED_CASES = {
    # every request within one 256-key tile: one piece each, rows written directly
    "direct": dict(lens=[17, 200, 256, 1, 0], H=(8, 2)),
    # up to 8 pieces per request: one level of the ticket tree
    "few": dict(lens=[3000, 900, 40, 0], H=(8, 2), budget=64, max_partitions=8),
    # 36 pieces: two levels
    "two_levels": dict(lens=[9000, 40, 2600], H=(8, 1), budget=4096),
    # 157 and 36 pieces: three levels
    "three_levels": dict(lens=[40000, 9000, 300, 1], H=(8, 1), budget=4096),
    # one slot cut into pieces by the split kernel (budget 32: one partition each)
    "pieces": dict(lens=[40000] + [300 + 37 * i for i in range(15)], H=(8, 2), budget=32),
    # 16 and 32 q heads per kv head: passes of two and four 8-row groups (on
    # tensor memory for fp8)
    "g16": dict(lens=[9000, 40, 2600, 300], H=(16, 1), budget=64),
    "g32": dict(lens=[5000, 1, 700], H=(32, 2), budget=48),
    # multi-token rows (tokens x G in one work item): 3 x 8 rows, 4 x 8 rows
    # (on tensor memory for fp8), 3 x 6 rows at head dim 256 (MTP verify)
    "verify3": dict(lens=[9000, 40, 2600, 300], ql=[3, 3, 1, 3], H=(8, 1), budget=64, pad=2),
    "verify4": dict(lens=[40000, 700, 5000], ql=[4, 4, 4], H=(8, 1), budget=4096),
    "verify3_d256": dict(lens=[16384, 3000, 40], ql=[3, 3, 3], H=(6, 1), D=256, bs=64, budget=304),
}


@pytest.mark.parametrize("case", list(FUSED_CASES))
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_merge(dev, case, kv):
    """Plans whose requests' query rows fit one work item (decode, and
    multi-token verify rows) can merge the pieces' partials inside the split
    kernel (ticket tree of fan-in 8, every token of the request merged by the
    CTA that took the group's last ticket) and launch no merge kernel: the
    result matches the oracle, matches the separate merge kernel's within the
    bounds, and a second call on the same plan gives the same bits (every
    ticket was reset).  Sharp queries (q std 6) so that a wrong weight or a
    lost piece shows."""
    c = dict(FUSED_CASES[case])
    lens, H = c.pop("lens"), c.pop("H")
    w = batch(dev, lens, H=H, kv=kv, seed=81 + len(lens), q_std=6.0, **c)
    ref = oracle_decode(w.to("cpu"))
    plan = binding.plan_for(w)
    assert not plan.fused_merge  # the merge kernel is the default
    plan.set_fused_merge(True)
    assert plan.fused_merge and plan.kernels_per_decode() == 1
    plan.refresh(w.context_lens, w.cu_query_lens)
    a = binding.decode_workload(plan, w)
    b = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    parity(a, ref, None, what=f"fused {case}")
    assert torch.equal(a, b), "a second fused call differs: tickets not reset"
    plan.set_fused_merge(False)
    assert plan.kernels_per_decode() == 2
    m = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    parity(m, ref, None, what=f"merge kernel {case}")
    parity(a, m.float().cpu().numpy(), None, what=f"fused vs merge kernel {case}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_merge_with_window_and_sinks(dev, kv):
    w = batch(dev, [40000, 9000, 300, 1], H=(8, 1), kv=kv, seed=91, budget=4096, q_std=6.0)
    sinks = np.linspace(-2, 2, 8)
    for window in (0, 9000):
        out, plan = run_ext(w, window=window, sinks=sinks, fused=True)
        assert plan.fused_merge
        parity(out, oracle_decode(w.to("cpu"), window=window, sinks=sinks), None, what=window)
        assert plan.read_errors() == 0


def test_fused_merge_needs_one_work_item_per_request(dev):
    """The fused merge needs every query row of a request (tokens x GQA group)
    in one work item (at most 32 rows) and a head dim of at most 256."""
    plan = binding.Plan(3, 6, 1, 256, max_query_len=3, max_tokens=12, device=dev)  # 18 rows
    assert plan.kernels_per_decode() == 2
    plan.set_fused_merge(True)
    assert plan.fused_merge and plan.kernels_per_decode() == 1
    for args, kw in (((3, 6, 1, 256), dict(max_query_len=6, max_tokens=18)),  # 36 rows
                     ((3, 64, 1, 128), {}),                                     # a group of 64
                     ((3, 8, 1, 512), {})):                                     # a wide head
        plan = binding.Plan(*args, device=dev, **kw)
        assert not plan.fused_merge and plan.kernels_per_decode() == 2
        with pytest.raises(binding.PaError) as e:
            plan.set_fused_merge(True)
        assert e.value.status == binding.PA_ERR_UNSUPPORTED


def test_set_kv_dtype_rejects_other_values(dev):
    plan = binding.Plan(4, 8, 2, 128, device=dev)
    with pytest.raises(binding.PaError):
        plan.set_kv_dtype(7)


# ------------------------------------------------- sliding window and sinks

def run_ext(w, window=0, sinks=None, budget=None, max_partitions=None, fused=False):
    plan = binding.plan_for(w, binding.PROPORTIONAL, budget, max_partitions)
    if fused:
        plan.set_fused_merge(True)
    plan.set_window(window)
    plan.refresh(w.context_lens, w.cu_query_lens)
    sk = None if sinks is None else torch.tensor(sinks, dtype=torch.float32, device=w.q.device)
    o = binding.decode_workload(plan, w, sinks=sk)
    torch.cuda.synchronize()
    return o, plan


@pytest.mark.parametrize("window", [1, 3, 50, 500])
@pytest.mark.parametrize("kv,D,bs", [("bf16", 128, 16), ("fp8", 128, 16), ("bf16", 64, 64),
                                     ("fp16", 256, 128)])
def test_sliding_window_decode(dev, window, kv, D, bs):
    q = "fp16" if kv == "fp16" else "bf16"
    w = batch(dev, RAGGED + [6000], H=(8, 2), D=D, bs=bs, kv=kv, q=q, seed=window + D)
    out, plan = run_ext(w, window=window)
    ref = oracle_decode(w.to("cpu"), window=window)
    assert max_diff(out, ref) <= TOL[kv]
    assert plan.read_errors() == 0


@pytest.mark.parametrize("window", [1, 50])
def test_sliding_window_verify_rows(dev, window):
    w = batch(dev, [600, 40, 3000, 2], ql=[3, 3, 3, 3], H=(6, 1), D=256, bs=64, pad=5, seed=21)
    out, plan = run_ext(w, window=window)
    ref = oracle_decode(w.to("cpu"), window=window)
    assert max_diff(out, ref) <= TOL["bf16"]
    assert torch.all(out[12:] == 0)


@pytest.mark.parametrize("window", [37, 700])
def test_windowed_plan_is_bit_exact(dev, window):
    for w in (wl.skewed(0, dev), batch(dev, [600, 40, 3000, 2], ql=[3, 3, 3, 3], H=(6, 1), D=256,
                                       bs=64, seed=22)):
        plan = binding.plan_for(w)
        plan.set_window(window)
        plan.refresh(w.context_lens, w.cu_query_lens)
        work, red = plan.download()
        ow, orr = oracle_plan(w, plan.info()["budget"], window=window)
        assert np.array_equal(work.numpy(), ow) and np.array_equal(red.numpy(), orr)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("P,W", [(1, 8), (8, 64), (256, 4096)])
def test_sinks_direct_few_and_many_pieces(dev, kv, P, W):
    """Sinks on rows written by one CTA (P = 1), merged by a warp (a few
    partitions) and merged by a CTA (hundreds of partitions), with and without
    a window; one head's sink at -inf is no sink."""
    w = batch(dev, [9000, 40, 2600, 0, 700], H=(8, 2), D=128, kv=kv, seed=23)
    rng = np.random.default_rng(5)
    sinks = rng.normal(0.0, 3.0, 8)
    sinks[3] = -np.inf
    for window in (0, 300):
        out, plan = run_ext(w, window=window, sinks=sinks, budget=W, max_partitions=P)
        ref = oracle_decode(w.to("cpu"), window=window, sinks=sinks)
        assert max_diff(out, ref) <= TOL[kv], window
        assert plan.read_errors() == 0


def test_window_with_pieces(dev):
    w = batch(dev, [40000] + [300 + 37 * i for i in range(15)], H=(8, 2), D=128, seed=24,
              budget=32)
    for window in (5000, 20000):
        out, _ = run_ext(w, window=window, sinks=np.linspace(-2, 2, 8))
        ref = oracle_decode(w.to("cpu"), window=window, sinks=np.linspace(-2, 2, 8))
        assert max_diff(out, ref) <= TOL["bf16"], window


# ------------------------------------------ K in the grouped 5-D layout

@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16")])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_grouped_k_sweep(dev, D, kv, q, bs):
    """K as [num_blocks, Hkv, D/16, bs, 16]: the oracle reads that layout by its
    own indexing; with 16-bit caches the result also equals the row-major run
    bit for bit (the same MMA k-steps in the same order)."""
    w = batch(dev, RAGGED + [5000], H=(8, 2), D=D, bs=bs, kv=kv, q=q, seed=3 * D + bs)
    w5 = wl.with_k_groups(w)
    out5, plan = run(w5)
    ref = oracle_decode(w5.to("cpu"))
    assert max_diff(out5, ref) <= TOL[kv]
    assert plan.read_errors() == 0
    if kv != "fp8":
        out4, _ = run(w)
        assert torch.equal(out4, out5)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_grouped_k_rows_window_sinks_pieces(dev, kv):
    """Grouped K through every other path: multi-token rows with padding, a
    sliding window with sinks, and a slot run as pieces with a CTA merge."""
    w = wl.with_k_groups(batch(dev, [600, 40, 3000, 2, 0], ql=[3, 3, 3, 3, 1], H=(6, 1), D=256,
                               bs=64, kv=kv, pad=5, seed=31))
    check(w)
    w = wl.with_k_groups(batch(dev, [40000] + [300 + 37 * i for i in range(15)], H=(8, 2), D=128,
                               kv=kv, seed=32, budget=32))
    sinks = np.linspace(-2, 2, 8)
    for window in (0, 7000):
        out, plan = run_ext(w, window=window, sinks=sinks)
        ref = oracle_decode(w.to("cpu"), window=window, sinks=sinks)
        assert max_diff(out, ref) <= TOL[kv], window
        assert plan.read_errors() == 0


def test_grouped_k_layout_checks(dev):
    w = batch(dev, [300, 20], H=(8, 2), D=128, seed=33)
    w5 = wl.with_k_groups(w)
    plan = binding.plan_for(w5)
    plan.refresh(w5.context_lens)
    bad_v = w5.v_cache[:, :, :8]  # V must be [nb, Hkv, bs, D] with K's nb, Hkv and bs
    with pytest.raises(ValueError):
        plan.decode(w5.q, w5.k_cache, bad_v, w5.block_tables, w5.context_lens)
    bad_k = w5.k_cache.reshape(*w5.k_cache.shape[:3], 8, 32)
    with pytest.raises(ValueError):
        plan.decode(w5.q, bad_k, w5.v_cache, w5.block_tables, w5.context_lens)
    lib = binding.load()
    st = lib.pa_decode_ex(plan._h, binding._ptr(w5.q), binding.BF16, 2, 8, 128,
                          binding._ptr(w5.k_cache), binding._ptr(w5.v_cache), binding.BF16,
                          1.0, 1.0, w5.v_cache.shape[0], 2, 16, binding._ptr(w5.block_tables),
                          w5.block_tables.shape[1], binding._ptr(w5.context_lens), None, 2,
                          0.1, None, 2, binding._ptr(torch.empty_like(w5.q)), None)
    assert st == binding.PA_ERR_UNSUPPORTED  # no third K layout


# -------------------------------------------- head dims 384 to 1024

WIDE = [384, 512, 640, 768, 896, 1024]


@pytest.mark.parametrize("D", WIDE)
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16")])
def test_wide_head_dims(dev, D, kv, q):
    """Head dims above 256 run one warp per 128- or 256-dim slice with the partial
    logits summed through shared memory; K row-major and grouped."""
    bs = 16 if D % 256 else 128
    w = batch(dev, [1, 15, 17, 255, 257, 700, 2100], H=(8, 1), D=D, bs=bs, kv=kv, q=q, seed=D)
    check(w)
    w5 = wl.with_k_groups(w)
    out5, plan = run(w5)
    assert max_diff(out5, oracle_decode(w5.to("cpu"))) <= TOL[kv]
    assert plan.read_errors() == 0


@pytest.mark.parametrize("D", [512, 1024])
def test_wide_head_dims_rows_groups_and_merges(dev, D):
    """Wide heads with GQA groups of 16 (two row groups, or two row chunks),
    multi-token rows with padding, and partitions merged by warps (few pieces)
    and by CTAs (many pieces)."""
    check(batch(dev, [300, 5000, 40], H=(32, 2), D=D, kv="bf16", seed=D + 1))
    check(batch(dev, [600, 40, 3000, 2, 0], ql=[3, 3, 3, 3, 1], H=(8, 1), D=D, bs=64, kv="fp8",
                pad=5, seed=D + 2))
    for P, W in ((4, 16), (64, 512)):
        check(batch(dev, [20000, 900, 40], H=(8, 1), D=D, kv="bf16", seed=D + 3, budget=W,
                    max_partitions=P))


def test_wide_head_dims_window_sinks_pieces(dev):
    w = batch(dev, [40000] + [300 + 37 * i for i in range(15)], H=(8, 1), D=640, kv="fp8",
              seed=41, budget=32)
    sinks = np.linspace(-2, 2, 8)
    for window in (0, 9000):
        out, plan = run_ext(w, window=window, sinks=sinks)
        assert max_diff(out, oracle_decode(w.to("cpu"), window=window, sinks=sinks)) <= TOL["fp8"]
        assert plan.read_errors() == 0


# ---------------------------------------------------- multi-token rows (cu)

def test_verify_rows_and_padding(dev):
    w = batch(dev, [600, 40, 3000, 2], ql=[3, 3, 3, 3], H=(6, 1), D=256, bs=64, pad=5, seed=1)
    out, _, _ = check(w)
    assert torch.all(out[12:] == 0)


def test_mixed_decode_and_prompt(dev):
    w = batch(dev, [700, 100, 0, 900, 5], ql=[1, 100, 2, 1, 0], H=(12, 2), D=256, bs=64, pad=3,
              seed=2)
    out, _, _ = check(w)
    cu = w.cu_query_lens.tolist()
    assert torch.all(out[cu[2]:cu[3]] == 0)       # zero-length request
    assert torch.all(out[cu[-1]:] == 0)          # graph padding rows


def test_rows_with_no_visible_key_are_zero(dev):
    w = batch(dev, [2, 300], ql=[5, 2], H=(8, 2), D=64, pad=1, seed=3)
    out, _, _ = check(w)
    assert torch.all(out[0:3] == 0)  # tokens 0..2 of request 0 see S-(L-1-i) <= 0 keys


@pytest.mark.parametrize("ql", [2, 4, 8])
def test_verify_row_groups(dev, ql):
    check(batch(dev, [5000, 900, 64], ql=[ql] * 3, H=(8, 1), D=128, kv="fp8", seed=ql))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("ql,H", [(2, (8, 1)), (3, (8, 1)), (3, (6, 1)), (2, (12, 2)), (4, (8, 1))])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_fp8_verify_rows(dev, D, ql, H, bs):
    """fp8 caches with two to four query-row groups per pass (speculative
    verify rows on an fp8 cache; at D 128 the tensor-memory consumer, 16, 24
    and 32 rows, row sums per thread and by the ones MMA; pages of 16 keys
    (two producer warps), 64 and 128 (one copy per tensor and stage)).
    Ragged lengths (one-key requests, rows with no visible key, a
    zero-length request), graph padding, fp16 and bf16 q, against the
    oracle."""
    lens = [5000, 900, 64, 1, 2, 257, 3000]
    q = "fp16" if (D + ql) % 2 else "bf16"
    w = batch(dev, lens, ql=[ql] * len(lens), H=H, D=D, bs=bs, kv="fp8", q=q, pad=3,
              seed=D + 10 * ql + bs)
    out, _, _ = check(w)
    assert torch.all(out[int(w.cu_query_lens[-1]):] == 0)


@pytest.mark.parametrize("D", [128, 256])
def test_fp8_verify_rows_window_sinks_sharp(dev, D):
    """fp8 verify rows with a sliding window, sinks, partitions merged by the
    merge kernel (a few and many), and sharp queries."""
    w = batch(dev, [20000, 700, 3000, 0], ql=[3, 3, 3, 1], H=(8, 1), D=D, kv="fp8", pad=2,
              seed=D + 7, q_std=6.0)
    sinks = np.linspace(-2, 2, 8)
    for window, P, W in ((0, 256, 2048), (500, 8, 64), (9000, 256, 2048)):
        out, plan = run_ext(w, window=window, sinks=sinks, budget=W, max_partitions=P)
        parity(out, oracle_decode(w.to("cpu"), window=window, sinks=sinks), None,
               what=(window, P))
        assert plan.read_errors() == 0


def test_cu_arange_matches_no_cu(dev):
    w = batch(dev, RAGGED, H=(8, 2), D=128, seed=9)
    a, _ = run(w)
    w2 = wl.Workload(**{**w.__dict__, "cu_query_lens": torch.arange(
        len(RAGGED) + 1, dtype=torch.int32, device=dev)})
    b, _ = run(w2)
    assert torch.equal(a, b)


# ------------------------------------------------------------ robustness

def _poison(w):
    """NaN in every cache slot that no request may read: the tail of each
    request's last page and every unused page."""
    nan = 0x7F if w.kv_dtype == "fp8" else float("nan")
    used = torch.zeros(w.k_cache.shape[0], dtype=torch.bool)
    bs = w.block_size
    for r, S in enumerate(w.context_lens.tolist()):
        np_ = -(-S // bs)
        pages = w.block_tables[r, :np_].long().cpu()
        used[pages] = True
        if S % bs:
            last = int(pages[-1])
            w.k_cache[last, :, S % bs:] = nan
            w.v_cache[last, :, S % bs:] = nan
    idx = (~used).nonzero().flatten().to(w.k_cache.device)
    w.k_cache[idx] = nan
    w.v_cache[idx] = nan


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_nan_poisoned_unread_slots(dev, kv):
    w = batch(dev, [17, 300, 1000, 5], H=(8, 2), D=128, kv=kv, seed=4, pool_pages=200)
    _poison(w)
    check(w)


GUARD = 0x7FC1  # a NaN in both bf16 and fp16


@pytest.mark.parametrize("case", ["decode_bf16", "decode_fp8", "verify_d256", "wide_d1024",
                                  "fp16_pieces"])
def test_output_guard_regions(dev, case):
    """The output sits inside a larger buffer whose every element holds a NaN
    sentinel: after the call the elements before and after it are untouched
    (no write out of bounds) and none inside it still holds the sentinel
    (every row written: outputs, merged rows, zero rows of padding and empty
    requests)."""
    mk = {
        "decode_bf16": lambda: batch(dev, [17, 300, 1000, 5000, 0], H=(8, 2), D=128),
        "decode_fp8": lambda: batch(dev, [17, 300, 1000, 5000, 0], H=(32, 4), D=128, kv="fp8"),
        "verify_d256": lambda: batch(dev, [600, 40, 3000, 2, 0], ql=[3, 3, 3, 3, 1], H=(6, 1),
                                     D=256, bs=64, pad=5),
        "wide_d1024": lambda: batch(dev, [700, 3000, 0], ql=[2, 1, 1], H=(16, 2), D=1024, pad=3),
        "fp16_pieces": lambda: batch(dev, [9000, 64, 300], H=(8, 1), D=64, bs=64, kv="fp16",
                                     q="fp16"),
    }
    w = mk[case]()
    n, g = w.q.numel(), 4096
    buf = torch.full((n + 2 * g,), GUARD, dtype=torch.int16, device=dev)
    out = buf[g:g + n].view(w.q.dtype).view(w.q.shape)
    kw = {"budget": 64} if case == "fp16_pieces" else {}
    check(w, out=out, **kw)
    assert torch.all(buf[:g] == GUARD) and torch.all(buf[g + n:] == GUARD), "write out of bounds"
    assert not torch.any(buf[g:g + n] == GUARD), "output element never written"


def test_deterministic(dev):
    w = wl.tiny(0, dev)
    a, _ = run(w)
    b, _ = run(w)
    assert torch.equal(a, b)


def test_stale_plan_is_reported_and_zeroed(dev):
    w = batch(dev, [3000, 800, 1200], H=(8, 2), D=128, seed=6)
    plan = binding.plan_for(w)
    plan.refresh(w.context_lens)
    w.context_lens[1] += 1  # a draft step bumps a length without re-planning
    out = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() & binding.DEVERR_STALE_PLAN
    assert torch.all(out[1] == 0)
    ref = oracle_decode(w.to("cpu"))
    assert max_diff(out[[0, 2]], ref[[0, 2]]) <= TOL["bf16"]


@pytest.mark.parametrize("grouped", [False, True])
def test_bad_page_is_reported_not_faulted(dev, grouped):
    w = batch(dev, [3000, 800], H=(8, 2), D=128, seed=7)
    w.block_tables[0, 3] = w.k_cache.shape[0] + 5
    out, plan = run(wl.with_k_groups(w) if grouped else w)
    assert plan.read_errors() & binding.DEVERR_BAD_PAGE
    ref = oracle_decode(wl.subset(w, [1]))
    assert max_diff(out[[1]], ref) <= TOL["bf16"]


@pytest.mark.parametrize("case", ["d128", "d128_two_rows", "d512_slices", "fp8_two_rows",
                                  "fp8_four_rows"])
def test_a_wait_that_runs_out_sets_the_timeout_bit(dev, case):
    """The timeout path, made to run on purpose: with a 100 us wait limit and
    the test hook that leaves every CTA's second pipeline stage un-issued, the
    consumers' bounded waits give up, PA_DEVERR_TIMEOUT is raised, the call
    returns (every barrier is still met on the abort path: the single-slice
    kernel, the two-row-group exchange epilogue, a 512-dim head whose slice
    warps meet a named barrier per stage, and the tensor-memory consumer --
    its issuing thread gives up on the missing tile, the softmax warps on
    its S, and the tensor memory is released after a last commit -- with
    per-thread row sums (16 rows) and the ones MMA (32 rows)), and the next
    call on the same plan, with the hook off and the default limit, is
    correct."""
    if case == "d128":
        w = batch(dev, [3000, 800, 1200, 17], H=(8, 2), D=128, seed=71)
    elif case == "d128_two_rows":
        w = batch(dev, [3000, 800, 1200], ql=[2, 2, 2], H=(8, 1), D=128, pad=2, seed=72)
    elif case.startswith("fp8"):
        ql = 2 if case == "fp8_two_rows" else 4
        w = batch(dev, [3000, 800, 1200], ql=[ql] * 3, H=(8, 1), D=128, kv="fp8", pad=2,
                  seed=74 + ql)
    else:
        w = batch(dev, [3000, 800, 1200], H=(8, 1), D=512, seed=73)
    plan = binding.plan_for(w)
    plan.refresh(w.context_lens, w.cu_query_lens)
    plan.set_wait_limit(100_000)
    plan.skip_stage_for_test(1)
    binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() & binding.DEVERR_TIMEOUT
    plan.skip_stage_for_test(-1)
    plan.set_wait_limit(0)
    out = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    assert max_diff(out, oracle_decode(w.to("cpu"))) <= TOL[w.kv_dtype]


def test_wait_limit_arguments(dev):
    plan = binding.Plan(4, 8, 2, 128, device=dev)
    for bad in (-1, 5):
        with pytest.raises(binding.PaError):
            plan.set_wait_limit(bad)
    with pytest.raises(binding.PaError):
        plan.skip_stage_for_test(-2)
    plan.set_wait_limit(10_000)
    plan.set_wait_limit(0)


def test_overflowing_query_rows_empty_the_plan(dev):
    w = batch(dev, [500, 500], ql=[2, 2], H=(8, 2), D=64, seed=8)
    plan = binding.Plan(2, 8, 2, 64, max_query_len=1, max_tokens=4, device=dev)
    plan.refresh(w.context_lens, w.cu_query_lens)
    out = binding.decode_workload(plan, w)
    torch.cuda.synchronize()
    assert plan.read_errors() & binding.DEVERR_PLAN_OVERFLOW
    assert torch.all(out == 0)


def test_validation_errors(dev):
    w = wl.tiny(0, dev)
    plan = binding.plan_for(w)
    with pytest.raises(binding.PaError) as e:  # decode before any refresh
        binding.decode_workload(plan, w)
    assert e.value.status == binding.PA_ERR_PLAN_MISMATCH
    plan.refresh(w.context_lens)
    with pytest.raises(binding.PaError) as e:  # refreshed without cu, called with cu
        plan.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                    torch.arange(5, dtype=torch.int32, device=dev))
    assert e.value.status == binding.PA_ERR_PLAN_MISMATCH
    with pytest.raises(binding.PaError) as e:  # fp16 q with a bf16 cache
        plan.decode(w.q.half(), w.k_cache, w.v_cache, w.block_tables, w.context_lens)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED
    k32 = w.k_cache.view(64, 2, 32, 64)
    with pytest.raises(binding.PaError) as e:  # block size 32 is outside the domain
        plan.decode(w.q, k32, k32, w.block_tables, w.context_lens)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED
    other = binding.Plan(5, 8, 2, 64, device=dev)
    other.refresh(torch.ones(5, dtype=torch.int32, device=dev))
    with pytest.raises(binding.PaError) as e:  # plan built for another batch size
        binding.decode_workload(other, w)
    assert e.value.status == binding.PA_ERR_PLAN_MISMATCH
    lib = binding.load()
    import ctypes
    st = lib.pa_decode(plan._h, ctypes.c_void_p(w.q.data_ptr() + 2), 0, 4, 8, 64,
                       ctypes.c_void_p(w.k_cache.data_ptr()), ctypes.c_void_p(w.v_cache.data_ptr()),
                       0, 1.0, 1.0, 128, 2, 16, ctypes.c_void_p(w.block_tables.data_ptr()),
                       w.block_tables.shape[1], ctypes.c_void_p(w.context_lens.data_ptr()), None,
                       4, 0.125, ctypes.c_void_p(w.q.data_ptr()), None)
    assert st == binding.PA_ERR_INVALID_ARG  # misaligned q


def test_graph_capture_refresh_and_decode(dev):
    """refresh + decode captured once, replayed after the lengths change in place."""
    w = batch(dev, [3000, 800, 64, 2000], H=(8, 2), D=128, seed=10, spare_blocks=40)
    plan = binding.plan_for(w)
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.refresh(w.context_lens, stream=s)
        binding.decode_workload(plan, w, out=out, stream=s)  # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.refresh(w.context_lens)
        binding.decode_workload(plan, w, out=out)
    # extend the batch inside the allocated pages and replay
    g2 = torch.Generator().manual_seed(0)
    for step in range(3):
        grow = torch.tensor([100, 257, 1, 300], dtype=torch.int32)
        new = w.context_lens.cpu() + grow
        bs = w.block_size
        for r in range(w.num_seqs):  # give the grown requests pages
            need = -(-int(new[r]) // bs)
            have = int((w.block_tables[r] >= 0).sum())
            if need > have:
                free = torch.randperm(w.k_cache.shape[0], generator=g2)[: need - have]
                w.block_tables[r, have:need] = free.to(torch.int32).to(dev)
        w.context_lens.copy_(new.to(dev))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_decode(w.to("cpu"))
        assert max_diff(out, ref) <= TOL["bf16"]
    assert plan.read_errors() == 0


def test_profiling_events_bracket_the_call_and_the_split(dev):
    """The call events enclose the split events, eagerly and in a replayed graph."""
    w = batch(dev, [3000, 800, 64, 2000], H=(8, 2), D=128, seed=11)
    plan = binding.plan_for(w)
    out = torch.empty_like(w.q)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev:
        e.record()
    plan.refresh(w.context_lens)
    plan.set_call_events(ev[1], ev[4])
    plan.set_split_events(ev[2], ev[3])
    ev[0].record()
    binding.decode_workload(plan, w, out=out)
    torch.cuda.synchronize()
    call, split = ev[1].elapsed_time(ev[4]), ev[2].elapsed_time(ev[3])
    assert 0 < split <= call and ev[0].elapsed_time(ev[1]) >= 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.decode_workload(plan, w, out=out)
    plan.set_call_events(None, None)
    plan.set_split_events(None, None)
    g.replay()
    torch.cuda.synchronize()
    assert 0 < ev[2].elapsed_time(ev[3]) <= ev[1].elapsed_time(ev[4])
    assert max_diff(out, oracle_decode(w.to("cpu"))) <= TOL["bf16"]


def test_largest_batch_4096_requests(dev):
    """The planner's domain limit: 4096 requests (lengths 0..3000, a few empty),
    with and without multi-token rows; sampled rows against the oracle."""
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 3000, 4096).tolist()
    lens[:3] = [0, 1, 2999]
    w = batch(dev, lens, H=(8, 1), D=64, bs=16, seed=31)
    out, plan = run(w)
    assert plan.read_errors() == 0
    pick = [0, 1, 2, 5, 100, 2047, 4095]
    assert _sampled(w, out, pick) <= TOL["bf16"]
    assert torch.all(out[0] == 0)  # the empty request
    ql = rng.integers(0, 3, 4096).tolist()
    w = batch(dev, lens, ql=ql, H=(4, 1), D=64, bs=16, pad=7, seed=32)
    out, plan = run(w)
    assert plan.read_errors() == 0
    assert _sampled(w, out, [r for r in pick if ql[r] > 0]) <= TOL["bf16"]
    assert torch.all(out[int(w.cu_query_lens[-1]):] == 0)


# ------------------------------------------------ full-size configurations

def _sampled(w, out, requests):
    sub = wl.subset(w, requests)
    ref = oracle_decode(sub, window=w.window)
    if w.cu_query_lens is None:
        rows = torch.tensor(requests)
    else:
        cu = w.cu_query_lens.cpu()
        rows = torch.cat([torch.arange(int(cu[r]), int(cu[r + 1])) for r in requests])
    return max_diff(out[rows.to(out.device)], ref)


def _pick(w, k=4):
    lens = w.context_lens.cpu()
    order = torch.argsort(lens)
    picks = {int(order[-1]), int(order[0]), int(order[len(order) // 2])}
    g = torch.Generator().manual_seed(1)
    while len(picks) < min(k, w.num_seqs):
        picks.add(int(torch.randint(w.num_seqs, (1,), generator=g)))
    return sorted(picks)


FULL = ["uniform", "skewed", "mtp_verify", "mixed_prompt", "large_bf16", "large_fp8",
        "uniform_w1024", "skewed_w4096", "uniform_k5", "skewed_k5", "uniform_d512",
        "skewed_d1024", "uniform_d1024", "uniform_n64_h8", "skewed_mtp3", "rows_fp8_t3",
        "rows_bf16_t4"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(dev, name):
    w = wl.CONFIGS[name](0, dev)
    for kind in (binding.PROPORTIONAL, binding.UNIFORM):
        out, plan = run(w, kind=kind)
        assert plan.read_errors() == 0
        d = _sampled(w, out, _pick(w))
        assert d <= TOL[w.kv_dtype], (name, kind, d)
        if w.cu_query_lens is not None:
            assert torch.all(out[int(w.cu_query_lens[-1]):] == 0)
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("seed", [1, 2])
def test_skewed_seeds_sampled(dev, seed):
    w = wl.skewed(seed, dev)
    out, plan = run(w)
    assert _sampled(w, out, _pick(w)) <= TOL["fp8"]
