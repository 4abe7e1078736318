"""Long contexts with sharp attention, and the error's growth with the split count.

With q, K, V ~ N(0, 1) and scale 1/sqrt(D) the logits spread over about one
unit, so over thousands of keys the softmax is nearly flat and the output rows
are small (standard deviation ~ 1/sqrt(S)): an absolute bound alone could not
see a dropped partition or a wrong merge weight on such rows.  Here q is drawn
with standard deviation 6 instead (logits over tens of units, attention
dominated by a few keys, outputs of order 1), and every case sits on the paths
that only long requests take: a slot cut into pieces, grids of more than one
wave, requests of more than 8 pieces (merged by a whole CTA), sliding windows
of 5000 keys and more, sparse top-k decode.

These cases are held to the relative bounds of helpers.parity (whole output
and every row; zero rows exactly zero), not to the absolute 1e-2 / 3e-2: that
bound is stated for the N(0, 1) configurations, whose outputs stay below 1,
while sharp outputs reach ~4, where the output's own rounding to bf16 moves an
element by up to 2^-8 x 4 ~ 0.016 however exact the rest is.

The drift check follows "[MiniMax-M3] Route the paged decode to aiter's FlyDSL
kernel with work planner", section 5 ("Planner drift at the real ceiling"):
the planned result against one reference per batch, for partition ceilings
8 ... 256 on contexts beyond 100k keys at batch 1, 8 and 24.  The error must
not grow with the number of partitions."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import oracle_decode, parity, bits16, kv_bits, q_code, DT_CODE
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

SHARP = 6.0  # standard deviation of q


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def batch(dev, lens, ql=None, H=(8, 2), D=128, bs=16, kv="bf16", q="bf16", pad=0, seed=0,
          q_std=SHARP, **kw):
    return wl.make_batch("long", lens, ql, H[0], H[1], D, bs, kv, q, seed=seed, pad_tokens=pad,
                         kv_scale=0.05, device=dev, q_std=q_std, **kw)


def run(w, window=0, sinks=None, budget=None, max_partitions=None, kind=binding.PROPORTIONAL):
    plan = binding.plan_for(w, kind, budget, max_partitions)
    plan.set_window(window)
    plan.refresh(w.context_lens, w.cu_query_lens)
    sk = None if sinks is None else torch.tensor(sinks, dtype=torch.float32, device=w.q.device)
    out = binding.decode_workload(plan, w, sinks=sk)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    return out, plan


def partitions(plan):
    """The plan's partition count per request (reduce_info word 1)."""
    _, red = plan.download()
    return red[:, 1]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sharp_pieces_of_one_long_slot(dev, kv):
    """One slot of 40000 keys among 15 short ones (budget 32: one partition per
    request), run as pieces and merged by a warp."""
    w = batch(dev, [40000] + [300 + 37 * i for i in range(15)], kv=kv, seed=51, budget=32)
    out, plan = run(w)
    assert bool((partitions(plan) == 1).all())
    parity(out, oracle_decode(w.to("cpu")), None)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sharp_many_partitions_cta_merge(dev, kv):
    """157 and 36 partitions (more than 8: a CTA merges each row), a two-tile
    request and a one-key request, G = 8."""
    w = batch(dev, [40000, 9000, 300, 1], H=(8, 1), kv=kv, seed=52, budget=4096)
    out, plan = run(w)
    parts = partitions(plan)
    assert int(parts[0]) == 157 and int(parts[1]) == 36
    parity(out, oracle_decode(w.to("cpu")), None)


@pytest.mark.parametrize("case", ["d128_48x8", "d1024_bf16", "d1024_fp8"])
def test_sharp_more_ctas_than_one_wave(dev, case):
    """Grids of more CTAs than run at once: slots cut into short pieces shared
    by the first wave, later CTAs starting at the work counter."""
    if case == "d128_48x8":
        w = batch(dev, [2048] * 40 + [1900, 2100, 1, 0, 700, 2048, 300, 2040], H=(64, 8),
                  seed=53)
    else:
        w = batch(dev, [12000, 9000, 15000, 20000], H=(32, 4), D=1024, kv=case.split("_")[1],
                  seed=54, max_partitions=16)
    out, plan = run(w)
    assert plan.capacity * w.num_kv_heads > 152
    parity(out, oracle_decode(w.to("cpu")), None)


@pytest.mark.parametrize("window", [5000, 20000])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sharp_long_windows_with_pieces_and_sinks(dev, window, kv):
    w = batch(dev, [40000, 26000] + [300 + 37 * i for i in range(14)], kv=kv, seed=55, budget=32)
    sinks = np.linspace(-2, 2, 8)
    out, _ = run(w, window=window, sinks=sinks)
    parity(out, oracle_decode(w.to("cpu"), window=window, sinks=sinks), None)


def test_sharp_long_window_many_partitions(dev):
    w = batch(dev, [60000, 7000], H=(8, 1), seed=56, budget=4096)
    out, _ = run(w, window=9000)
    parity(out, oracle_decode(w.to("cpu"), window=9000), None)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sharp_verify_rows_long_context(dev, kv):
    """8 requests x 3 tokens at 16384 keys (the MTP-verify shape), G = 6."""
    w = batch(dev, [16384] * 8, ql=[3] * 8, H=(6, 1), D=256, bs=64, kv=kv, pad=8, seed=57)
    out, _ = run(w)
    parity(out, oracle_decode(w.to("cpu")), None)
    assert torch.all(out[24:] == 0)


def test_sharp_mixed_prompt_long_context(dev):
    w = batch(dev, [16384] * 7 + [100], ql=[1] * 7 + [100], H=(12, 2), D=256, bs=64, pad=21,
              seed=58)
    out, _ = run(w)
    parity(out, oracle_decode(w.to("cpu")), None)


def test_sharp_sparse_decode(dev):
    """Top-32 block selection over the skewed length mix, sharp queries."""
    sw = wl.sparse(0, dev)
    w = sw.base
    w.q.copy_((w.q.float() * SHARP).to(w.q.dtype))
    plan = binding.Plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                        max_partitions=sw.max_partitions, budget=w.budget or 0, device=dev)
    sel, sl = binding.sparse_select(sw.scores, w.context_lens, w.block_tables, w.block_size,
                                    sw.top_k, sw.init_blocks, sw.local_blocks)
    plan.refresh(sl)
    out = plan.decode(w.q, w.k_cache, w.v_cache, sel, sl, None, w.scale, w.k_scale, w.v_scale)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    ref = oracle.sparse_decode(bits16(w.q), q_code(w), kv_bits(w.k_cache, w.kv_dtype),
                               kv_bits(w.v_cache, w.kv_dtype), DT_CODE[w.kv_dtype], w.k_scale,
                               w.v_scale, w.block_tables.cpu().numpy(),
                               w.context_lens.cpu().numpy(), w.scale,
                               sw.scores.cpu().numpy(), w.block_size, sw.top_k, sw.init_blocks,
                               sw.local_blocks)
    parity(out, ref, None)


def test_sharp_full_size_skewed_sampled(dev):
    """The skewed fp8 batch at full size with sharp queries: the longest, the
    shortest, the median and a random request against the oracle."""
    base = wl.skewed(0, dev)
    base.q.copy_((base.q.float() * SHARP).to(base.q.dtype))
    out, _ = run(base)
    lens = base.context_lens.cpu()
    order = torch.argsort(lens)
    picks = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2]), 5})
    parity(out[torch.tensor(picks, device=dev)], oracle_decode(wl.subset(base, picks)), None)


# ------------------------------------------------------ drift vs split count

DRIFT_P = [8, 32, 64, 128, 256]


def _drift_lens(n: int, seed: int) -> list[int]:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(100_000, 130_001, n)]


@pytest.mark.parametrize("n,q_std,kv,ql", [(1, 1.0, "bf16", 1), (1, SHARP, "bf16", 1),
                                           (8, 1.0, "bf16", 1), (8, SHARP, "bf16", 1),
                                           (24, 1.0, "bf16", 1), (8, 1.0, "fp8", 3),
                                           (8, SHARP, "fp8", 3)])
def test_error_does_not_grow_with_split_count(dev, n, q_std, kv, ql):
    """One batch, one fp64 reference; the planned GPU result for partition
    ceilings 8 ... 256 (budget n x P x Hkv, so a request of mean length gets P
    partitions).  ||gpu - ref|| / ||ref|| and max |gpu - ref| / max |ref| stay
    below the relative bounds at every P, and at P = 256 within 1.5x their
    value at P = 8.  The fp8 3-token cases (24 rows per pass) run on the
    tensor-memory consumer."""
    w = batch(dev, _drift_lens(n, 60 + n), ql=None if ql == 1 else [ql] * n, H=(8, 1), kv=kv,
              seed=61 + n + ql, q_std=q_std)
    ref = oracle_decode(w.to("cpu"))
    rows = []
    for P in DRIFT_P:
        out, plan = run(w, budget=n * P * w.num_kv_heads, max_partitions=P)
        e = parity(out, ref, None if q_std > 1 else kv, what=f"P={P}")
        rows.append({"P": P, "max_parts": int(partitions(plan).max()), **e})
    table = {"n": n, "q_std": q_std, "kv": kv, "ql": ql, "lens": w.context_lens.tolist()[:4],
             "rows": rows}
    print("DRIFT " + json.dumps(table))
    out_dir = os.environ.get("PA_DRIFT_OUT")
    if out_dir:
        with open(os.path.join(out_dir, f"drift_n{n}_q{q_std:g}_{kv}_l{ql}.json"), "w") as f:
            json.dump(table, f)
    assert rows[-1]["max_parts"] == 256 or n > 1
    e8, e256 = rows[0], rows[-1]
    assert e256["rel_norm"] <= 1.5 * e8["rel_norm"], rows
    assert e256["rel_max"] <= 1.5 * e8["rel_max"], rows
