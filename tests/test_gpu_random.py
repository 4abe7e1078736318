"""Randomised parity: many small batches whose every knob is drawn at random --
head dim, cache dtype, page size, GQA group, query rows per request, padding,
sliding window, sinks, K layout, plan kind, budget and partition ceiling,
ragged lengths (empty requests and one-key requests included) -- each compared
with the fp64 oracle element by element.  The draws are seeded, so a failure
names a reproducible case."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import oracle_decode, parity
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu
HEAD_DIMS = [64, 128, 256, 384, 512, 640, 768, 896, 1024]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def draw(seed: int, dev):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice(HEAD_DIMS, p=[.2, .2, .2, .06, .06, .06, .06, .08, .08]))
    kv = str(rng.choice(["bf16", "fp16", "fp8"]))
    q = "fp16" if kv == "fp16" else str(rng.choice(["bf16", "fp16"])) if kv == "fp8" else "bf16"
    bs = int(rng.choice([16, 64, 128]))
    hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 6, 8, 16]))
    n = int(rng.integers(1, 9 if D <= 256 else 4))  # keep the fp64 oracle quick
    lens = [int(x) for x in rng.choice([0, 1, 2, 15, 16, 17, 255, 257, 700, 1500, 4000, 9000], n)]
    ql = None
    pad = 0
    if rng.random() < 0.5:
        ql = [int(x) for x in rng.integers(0, 5, n)]
        pad = int(rng.integers(0, 4))
    if ql is not None and sum(ql) + pad == 0:
        pad = 1  # at least one output row
    window = int(rng.choice([0, 0, 1, 7, 300, 2000]))
    sinks = rng.normal(0.0, 2.0, G * hkv) if rng.random() < 0.3 else None
    grouped = rng.random() < 0.3
    kind = int(rng.choice([binding.PROPORTIONAL, binding.UNIFORM]))
    budget = int(rng.choice([0, 8, 32, 296]))
    P = int(rng.choice([1, 4, 256]))
    w = wl.make_batch(f"rand{seed}", lens, ql, G * hkv, hkv, D, bs, kv, q, seed=seed,
                      pad_tokens=pad, kv_scale=0.05, device=dev, budget=budget or None,
                      max_partitions=P)
    return w, dict(window=window, sinks=sinks, grouped=grouped, kind=kind)


@pytest.mark.parametrize("seed", range(160))
def test_random_batch(dev, seed):
    w, o = draw(seed, dev)
    plan = binding.plan_for(w, o["kind"])
    plan.set_window(o["window"])
    plan.refresh(w.context_lens, w.cu_query_lens)
    wk = wl.with_k_groups(w) if o["grouped"] else w
    sk = None if o["sinks"] is None else torch.tensor(o["sinks"], dtype=torch.float32,
                                                      device=dev)
    out = binding.decode_workload(plan, wk, sinks=sk)
    torch.cuda.synchronize()
    assert plan.read_errors() == 0
    ref = oracle_decode(w.to("cpu"), window=o["window"], sinks=o["sinks"])
    parity(out, ref, w.kv_dtype, what=f"seed {seed} {o}")
    if w.cu_query_lens is not None:  # graph padding rows are zero
        assert torch.all(out[int(w.cu_query_lens[-1]):] == 0)
