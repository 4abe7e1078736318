"""Pins of the fp64 CPU oracle against facts that do not come from the oracle:
number-format definitions checked against torch's own casts, a library attention
routine (torch SDPA in float64) on tiny batches, closed forms, invariants of the
method, and the values the source pages print (tests/golden/plan_points.json)."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import bits16, oracle_args, oracle_decode, oracle_decode_planned, oracle_plan
from paged_kv_decode_split_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_points.json")


# ------------------------------------------------------------------ number formats

def test_e4m3fn_all_256_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3fn_to_double(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF only: e4m3fn has no infinities
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_and_fp16_all_codes_match_torch():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    for dt, fn in ((torch.bfloat16, oracle.bf16_to_double), (torch.float16, oracle.fp16_to_double)):
        ref = codes.view(dt).to(torch.float64).numpy()
        got = np.array([fn(b) for b in range(65536)])
        nan = np.isnan(ref)
        assert np.array_equal(nan, np.isnan(got))
        assert np.array_equal(ref[~nan], got[~nan])


# ------------------------------------------------------------ attention: library routine

def _dequant(t: torch.Tensor, kv_dtype: str, scale: float) -> torch.Tensor:
    if kv_dtype == "fp8":
        return t.view(torch.float8_e4m3fn).to(torch.float64) * scale
    return t.to(torch.float64)


def sdpa_reference(w) -> torch.Tensor:
    """Each request's keys gathered densely with torch indexing, then torch's
    scaled_dot_product_attention in float64 with the end-aligned causal mask
    (token i of L sees the first S-(L-1-i) keys); rows of padding, empty requests
    and rows with no visible key are zero."""
    n, G = w.num_seqs, w.num_q_heads // w.num_kv_heads
    out = torch.zeros(w.num_tokens, w.num_q_heads, w.head_dim, dtype=torch.float64)
    cu = w.cu_query_lens
    for r in range(n):
        S = int(w.context_lens[r])
        rows = list(range(int(cu[r]), int(cu[r + 1]))) if cu is not None else [r]
        L = len(rows)
        if S <= 0 or L == 0:
            continue
        pages = w.block_tables[r, : -(-S // w.block_size)].long()
        K = _dequant(w.k_cache[pages], w.kv_dtype, w.k_scale)  # [p, Hkv, bs, D]
        V = _dequant(w.v_cache[pages], w.kv_dtype, w.v_scale)
        K = K.permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim)[:, :S]
        V = V.permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim)[:, :S]
        K = K.repeat_interleave(G, dim=0)  # q head hq uses kv head hq // G
        V = V.repeat_interleave(G, dim=0)
        q = w.q[rows].to(torch.float64).permute(1, 0, 2)  # [Hq, L, D]
        mask = torch.ones(L, S, dtype=torch.bool).tril(diagonal=S - L)
        o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=w.scale)
        visible = mask.any(dim=1)
        o[:, ~visible] = 0.0
        out[rows] = o.permute(1, 0, 2)
    return out


CASES = [
    dict(name="decode_bf16", lens=[17, 64, 200, 1000], ql=None, H=(8, 2), D=64, bs=16, kv="bf16"),
    dict(name="decode_fp8", lens=[1, 33, 300], ql=None, H=(8, 1), D=128, bs=16, kv="fp8"),
    dict(name="decode_fp16", lens=[5, 129], ql=None, H=(4, 4), D=64, bs=64, kv="fp16"),
    dict(name="verify", lens=[40, 7, 130], ql=[3, 3, 3], H=(6, 1), D=64, bs=16, kv="bf16", pad=2),
    dict(name="mixed", lens=[50, 0, 20, 9], ql=[1, 2, 20, 0], H=(4, 2), D=64, bs=16, kv="bf16",
         pad=3),
    dict(name="short_ctx", lens=[2, 3], ql=[4, 1], H=(2, 1), D=64, bs=16, kv="fp8", pad=1),
]


def _case(c, seed=0, **kw):
    return wl.make_batch(c["name"], c["lens"], c["ql"], c["H"][0], c["H"][1], c["D"], c["bs"],
                         c["kv"], seed=seed, pad_tokens=c.get("pad", 0), kv_scale=0.05, **kw)


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_dense_matches_torch_sdpa(c):
    w = _case(c)
    got = oracle_decode(w)
    ref = sdpa_reference(w).numpy()
    assert np.abs(got - ref).max() < 1e-12


def test_sdpa_reference_sees_the_per_token_causal_range():
    # "short_ctx": request 0 has S=2 keys and L=4 tokens: tokens 0 and 1 see no key
    # (S-(L-1-i) <= 0) and must be zero; tokens 2 and 3 see 1 and 2 keys.
    w = _case(CASES[-1])
    out = oracle_decode(w)
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    assert np.any(out[2] != 0) and np.any(out[3] != 0)


# ------------------------------------------------------------------- closed forms

def _single(S, L=1, H=(4, 2), D=64, bs=16, kv="bf16", seed=3):
    return wl.make_batch("single", [S], None if L == 1 else [L], H[0], H[1], D, bs, kv,
                         seed=seed, kv_scale=0.05)


def test_one_key_returns_that_value_row():
    w = _single(1)
    out = oracle_decode(w)
    page = int(w.block_tables[0, 0])
    for hq in range(w.num_q_heads):
        v = w.v_cache[page, hq // 2, 0].to(torch.float64).numpy()
        assert np.array_equal(out[0, hq], v)


def test_zero_query_gives_mean_of_visible_values():
    w = _single(77, L=3)
    w.q.zero_()
    out = oracle_decode(w)
    for i in range(3):
        K = 77 - (3 - 1 - i)
        pages = w.block_tables[0].long()
        V = w.v_cache[pages].to(torch.float64).permute(1, 0, 2, 3).reshape(2, -1, 64)[:, :K]
        for hq in range(4):
            assert np.allclose(out[i, hq], V[hq // 2].mean(0).numpy(), atol=1e-13, rtol=0)


def test_constant_values_give_that_constant():
    w = _single(300, kv="fp8")
    w.v_cache.fill_(0x38)  # e4m3fn 0x38 = 1.0
    out = oracle_decode(w)
    assert np.allclose(out, 1.0 * w.v_scale, atol=1e-14, rtol=0)


def test_dominant_key_selects_its_value():
    w = _single(100)
    w.k_cache.zero_()
    pages = w.block_tables[0].long()
    j = 57
    w.k_cache[pages[j // 16], :, j % 16] = w.q[0].reshape(2, 2, 64)[:, 0] * 64  # huge logit
    out = oracle_decode(w)
    v = w.v_cache[pages[j // 16], 0, j % 16].to(torch.float64).numpy()
    assert np.allclose(out[0, 0], v, atol=1e-12)


# -------------------------------------------------------------------- invariants

def _repage(w, new_bs: int, seed: int):
    """The same logical keys stored under another page size and a fresh random
    physical page order."""
    g = torch.Generator().manual_seed(seed)
    n = w.num_seqs
    dense_k, dense_v = [], []
    for r in range(n):
        S = int(w.context_lens[r])
        p = -(-S // w.block_size) if S > 0 else 0
        pages = w.block_tables[r, :p].long()
        dense_k.append(w.k_cache[pages].permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim))
        dense_v.append(w.v_cache[pages].permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim))
    need = [(-(-int(s) // new_bs) if s > 0 else 0) for s in w.context_lens.tolist()]
    nb = sum(need) + 5
    perm = torch.randperm(nb, generator=g)
    shape = (nb, w.num_kv_heads, new_bs, w.head_dim)
    k = torch.full(shape, 0x7F if w.kv_dtype == "fp8" else 0, dtype=w.k_cache.dtype)
    v = k.clone()
    bt = torch.full((n, max(1, max(need))), -1, dtype=torch.int32)
    at = 0
    for r in range(n):
        for b in range(need[r]):
            page = int(perm[at]); at += 1
            bt[r, b] = page
            lo, hi = b * new_bs, min((b + 1) * new_bs, dense_k[r].shape[1])
            k[page, :, : hi - lo] = dense_k[r][:, lo:hi]
            v[page, :, : hi - lo] = dense_v[r][:, lo:hi]
    return wl.Workload(w.name, w.q, k, v, w.kv_dtype, w.k_scale, w.v_scale, bt, w.context_lens,
                       w.cu_query_lens, w.scale, w.num_q_heads, w.num_kv_heads, w.head_dim,
                       new_bs, w.budget, w.max_partitions)


@pytest.mark.parametrize("c", CASES[:4], ids=[c["name"] for c in CASES[:4]])
def test_output_independent_of_paging(c):
    w = _case(c)
    base = oracle_decode(w)
    for i, bs in enumerate((16, 64, 128)):
        other = oracle_decode(_repage(w, bs, seed=11 + i))
        assert np.abs(other - base).max() < 1e-12


def test_cu_arange_is_bitwise_the_no_cu_path():
    w = _case(CASES[0])
    a = oracle_decode(w)
    w2 = wl.Workload(**{**w.__dict__, "cu_query_lens": torch.arange(5, dtype=torch.int32)})
    b = oracle_decode(w2)
    assert np.array_equal(a, b)


def test_padding_rows_and_empty_requests_are_zero():
    w = _case(CASES[4])  # lens [50, 0, 20, 9], ql [1, 2, 20, 0], 3 padding rows
    out = oracle_decode(w)
    cu = w.cu_query_lens.tolist()
    assert np.all(out[cu[1]:cu[2]] == 0)          # request 1 has S = 0
    assert np.all(out[cu[-1]:] == 0)             # graph padding rows
    assert np.all(np.isfinite(out))
    # request 2 (S=20, L=20): token 0 sees exactly one key -> that key's value
    page = int(w.block_tables[2, 0])
    t0 = cu[2]
    for hq in range(4):
        assert np.array_equal(out[t0, hq], w.v_cache[page, hq // 2, 0].to(torch.float64).numpy())


def test_adding_a_padding_row_changes_no_other_row():
    c = dict(CASES[3]); c["pad"] = 0
    w = _case(c)
    a = oracle_decode(w)
    extra = torch.randn(5, w.num_q_heads, w.head_dim).to(w.q.dtype)
    w2 = wl.Workload(**{**w.__dict__, "q": torch.cat([w.q, extra])})
    b = oracle_decode(w2)
    assert np.array_equal(a, b[: a.shape[0]]) and np.all(b[a.shape[0]:] == 0)


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_merge_identity_for_any_split_count(c):
    """Partial softmaxes over the plan's tasks plus the LSE merge give the dense
    result, whatever the split count (1 ... 256) and the plan kind."""
    w = _case(c)
    dense = oracle_decode(w)
    for P, W in ((1, 8), (2, 8), (7, 100), (256, 512), (256, 4096)):
        for kind in (oracle.PLAN_PROPORTIONAL, oracle.PLAN_UNIFORM):
            work, red = oracle_plan(w, W, kind, max_partitions=P)
            got = oracle_decode_planned(w, work, red)
            assert np.abs(got - dense).max() < 1e-12, (P, W, kind)


def test_merge_identity_uses_every_partition():
    # a plan whose tasks split a 1000-token request in several parts
    w = _case(CASES[0])
    work, red = oracle_plan(w, 4096, max_partitions=256)
    assert red[3, 1] == 4
    dense = oracle_decode(w)
    bad = work.copy()
    bad[red[3, 0], 2] -= 1  # drop the last tile of the first part
    got = oracle_decode_planned(w, bad, red)
    assert np.abs(got[3] - dense[3]).max() > 1e-3


# ---------------------------------------------------------------------- work plan

def test_golden_capacities():
    g = json.load(open(GOLDEN))
    for e in g["capacity"]:
        assert oracle.plan_capacity(e["n"], e["num_kv_heads"], e["max_partitions"],
                                    e["budget"]) == e["capacity"], e["cite"]


def _lens(e):
    if "context_lens" in e:
        return e["context_lens"]
    v, k = e["context_lens_repeat"]
    return [v] * k


def test_golden_partition_counts():
    g = json.load(open(GOLDEN))
    for e in g["partitions"]:
        lens = np.array(_lens(e), dtype=np.int32)
        want = e["parts"] if "parts" in e else [e["parts_repeat"][0]] * e["parts_repeat"][1]
        _, red = oracle.plan(lens, None, e["num_kv_heads"], e["max_partitions"], e["budget"])
        assert red[:, 1].tolist() == want, e["cite"]
        if "same_with_max_partitions" in e:
            _, red2 = oracle.plan(lens, None, e["num_kv_heads"], e["same_with_max_partitions"],
                                  e["budget"])
            assert red2[:, 1].tolist() == want, e["cite"]


def test_golden_tile_counts():
    g = json.load(open(GOLDEN))
    for e in g["tiles"]:
        for S, nt in zip(e["context_lens"], e["tiles"]):
            work, red = oracle.plan(np.array([S], np.int32), None, 1, 100000, 10 ** 6)
            p = red[0, 1]
            assert p == nt  # one tile per partition when the budget is unbounded
            assert work[p - 1, 2] == nt and work[0, 1] == 0


def test_capacity_ceil_and_floor():
    assert oracle.plan_capacity(1, 3, 256, 10) == 4      # ceil(10 / 3)
    assert oracle.plan_capacity(32, 4, 256, 296) == 74
    assert oracle.plan_capacity(512, 8, 256, 304) == 512  # never below the batch
    assert oracle.plan_capacity(2, 1, 3, 512) == 6        # never above n * P


def _check_plan(lens, qlens, Hkv, P, W, kind):
    lens = np.asarray(lens, np.int32)
    cu = None if qlens is None else np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    work, red = oracle.plan(lens, cu, Hkv, P, W, kind)
    n, C = len(lens), work.shape[0]
    ql = np.ones(n, int) if qlens is None else np.asarray(qlens)
    active = (lens > 0) & (ql > 0)
    parts = red[:, 1]
    T = oracle.TILE
    tiles = -(-lens.astype(np.int64) // T)
    assert parts.sum() <= C
    assert np.all(parts[~active] == 0)
    assert np.all(parts[active] >= 1)
    assert np.all(parts[active] <= np.minimum(P, tiles[active]))
    assert np.array_equal(red[:, 0], np.concatenate([[0], np.cumsum(parts)[:-1]]))
    for r in range(n):
        f, p = red[r]
        if p == 0:
            continue
        seg = work[f:f + p]
        assert np.all(seg[:, 0] == r) and np.all(seg[:, 3] == lens[r])
        assert seg[0, 1] == 0 and seg[-1, 2] == tiles[r]
        assert np.all(seg[1:, 1] == seg[:-1, 2]) and np.all(seg[:, 2] > seg[:, 1])
        sizes = seg[:, 2] - seg[:, 1]
        assert sizes.max() - sizes.min() <= 1     # even chunking
    assert np.all(work[parts.sum():, 0] == -1)
    return work, red, active


@pytest.mark.parametrize("kind", [oracle.PLAN_PROPORTIONAL, oracle.PLAN_UNIFORM])
@pytest.mark.parametrize("seed", range(6))
def test_plan_invariants_random(kind, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    lens = np.clip(np.round(np.exp(rng.normal(np.log(4096), 1.5, n))), 1, 131072).astype(np.int32)
    lens[rng.random(n) < 0.1] = 0
    qlens = None if seed % 2 == 0 else rng.integers(0, 5, n)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    P = int(rng.choice([1, 8, 64, 256]))
    W = int(rng.choice([296, 304, 512, 2048]))
    work, red, active = _check_plan(lens, qlens, Hkv, P, W, kind)
    parts = red[:, 1]
    if kind == oracle.PLAN_PROPORTIONAL:
        # monotone in context length among active requests
        idx = np.where(active)[0]
        order = idx[np.argsort(lens[idx], kind="stable")]
        assert np.all(np.diff(parts[order]) >= 0)
    else:
        C = work.shape[0]
        tiles = -(-lens.astype(np.int64) // oracle.TILE)
        cap = min(P, C // max(1, active.sum()))
        assert np.array_equal(parts[active], np.minimum(cap, tiles[active]))


def test_plan_proportional_rule_by_hand():
    # C = min(3*256, max(3, ceil(304/4))) = 76; n_act = 3; sum S = 11000
    lens = np.array([1000, 2000, 8000], np.int32)
    work, red = oracle.plan(lens, None, 4, 256, 304)
    assert work.shape[0] == 76
    # 1 + floor(73*S/11000): 1000 -> 7 (cap 4 tiles), 2000 -> 14 (cap 8), 8000 -> 54 (cap 32)
    assert red[:, 1].tolist() == [4, 8, 32]
    lens = np.array([100000, 5000, 300], np.int32)
    _, red = oracle.plan(lens, None, 4, 256, 304)
    # 1 + floor(73*S/105300): 100000 -> 70, 5000 -> 4, 300 -> 1
    assert red[:, 1].tolist() == [70, 4, 1]
    _, red = oracle.plan(lens, None, 4, 256, 304, kind=oracle.PLAN_UNIFORM)
    # floor(76/3) = 25 each, capped by tiles: 391 -> 25, 20 -> 20, 2 -> 2
    assert red[:, 1].tolist() == [25, 20, 2]


def test_plan_skips_zero_length_and_rowless_requests():
    lens = np.array([500, 0, 700, 300], np.int32)
    cu = np.array([0, 1, 2, 2, 5], np.int32)   # request 2 owns no query row
    work, red = oracle.plan(lens, cu, 1, 256, 16)
    assert red[:, 1].tolist()[1:3] == [0, 0]
    # n_act = 2, sum S = 800, C = 16: 1 + floor(14*500/800) = 9 -> 2 tiles; 1 + floor(14*300/800) = 6 -> 2
    assert red[:, 1].tolist() == [2, 0, 0, 2]
    assert red[:, 0].tolist() == [0, 2, 2, 2]


# ------------------------------------------------- sliding window and attention sinks

def sdpa_window_reference(w, window: int, sinks=None) -> torch.Tensor:
    """torch SDPA in float64 with a banded mask: token i (end-aligned causal range
    [0, K_i)) sees only keys [K_i - window, K_i).  A sink is an extra key whose
    logit is the sink and whose value row is zero, appended to every row."""
    n, G = w.num_seqs, w.num_q_heads // w.num_kv_heads
    out = torch.zeros(w.num_tokens, w.num_q_heads, w.head_dim, dtype=torch.float64)
    cu = w.cu_query_lens
    for r in range(n):
        S = int(w.context_lens[r])
        rows = list(range(int(cu[r]), int(cu[r + 1]))) if cu is not None else [r]
        L = len(rows)
        if S <= 0 or L == 0:
            continue
        pages = w.block_tables[r, : -(-S // w.block_size)].long()
        K = _dequant(w.k_cache[pages], w.kv_dtype, w.k_scale)
        V = _dequant(w.v_cache[pages], w.kv_dtype, w.v_scale)
        K = K.permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim)[:, :S]
        V = V.permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim)[:, :S]
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        q = w.q[rows].to(torch.float64).permute(1, 0, 2)  # [Hq, L, D]
        mask = torch.ones(L, S, dtype=torch.bool).tril(diagonal=S - L)
        if window > 0:
            mask &= ~torch.ones(L, S, dtype=torch.bool).tril(diagonal=S - L - window)
        visible = mask.any(dim=1)
        if sinks is None:
            o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=w.scale)
        else:
            # the sink as one more key: a key vector along q with logit = sink (per
            # head and row), and a zero value row
            sk = torch.as_tensor(sinks, dtype=torch.float64)  # [Hq]
            qn = (q * q).sum(-1, keepdim=True)  # [Hq, L, 1]
            ksink = q * (sk[:, None, None] / (w.scale * qn))  # scale * q . ksink = sink
            Kx = torch.cat([K[:, None].expand(-1, L, -1, -1), ksink[:, :, None]], dim=2)
            Vx = torch.cat([V[:, None].expand(-1, L, -1, -1),
                            torch.zeros(w.num_q_heads, L, 1, w.head_dim, dtype=torch.float64)], dim=2)
            mx = torch.cat([mask, torch.ones(L, 1, dtype=torch.bool)], dim=1)
            o = F.scaled_dot_product_attention(q[:, :, None], Kx, Vx, attn_mask=mx[:, None],
                                               scale=w.scale)[:, :, 0]
        o[:, ~visible] = 0.0
        out[rows] = o.permute(1, 0, 2)
    return out


WINDOW_CASES = [c for c in CASES if c["name"] in ("decode_bf16", "decode_fp8", "verify", "mixed")]


@pytest.mark.parametrize("window", [1, 3, 50, 500])
@pytest.mark.parametrize("c", WINDOW_CASES, ids=[c["name"] for c in WINDOW_CASES])
def test_window_matches_torch_sdpa_banded(c, window):
    w = _case(c)
    got = oracle_decode(w, window=window)
    ref = sdpa_window_reference(w, window).numpy()
    assert np.abs(got - ref).max() < 1e-12


def test_window_wider_than_every_row_is_no_window():
    w = _case(CASES[0])  # longest request: 1000 keys
    assert np.array_equal(oracle_decode(w, window=1000), oracle_decode(w))
    assert np.array_equal(oracle_decode(w, window=5000), oracle_decode(w))


def test_window_one_returns_the_last_visible_value_row():
    w = _single(300, H=(4, 2))
    out = oracle_decode(w, window=1)
    G = 2
    page = int(w.block_tables[0, 299 // w.block_size])
    for hq in range(4):
        v = w.v_cache[page, hq // G, 299 % w.block_size].to(torch.float64).numpy()
        assert np.abs(out[0, hq] - v).max() < 1e-15


@pytest.mark.parametrize("c", WINDOW_CASES, ids=[c["name"] for c in WINDOW_CASES])
def test_sinks_match_torch_sdpa_with_an_extra_key(c):
    w = _case(c)
    rng = np.random.default_rng(4)
    sinks = rng.normal(0.0, 2.0, w.num_q_heads)
    for window in (0, 50):
        got = oracle_decode(w, window=window, sinks=sinks)
        ref = sdpa_window_reference(w, window, sinks).numpy()
        assert np.abs(got - ref).max() < 1e-12, window


def test_sink_at_minus_infinity_is_no_sink_and_a_huge_sink_silences_the_row():
    w = _case(CASES[0])
    none = oracle_decode(w)
    assert np.array_equal(oracle_decode(w, sinks=np.full(w.num_q_heads, -np.inf)), none)
    quiet = oracle_decode(w, sinks=np.full(w.num_q_heads, 800.0))
    assert np.abs(quiet).max() < 1e-300


@pytest.mark.parametrize("window", [1, 37, 300, 5000])
@pytest.mark.parametrize("c", WINDOW_CASES, ids=[c["name"] for c in WINDOW_CASES])
def test_windowed_plan_covers_the_read_range_and_merges_to_dense(c, window):
    """The windowed plan covers, for each request, the tiles from the one holding
    its first token's first visible key up to ceil(S/T), once each; its partials
    merge to the dense windowed result, with and without sinks."""
    w = _case(c)
    lens = w.context_lens.numpy()
    cu = None if w.cu_query_lens is None else w.cu_query_lens.numpy()
    sinks = np.linspace(-1.0, 1.0, w.num_q_heads)
    for P, W in ((1, 8), (7, 100), (256, 4096)):
        work, red = oracle_plan(w, W, max_partitions=P, window=window)
        for r in range(w.num_seqs):
            f, p = red[r]
            if p == 0:
                continue
            L = 1 if cu is None else int(cu[r + 1] - cu[r])
            first = max(0, int(lens[r]) - (L - 1) - window)
            seg = work[f:f + p]
            assert seg[0, 1] == first // oracle.TILE
            assert seg[-1, 2] == -(-int(lens[r]) // oracle.TILE)
            assert np.all(seg[1:, 1] == seg[:-1, 2])
        for sk in (None, sinks):
            got = oracle_decode_planned(w, work, red, window=window, sinks=sk)
            dense = oracle_decode(w, window=window, sinks=sk)
            assert np.abs(got - dense).max() < 1e-12, (P, W)


def test_windowed_plan_with_no_window_is_the_plain_plan():
    lens = np.array([100000, 5000, 300, 0, 70000], np.int32)
    for kind in (oracle.PLAN_PROPORTIONAL, oracle.PLAN_UNIFORM):
        a = oracle.plan(lens, None, 4, 256, 304, kind)
        b = oracle.plan(lens, None, 4, 256, 304, kind, window=200000)  # wider than every S
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_windowed_plan_sizes_requests_by_their_window():
    # A window of 1000 keys makes every request read at most 1000 (+ alignment)
    # keys: the proportional shares follow the read ranges, not S.
    lens = np.array([100000, 5000, 300], np.int32)
    work, red = oracle.plan(lens, None, 4, 256, 304, window=1000)
    # read ranges from the first visible key's tile: 100000-1000=99000 -> tile 386
    # (98816): 1184 keys, 5 tiles; 5000-1000=4000 -> tile 15 (3840): 1160, 5
    # tiles; 300: 300 keys, 2 tiles.  sum = 2644; C - n_act = 73:
    # 1 + floor(73*1184/2644) = 33 -> 5; 1 + floor(73*1160/2644) = 33 -> 5; 1 + 8 -> 2
    assert red[:, 1].tolist() == [5, 5, 2]
    assert work[0, 1] == 386 and work[4, 2] == 391


# ------------------------------------------------------ K in 16-element groups

@pytest.mark.parametrize("c", WINDOW_CASES, ids=[c["name"] for c in WINDOW_CASES])
def test_grouped_k_layout_gives_the_same_result(c):
    """K rearranged into [num_blocks, Hkv, D/16, block_size, 16] (torch permute)
    must give exactly the same outputs, dense and planned, with a window and
    sinks."""
    w = _case(c)
    w5 = wl.with_k_groups(w)
    assert w5.k_cache.dim() == 5
    sinks = np.linspace(-1.0, 1.0, w.num_q_heads)
    assert np.array_equal(oracle_decode(w5), oracle_decode(w))
    assert np.array_equal(oracle_decode(w5, window=30, sinks=sinks),
                          oracle_decode(w, window=30, sinks=sinks))
    work, red = oracle_plan(w, 100, max_partitions=7)
    assert np.array_equal(oracle_decode_planned(w5, work, red), oracle_decode_planned(w, work, red))


def test_grouped_k_layout_element_positions():
    # element (page p, head h, key slot j, dim d) of the 5-D K sits at
    # [p, h, d // 16, j, d % 16]: a cache whose every element encodes its own
    # (j, d) checks the permutation, independent of the oracle
    w = _single(40, H=(2, 2), D=64, bs=16)
    nb, hkv, bs, d = w.k_cache.shape
    jj = torch.arange(bs).view(1, 1, bs, 1).expand(nb, hkv, bs, d)
    dd = torch.arange(d).view(1, 1, 1, d).expand(nb, hkv, bs, d)
    code = ((jj << 8) | dd).to(torch.int16)  # distinct bit patterns
    w.k_cache.view(torch.int16).copy_(code)
    k5 = wl.with_k_groups(w).k_cache.view(torch.int16)
    for j, dim in ((0, 0), (3, 17), (15, 63), (7, 48)):
        assert int(k5[1, 1, dim // 16, j, dim % 16]) == (j << 8) | dim


# ------------------------------------------------------- sparse top-k decode

def test_sparse_select_order_by_hand():
    """Seven blocks, no fixed blocks: the scores rank NaN > 2.0 (block 3) = 2.0
    (block 4, the higher index loses the tie) > 1.0 > +0 > -0 > -inf, so the
    top k for k = 0..7 adds blocks 1, 3, 4, 0, 6, 5, 2 in that order."""
    sc = np.array([[1.0, np.nan, -np.inf, 2.0, 2.0, -0.0, 0.0]], dtype=np.float32)
    bt = np.arange(10, 17, dtype=np.int32)[None]
    rank = [1, 3, 4, 0, 6, 5, 2]
    for k in range(8):
        sel, sl = oracle.sparse_select(sc, np.array([7 * 16], np.int32), bt, 16, k, 0, 0)
        want = sorted(10 + b for b in rank[:k])
        assert sel[0].tolist() == want, k
        assert sl[0] == 16 * k


def _order_key(x: np.float32) -> int:
    u = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
    return (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)


def _select_by_repeated_argmax(scores, S, bs, top_k, init, local, max_blocks):
    """The same selection found another way: fixed blocks, then top_k times the
    remaining candidate with the largest (key, -index)."""
    nb = min(-(-S // bs) if S > 0 else 0, max_blocks)
    chosen = {b for b in range(nb) if b < init or b >= nb - local}
    rest = [b for b in range(nb) if b not in chosen]
    for _ in range(top_k):
        if not rest:
            break
        best = max(rest, key=lambda b: (_order_key(scores[b]), -b))
        chosen.add(best)
        rest.remove(best)
    blocks = sorted(chosen)
    tokens = sum(min((b + 1) * bs, S) - b * bs for b in blocks)
    return blocks, tokens


@pytest.mark.parametrize("seed", range(6))
def test_sparse_select_matches_repeated_argmax(seed):
    rng = np.random.default_rng(seed)
    n, bs, max_blocks = 12, 16, 20
    palette = np.array([0.5, -1.0, 3.0, 0.0, -0.0, np.inf, -np.inf, np.nan, 3.0], np.float32)
    scores = palette[rng.integers(0, len(palette), (n, max_blocks))]  # many ties
    lens = rng.integers(0, max_blocks * bs + 1, n).astype(np.int32)
    lens[0], lens[1], lens[2] = 0, 5, bs  # empty, one partial block, one full block
    bt = rng.permutation(1000)[: n * max_blocks].reshape(n, max_blocks).astype(np.int32)
    for top_k, init, local in [(0, 1, 1), (3, 0, 1), (4, 1, 2), (5, 2, 0), (25, 1, 1), (2, 9, 9)]:
        sel, sl = oracle.sparse_select(scores, lens, bt, bs, top_k, init, local)
        for r in range(n):
            blocks, tokens = _select_by_repeated_argmax(scores[r], int(lens[r]), bs, top_k, init,
                                                        local, max_blocks)
            want = [int(bt[r, b]) for b in blocks]
            assert sel[r, : len(want)].tolist() == want, (r, top_k, init, local)
            assert (sel[r, len(want):] == -1).all()
            assert sl[r] == tokens


def test_sparse_select_without_scores_keeps_only_fixed_blocks():
    lens = np.array([0, 10, 100, 1000], np.int32)
    bt = np.arange(4 * 70, dtype=np.int32).reshape(4, 70)
    sel, sl = oracle.sparse_select(None, lens, bt, 16, 0, 2, 1)
    assert sel.tolist() == [[-1, -1, -1], [70, -1, -1], [140, 141, 146], [210, 211, 272]]
    assert sl.tolist() == [0, 10, 16 + 16 + 4, 16 + 16 + 8]


def _sparse_case(kv="bf16", seed=0):
    return wl.make_batch("sparse", [1, 40, 300, 777, 1500], None, 8, 2, 64, 16, kv, seed=seed,
                         kv_scale=0.05)


def test_sparse_decode_with_every_block_selected_is_dense():
    w = _sparse_case()
    a = oracle_args(w)
    nbmax = w.block_tables.shape[1]
    scores = np.random.default_rng(1).normal(size=(w.num_seqs, nbmax)).astype(np.float32)
    sparse = oracle.sparse_decode(*a[:9], a[10], scores, w.block_size, nbmax, 1, 1)
    assert np.array_equal(sparse, oracle_decode(w))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_sparse_decode_matches_sdpa_over_the_selected_keys(kv):
    """torch SDPA in float64 over the explicit token positions of the selected
    blocks (gathered from the request's own block table)."""
    w = _sparse_case(kv, seed=2)
    a = oracle_args(w)
    nbmax = w.block_tables.shape[1]
    scores = np.random.default_rng(3).normal(size=(w.num_seqs, nbmax)).astype(np.float32)
    top_k, init, local = 5, 1, 2
    got = oracle.sparse_decode(*a[:9], a[10], scores, w.block_size, top_k, init, local)
    G = w.num_q_heads // w.num_kv_heads
    for r in range(w.num_seqs):
        S = int(w.context_lens[r])
        blocks, _ = _select_by_repeated_argmax(scores[r], S, w.block_size, top_k, init, local,
                                               nbmax)
        pos = [j for b in blocks for j in range(b * w.block_size, min((b + 1) * w.block_size, S))]
        pages = w.block_tables[r, torch.tensor(pos) // w.block_size].long()
        slot = torch.tensor(pos) % w.block_size
        K = _dequant(w.k_cache[pages, :, slot], w.kv_dtype, w.k_scale)  # [keys, Hkv, D]
        V = _dequant(w.v_cache[pages, :, slot], w.kv_dtype, w.v_scale)
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        q = w.q[r].to(torch.float64)[:, None, :]
        o = F.scaled_dot_product_attention(q, K, V, scale=w.scale)[:, 0]
        assert np.abs(got[r] - o.numpy()).max() < 1e-12, r
