"""Seeded synthetic inputs for paged-KV decode.

This module holds no arithmetic of the attention method or of the work plan:
it only draws random numbers and lays them out as a paged KV cache.  Both the
CUDA path and the CPU oracle consume what it produces.

Workload shapes follow the batches the source pages describe:
  * context-length skew of agentic decode batches ("[MiniMax-M3] Route the
    paged decode to aiter's FlyDSL kernel with work planner", section 1,
    Motivation: step-internal max/min context ratio p50 2.49, p90 22.2, max
    1610) -- modelled as a clipped lognormal;
  * the MTP-verify and mixed decode+prompt launch shapes of vllm-rdna pull 29
    (Problem table: 8 req x 3 tok at 16k with H 6/1; 7 decodes at 16k plus a
    100-token prompt with H 12/2, D=256);
  * fp8 page-16 KV caches with a per-tensor scale.

Layouts: q [num_tokens, Hq, D]; k_cache/v_cache [num_blocks, Hkv, block_size, D]
(bf16/fp16 tensors, or uint8 bytes holding OCP float8 e4m3fn codes);
block_tables int32 [n, max_blocks] with -1 in unused entries; context_lens
int32 [n]; cu_query_lens int32 [n+1] or None.  Physical pages are a random
permutation of the pool.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

KV_DTYPES = ("bf16", "fp16", "fp8")


@dataclass
class Workload:
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    kv_dtype: str
    k_scale: float
    v_scale: float
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    cu_query_lens: Optional[torch.Tensor]
    scale: float
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    budget: Optional[int] = None        # None: 2 x SM count of the device
    max_partitions: int = 256
    meta: dict = field(default_factory=dict)
    window: int = 0                     # sliding window (0: none)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    def kv_bytes_per_request(self) -> torch.Tensor:
        """Algorithmic KV bytes of each request (int64, CPU): every key and
        value row its tokens can see, per kv head, read once (under a sliding
        window W: the last W + L - 1 keys of a request with L tokens)."""
        lens = self.context_lens.clamp(min=0).to(torch.int64).cpu()
        if self.window > 0:
            if self.cu_query_lens is None:
                L = torch.ones_like(lens)
            else:
                cu = self.cu_query_lens.to(torch.int64).cpu()
                L = cu[1:] - cu[:-1]
            lens = torch.minimum(lens, self.window + L - 1)
            lens[L == 0] = 0
        return lens * self.num_kv_heads * self.head_dim * 2 * self.kv_elem_bytes

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of one decode call (kv_bytes_per_request summed)."""
        return int(self.kv_bytes_per_request().sum().item())

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return Workload(self.name, mv(self.q), mv(self.k_cache), mv(self.v_cache), self.kv_dtype,
                        self.k_scale, self.v_scale, mv(self.block_tables), mv(self.context_lens),
                        mv(self.cu_query_lens), self.scale, self.num_q_heads, self.num_kv_heads,
                        self.head_dim, self.block_size, self.budget, self.max_partitions,
                        dict(self.meta), self.window)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def lognormal_lengths(n: int, median: float, sigma: float, lo: int, hi: int,
                      seed: int) -> list[int]:
    """n context lengths ~ round(lognormal(ln median, sigma)) clipped to [lo, hi]."""
    g = _gen(seed, "cpu")
    z = torch.randn(n, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return [int(v) for v in x.tolist()]


def _kv_values(shape, kv_dtype: str, scale: float, g: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if kv_dtype == "bf16":
        return x.to(torch.bfloat16)
    if kv_dtype == "fp16":
        return x.to(torch.float16)
    if kv_dtype == "fp8":
        # stored code = float8_e4m3fn(x / scale), round-to-nearest-even; |x/scale| is
        # kept inside the format's finite range +-448.
        return (x / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


def make_batch(name: str, context_lens: Sequence[int], query_lens: Optional[Sequence[int]],
               num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
               kv_dtype: str = "bf16", q_dtype: str = "bf16", seed: int = 0,
               pool_pages: Optional[int] = None, pad_tokens: int = 0,
               kv_scale: float = 0.05, scale: Optional[float] = None, device="cpu",
               budget: Optional[int] = None, max_partitions: int = 256,
               spare_blocks: int = 0, q_std: float = 1.0) -> Workload:
    """A paged batch.  query_lens=None means one query token per request and no
    cu_query_lens; otherwise cu_query_lens is the running sum of query_lens and
    pad_tokens graph-padding rows follow the last request's rows.  q is drawn
    N(0, q_std^2): q_std = 1 gives logits of about unit spread (a nearly flat
    softmax over a long context); a larger q_std (e.g. 6) gives sharp
    attention, dominated by a few keys, whose outputs stay of order 1 however
    long the context."""
    n = len(context_lens)
    g = _gen(seed, device)
    gc = _gen(seed + 7919, "cpu")
    pages = [max(0, -(-int(s) // block_size)) for s in context_lens]
    max_blocks = max(1, max(pages) + spare_blocks)
    need = sum(pages)
    nb = max(need, 1) if pool_pages is None else pool_pages
    if nb < need:
        raise ValueError(f"pool of {nb} pages cannot hold {need}")
    perm = torch.randperm(nb, generator=gc).to(torch.int32)
    bt = torch.full((n, max_blocks), -1, dtype=torch.int32)
    at = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[at:at + p]
        at += p

    if query_lens is None:
        cu = None
        num_tokens = n
    else:
        assert len(query_lens) == n
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(list(query_lens), dtype=torch.int64), 0).to(torch.int32)
        num_tokens = int(cu[-1]) + pad_tokens

    qdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[q_dtype]
    q = (torch.randn((num_tokens, num_q_heads, head_dim), generator=g, device=device,
                     dtype=torch.float32) * q_std).to(qdt)
    shape = (nb, num_kv_heads, block_size, head_dim)
    k = _kv_values(shape, kv_dtype, kv_scale, g, device)
    v = _kv_values(shape, kv_dtype, kv_scale, g, device)
    ks = kv_scale if kv_dtype == "fp8" else 1.0
    return Workload(
        name=name, q=q, k_cache=k, v_cache=v, kv_dtype=kv_dtype, k_scale=ks, v_scale=ks,
        block_tables=bt.to(device), context_lens=torch.tensor(list(context_lens),
                                                              dtype=torch.int32).to(device),
        cu_query_lens=None if cu is None else cu.to(device),
        scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale,
        num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, budget=budget, max_partitions=max_partitions,
        meta={"seed": seed})


# ------------------------------------------------------------------ named configs

def tiny(seed: int = 0, device="cpu") -> Workload:
    """4 decodes with context {17, 64, 200, 1000}, Hq/Hkv 8/2, D 64, page 16, bf16,
    pages permuted inside a 128-page pool, scale 1/sqrt(64)."""
    return make_batch("tiny", [17, 64, 200, 1000], None, 8, 2, 64, 16, "bf16", seed=seed,
                      pool_pages=128, device=device)


def uniform(seed: int = 0, device="cpu") -> Workload:
    """32 decodes x 8192 context, Hq/Hkv 32/4, D 128, page 16, bf16."""
    return make_batch("uniform", [8192] * 32, None, 32, 4, 128, 16, "bf16", seed=seed,
                      device=device)


def skewed(seed: int = 0, device="cpu") -> Workload:
    """32 decodes, context lognormal(median 4096, sigma 1.5) clipped to [64, 131072],
    Hq/Hkv 32/4, D 128, page 16, fp8 e4m3fn KV with scale 0.05, bf16 q, budget
    2 x 148, partition cap 256."""
    lens = lognormal_lengths(32, 4096, 1.5, 64, 131072, seed)
    w = make_batch("skewed", lens, None, 32, 4, 128, 16, "fp8", seed=seed, kv_scale=0.05,
                   device=device, budget=296, max_partitions=256)
    w.meta["max_over_min"] = max(lens) / min(lens)
    return w


def skewed_mtp3(seed: int = 0, device="cpu") -> Workload:
    """MTP verify on the skewed agentic batch: the skewed lengths (32 requests,
    lognormal median 4096, sigma 1.5, clipped to [64, 131072]), 3 query tokens
    per request (the target token and two drafts), Hq/Hkv 32/4, D 128, page 16,
    fp8 e4m3fn KV (scale 0.05), bf16 q, budget 2 x 148, cap 256 -- the pages'
    production shape, fp8 page-16 KV with speculative-decoding verify rows."""
    lens = lognormal_lengths(32, 4096, 1.5, 64, 131072, seed)
    w = make_batch("skewed_mtp3", lens, [3] * 32, 32, 4, 128, 16, "fp8", seed=seed,
                   kv_scale=0.05, device=device, budget=296, max_partitions=256)
    w.meta["max_over_min"] = max(lens) / min(lens)
    return w


def mtp_verify(seed: int = 0, device="cpu", pad_tokens: int = 8) -> Workload:
    """MTP verify: 8 requests x 3 query tokens at 16384 context, Hq/Hkv 6/1, D 256,
    page 64, bf16, per-token causal ranges, graph padding rows after cu[-1]."""
    return make_batch("mtp_verify", [16384] * 8, [3] * 8, 6, 1, 256, 64, "bf16", seed=seed,
                      pad_tokens=pad_tokens, device=device)


def mixed_prompt(seed: int = 0, device="cpu", pad_tokens: int = 21) -> Workload:
    """Mixed batch: 7 single-token decodes at 16384 plus one 100-token prompt of
    context 100, Hq/Hkv 12/2, D 256, page 64, bf16, graph padding rows."""
    return make_batch("mixed_prompt", [16384] * 7 + [100], [1] * 7 + [100], 12, 2, 256, 64,
                      "bf16", seed=seed, pad_tokens=pad_tokens, device=device)


def verify_rows(kv_dtype: str, tokens: int, seed: int = 0, device="cpu") -> Workload:
    """Verify rows at head dim 128: 16 requests x 16384 keys, `tokens` query
    tokens each (per-token causal ranges), Hq/Hkv 32/4, page 16, bf16 or fp8
    KV (scale 0.05)."""
    return make_batch(f"rows_{kv_dtype}_t{tokens}", [16384] * 16, [tokens] * 16, 32, 4, 128, 16,
                      kv_dtype, seed=seed, kv_scale=0.05, device=device)


def large(kv_dtype: str = "bf16", seed: int = 0, device="cpu") -> Workload:
    """512 decodes, context lognormal(median 2048, sigma 1.2) clipped to [16, 65536],
    Hq/Hkv 64/8, D 128, page 128, bf16 or fp8 KV, budget 2 x SM, cap 256."""
    lens = lognormal_lengths(512, 2048, 1.2, 16, 65536, seed)
    return make_batch(f"large_{kv_dtype}", lens, None, 64, 8, 128, 128, kv_dtype, seed=seed,
                      kv_scale=0.05, device=device)


def large_quarter(kv_dtype: str = "bf16", seed: int = 0, device="cpu") -> Workload:
    """The first 128 requests of the Large batch's length draw (same shapes:
    Hq/Hkv 64/8, D 128, page 128): about 2 GB of bf16 KV, a profiling-sized
    case of the same kernel (larger than L2, a few GB on the device)."""
    lens = lognormal_lengths(512, 2048, 1.2, 16, 65536, seed)[:128]
    return make_batch(f"large_{kv_dtype}_quarter", lens, None, 64, 8, 128, 128, kv_dtype,
                      seed=seed, kv_scale=0.05, device=device)


def uniform_window(seed: int = 0, device="cpu") -> Workload:
    """The uniform batch under a 1024-key sliding window (each request reads its
    last 1024 keys)."""
    w = uniform(seed, device)
    w.name, w.window = "uniform_w1024", 1024
    return w


def skewed_window(seed: int = 0, device="cpu") -> Workload:
    """The skewed batch under a 4096-key sliding window."""
    w = skewed(seed, device)
    w.name, w.window = "skewed_w4096", 4096
    return w


CONFIGS = {
    "tiny": tiny,
    "uniform": uniform,
    "skewed": skewed,
    "mtp_verify": mtp_verify,
    "mixed_prompt": mixed_prompt,
    "large_bf16": lambda seed=0, device="cpu": large("bf16", seed, device),
    "large_fp8": lambda seed=0, device="cpu": large("fp8", seed, device),
    "large_bf16_quarter": lambda seed=0, device="cpu": large_quarter("bf16", seed, device),
    "uniform_w1024": uniform_window,
    "skewed_w4096": skewed_window,
}


def with_k_groups(w: Workload) -> Workload:
    """The same batch with K stored in the 5-D layout [num_blocks, Hkv, D/16,
    block_size, 16] (the head dim in 16-element groups; V unchanged)."""
    nb, hkv, bs, d = w.k_cache.shape
    k5 = w.k_cache.view(nb, hkv, bs, d // 16, 16).permute(0, 1, 3, 2, 4).contiguous()
    return Workload(w.name + "_k5", w.q, k5, w.v_cache, w.kv_dtype, w.k_scale, w.v_scale,
                    w.block_tables, w.context_lens, w.cu_query_lens, w.scale, w.num_q_heads,
                    w.num_kv_heads, w.head_dim, w.block_size, w.budget, w.max_partitions,
                    dict(w.meta), w.window)


# The uniform and skewed batches with K in the grouped 5-D layout (same bytes).
CONFIGS["uniform_k5"] = lambda seed=0, device="cpu": with_k_groups(uniform(seed, device))
CONFIGS["skewed_k5"] = lambda seed=0, device="cpu": with_k_groups(skewed(seed, device))


def uniform_d512(seed: int = 0, device="cpu") -> Workload:
    """16 decodes x 8192 context, Hq/Hkv 32/4, D 512, page 16, bf16."""
    return make_batch("uniform_d512", [8192] * 16, None, 32, 4, 512, 16, "bf16", seed=seed,
                      device=device)


def uniform_d1024(seed: int = 0, device="cpu") -> Workload:
    """16 decodes x 8192 context, Hq/Hkv 32/4, D 1024, page 16, bf16."""
    return make_batch("uniform_d1024", [8192] * 16, None, 32, 4, 1024, 16, "bf16", seed=seed,
                      device=device)


def skewed_d1024(seed: int = 0, device="cpu") -> Workload:
    """The skewed length mix (32 decodes, lognormal median 4096, sigma 1.5) with
    Hq/Hkv 16/2, D 1024, page 16, fp8 e4m3fn KV (scale 0.05), K in the grouped
    5-D layout, budget 2 x 148, partition cap 256."""
    lens = lognormal_lengths(32, 4096, 1.5, 64, 131072, seed)
    w = make_batch("skewed_d1024", lens, None, 16, 2, 1024, 16, "fp8", seed=seed,
                   kv_scale=0.05, device=device, budget=296, max_partitions=256)
    w.meta["max_over_min"] = max(lens) / min(lens)
    w = with_k_groups(w)
    w.name = "skewed_d1024"
    return w


def uniform_n64_h8(seed: int = 0, device="cpu") -> Workload:
    """64 decodes x 4096 context, Hq/Hkv 64/8, D 128, page 16, bf16: the plan
    keeps one partition per request (C = n = 64), so its 512 CTAs are more
    than the 2 x SM count that run at once."""
    return make_batch("uniform_n64_h8", [4096] * 64, None, 64, 8, 128, 16, "bf16", seed=seed,
                      device=device)


CONFIGS["uniform_d512"] = uniform_d512
CONFIGS["uniform_d1024"] = uniform_d1024
CONFIGS["skewed_d1024"] = skewed_d1024
CONFIGS["uniform_n64_h8"] = uniform_n64_h8
CONFIGS["skewed_mtp3"] = skewed_mtp3
for _kv in ("fp8", "bf16"):
    for _t in (1, 2, 3, 4):
        CONFIGS[f"rows_{_kv}_t{_t}"] = (lambda seed=0, device="cpu", kv=_kv, t=_t:
                                        verify_rows(kv, t, seed, device))


@dataclass
class SparseWorkload:
    """A decode batch whose requests attend to a top-k selection of their KV
    blocks: `base` is the batch (caches, block tables, context lengths, one
    query token per request), `scores` the per-block indexer scores [n,
    max_blocks] fp32; the selection keeps the first `init_blocks`, the last
    `local_blocks` and the `top_k` best-scored blocks between them."""
    name: str
    base: Workload
    scores: torch.Tensor
    top_k: int
    init_blocks: int
    local_blocks: int
    max_partitions: int = 8             # the sparse partition ceiling

    @property
    def sel_stride(self) -> int:
        return self.init_blocks + self.top_k + self.local_blocks

    def selected_tokens(self) -> torch.Tensor:
        """Tokens each request's selection holds, from the lengths alone (the
        count of selected blocks is fixed; with local_blocks >= 1 the tail
        block is one of them)."""
        assert self.local_blocks >= 1
        bs = self.base.block_size
        S = self.base.context_lens.clamp(min=0).to(torch.int64).cpu()
        nb = (S + bs - 1) // bs
        lo = torch.clamp(nb, max=self.init_blocks)
        hi = torch.maximum(lo, nb - self.local_blocks)
        count = lo + (nb - hi) + torch.clamp(hi - lo, max=self.top_k)
        return torch.where(nb > 0, count * bs - (nb * bs - S), torch.zeros_like(S))

    def kv_bytes(self) -> int:
        w = self.base
        return int(self.selected_tokens().sum()) * w.num_kv_heads * w.head_dim * 2 * \
            w.kv_elem_bytes

    def to(self, device) -> "SparseWorkload":
        return SparseWorkload(self.name, self.base.to(device), self.scores.to(device), self.top_k,
                              self.init_blocks, self.local_blocks, self.max_partitions)


def sparse(seed: int = 0, device="cpu") -> SparseWorkload:
    """Sparse top-k decode: 32 decodes, context lognormal(median 4096, sigma 1.5)
    clipped to [64, 131072], Hq/Hkv 32/4, D 128, page 64, fp8 e4m3fn KV (scale
    0.05), bf16 q; per-block scores N(0, 1); the first block, the last block and
    the top 32 blocks between them (at most 34 blocks = 2176 tokens per
    request); partition ceiling 8, budget 2 x 148."""
    lens = lognormal_lengths(32, 4096, 1.5, 64, 131072, seed)
    w = make_batch("sparse", lens, None, 32, 4, 128, 64, "fp8", seed=seed, kv_scale=0.05,
                   device=device, budget=296, max_partitions=8)
    g = _gen(seed + 104729, device)
    scores = torch.randn(tuple(w.block_tables.shape), generator=g, device=device,
                         dtype=torch.float32)
    return SparseWorkload("sparse", w, scores, 32, 1, 1)


SPARSE_CONFIGS = {"sparse": sparse}


def subset(w: Workload, requests: Sequence[int]) -> Workload:
    """The sub-batch of the given requests, with their pages copied into a compact
    pool (same bytes, same page order inside each request).  Every output row of a
    request depends only on that request, so the sub-batch's rows equal the full
    batch's rows for those requests."""
    requests = list(requests)
    bs = w.block_size
    lens = w.context_lens.cpu()
    cu = None if w.cu_query_lens is None else w.cu_query_lens.cpu()
    bt = w.block_tables.cpu()
    new_pages, rows, qlens = [], [], []
    for r in requests:
        p = max(0, -(-int(lens[r]) // bs))
        new_pages.append(bt[r, :p])
        if cu is None:
            rows.append(torch.tensor([r]))
            qlens.append(1)
        else:
            rows.append(torch.arange(int(cu[r]), int(cu[r + 1])))
            qlens.append(int(cu[r + 1] - cu[r]))
    src = torch.cat(new_pages).long() if new_pages else torch.zeros(0, dtype=torch.long)
    k = w.k_cache[src.to(w.k_cache.device)].cpu()
    v = w.v_cache[src.to(w.v_cache.device)].cpu()
    max_blocks = max(1, max(len(p) for p in new_pages))
    nbt = torch.full((len(requests), max_blocks), -1, dtype=torch.int32)
    at = 0
    for i, p in enumerate(new_pages):
        nbt[i, :len(p)] = torch.arange(at, at + len(p), dtype=torch.int32)
        at += len(p)
    q = w.q.cpu()[torch.cat(rows)]
    ncu = None
    if cu is not None:
        ncu = torch.zeros(len(requests) + 1, dtype=torch.int32)
        ncu[1:] = torch.cumsum(torch.tensor(qlens), 0).to(torch.int32)
    return Workload(w.name + "_subset", q, k, v, w.kv_dtype, w.k_scale, w.v_scale, nbt,
                    lens[requests].clone(), ncu, w.scale, w.num_q_heads, w.num_kv_heads,
                    w.head_dim, w.block_size, w.budget, w.max_partitions, dict(w.meta), w.window)
