"""Sparse top-k decode on the GPU: the selection kernel (pa_sparse_select)
bit-exact against the oracle's selection, and selection + plan refresh +
decode against the oracle's sparse decode, element by element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import kv_bits, bits16, q_code, DT_CODE, parity
from paged_kv_decode_split_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _select_both(scores, lens, bt, bs, top_k, init, local, stride=None):
    sel, sl = binding.sparse_select(scores, lens, bt, bs, top_k, init, local,
                                    sel_block_tables=None if stride is None else torch.empty(
                                        (bt.shape[0], stride), dtype=torch.int32,
                                        device=bt.device))
    torch.cuda.synchronize()
    osel, osl = oracle.sparse_select(None if scores is None else scores.cpu().numpy(),
                                     lens.cpu().numpy(), bt.cpu().numpy(), bs, top_k, init,
                                     local, sel.shape[1])
    return sel.cpu().numpy(), sl.cpu().numpy(), osel, osl


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("top_k,init,local", [(0, 1, 1), (1, 0, 0), (7, 1, 1), (32, 2, 3),
                                              (300, 0, 1), (5000, 1, 1)])
def test_select_bit_exact(dev, seed, top_k, init, local):
    """Random scores drawn from a small palette (many ties, +-0, +-inf, NaN),
    lengths from 0 to the table width, block tables with random physical ids."""
    rng = np.random.default_rng(seed)
    n, bs, max_blocks = 64, 16, 700
    palette = np.array([0.5, -1.0, 3.0, 0.0, -0.0, np.inf, -np.inf, np.nan, 1e-30, -1e30],
                       np.float32)
    scores = palette[rng.integers(0, len(palette), (n, max_blocks + 3))]
    scores[: n // 2] = rng.normal(size=(n // 2, max_blocks + 3)).astype(np.float32)
    lens = rng.integers(0, max_blocks * bs + 1, n).astype(np.int32)
    lens[:4] = [0, 1, bs, bs + 1]
    bt = rng.integers(0, 1 << 20, (n, max_blocks)).astype(np.int32)
    t = lambda a: torch.from_numpy(a).to(dev)
    sel, sl, osel, osl = _select_both(t(scores) if top_k else None, t(lens), t(bt), bs, top_k,
                                      init, local)
    assert np.array_equal(sel, osel)
    assert np.array_equal(sl, osl)


def test_select_wider_rows_are_padded(dev):
    rng = np.random.default_rng(9)
    scores = torch.from_numpy(rng.normal(size=(5, 40)).astype(np.float32)).to(dev)
    lens = torch.tensor([0, 100, 300, 600, 640], dtype=torch.int32, device=dev)
    bt = torch.arange(5 * 40, dtype=torch.int32, device=dev).reshape(5, 40)
    sel, sl, osel, osl = _select_both(scores, lens, bt, 16, 4, 1, 1, stride=50)
    assert np.array_equal(sel, osel) and np.array_equal(sl, osl)
    assert (sel[:, 6:] == -1).all()


def test_select_too_long_request_is_reported(dev):
    scores = torch.zeros((2, 8), dtype=torch.float32, device=dev)
    lens = torch.tensor([100, 8 * 16 + 5], dtype=torch.int32, device=dev)  # r1 needs 9 blocks
    bt = torch.arange(16, dtype=torch.int32, device=dev).reshape(2, 8)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sel, sl = binding.sparse_select(scores, lens, bt, 16, 2, 1, 1, device_errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.DEVERR_BAD_PAGE
    osel, osl = oracle.sparse_select(scores.cpu().numpy(), lens.cpu().numpy(), bt.cpu().numpy(),
                                     16, 2, 1, 1)
    assert np.array_equal(sel.cpu().numpy(), osel) and np.array_equal(sl.cpu().numpy(), osl)


def test_select_rejects_bad_arguments(dev):
    lens = torch.ones(2, dtype=torch.int32, device=dev)
    bt = torch.zeros((2, 4), dtype=torch.int32, device=dev)
    with pytest.raises(binding.PaError):  # top_k > 0 without scores
        binding.sparse_select(None, lens, bt, 16, 2, 1, 1)
    with pytest.raises(binding.PaError):  # rows narrower than init + top_k + local
        binding.sparse_select(torch.zeros((2, 4), device=dev), lens, bt, 16, 2, 1, 1,
                              sel_block_tables=torch.empty((2, 3), dtype=torch.int32,
                                                           device=dev))
    with pytest.raises(binding.PaError):  # score rows shorter than the block table
        binding.sparse_select(torch.zeros((2, 3), device=dev), lens, bt, 16, 2, 1, 1)


# ------------------------------------------------------------- sparse decode

def _oracle_sparse(sw):
    w = sw.base.to("cpu")
    return oracle.sparse_decode(bits16(w.q), q_code(w), kv_bits(w.k_cache, w.kv_dtype),
                                kv_bits(w.v_cache, w.kv_dtype), DT_CODE[w.kv_dtype], w.k_scale,
                                w.v_scale, w.block_tables.numpy(), w.context_lens.numpy(),
                                w.scale, sw.scores.cpu().numpy(), w.block_size, sw.top_k,
                                sw.init_blocks, sw.local_blocks)


def _run_sparse(sw, kind=binding.PROPORTIONAL, grouped=False):
    w = sw.base
    plan = binding.Plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                        max_partitions=sw.max_partitions, budget=w.budget or 0, kind=kind,
                        device=w.q.device)
    sel, sl = binding.sparse_select(sw.scores, w.context_lens, w.block_tables, w.block_size,
                                    sw.top_k, sw.init_blocks, sw.local_blocks)
    plan.refresh(sl)
    k = wl.with_k_groups(w).k_cache if grouped else w.k_cache
    out = plan.decode(w.q, k, w.v_cache, sel, sl, None, w.scale, w.k_scale, w.v_scale)
    torch.cuda.synchronize()
    return out, plan, sel, sl


def _small(dev, kv="bf16", bs=16, seed=0, top_k=5, init=1, local=2, D=128):
    lens = [1, 16, 17, 200, 777, 1500, 3000, 0]
    w = wl.make_batch("sparse_small", lens, None, 8, 2, D, bs, kv, "fp16" if kv == "fp16" else
                      "bf16", seed=seed, kv_scale=0.05, device=dev, max_partitions=8)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 1)
    scores = torch.randn(tuple(w.block_tables.shape), generator=g, device=dev)
    return wl.SparseWorkload("sparse_small", w, scores, top_k, init, local)


@pytest.mark.parametrize("kv,bs,D", [("bf16", 16, 128), ("fp8", 64, 128), ("fp16", 128, 64),
                                      ("bf16", 16, 512)])
@pytest.mark.parametrize("top_k,init,local", [(5, 1, 2), (0, 1, 1), (64, 0, 1)])
def test_sparse_decode_parity(dev, kv, bs, D, top_k, init, local):
    sw = _small(dev, kv, bs, seed=bs + top_k, top_k=top_k, init=init, local=local, D=D)
    out, plan, _, sl = _run_sparse(sw)
    ref = _oracle_sparse(sw)
    parity(out, ref, kv)
    assert plan.read_errors() == 0
    assert torch.all(out[sw.base.context_lens == 0] == 0)


def test_sparse_decode_grouped_k_and_uniform_plan(dev):
    sw = _small(dev, "fp8", 16, seed=5)
    ref = _oracle_sparse(sw)
    for kind, grouped in ((binding.UNIFORM, False), (binding.PROPORTIONAL, True)):
        out, plan, _, _ = _run_sparse(sw, kind=kind, grouped=grouped)
        parity(out, ref, "fp8", what=f"kind {kind} grouped {grouped}")


def test_sparse_full_size(dev):
    """The sparse benchmark batch at full size, every output element."""
    sw = wl.sparse(0, dev)
    out, plan, sel, sl = _run_sparse(sw)
    assert np.array_equal(sl.cpu().numpy(), sw.selected_tokens().numpy().astype(np.int32))
    ref = _oracle_sparse(sw)
    parity(out, ref, "fp8")
    assert plan.read_errors() == 0
    work, red = plan.download()
    assert int(red[:, 1].max()) <= 8  # the sparse partition ceiling


def test_sparse_step_in_a_cuda_graph(dev):
    """Selection, refresh and decode captured once and replayed after the
    scores and lengths change in place (one refresh per step, inside the
    graph)."""
    sw = _small(dev, "bf16", 16, seed=11)
    w = sw.base
    plan = binding.Plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                        max_partitions=8, device=dev)
    sel = torch.empty((w.num_seqs, sw.sel_stride), dtype=torch.int32, device=dev)
    sl = torch.empty(w.num_seqs, dtype=torch.int32, device=dev)
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def step():
        binding.sparse_select(sw.scores, w.context_lens, w.block_tables, w.block_size, sw.top_k,
                              sw.init_blocks, sw.local_blocks, sel, sl, stream=s)
        plan.refresh(sl, stream=s)
        plan.decode(w.q, w.k_cache, w.v_cache, sel, sl, None, w.scale, out=out, stream=s)

    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for trial in range(2):
        sw.scores.copy_(torch.randn(sw.scores.shape, device=dev))
        w.context_lens.copy_(torch.clamp(w.context_lens - 3 * trial, min=0))
        g.replay()
        torch.cuda.synchronize()
        ref = _oracle_sparse(sw)
        parity(out, ref, "bf16", what=f"trial {trial}")
    assert plan.read_errors() == 0
