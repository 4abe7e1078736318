"""Shared test helpers: turn a Workload into the oracle's raw-bit inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

DT_CODE = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp8": oracle.FP8_E4M3}


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def kv_bits(t: torch.Tensor, kv_dtype: str) -> np.ndarray:
    if kv_dtype == "fp8":
        return t.detach().cpu().contiguous().view(torch.uint8).numpy()
    return bits16(t)


def q_code(w) -> int:
    return oracle.FP16 if w.q.dtype == torch.float16 else oracle.BF16


def oracle_args(w):
    cu = None if w.cu_query_lens is None else w.cu_query_lens.cpu().numpy()
    return (bits16(w.q), q_code(w), kv_bits(w.k_cache, w.kv_dtype), kv_bits(w.v_cache, w.kv_dtype),
            DT_CODE[w.kv_dtype], w.k_scale, w.v_scale, w.block_tables.cpu().numpy(),
            w.context_lens.cpu().numpy(), cu, w.scale)


def oracle_decode(w, window: int = 0, sinks=None) -> np.ndarray:
    return oracle.decode(*oracle_args(w), window=window, sinks=sinks)


def oracle_decode_planned(w, work, red, window: int = 0, sinks=None) -> np.ndarray:
    return oracle.decode_planned(*oracle_args(w), work, red, window=window, sinks=sinks)


def oracle_plan(w, budget: int, kind: int = oracle.PLAN_PROPORTIONAL, max_partitions=None,
                window: int = 0):
    cu = None if w.cu_query_lens is None else w.cu_query_lens.cpu().numpy()
    return oracle.plan(w.context_lens.cpu().numpy(), cu, w.num_kv_heads,
                       w.max_partitions if max_partitions is None else max_partitions,
                       budget, kind, window=window)
