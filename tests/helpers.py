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


# ------------------------------------------------------------ parity bounds
#
# Absolute bound (the stated target): max |gpu - oracle| over every output
# element, 1e-2 with 16-bit caches and 3e-2 with fp8-e4m3 caches.
TOL = {"bf16": 1e-2, "fp16": 1e-2, "fp8": 3e-2}
# Relative bounds, which still discriminate where the outputs are small (long,
# flat softmaxes give output rows of standard deviation ~1/sqrt(S)).  From the
# arithmetic of the path: the output is rounded once to bf16 (unit roundoff
# u = 2^-8; fp16 2^-11) and the probabilities enter the P.V products rounded to
# bf16 (16-bit caches) or fp16 (fp8 caches); every other step is fp32 with
# errors near 2^-24.  Both roundings are unbiased, so the relative error of a
# row is about sqrt(2) u / sqrt(3) ~ 3e-3 RMS and at most ~2u per element;
# the bounds leave about 3x on each.
REL_NORM = 1e-2  # ||gpu - oracle|| / ||oracle||, whole output and every row
REL_MAX = 2e-2   # max |gpu - oracle| / max |oracle|


def parity(out, ref: np.ndarray, kv_dtype=None, what: str = "") -> dict:
    """Checks one output against the oracle: finite, max-abs within TOL (unless
    kv_dtype is None: the caller checks it), the
    relative bounds over the whole output and over every row (the first
    dimension: a query row, all its heads and dims), and rows whose oracle
    result is zero (padding, empty requests, no visible key) exactly zero.
    Returns the measured errors."""
    got = out.float().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if ref.size == 0:
        return {"max_abs": 0.0, "rel_norm": 0.0, "rel_max": 0.0, "row_rel": 0.0}
    d = got.astype(np.float64) - ref
    max_abs = float(np.abs(d).max())
    ref_norm = float(np.sqrt((ref * ref).sum()))
    rel_norm = float(np.sqrt((d * d).sum()) / ref_norm) if ref_norm > 0 else 0.0
    ref_max = float(np.abs(ref).max())
    rel_max = max_abs / ref_max if ref_max > 0 else 0.0
    rows_ref = np.sqrt((ref.reshape(ref.shape[0], -1) ** 2).sum(axis=1))
    rows_d = np.sqrt((d.reshape(d.shape[0], -1) ** 2).sum(axis=1))
    zero = rows_ref == 0
    assert np.all(rows_d[zero] == 0), f"{what}: rows {np.nonzero(zero & (rows_d > 0))[0][:8]} " \
                                      "must be exactly zero"
    row_rel = float((rows_d[~zero] / rows_ref[~zero]).max()) if np.any(~zero) else 0.0
    e = {"max_abs": max_abs, "rel_norm": rel_norm, "rel_max": rel_max, "row_rel": row_rel}
    if kv_dtype is not None:
        assert max_abs <= TOL[kv_dtype], (what, e)
    if ref_max > 0:
        assert rel_norm <= REL_NORM and rel_max <= REL_MAX, (what, e)
        assert row_rel <= REL_NORM, (what, e)
    return e
