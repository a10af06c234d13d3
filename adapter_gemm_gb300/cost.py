"""Algorithmic work of the multi-LoRA linear layer, for roofline reporting.

Counts are what the method must do, not what a kernel happens to move:
  layer FLOPs = 2 T d_in d_out + sum over adapter rows of 2 r_s (d_in + d_out)
  layer bytes = 2 (T d_in + d_in d_out + T d_out) + sum over active slots of
                2 r_s (d_in + d_out)          (bf16; true ranks, not R_max)
The correction's share of a square d x d projection at rank r is
r (d_in + d_out) / (d_in d_out) (0.78 % at r = 16, d = 4096: the LoRA-serving
page's intro), and an adapter has r (d_in + d_out) parameters per target
("Adapter size").

Per kernel (the layer runs as plan -> shrink -> GEMM with fused expand):
  GEMM   FLOPs 2 T d_in d_out + sum_rows 2 r d_out;
         bytes 2 (T d_in + d_in d_out + T d_out) + sum_active 2 r d_out
               + sum_rows 4 r (reading the fp32 shrink result)
  shrink bytes sum_rows 2 d_in (x rows on adapters) + sum_active 2 r d_in
               + sum_rows 4 r (writing U) [+ 4 T d_in when it also writes
               the plan-ordered copy of x for the wide GEMM]
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Work:
    flops: float
    bytes: float


def _row_ranks(ids, ranks):
    ids = np.asarray(ids)
    ranks = np.asarray(ranks)
    S = len(ranks)
    ok = (ids > 0) & (ids < S)
    return np.where(ok, ranks[np.clip(ids, 0, S - 1)], 0)


def _active_ranks(ids, ranks):
    ids = np.asarray(ids)
    S = len(ranks)
    act = np.unique(ids[(ids > 0) & (ids < S)])
    return np.asarray(ranks)[act] if act.size else np.zeros(0, dtype=np.int64)


def layer(T: int, d_in: int, d_out: int, ids, ranks) -> Work:
    rr = _row_ranks(ids, ranks).astype(np.float64)
    ar = _active_ranks(ids, ranks).astype(np.float64)
    flops = 2.0 * T * d_in * d_out + float((2.0 * rr * (d_in + d_out)).sum())
    nbytes = 2.0 * (T * d_in + d_in * d_out + T * d_out) + float((2.0 * ar * (d_in + d_out)).sum())
    return Work(flops, nbytes)


def gemm_kernel(T: int, d_in: int, d_out: int, ids=None, ranks=None) -> Work:
    flops = 2.0 * T * d_in * d_out
    nbytes = 2.0 * (T * d_in + d_in * d_out + T * d_out)
    if ids is not None:
        rr = _row_ranks(ids, ranks).astype(np.float64)
        ar = _active_ranks(ids, ranks).astype(np.float64)
        flops += float((2.0 * rr * d_out).sum())
        nbytes += float((2.0 * ar * d_out).sum()) + float((4.0 * rr).sum())
    return Work(flops, nbytes)


def shrink_kernel(T: int, d_in: int, ids, ranks, writes_sorted_x: bool) -> Work:
    rr = _row_ranks(ids, ranks).astype(np.float64)
    ar = _active_ranks(ids, ranks).astype(np.float64)
    n_rows = float((rr > 0).sum())
    flops = float((2.0 * rr * d_in).sum())
    nbytes = 2.0 * n_rows * d_in + float((2.0 * ar * d_in).sum()) + float((4.0 * rr).sum())
    if writes_sorted_x:
        nbytes += 4.0 * T * d_in - 2.0 * n_rows * d_in   # read every row once, write it once
    return Work(flops, nbytes)


def correction_ratio(rank: int, d_in: int, d_out: int) -> float:
    return rank * (d_in + d_out) / (d_in * d_out)


def adapter_params(rank: int, shapes) -> int:
    return sum(rank * (k + n) for k, n in shapes)


def roofline_time(w: Work, peak_tflops: float, peak_gbs: float) -> tuple[float, str]:
    """Lower bound on time (s) and which roof binds."""
    t_c = w.flops / (peak_tflops * 1e12)
    t_m = w.bytes / (peak_gbs * 1e9)
    return (t_c, "tensor") if t_c >= t_m else (t_m, "hbm")


def sliced_layer(T: int, d_in: int, d_outs, ids, ranks_list) -> Work:
    """Projections that share x: each slice's layer, with x read once."""
    ws = [layer(T, d_in, n, ids, r) for n, r in zip(d_outs, ranks_list)]
    return Work(sum(w.flops for w in ws), sum(w.bytes for w in ws) - 2.0 * T * d_in * (len(ws) - 1))


def sliced_gemm_kernel(T: int, d_in: int, d_outs, ids=None, ranks_list=None) -> Work:
    """The GEMM over every slice, with x read once."""
    ws = [gemm_kernel(T, d_in, n, ids, r) for n, r in zip(d_outs, ranks_list or [None] * len(d_outs))]
    return Work(sum(w.flops for w in ws), sum(w.bytes for w in ws) - 2.0 * T * d_in * (len(ws) - 1))
