"""Seeded synthetic workloads for the multi-LoRA linear layer.

This module only draws inputs: token slot ids, activations, base weights and
adapter factors, rounded to bf16. It holds none of the layer's arithmetic, so
both the CPU oracle (through the tests) and the CUDA path can consume it.

Shapes and value distributions follow the pages' setting: Llama-3-8B-shaped
projections (d = 4096, d_kv = 1024, FFN 14336; "LoRA serving, embeddings,
rerankers, pooling", symbols paragraph), rank-16 adapters with alpha = 32,
x ~ N(0, 1), W, A, B ~ N(0, 0.02) drawn in fp32 and rounded to bf16 (round to
nearest even). Slot 0 is the zero adapter; it is never given weights.

Workloads:
  tiny          T=64,  256->256,     slots 1-3 rank 8, alpha 16, ids uniform {0..3}
  q_decode      T=64,  4096->4096,   8 adapters r16, 8 contiguous rows each
  qkv_decode    q_decode's batch over the q/k/v projections (4096 -> 4096 +
                1024 + 1024) as one call over three output slices
  lm_head_prefill  64 sequences x 64 tokens; the LM head (4096 -> 128256) on
                each sequence's last position, 8 adapters r16
  skewed_prefill  T=4096, 4096->4096, 90 % of rows on one adapter, 5 % on
                slot 0, the rest over 15 adapters r16
  gateup_prefill T=4096, 4096->14336, 16 adapters r16, power-law (1.1) segment
                lengths by largest remainder, 10 % of rows on slot 0, contiguous
                segments in a seeded order
  mixed_down    T=256, 14336->4096,  31 adapters, ranks from {8,16,64}, ids
                i.i.d.: 25 % slot 0, else truncated power law (1.2), interleaved
  layer_sweep   the seven Llama-3-8B targets, 50 resident adapters r16 per
                target, T in {1,8,64,512,4096}, ids i.i.d.: 10 % slot 0 else
                uniform over 1..50; layer_sweep_sliced runs q/k/v and gate/up
                as one call each
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# Llama-3-8B decoder-layer projections (in, out), the seven usual targets.
LLAMA3_8B_TARGETS = (
    ("q_proj", 4096, 4096),
    ("k_proj", 4096, 1024),
    ("v_proj", 4096, 1024),
    ("o_proj", 4096, 4096),
    ("gate_proj", 4096, 14336),
    ("up_proj", 4096, 14336),
    ("down_proj", 14336, 4096),
)

SWEEP_T = (1, 8, 64, 512, 4096)


@dataclass
class Target:
    """One adapted linear: base weight plus its slot pool (host bf16 tensors)."""
    name: str
    d_in: int
    d_out: int
    W: torch.Tensor            # [d_out, d_in] bf16
    A: torch.Tensor            # [S, R_max, d_in] bf16, zero past each slot's rank
    B: torch.Tensor            # [S, d_out, R_max] bf16, zero past each slot's rank
    rank: np.ndarray           # [S] int32, rank[0] = 0
    alpha: np.ndarray          # [S] float32, alpha[0] = 0
    x_in: torch.Tensor | None = None   # own input when d_in differs from the step's x


@dataclass
class Workload:
    name: str
    T: int
    S: int
    R_max: int
    ids: np.ndarray            # [T] int32 token slot ids
    x: torch.Tensor            # [T, d_in] bf16 (d_in of the first target)
    targets: list = field(default_factory=list)
    # targets that share their input and run as one call over output slices
    # (tuples of target indices); every other target runs on its own
    groups: list = field(default_factory=list)
    # the layer runs on these rows of x only (the LM head's sampled positions);
    # T and ids then count the selected rows
    sel: np.ndarray | None = None

    def units(self) -> list:
        """The calls of one step, in target order: tuples of target indices."""
        grouped = {i: g for g in self.groups for i in g}
        out, seen = [], set()
        for i in range(len(self.targets)):
            if i in seen:
                continue
            g = tuple(grouped.get(i, (i,)))
            seen.update(g)
            out.append(g)
        return out

    @property
    def d_in(self) -> int:
        return self.targets[0].d_in

    @property
    def d_out(self) -> int:
        return self.targets[0].d_out


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 array -> bf16 tensor, round to nearest even (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def make_target(rng: np.random.Generator, name: str, d_in: int, d_out: int,
                ranks, alphas, R_max: int) -> Target:
    """Draw W and a slot pool. Slot s >= 1 gets A_s [r_s, d_in], B_s [d_out, r_s]
    in the leading rows/columns of its padded block; padding stays zero."""
    S = len(ranks)
    W = to_bf16(_normal(rng, (d_out, d_in), 0.02))
    A = torch.zeros((S, R_max, d_in), dtype=torch.bfloat16)
    B = torch.zeros((S, d_out, R_max), dtype=torch.bfloat16)
    for s in range(1, S):
        r = int(ranks[s])
        if r == 0:
            continue
        A[s, :r] = to_bf16(_normal(rng, (r, d_in), 0.02))
        B[s, :, :r] = to_bf16(_normal(rng, (d_out, r), 0.02))
    return Target(name, d_in, d_out, W, A, B,
                  np.asarray(ranks, dtype=np.int32), np.asarray(alphas, dtype=np.float32))


def largest_remainder(total: int, weights: np.ndarray) -> np.ndarray:
    """Integer split of `total` proportional to `weights`, every share >= 1."""
    w = np.asarray(weights, dtype=np.float64)
    quota = total * w / w.sum()
    base = np.maximum(np.floor(quota).astype(np.int64), 1)
    left = total - int(base.sum())
    order = np.argsort(-(quota - np.floor(quota)), kind="stable")
    i = 0
    while left > 0:
        base[order[i % len(order)]] += 1
        left -= 1
        i += 1
    while left < 0:                       # only if the >=1 floor overshot
        j = int(np.argmax(base))
        base[j] -= 1
        left += 1
    return base


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def tiny(seed: int = 1001) -> Workload:
    T, K, N, S, r = 64, 256, 256, 4, 8
    g_ids, g_x, g_w = _streams(seed, 3)
    ids = g_ids.integers(0, S, size=T).astype(np.int32)
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    ranks = [0] + [r] * (S - 1)
    alphas = [0.0] + [16.0] * (S - 1)
    t = make_target(g_w, "proj", K, N, ranks, alphas, r)
    return Workload("tiny", T, S, r, ids, x, [t])


def q_decode(seed: int = 1002) -> Workload:
    T, K, N, S, r = 64, 4096, 4096, 9, 16
    _, g_x, g_w = _streams(seed, 3)
    ids = np.repeat(np.arange(1, S, dtype=np.int32), T // (S - 1))
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    t = make_target(g_w, "q_proj", K, N, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
    return Workload("q_decode", T, S, r, ids, x, [t])


def qkv_decode(seed: int = 1005) -> Workload:
    """The query, key and value projections of one decode step as one call over
    three output slices (4096 + 1024 + 1024), with q_decode's batch: T=64, 8
    adapters of rank 16, 8 contiguous rows each; each slice has its own
    adapter factors."""
    T, K, S, r = 64, 4096, 9, 16
    streams = _streams(seed, 5)
    g_x = streams[1]
    ids = np.repeat(np.arange(1, S, dtype=np.int32), T // (S - 1))
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    tl = [make_target(g, name, K, n, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
          for (name, _, n), g in zip(LLAMA3_8B_TARGETS[:3], streams[2:])]
    return Workload("qkv_decode", T, S, r, ids, x, tl, groups=[(0, 1, 2)])


def skewed_prefill(seed: int = 1007) -> Workload:
    """A skewed load: T=4096 rows of a 4096 -> 4096 projection, 90 % of the
    rows on one adapter, 5 % on slot 0, the rest spread over 15 more adapters
    (rank 16), rows shuffled."""
    T, K, N, S, r = 4096, 4096, 4096, 17, 16
    g_ids, g_x, g_w = _streams(seed, 3)
    n_hot, n_base = int(0.9 * T), int(0.05 * T)
    ids = np.concatenate([np.full(n_hot, 1, np.int32), np.zeros(n_base, np.int32),
                          g_ids.integers(2, S, size=T - n_hot - n_base).astype(np.int32)])
    ids = ids[g_ids.permutation(T)].astype(np.int32)
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    t = make_target(g_w, "o_proj", K, N, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
    return Workload("skewed_prefill", T, S, r, ids, x, [t])


def lm_head_prefill(seed: int = 1006) -> Workload:
    """The LM head's adapter on a prefill batch: 64 sequences of 64 tokens
    (x [4096, 4096]); the head runs on each sequence's last position only (64
    selected rows), into the 128256-entry vocabulary of Llama 3. Eight adapters
    of rank 16, eight sequences each."""
    n_seq, L_seq, K, N, S, r = 64, 64, 4096, 128256, 9, 16
    g_x, g_w = _streams(seed, 2)
    x = to_bf16(_normal(g_x, (n_seq * L_seq, K), 1.0))
    sel = (np.arange(n_seq, dtype=np.int32) + 1) * L_seq - 1
    ids = np.repeat(np.arange(1, S, dtype=np.int32), n_seq // (S - 1))
    t = make_target(g_w, "lm_head", K, N, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
    return Workload("lm_head_prefill", n_seq, S, r, ids, x, [t], sel=sel)


def gateup_ids(rng: np.random.Generator, T: int = 4096, n_adapters: int = 16,
               base_frac: float = 0.1, power: float = 1.1) -> np.ndarray:
    n0 = int(round(base_frac * T))
    weights = np.arange(1, n_adapters + 1, dtype=np.float64) ** (-power)
    lengths = largest_remainder(T - n0, weights)
    slot_of_rank = rng.permutation(n_adapters) + 1       # weight rank -> slot
    segs = [(0, n0)] + [(int(slot_of_rank[i]), int(lengths[i])) for i in range(n_adapters)]
    order = rng.permutation(len(segs))
    return np.concatenate([np.full(segs[i][1], segs[i][0], dtype=np.int32) for i in order])


def gateup_prefill(seed: int = 1003) -> Workload:
    T, K, N, S, r = 4096, 4096, 14336, 17, 16
    g_ids, g_x, g_w = _streams(seed, 3)
    ids = gateup_ids(g_ids, T, S - 1)
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    t = make_target(g_w, "gate_proj", K, N, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
    return Workload("gateup_prefill", T, S, r, ids, x, [t])


def mixed_down(seed: int = 1004) -> Workload:
    T, K, N, S, R = 256, 14336, 4096, 32, 64
    g_ids, g_x, g_w, g_r = _streams(seed, 4)
    ranks = [0] + [int(v) for v in g_r.choice(np.array([8, 16, 64]), size=S - 1)]
    p = np.arange(1, S, dtype=np.float64) ** (-1.2)
    p /= p.sum()
    base = g_ids.random(T) < 0.25
    pick = g_ids.choice(np.arange(1, S), size=T, p=p)
    ids = np.where(base, 0, pick).astype(np.int32)
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    t = make_target(g_w, "down_proj", K, N, ranks, [0.0] + [32.0] * (S - 1), R)
    return Workload("mixed_down", T, S, R, ids, x, [t])


def sweep_ids(rng: np.random.Generator, T: int, n_adapters: int = 50,
              base_frac: float = 0.1) -> np.ndarray:
    base = rng.random(T) < base_frac
    pick = rng.integers(1, n_adapters + 1, size=T)
    return np.where(base, 0, pick).astype(np.int32)


def layer_sweep(T: int, seed: int | None = None, targets=LLAMA3_8B_TARGETS, sliced: bool = False) -> Workload:
    """All seven targets of one decoder layer share the step's ids. x is drawn
    for d_in = 4096; the down projection gets its own [T, 14336] input, stored
    on that target as `x_in` (use `input_for`). With `sliced`, q/k/v and
    gate/up run as one call each over their output slices."""
    seed = 5000 + T if seed is None else seed
    S, r = 51, 16
    streams = _streams(seed, 3 + len(targets))
    g_ids, g_x, g_x2 = streams[:3]
    ids = sweep_ids(g_ids, T, S - 1)
    x = to_bf16(_normal(g_x, (T, 4096), 1.0))
    x_ffn = None
    tl = []
    for (name, k, n), g in zip(targets, streams[3:]):
        t = make_target(g, name, k, n, [0] + [r] * (S - 1), [0.0] + [32.0] * (S - 1), r)
        if k != 4096:
            if x_ffn is None:
                x_ffn = to_bf16(_normal(g_x2, (T, k), 1.0))
            t.x_in = x_ffn
        tl.append(t)
    if sliced:
        return Workload(f"layer_sweep_sliced_T{T}", T, S, r, ids, x, tl, groups=[(0, 1, 2), (4, 5)])
    return Workload(f"layer_sweep_T{T}", T, S, r, ids, x, tl)


def input_for(w: Workload, t: Target) -> torch.Tensor:
    return t.x_in if t.x_in is not None else w.x


def rows_input(w: Workload, t: Target) -> torch.Tensor:
    """The rows the layer sees: the target's input, or its selected rows."""
    x = input_for(w, t)
    return x if w.sel is None else x[torch.from_numpy(w.sel.astype(np.int64))]


def by_name(name: str) -> Workload:
    if name == "tiny":
        return tiny()
    if name == "q_decode":
        return q_decode()
    if name == "gateup_prefill":
        return gateup_prefill()
    if name == "mixed_down":
        return mixed_down()
    if name == "qkv_decode":
        return qkv_decode()
    if name == "lm_head_prefill":
        return lm_head_prefill()
    if name == "skewed_prefill":
        return skewed_prefill()
    if name.startswith("layer_sweep_sliced_T"):
        return layer_sweep(int(name[len("layer_sweep_sliced_T"):]), sliced=True)
    if name.startswith("layer_sweep_T"):
        return layer_sweep(int(name[len("layer_sweep_T"):]))
    raise KeyError(name)


def random_case(seed: int, T: int, K: int, N: int, S: int, R_max: int,
                ranks=None, alpha: float = 32.0, base_frac: float = 0.2,
                sorted_ids: bool = False) -> Workload:
    """A generic seeded case for parity sweeps (ragged sizes, odd ranks)."""
    g_ids, g_x, g_w, g_r = _streams(seed, 4)
    if ranks is None:
        ranks = [0] + [int(v) for v in g_r.integers(1, R_max + 1, size=S - 1)]
    base = g_ids.random(T) < base_frac
    pick = g_ids.integers(1, S, size=T) if S > 1 else np.zeros(T, dtype=np.int64)
    ids = np.where(base, 0, pick).astype(np.int32)
    if sorted_ids:
        ids = np.sort(ids).astype(np.int32)
    x = to_bf16(_normal(g_x, (T, K), 1.0))
    t = make_target(g_w, "proj", K, N, ranks, [0.0] + [alpha] * (S - 1), R_max)
    return Workload(f"case{seed}", T, S, R_max, ids, x, [t])
