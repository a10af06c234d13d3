"""CPU oracle for the multi-LoRA linear layer. TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this module. It shares no code with the CUDA path and imports nothing from it.
Everything is computed in float64 from inputs that were widened exactly from
their bf16 bit patterns (a bf16 value is exactly representable in float64).

What it computes, and where the pages define it:

* The layer (Chapter 43, "Many adapters, one base-model batch", the per-row
  equation; "LoRA serving, embeddings, rerankers, pooling", the W' = W + (a/r)BA
  paragraph and its row-vector form; "LoRA adapter application at serve time",
  the conventions table): for token row t with slot s = ids[t],
      y[t, :] = x[t] W^T + (alpha_s / r_s) (x[t] A_s^T) B_s^T,
  with W [d_out, d_in], A_s [r_s, d_in], B_s [d_out, r_s]. Slot 0 is the zero
  adapter (mstar lora.pool module docstring): its rows get the base output and no
  correction at all. alpha_s / r_s uses the adapter's true rank (Chapter 43,
  AdapterBank.load; conventions table "alpha / rank (PEFT convention)").

* Several projections that share x (LoRA serving page, the vLLM section's
  per-slice stacked A and B): each output slice is the layer above with its
  own adapters; the slices' outputs sit side by side.

* The plan (LoRA serving page, "The metadata is a sort and a unique" and the
  worked three-request example; mstar LoraAddressing): a stable sort of token
  rows by slot, the per-slot counts, their exclusive prefix sum (segment start
  offsets), and the list of adapter slots that occur.

Readings where the pages are silent or disagree:
  - the base-only id is slot 0 (the mstar page), not -1 (the vLLM page); an id
    outside [0, S) is invalid, counted, and treated as slot 0;
  - the scale alpha_s / r_s is formed in fp32, as the device stores it, then
    widened; A and B stay unscaled in the pool;
  - a slot with rank 0 adds nothing (the SGLang rank-0 early return).

Parity pins for every function here live in tests/test_oracle.py.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# plan: stable grouping of token rows by slot
# --------------------------------------------------------------------------

def sanitize_ids(ids, S: int):
    """Map invalid slot ids (outside [0, S)) to slot 0 and count them."""
    ids = np.asarray(ids, dtype=np.int64)
    bad = (ids < 0) | (ids >= S)
    return np.where(bad, 0, ids), int(bad.sum())


def plan(ids, S: int, tile_rows: int | None = None) -> dict:
    """The per-step addressing of a batch.

    counts[s]     number of rows on slot s (vLLM's num_tokens_per_lora)
    indptr[s]     exclusive prefix sum of counts, S + 1 entries
                  (vLLM's lora_token_start_loc; mstar's slot_indptr)
    token_order   row ids grouped by slot, slots ascending, rows ascending
                  inside a slot (a stable sort; vLLM's
                  token_indices_sorted_by_lora_ids; mstar's token_order)
    active        slots s >= 1 with counts[s] > 0, ascending
    slot_of_token ids with invalid entries mapped to 0
    n_invalid     how many ids were outside [0, S)
    tiles         if tile_rows is given: (slot, begin, end) over every slot's
                  segment (slot 0 included), cut every tile_rows rows
    """
    slot, n_invalid = sanitize_ids(ids, S)
    T = len(slot)
    counts = np.zeros(S, dtype=np.int64)
    for s in range(S):
        counts[s] = int(np.count_nonzero(slot == s))
    indptr = np.zeros(S + 1, dtype=np.int64)
    for s in range(S):
        indptr[s + 1] = indptr[s] + counts[s]
    token_order = np.zeros(T, dtype=np.int64)
    for s in range(S):
        rows = np.nonzero(slot == s)[0]          # ascending row ids
        token_order[indptr[s]:indptr[s + 1]] = rows
    active = np.array([s for s in range(1, S) if counts[s] > 0], dtype=np.int64)
    out = dict(counts=counts, indptr=indptr, token_order=token_order,
               active=active, slot_of_token=slot, n_invalid=n_invalid)
    if tile_rows is not None:
        tiles = []
        for s in range(S):
            for b in range(int(indptr[s]), int(indptr[s + 1]), tile_rows):
                tiles.append((s, b, min(b + tile_rows, int(indptr[s + 1]))))
        out["tiles"] = np.array(tiles, dtype=np.int64).reshape(-1, 3)
    return out


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------

def slot_scale(alpha, rank) -> float:
    """alpha / r as the fp32 quotient the pool stores, widened to float64."""
    if int(rank) == 0:
        return 0.0
    return float(np.float32(alpha) / np.float32(rank))


def base_linear(x, W, rows=None) -> np.ndarray:
    """x W^T in float64 (the base projection, computed once for all rows)."""
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    if rows is not None:
        x = x[np.asarray(rows)]
    return x @ W.T


def lora_linear(x, W, A, B, rank, alpha, ids, rows=None) -> np.ndarray:
    """The layer in the grouped form: base projection once, then for each
    adapter slot gather its rows, shrink to rank, expand, add, scatter back
    (Chapter 43's grouped PyTorch reference, with the slot-0 convention).

    x [T, d_in]; W [d_out, d_in]; A [S, R_max, d_in]; B [S, d_out, R_max];
    rank [S]; alpha [S]; ids [T]. Returns float64 [len(rows) or T, d_out].
    """
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    S = A.shape[0]
    slot, _ = sanitize_ids(ids, S)
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    y = x[rows] @ W.T
    row_slot = slot[rows]
    for s in range(1, S):
        r = int(rank[s])
        if r == 0:
            continue
        sel = np.nonzero(row_slot == s)[0]
        if sel.size == 0:
            continue
        xs = x[rows[sel]]                      # gathered rows of slot s
        u = xs @ A[s, :r].T                    # shrink: [n, r]
        y[sel] += slot_scale(alpha[s], r) * (u @ B[s, :, :r].T)   # expand + add
    return y


def lora_linear_sliced(x, Ws, As, Bs, ranks, alphas, ids, rows=None) -> np.ndarray:
    """Projections that share x, such as query/key/value or gate/up (LoRA
    serving page, "vLLM: preallocated stacked buffers plus a Punica-style
    Triton kernel": one stacked A and one stacked B per output slice, a shrink
    into [num_slices, num_tokens, rank], an expand over output_slices). Slice i
    is the layer of (x, Ws[i], As[i], Bs[i], ranks[i], alphas[i]) with the
    common ids; the slices' outputs are placed side by side, in slice order.
    Returns float64 [len(rows) or T, sum of the slices' d_out]."""
    return np.concatenate([lora_linear(x, W, A, B, r, a, ids, rows=rows)
                           for W, A, B, r, a in zip(Ws, As, Bs, ranks, alphas)], axis=1)


def lora_linear_rows(x_all, sel, W, A, B, rank, alpha, ids) -> np.ndarray:
    """The layer on selected positions only: the LM head's adapter runs on the
    sampled positions, each mapped to its own adapter (LoRA serving page, the
    worked example's step 6: sampler_indices, one entry per sampled position).
    Row i is the layer of x_all[sel[i]] (a zero row when sel[i] is outside
    [0, T_all)) with slot ids[i]."""
    x_all = np.asarray(x_all, dtype=np.float64)
    sel = np.asarray(sel)
    ok = (sel >= 0) & (sel < x_all.shape[0])
    x = np.zeros((len(sel), x_all.shape[1]))
    x[ok] = x_all[sel[ok]]
    return lora_linear(x, W, A, B, rank, alpha, ids)


def lora_linear_indexed(x, W, A, B, rank, alpha, ids) -> np.ndarray:
    """The same layer row by row, in the indexed (BGMV-like) form: each row
    looks up its own slot. Slow; for small cases only."""
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    S = A.shape[0]
    T = x.shape[0]
    y = np.zeros((T, W.shape[0]), dtype=np.float64)
    for t in range(T):
        s = int(ids[t])
        y[t] = W @ x[t]
        if 1 <= s < S and int(rank[s]) > 0:
            r = int(rank[s])
            u = A[s, :r] @ x[t]
            y[t] += slot_scale(alpha[s], r) * (B[s, :, :r] @ u)
    return y


def merged_weight(W, A_s, B_s, sc) -> np.ndarray:
    """W' = W + sc * B_s A_s (the merged adapter, in float64)."""
    return np.asarray(W, np.float64) + sc * (np.asarray(B_s, np.float64) @ np.asarray(A_s, np.float64))


# --------------------------------------------------------------------------
# operation counts of the layer as the oracle evaluates it
# --------------------------------------------------------------------------

def correction_macs_per_row(rank: int, d_in: int, d_out: int) -> int:
    """Multiply-adds of one row's correction: shrink r*d_in, expand d_out*r."""
    return rank * d_in + d_out * rank


def base_macs_per_row(d_in: int, d_out: int) -> int:
    return d_in * d_out


def correction_flop_ratio(rank: int, d_in: int, d_out: int) -> float:
    """Correction FLOPs over base FLOPs for one adapted row."""
    return correction_macs_per_row(rank, d_in, d_out) / base_macs_per_row(d_in, d_out)


def adapter_params(rank: int, shapes) -> int:
    """Parameters of one adapter over (d_in, d_out) targets: r (d_in + d_out) each."""
    return sum(rank * (k + n) for k, n in shapes)
