"""Pins of the CPU oracle against facts the pages and the mathematics fix.

None of these compare the oracle with itself: the plan is pinned to the pages'
worked example and to Python's stable sort; the layer to the merged-weight
identity, to exact integer arithmetic, to the slot-0 rule and to the grouped vs
indexed forms; the counters to the pages' printed arithmetic.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import lora_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- plan ----

def test_plan_worked_example():
    """LoRA serving page, three-request worked example: counts [3, 5, 4],
    start offsets [0, 3, 8, 12], sorted order [9,10,11, 0..4, 5..8]."""
    g = json.load(open(os.path.join(GOLDEN, "plan_worked_example.json")))
    p = O.plan(g["ids"], g["S"])
    assert p["counts"].tolist() == g["counts"]
    assert p["indptr"].tolist() == g["indptr"]
    assert p["token_order"].tolist() == g["token_order"]
    assert p["active"].tolist() == g["active"]
    assert p["n_invalid"] == 0


@pytest.mark.parametrize("S", [1, 2, 3])
def test_plan_bruteforce_vs_stable_sort(S):
    """Every id vector (with out-of-range ids) up to T = 5 against Python's
    stable sorted() and collections counting."""
    alphabet = list(range(-1, S + 1))          # -1 and S are invalid
    for T in range(0, 6 if S < 3 else 5):
        for ids in itertools.product(alphabet, repeat=T):
            key = [i if 0 <= i < S else 0 for i in ids]
            p = O.plan(list(ids), S, tile_rows=2)
            order = sorted(range(T), key=lambda t: key[t])      # stable
            assert p["token_order"].tolist() == order
            counts = [key.count(s) for s in range(S)]
            assert p["counts"].tolist() == counts
            assert p["indptr"].tolist() == [sum(counts[:s]) for s in range(S + 1)]
            assert p["active"].tolist() == [s for s in range(1, S) if counts[s]]
            assert p["n_invalid"] == sum(1 for i in ids if not 0 <= i < S)
            # tiles: cover each segment exactly once, in order, at most 2 rows
            cover = []
            for s, b, e in p["tiles"].tolist():
                assert 0 < e - b <= 2
                assert all(key[order[i]] == s for i in range(b, e))
                cover.extend(range(b, e))
            assert cover == list(range(T))


def test_plan_empty():
    p = O.plan([], 4)
    assert p["counts"].tolist() == [0, 0, 0, 0]
    assert p["indptr"].tolist() == [0, 0, 0, 0, 0]
    assert p["token_order"].tolist() == [] and p["active"].tolist() == []


# ---------------------------------------------------------------- layer ----

def _case(seed, T, K, N, S, R, ranks=None, alpha=None):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((N, K))
    A = np.zeros((S, R, K))
    B = np.zeros((S, N, R))
    ranks = ranks if ranks is not None else [0] + list(rng.integers(1, R + 1, size=S - 1))
    for s in range(1, S):
        A[s, :ranks[s]] = rng.standard_normal((ranks[s], K))
        B[s, :, :ranks[s]] = rng.standard_normal((N, ranks[s]))
    alpha = alpha if alpha is not None else [0.0] + [float(a) for a in rng.integers(1, 64, size=S - 1)]
    ids = rng.integers(-1, S + 1, size=T)      # includes invalid ids
    return x, W, A, B, np.array(ranks), np.array(alpha, dtype=np.float32), ids


def test_merged_identity_page_case():
    """LoRA serving page, "the row-vector formula must agree with merging the
    stored [out, in] weight": seed 5, x 3x4, W 6x4, A 2x4, B 6x2, scale 0.5,
    merged and unmerged agree to 1e-12."""
    rng = np.random.default_rng(5)
    x = rng.normal(size=(3, 4))
    w = rng.normal(size=(6, 4))
    a = rng.normal(size=(2, 4))
    b = rng.normal(size=(6, 2))
    A = np.zeros((2, 2, 4)); A[1] = a
    B = np.zeros((2, 6, 2)); B[1] = b
    # scale 0.5 = alpha / rank with rank 2, alpha 1
    y = O.lora_linear(x, w, A, B, [0, 2], [0.0, 1.0], [1, 1, 1])
    merged = x @ O.merged_weight(w, a, b, 0.5).T
    np.testing.assert_allclose(y, merged, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merged_identity_per_row(seed):
    """Each row equals x_t (W + sc_s B_s A_s)^T for its own slot (conventions
    table: delta W' = W + (B @ A) * (alpha / rank))."""
    x, W, A, B, rank, alpha, ids = _case(seed, 11, 9, 7, 5, 4)
    y = O.lora_linear(x, W, A, B, rank, alpha, ids)
    for t in range(len(ids)):
        s = int(ids[t])
        if 1 <= s < 5:
            r = rank[s]
            Wm = O.merged_weight(W, A[s, :r], B[s, :, :r], float(np.float32(alpha[s]) / np.float32(r)))
        else:
            Wm = W
        ref = Wm @ x[t]
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-12)


def test_slot0_rows_equal_base_exactly():
    """Slot 0 is the zero adapter: its rows are the base output, bit for bit."""
    x, W, A, B, rank, alpha, ids = _case(3, 40, 32, 24, 6, 8)
    y = O.lora_linear(x, W, A, B, rank, alpha, ids)
    base = O.base_linear(x, W)
    slot0 = (ids == 0) | (ids < 0) | (ids >= 6)
    assert slot0.any()
    assert np.array_equal(y[slot0], base[slot0])
    assert not np.allclose(y[~slot0], base[~slot0])


def test_grouped_equals_indexed():
    for seed in range(4):
        x, W, A, B, rank, alpha, ids = _case(10 + seed, 23, 19, 13, 6, 5)
        g = O.lora_linear(x, W, A, B, rank, alpha, ids)
        i = O.lora_linear_indexed(x, W, A, B, rank, alpha, ids)
        np.testing.assert_allclose(g, i, rtol=1e-12, atol=1e-12)


def test_rows_subset_matches_full():
    x, W, A, B, rank, alpha, ids = _case(7, 30, 16, 12, 4, 3)
    full = O.lora_linear(x, W, A, B, rank, alpha, ids)
    rows = [29, 0, 5, 5, 17]
    np.testing.assert_array_equal(O.lora_linear(x, W, A, B, rank, alpha, ids, rows=rows), full[rows])


def _exact_int_layer(x, W, A, B, ranks, scales, ids):
    """y with Python integers and Fractions; no numpy arithmetic."""
    T, K = len(x), len(x[0])
    N = len(W)
    out = []
    for t in range(T):
        s = ids[t]
        row = []
        for n in range(N):
            acc = Fraction(sum(int(x[t][k]) * int(W[n][k]) for k in range(K)))
            if 1 <= s < len(ranks) and ranks[s] > 0:
                u = [sum(int(x[t][k]) * int(A[s][j][k]) for k in range(K)) for j in range(ranks[s])]
                acc += scales[s] * sum(u[j] * int(B[s][n][j]) for j in range(ranks[s]))
            row.append(acc)
        out.append(row)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_integer_bruteforce_exact(seed):
    """Integer inputs in {-2..2}, power-of-two scales: the exact result
    computed with Python integers must equal the oracle exactly."""
    rng = np.random.default_rng(100 + seed)
    T, K, N, S, R = int(rng.integers(1, 9)), int(rng.integers(1, 17)), int(rng.integers(1, 17)), 4, 4
    ranks = [0] + [int(v) for v in rng.integers(0, R + 1, size=S - 1)]
    # alpha / rank in {0.5, 1, 2, 4}
    alpha = [0.0] + [float(r * 2.0 ** int(rng.integers(-1, 3))) for r in ranks[1:]]
    x = rng.integers(-2, 3, size=(T, K))
    W = rng.integers(-2, 3, size=(N, K))
    A = np.zeros((S, R, K), dtype=np.int64)
    B = np.zeros((S, N, R), dtype=np.int64)
    for s in range(1, S):
        A[s, :ranks[s]] = rng.integers(-2, 3, size=(ranks[s], K))
        B[s, :, :ranks[s]] = rng.integers(-2, 3, size=(N, ranks[s]))
    ids = rng.integers(-1, S + 1, size=T)
    scales = [Fraction(0)] + [Fraction(alpha[s]) / ranks[s] if ranks[s] else Fraction(0) for s in range(1, S)]
    exact = _exact_int_layer(x.tolist(), W.tolist(), A.tolist(), B.tolist(), ranks, scales, ids.tolist())
    y = O.lora_linear(x, W, A, B, ranks, alpha, ids)
    for t in range(T):
        for n in range(N):
            assert Fraction(y[t, n]) == exact[t][n], (t, n)


@pytest.mark.parametrize("seed", range(4))
def test_sliced_integer_exact(seed):
    """Slices with their own adapters, integer inputs: each slice's columns
    equal the exact integer layer of that slice, in slice order."""
    rng = np.random.default_rng(300 + seed)
    T, K, S, R = int(rng.integers(1, 7)), int(rng.integers(1, 13)), 4, 4
    n_sl = int(rng.integers(1, 4))
    d_outs = [int(rng.integers(1, 9)) for _ in range(n_sl)]
    ids = rng.integers(-1, S + 1, size=T)
    x = rng.integers(-2, 3, size=(T, K))
    Ws, As, Bs, ranks_l, alphas_l, exact_cols = [], [], [], [], [], []
    for n in d_outs:
        ranks = [0] + [int(v) for v in rng.integers(0, R + 1, size=S - 1)]
        alpha = [0.0] + [float(r * 2.0 ** int(rng.integers(-1, 3))) for r in ranks[1:]]
        W = rng.integers(-2, 3, size=(n, K))
        A = np.zeros((S, R, K), dtype=np.int64)
        B = np.zeros((S, n, R), dtype=np.int64)
        for s in range(1, S):
            A[s, :ranks[s]] = rng.integers(-2, 3, size=(ranks[s], K))
            B[s, :, :ranks[s]] = rng.integers(-2, 3, size=(n, ranks[s]))
        scales = [Fraction(0)] + [Fraction(alpha[s]) / ranks[s] if ranks[s] else Fraction(0) for s in range(1, S)]
        exact_cols.append(_exact_int_layer(x.tolist(), W.tolist(), A.tolist(), B.tolist(), ranks, scales, ids.tolist()))
        Ws.append(W); As.append(A); Bs.append(B); ranks_l.append(ranks); alphas_l.append(alpha)
    y = O.lora_linear_sliced(x, Ws, As, Bs, ranks_l, alphas_l, ids)
    assert y.shape == (T, sum(d_outs))
    off = 0
    for n, ex in zip(d_outs, exact_cols):
        for t in range(T):
            for c in range(n):
                assert Fraction(y[t, off + c]) == ex[t][c], (t, off + c)
        off += n


def test_sliced_split_of_one_layer():
    """One adapter layer split by output rows into slices (W and B split, A
    shared) gives the unsliced layer's columns, in order."""
    rng = np.random.default_rng(7)
    T, K, N, S, R = 9, 24, 20, 5, 8
    x = rng.standard_normal((T, K))
    W = rng.standard_normal((N, K))
    A = rng.standard_normal((S, R, K))
    B = rng.standard_normal((S, N, R))
    ranks = [0, 8, 3, 5, 8]
    for s in range(S):
        A[s, ranks[s]:] = 0
        B[s, :, ranks[s]:] = 0
    alpha = [0.0, 16.0, 3.0, 10.0, 8.0]
    ids = rng.integers(0, S, size=T)
    cuts = [0, 7, 15, N]
    parts = list(zip(cuts[:-1], cuts[1:]))
    y = O.lora_linear_sliced(x, [W[a:b] for a, b in parts], [A] * 3, [B[:, a:b] for a, b in parts],
                             [ranks] * 3, [alpha] * 3, ids)
    full = O.lora_linear(x, W, A, B, ranks, alpha, ids)
    np.testing.assert_allclose(y, full, rtol=1e-12, atol=1e-12)
    # swapping two slices' inputs moves their columns
    y_sw = O.lora_linear_sliced(x, [W[7:15], W[0:7]], [A, A], [B[:, 7:15], B[:, 0:7]], [ranks] * 2, [alpha] * 2, ids)
    np.testing.assert_allclose(y_sw[:, :8], full[:, 7:15], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y_sw[:, 8:], full[:, 0:7], rtol=1e-12, atol=1e-12)


def test_rows_selection_pins():
    """The layer on selected positions: selecting every row in order is the
    layer itself; a reversed selection reverses the rows; an index outside x
    reads a zero row, which gets exactly zero."""
    rng = np.random.default_rng(11)
    T, K, N, S, R = 7, 12, 10, 4, 4
    x = rng.integers(-2, 3, size=(T, K)).astype(np.float64)
    W = rng.integers(-2, 3, size=(N, K)).astype(np.float64)
    A = np.zeros((S, R, K)); B = np.zeros((S, N, R))
    ranks = [0, 4, 2, 3]
    for s in range(1, S):
        A[s, :ranks[s]] = rng.integers(-2, 3, size=(ranks[s], K))
        B[s, :, :ranks[s]] = rng.integers(-2, 3, size=(N, ranks[s]))
    alpha = [0.0, 8.0, 4.0, 6.0]
    ids = rng.integers(0, S, size=T)
    full = O.lora_linear(x, W, A, B, ranks, alpha, ids)
    assert np.array_equal(O.lora_linear_rows(x, np.arange(T), W, A, B, ranks, alpha, ids), full)
    rev = np.arange(T)[::-1]
    assert np.array_equal(O.lora_linear_rows(x, rev, W, A, B, ranks, alpha, ids[rev]), full[rev])
    y = O.lora_linear_rows(x, np.array([2, -1, T, 5]), W, A, B, ranks, alpha, np.array([ids[2], 1, 2, ids[5]]))
    assert np.array_equal(y[0], full[2]) and np.array_equal(y[3], full[5])
    assert not y[1].any() and not y[2].any()


def test_transposed_or_dropped_terms_are_caught():
    """The integer pin distinguishes the plausible slips: a transposed B, a
    dropped scale, a rank-padded scale, a wrong sign."""
    rng = np.random.default_rng(9)
    T, K, N, S, R = 3, 5, 6, 2, 4
    x = rng.integers(-2, 3, size=(T, K)); W = rng.integers(-2, 3, size=(N, K))
    A = np.zeros((S, R, K)); B = np.zeros((S, N, R))
    A[1, :3] = rng.integers(-2, 3, size=(3, K)); B[1, :, :3] = rng.integers(-2, 3, size=(N, 3))
    ids = [1, 1, 1]
    y = O.lora_linear(x, W, A, B, [0, 3], [0.0, 6.0], ids)          # scale 2 (true rank 3)
    u = x @ A[1, :3].T
    good = x @ W.T + 2.0 * u @ B[1, :, :3].T
    assert np.array_equal(y, good)
    for wrong in (x @ W.T + u @ B[1, :, :3].T,                       # dropped scale
                  x @ W.T + (6.0 / R) * u @ B[1, :, :3].T,           # scale with R_max
                  x @ W.T - 2.0 * u @ B[1, :, :3].T):                # sign
        assert not np.array_equal(y, wrong)


# ------------------------------------------------------------- counters ----

LLAMA3_8B = [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096),
             (4096, 14336), (4096, 14336), (14336, 4096)]


def test_flop_ratio_square_r16():
    """LoRA serving page, intro: the rank-16 correction costs 0.78 % of the
    base GEMM for a square 4096 projection (16 * 8192 / 4096^2 = 0.0078125)."""
    assert O.correction_flop_ratio(16, 4096, 4096) == 0.0078125
    assert round(100 * O.correction_flop_ratio(16, 4096, 4096), 2) == 0.78


def test_adapter_param_arithmetic():
    """LoRA serving page: 41.9 M params for a rank-16 adapter on the seven
    targets over 32 layers; r * 5 MiB in bf16; attention-only per-layer sum
    26,624 -> 13.63 M params, 26 MiB; 0.52 % of 8.03 B; 0.56 % of the 15.01 GB
    decode stream; k*r about 286 for +10 % weight traffic."""
    per_layer_unit = O.adapter_params(1, LLAMA3_8B)
    assert per_layer_unit == 81920
    p16 = 32 * O.adapter_params(16, LLAMA3_8B)
    assert p16 == 41_943_040 and round(p16 / 1e6, 1) == 41.9
    assert 32 * O.adapter_params(1, LLAMA3_8B) * 2 == 5 * 2**20          # r * 5 MiB
    assert O.adapter_params(1, LLAMA3_8B[:4]) == 26_624
    p_att = 32 * O.adapter_params(16, LLAMA3_8B[:4])
    assert round(p_att / 1e6, 2) == 13.63 and p_att * 2 == 26 * 2**20
    assert round(100 * p16 / 8.03e9, 2) == 0.52
    assert round(100 * 2 * p16 / 15.01e9, 2) == 0.56
    assert round(0.1 * 15.01e9 / (32 * O.adapter_params(1, LLAMA3_8B) * 2)) == 286
    # fifty adapters: 4.2 GB
    assert round(50 * 2 * p16 / 1e9, 1) == 4.2
