"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded bf16 inputs. Plan arrays bit-exact; y within 2e-2 * (1 + |ref|);
slot-0 rows bitwise equal to the GPU's own base-only run."""
import numpy as np
import pytest
import torch

from adapter_gemm_gb300 import lora as L
from adapter_gemm_gb300 import workloads as WL
from oracle import lora_oracle as O

from _gpu_common import DeviceWorkload, assert_parity, f64, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from adapter_gemm_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    assert L.last_device_error() == 0


# ------------------------------------------------------------------ plan ----

def _plan_case(ids, S):
    T = len(ids)
    plan = L.Plan(T, S, 8, 64, device=DEV)
    plan.build(torch.tensor(np.asarray(ids, dtype=np.int32), device=DEV))
    n_bad = plan.check()
    ref = O.plan(ids, S, tile_rows=L.TILE_ROWS)
    assert n_bad == ref["n_invalid"]
    assert plan.n_invalid() == ref["n_invalid"]
    assert plan.counts().cpu().tolist() == ref["counts"].tolist()
    assert plan.indptr().cpu().tolist() == ref["indptr"].tolist()
    assert plan.token_order().cpu().tolist() == ref["token_order"].tolist()
    assert plan.slot_of_token().cpu().tolist() == ref["slot_of_token"].tolist()
    assert plan.active().cpu().tolist() == ref["active"].tolist()
    tiles = plan.tiles().cpu()[:, :3].tolist()
    assert tiles == ref["tiles"].tolist()


def test_plan_worked_example():
    _plan_case([1] * 5 + [2] * 4 + [0] * 3, 3)


@pytest.mark.parametrize("T,S,seed", [(0, 4, 0), (1, 2, 1), (31, 3, 2), (33, 5, 3), (64, 9, 4),
                                      (1000, 17, 5), (1024, 1024, 6), (4096, 51, 7), (5000, 2, 8),
                                      (70000, 300, 9)])
def test_plan_random(T, S, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-2, S + 2, size=T)     # includes invalid ids
    _plan_case(ids.tolist(), S)


def test_plan_all_one_slot_and_sorted_runs():
    _plan_case([3] * 777, 4)
    _plan_case([0] * 100 + [1] * 100, 2)
    _plan_case(sorted(np.random.default_rng(1).integers(0, 40, size=3000).tolist(), reverse=True), 40)


# --------------------------------------------------------------- configs ----

def _full_check(w, i=0):
    dw = DeviceWorkload(w, DEV)
    y = dw.run(i)
    assert_parity(y, dw.oracle(i), w.name)
    return dw, y


def test_tiny_full():
    _full_check(WL.tiny())


def test_q_decode_full():
    _full_check(WL.q_decode())


def test_mixed_down_full():
    _full_check(WL.mixed_down())


def test_gateup_prefill_full():
    """Every element of the 4096 x 14336 output against the oracle."""
    _full_check(WL.gateup_prefill())


@pytest.mark.parametrize("T", WL.SWEEP_T)
def test_layer_sweep(T):
    w = WL.layer_sweep(T)
    dw = DeviceWorkload(w, DEV)
    rows = np.arange(T) if T <= 64 else sample_rows(w.ids, 48)
    for i, t in enumerate(w.targets):
        y = dw.run(i)
        assert_parity(y[torch.as_tensor(rows, device=DEV)], dw.oracle(i, rows=rows), f"{w.name}/{t.name}")


def test_layer_sweep_T4096_whole_targets():
    """The prefill-sized sweep: every element of two targets' outputs (the
    widest, gate 4096 -> 14336, and the long-K down 14336 -> 4096)."""
    w = WL.layer_sweep(4096)
    dw = DeviceWorkload(w, DEV)
    for i, t in enumerate(w.targets):
        if t.name in ("gate_proj", "down_proj"):
            assert_parity(dw.run(i), dw.oracle(i), f"{w.name}/{t.name}")


# ------------------------------------------------------------ slot 0 rows ----

@pytest.mark.parametrize("name", ["tiny", "q_decode", "mixed_down", "gateup_prefill", "layer_sweep_T512"])
def test_slot0_rows_bitwise_equal_base_only(name):
    w = WL.by_name(name)
    dw = DeviceWorkload(w, DEV)
    for i in range(min(2, len(w.targets))):
        y = dw.run(i)
        yb = dw.run(i, base_only=True)
        slot0 = torch.as_tensor(w.ids == 0, device=DEV)
        if slot0.any():
            assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))
        # base-only run is itself the base projection
        rows = np.arange(min(w.T, 16))
        base = O.base_linear(f64(WL.input_for(w, w.targets[i])), f64(w.targets[i].W), rows=rows)
        assert_parity(yb[: len(rows)], base, name + " base-only")


# --------------------------------------------------------- exact integers ----

@pytest.mark.parametrize("T,K,N,R", [(9, 16, 24, 8), (64, 64, 136, 8), (300, 64, 264, 8), (513, 32, 520, 16),
                                     (2049, 64, 8704, 16)])    # CTA pairs, a last row block of one row
def test_integer_inputs_bit_exact(T, K, N, R):
    """Small-integer inputs with power-of-two scales: every partial sum is exact
    in fp32 and every output is an integer of magnitude <= 256, so the GPU must
    equal the exact result bit for bit."""
    rng = np.random.default_rng(T + K + N)
    S = 5
    ranks = [0, 1, 2, 2, 0]           # slot 4 stays empty (rank 0)
    alpha = np.array([0.0, 1.0, 2.0, 4.0, 0.0], dtype=np.float32)    # scales 1, 1, 2
    x = rng.integers(-1, 2, size=(T, K)).astype(np.float32)
    W = rng.integers(-1, 2, size=(N, K)).astype(np.float32)
    A = np.zeros((S, R, K), np.float32)
    B = np.zeros((S, N, R), np.float32)
    for s in range(1, S):
        A[s, :ranks[s]] = rng.integers(-1, 2, size=(ranks[s], K))
        B[s, :, :ranks[s]] = rng.integers(-1, 2, size=(N, ranks[s]))
    ids = rng.integers(0, S, size=T).astype(np.int32)
    ref = O.lora_linear(x, W, A, B, ranks, alpha, ids)
    assert np.abs(ref).max() <= 256 and np.array_equal(ref, np.round(ref))
    tgt = WL.Target("int", K, N, WL.to_bf16(W), WL.to_bf16(A), WL.to_bf16(B), np.array(ranks, np.int32), alpha)
    w = WL.Workload("int", T, S, R, ids, WL.to_bf16(x), [tgt])
    dw = DeviceWorkload(w, DEV)
    y = f64(dw.run(0))
    assert np.array_equal(y, ref)


# ------------------------------------------------------------ ragged sizes ----

RAGGED = [
    # T, K, N, S, R_max
    (1, 64, 8, 2, 8),
    (5, 200, 72, 3, 8),
    (17, 1000, 200, 6, 24),
    (100, 4096, 520, 9, 64),
    (256, 520, 1032, 33, 128),
    (257, 200, 264, 4, 16),
    (300, 1000, 520, 7, 24),
    (480, 4160, 264, 5, 16),
    (512, 1024, 392, 12, 32),
    (700, 4104, 1288, 40, 64),
    (1500, 2048, 776, 17, 128),
]


@pytest.mark.parametrize("T,K,N,S,R", RAGGED)
def test_ragged_shapes(T, K, N, S, R):
    w = WL.random_case(seed=T * 7 + K, T=T, K=K, N=N, S=S, R_max=R)
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    rows = np.arange(T) if T <= 400 else sample_rows(w.ids, 200)
    assert_parity(y[torch.as_tensor(rows, device=DEV)], dw.oracle(0, rows=rows), f"ragged {T},{K},{N}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


# Long projections (d_in or d_out of 8192 or more) of batches of 2048 rows or
# more run the prefill GEMM on CTA pairs (256-row tiles, one M = 256 MMA over
# the two CTAs of a cluster). The cases: the long side in d_in and in d_out; a
# last row block whose second half lies wholly past T (2100 = 8 x 256 + 52) or
# partly (2300); a last wave split into 256 x 128 halves (153 and 306 tiles on
# 76 pairs); slot-0 rows bit for bit against base-only calls, which take the
# same kernel.
@pytest.mark.parametrize("T,K,N,S,R", [(2100, 8192, 4352, 17, 32), (2300, 2048, 8704, 30, 16)])
def test_pair_prefill_ragged(T, K, N, S, R):
    assert L.linear_path(T, K, N) == 1
    w = WL.random_case(seed=T + K + N, T=T, K=K, N=N, S=S, R_max=R, base_frac=0.15)
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    rows = np.unique(np.concatenate([sample_rows(w.ids, 160), np.arange(T - 64, T), np.arange(2040, 2060)]))
    assert_parity(y[torch.as_tensor(rows, device=DEV)], dw.oracle(0, rows=rows), f"pairs T={T} {K}->{N}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


# Batches whose pool has R_max <= 16, at least 8 rows per group of G
# consecutive slot ids (G R_max <= 256) and fewer than 32 rows per slot take
# grouped shrink units: one MMA per K step over every slot of the group, each
# row keeping its own slot's columns. The cases: groups found in the ids
# (T <= 64) and on the plan (chunks of 128 rows), for the decode kernel and
# for the prefill kernel (its plan-ordered copy of x, slot 0's rows as
# copy-only units, U as bf16 high and low parts), R_max 8 and 16, d_in not a
# multiple of 64 (one slice per stage), ranks below R_max, uninstalled
# (rank-0) slots inside a group, a last group cut short by S, invalid ids,
# slot-0 rows; 7 groups of 16 slots beside a wide decode output (112 weight
# tiles).
GROUPED = [(64, 1024, 512, 40, 16), (48, 1000, 264, 20, 8), (100, 512, 256, 30, 16),
           (300, 768, 384, 51, 16), (256, 4096, 1024, 51, 16), (700, 512, 512, 51, 16),
           (900, 256, 264, 40, 8), (64, 4096, 14336, 100, 16)]


@pytest.mark.parametrize("T,K,N,S,R", GROUPED)
def test_grouped_shrink_units(T, K, N, S, R):
    rng = np.random.default_rng(T + S)
    ranks = [0] + [0 if s % 7 == 3 else int(rng.integers(1, R + 1)) for s in range(1, S)]
    w = WL.random_case(seed=900 + T, T=T, K=K, N=N, S=S, R_max=R, ranks=ranks)
    w.ids[::17] = -1                                   # invalid ids: counted, base rows
    w.ids[5::23] = S
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    assert_parity(y, dw.oracle(0), f"grouped shrink T={T} S={S} R={R}")
    base = torch.as_tensor((w.ids <= 0) | (w.ids >= S) | (np.asarray(ranks)[np.clip(w.ids, 0, S - 1)] == 0),
                           device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[base].view(torch.int16), yb[base].view(torch.int16))


# ---------------------------------------------------------- wiring & edges ----

def test_perturbing_a_slot_changes_exactly_its_rows():
    """Reinstall slot s with a different B: rows on s change, no other row does."""
    w = WL.layer_sweep(64, targets=WL.LLAMA3_8B_TARGETS[:1])
    dw = DeviceWorkload(w, DEV)
    y0 = dw.run(0)
    t = w.targets[0]
    for s in (int(w.ids[3]), int(w.ids[-1])):
        if s == 0:
            continue
        r = int(t.rank[s])
        A = t.A[s, :r].to(DEV).contiguous()
        Bn = (t.B[s, :, :r].float() * -1.5).to(torch.bfloat16).to(DEV).contiguous()
        dw.targets[0].pool.install(s, A, Bn, float(t.alpha[s]))
        y1 = dw.run(0)
        changed = (y1.view(torch.int16) != y0.view(torch.int16)).any(dim=1).cpu().numpy()
        assert np.array_equal(changed, w.ids == s), s
        dw.targets[0].pool.install(s, A, t.B[s, :, :r].to(DEV).contiguous(), float(t.alpha[s]))
        assert torch.equal(dw.run(0).view(torch.int16), y0.view(torch.int16))


def test_every_active_slot_contributes():
    w = WL.layer_sweep(512, targets=WL.LLAMA3_8B_TARGETS[:1])
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    yb = dw.run(0, base_only=True)
    differs = (y.view(torch.int16) != yb.view(torch.int16)).any(dim=1).cpu().numpy()
    for s in np.unique(w.ids):
        if s > 0:
            assert differs[w.ids == s].all(), s


def test_runs_are_deterministic():
    for w in (WL.mixed_down(), WL.layer_sweep(512, targets=WL.LLAMA3_8B_TARGETS[4:5])):
        dw = DeviceWorkload(w, DEV)
        a = dw.run(0)
        b = dw.run(0)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_invalid_ids_are_counted_and_get_base_rows():
    w = WL.random_case(seed=11, T=80, K=256, N=128, S=4, R_max=8)
    w.ids[[0, 7, 50]] = [-1, 4, 1000]
    dw = DeviceWorkload(w, DEV)
    assert dw.plan.check() == 3
    y = dw.run(0)
    assert_parity(y, dw.oracle(0), "invalid ids")
    yb = dw.run(0, base_only=True)
    for r in (0, 7, 50):
        assert torch.equal(y[r].view(torch.int16), yb[r].view(torch.int16))


def test_empty_batch_and_all_base_rows():
    W = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    pool = L.Pool(3, 8, 128, 64, device=DEV)
    plan = L.Plan(0, 3, 8, 128, device=DEV).build(torch.empty(0, dtype=torch.int32, device=DEV))
    y = L.linear(torch.empty(0, 128, dtype=torch.bfloat16, device=DEV), W, pool, plan)
    assert y.shape == (0, 64)
    x = torch.randn(40, 128, device=DEV).to(torch.bfloat16)
    plan = L.Plan(40, 3, 8, 128, device=DEV).build(torch.zeros(40, dtype=torch.int32, device=DEV))
    assert plan.n_active() == 0
    y = L.linear(x, W, pool, plan)
    yb = L.linear(x, W)
    assert torch.equal(y.view(torch.int16), yb.view(torch.int16))


def test_install_refuses_non_finite_and_keeps_slot():
    pool = L.Pool(3, 8, 64, 32, device=DEV)
    A = torch.randn(4, 64, device=DEV).to(torch.bfloat16)
    B = torch.randn(32, 4, device=DEV).to(torch.bfloat16)
    pool.install(1, A, B, 8.0)
    before = (pool.A.clone(), pool.B.clone(), pool.rank.clone(), pool.scale.clone())
    bad = B.clone()
    bad[3, 1] = float("nan")
    with pytest.raises(L.LoraError) as e:
        pool.install(1, A, bad, 8.0)
    assert e.value.name == "LORA_ENONFINITE"
    bad = A.clone()
    bad[0, 0] = float("inf")
    with pytest.raises(L.LoraError):
        pool.install(1, bad, B, 8.0)
    for t0, t1 in zip(before, (pool.A, pool.B, pool.rank, pool.scale)):
        assert torch.equal(t0, t1)
    # a smaller reinstall zeroes the old padding
    pool.install(1, A[:2].contiguous(), B[:, :2].contiguous(), 4.0)
    assert int(pool.rank[1]) == 2 and float(pool.scale[1]) == 2.0
    assert pool.A[1, 2:].abs().sum() == 0 and pool.B[1, :, 2:].abs().sum() == 0


def test_row_offsets_beyond_int32():
    """T * d_in > 2^31 elements: row offsets must be 64-bit everywhere
    (the LoRA-serving page's long-context int32 overflow)."""
    T, K, N, S, R = 150_000, 14_336, 64, 3, 8
    assert T * K > 2**31
    w = WL.random_case(seed=5, T=256, K=K, N=N, S=S, R_max=R)   # adapters and W only
    t = w.targets[0]
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn(T, K, device=DEV, generator=g).to(torch.bfloat16)
    ids_np = np.random.default_rng(4).integers(0, S, size=T).astype(np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    Wd = t.W.to(DEV)
    pool = L.Pool(S, R, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    plan = L.Plan(T, S, R, K, device=DEV).build(ids)
    y = L.linear(x, Wd, pool, plan)
    torch.cuda.synchronize()
    rows = np.array([0, 1, T // 2, T - 2, T - 1, 149_000, 100_001])
    xr = f64(x[torch.as_tensor(rows, device=DEV)])
    ref = O.lora_linear(xr, f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, ids_np[rows])
    assert_parity(y[torch.as_tensor(rows, device=DEV)], ref, "int64 offsets")
    del x, y, plan
    torch.cuda.empty_cache()


# --------------------------------------------- back-to-back calls, no sync ----
# The kernels start before the kernel ahead of them has finished (programmatic
# dependent launch) and request their first weight stages early; a call's
# first kernel reads x and the ids only after its wait. These tests chain calls
# on one stream with no synchronisation in between: each step's input is the
# previous step's output, and the same plan object (its arrays and U) is
# rebuilt for every step.

def _chained_steps(T, K, S, R, n_steps, base_only=False, seed=3):
    w = WL.random_case(seed=seed, T=T, K=K, N=K, S=S, R_max=R)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, K, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    rng = np.random.default_rng(seed + 1)
    ids_np = [rng.integers(0, S, size=T).astype(np.int32) for _ in range(n_steps)]
    ids = [torch.from_numpy(v).to(DEV) for v in ids_np]
    plan = L.Plan(T, S, R, K, device=DEV)
    xs = [w.x.to(DEV)]
    torch.cuda.synchronize()
    for k in range(n_steps):                 # no synchronisation inside the loop
        if base_only:
            xs.append(L.linear(xs[-1], W))
        else:
            plan.build(ids[k])
            xs.append(L.linear(xs[-1], W, pool, plan))
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    for k in range(n_steps):
        x_in = f64(xs[k])
        step_ids = np.zeros(T, np.int32) if base_only else ids_np[k]
        ref = O.lora_linear(x_in, f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, step_ids)
        assert_parity(xs[k + 1], ref, f"step {k}")


def test_chained_decode_steps_fused_shrink():
    _chained_steps(T=64, K=1024, S=9, R=16, n_steps=4)        # (S-1) R = 128: shrink fused in


def test_chained_decode_steps_shrink_kernel():
    _chained_steps(T=48, K=1024, S=20, R=16, n_steps=4)       # shrink kernel ahead of the GEMM


def test_chained_decode_steps_base_only():
    _chained_steps(T=64, K=1024, S=9, R=16, n_steps=4, base_only=True)


def test_chained_prefill_steps():
    _chained_steps(T=300, K=512, S=12, R=16, n_steps=3)       # the wide kernel


@pytest.mark.parametrize("T,K,S,R", [(64, 1024, 9, 16), (48, 1024, 20, 16), (300, 512, 12, 16)])
def test_input_written_two_calls_back_and_by_a_foreign_kernel(T, K, S, R):
    """Inputs that are not the previous call's output but may still be in
    flight: y1 = f(x0); y2 = f(x1); y3 = f(y1) (y1 written two calls back), and
    x written by a torch kernel right before the call, and ids written by a
    torch kernel right before the plan - all with no synchronisation. Covers
    the fused decode shrink, the shrink kernel ahead of the decode GEMM, and the
    prefill kernel."""
    w = WL.random_case(seed=77, T=T, K=K, N=K, S=S, R_max=R)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, K, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    ids_np = w.ids.astype(np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    plan = L.Plan(T, S, R, K, device=DEV).build(ids)
    x0 = w.x.to(DEV)
    x1 = (x0 * -1).contiguous()
    x_src = (x0 * 0.5).contiguous()
    ids_src = torch.from_numpy(np.roll(ids_np, 3)).to(DEV)
    ids_dst = torch.zeros_like(ids)
    x_dst = torch.empty_like(x0)
    plan2 = L.Plan(T, S, R, K, device=DEV)
    torch.cuda.synchronize()
    y1 = L.linear(x0, W, pool, plan)
    y2 = L.linear(x1, W, pool, plan)
    y3 = L.linear(y1, W, pool, plan)
    x_dst.copy_(x_src)                       # a torch kernel writes x ...
    y4 = L.linear(x_dst, W, pool, plan)      # ... right before the call reads it
    torch.add(ids_src, 0, out=ids_dst)       # a torch kernel writes the ids ...
    plan2.build(ids_dst)                     # ... right before the plan reads them
    y5 = L.linear(x0, W, pool, plan2)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    f = lambda x, i: O.lora_linear(f64(x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, i)
    r1 = f(x0, ids_np)
    assert_parity(y1, r1, "y1 = f(x0)")
    assert_parity(y2, f(x1, ids_np), "y2 = f(x1)")
    assert_parity(y3, f(y1, ids_np), "y3 = f(y1), y1 two calls back")
    assert_parity(y4, f(x_src, ids_np), "x written by a torch kernel")
    assert_parity(y5, f(x0, np.roll(ids_np, 3)), "ids written by a torch kernel")


def test_one_plan_many_targets_without_sync():
    """Several layers of one step share the plan (and its U), back to back."""
    T, K, S, R = 64, 512, 20, 16
    ws = [WL.random_case(seed=40 + i, T=T, K=K, N=K, S=S, R_max=R) for i in range(3)]
    ids_np = ws[0].ids
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(DEV)
    plan = L.Plan(T, S, R, K, device=DEV).build(ids)
    x = ws[0].x.to(DEV)
    outs = []
    for w in ws:
        t = w.targets[0]
        pool = L.Pool(S, R, K, K, device=DEV)
        pool.load_padded(t.A, t.B, t.rank, t.alpha)
        outs.append((t, L.linear(x, t.W.to(DEV), pool, plan)))
    torch.cuda.synchronize()
    for t, y in outs:
        ref = O.lora_linear(f64(x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, ids_np)
        assert_parity(y, ref, "shared plan")


# ------------------------------------------------ decode path selection ----

def test_fused_shrink_invalid_ids_and_mixed_ranks():
    """A pool whose adapters' A rows fit one 128-row tile computes U inside the
    GEMM: ids outside [0, S) give base rows, ranks below R_max (zero padding)
    and a rank-0 slot add nothing beyond their true rank."""
    w = WL.random_case(seed=21, T=48, K=512, N=384, S=5, R_max=32, ranks=[0, 8, 32, 17, 0])
    w.ids[[0, 5, 9]] = [-3, 5, 77]
    w.ids[[1, 2]] = 4                                    # the rank-0 slot
    dw = DeviceWorkload(w, DEV)
    assert dw.plan.check() == 3
    n0 = L.launch_count()
    y = dw.run(0)
    assert L.launch_count() - n0 == 1                    # one kernel: the shrink is fused in
    assert_parity(y, dw.oracle(0), "fused shrink")
    yb = dw.run(0, base_only=True)
    for r in (0, 1, 2, 5, 9):
        assert torch.equal(y[r].view(torch.int16), yb[r].view(torch.int16))


@pytest.mark.parametrize("T,S,R,kernels", [
    (40, 6, 16, 1),     # every slot's ranks fit one CTA's expand: the shrink fused in
    (40, 40, 32, 2),    # the expand's chunks dealt over the cluster, U from the shrink kernel
    (6, 40, 32, 2),     # a batch of at most 8 rows: the CUDA-core expand
])
def test_tensor_core_expand_with_ids_from_previous_output(T, S, R, kernels):
    """The step's ids lie in the previous call's output on the same stream, so
    no kernel may read them before its wait for the kernel ahead: the fused
    GEMM's idle warps wait before they build the token tables, the shrink
    kernel waits before it reads them."""
    K, N = 512, 256
    ranks = [0, 16, 5, 12, 16, 9] if S == 6 else None
    w = WL.random_case(seed=23 + S + T, T=T, K=K, N=N, S=S, R_max=R, ranks=ranks)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(w.S, w.R_max, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    x = w.x.to(DEV)
    ids_dev = torch.from_numpy(w.ids.astype(np.int32)).to(DEV)
    plan = L.Plan(T, w.S, w.R_max, K, device=DEV).build(ids_dev)
    buf = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
    L.linear(x, W, pool, plan, buf)
    first = buf.clone()                                  # ordered after the GEMM on this stream
    ids_in_y = buf.view(torch.int32).reshape(-1)[:T]     # overwrite part of that output with the ids
    ids_in_y.copy_(ids_dev)
    plan.build(ids_in_y)
    n0 = L.launch_count()
    y = L.linear(x, W, pool, plan)
    assert L.launch_count() - n0 == kernels
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    ref = O.lora_linear(f64(x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, w.ids)
    assert_parity(first, ref, "first call")
    assert_parity(y, ref, "ids from the previous output")


FUSED_EDGES = [
    # T, K, N, S, R_max: every adapter slot's ranks (rounded up to 16) fit 128 pairs
    (64, 256, 256, 2, 128),      # one slot of rank 128: eight chunks of pairs
    (64, 256, 256, 9, 8),        # rank 8 < 16: pad positions of every slot stay zero
    (16, 192, 136, 5, 24),       # R16 = 32; three K slices; a ragged weight tile
    (1, 64, 8, 3, 16),           # one row, one K slice, eight outputs
    (63, 4160, 264, 3, 64),      # 65 K slices; T one short of a full tile
]


@pytest.mark.parametrize("T,K,N,S,R", FUSED_EDGES)
def test_fused_shrink_edge_shapes(T, K, N, S, R):
    w = WL.random_case(seed=T * 13 + K + S, T=T, K=K, N=N, S=S, R_max=R)
    dw = DeviceWorkload(w, DEV)
    n0 = L.launch_count()
    y = dw.run(0)
    assert L.launch_count() - n0 == 1                    # the shrink is fused in
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    assert_parity(y, dw.oracle(0), f"fused {T},{K},{N},{S},{R}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


@pytest.mark.parametrize("T", [64, 300])
def test_most_slots(T):
    """S = 1024 slots, ids over all of them: the decode path's chunk-dealt
    expand and the prefill path's segment lists."""
    w = WL.random_case(seed=1024 + T, T=T, K=128, N=136, S=1024, R_max=8, base_frac=0.05)
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    assert_parity(y, dw.oracle(0), f"S=1024, T={T}")


@pytest.mark.parametrize("T,K,N,S,R", [
    (256, 64, 128, 33, 128),     # one CTA per cluster: 32 slots x 8 chunks, many batches
    (200, 192, 384, 40, 128),    # ragged token tile, two CTAs per cluster
    (9, 4096, 256, 60, 64),      # eight CTAs per cluster, a few chunks: some CTAs get none
])
def test_chunk_dealt_expand_batches(T, K, N, S, R):
    """The decode path's expand with U from the shrink kernel, when the slots'
    ranks exceed what one CTA's expand holds: the (slot, 16-rank chunk) pairs
    are dealt over the cluster's CTAs and added in batches."""
    w = WL.random_case(seed=T * 13 + S, T=T, K=K, N=N, S=S, R_max=R, base_frac=0.1)
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    assert_parity(y, dw.oracle(0), f"chunk-dealt expand {T},{K},{N},{S},{R}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


# The rank-aware kernel choice: from 257 to 640 rows a pool of at least 128
# (slot, 16-rank) chunks, or of at least 64 above 560 rows, takes the wide
# kernel; a base-only run given the pool takes the same one.
@pytest.mark.parametrize("T,K,N,S,R,path", [
    (300, 512, 512, 33, 64, 1),      # 128 chunks
    (600, 512, 520, 17, 64, 1),      # 64 chunks above 560 rows
    (400, 512, 512, 17, 64, 0),      # 64 chunks at 400 rows: the swap-AB kernel
    (500, 256, 384, 9, 128, 0),      # 64 chunks of rank 128 at 500 rows
])
def test_rank_aware_kernel_choice(T, K, N, S, R, path):
    assert L.linear_path(T, K, N) == 0
    w = WL.random_case(seed=T + 31 * S, T=T, K=K, N=N, S=S, R_max=R, base_frac=0.1)
    dw = DeviceWorkload(w, DEV)
    assert L.linear_path(T, K, N, dw.targets[0].pool) == path
    y = dw.run(0)
    assert_parity(y, dw.oracle(0), f"rank-aware T={T} S={S} R={R} path {path}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


@pytest.mark.parametrize("T,K,N,path", [
    (640, 512, 1024, 0),         # three token tiles on the swap-AB kernel
    (641, 512, 1024, 1),         # past the swap-AB kernel's range
    (300, 512, 20480, 1),        # too many weight tiles to split K: the persistent kernel
])
def test_mid_sized_batches_on_either_kernel(T, K, N, path):
    assert L.linear_path(T, K, N) == path
    w = WL.random_case(seed=T + N, T=T, K=K, N=N, S=20, R_max=32, base_frac=0.1)
    dw = DeviceWorkload(w, DEV)
    y = dw.run(0)
    rows = sample_rows(w.ids, 160)
    assert_parity(y[torch.as_tensor(rows, device=DEV)], dw.oracle(0, rows=rows), f"T={T} N={N} path {path}")
    slot0 = torch.as_tensor(w.ids == 0, device=DEV)
    yb = dw.run(0, base_only=True)
    assert torch.equal(y[slot0].view(torch.int16), yb[slot0].view(torch.int16))


def test_wide_output_takes_the_shrink_kernel():
    """Many weight tiles would re-read the A tile too often: U comes from the
    shrink kernel ahead (two kernels) and the expand runs on the tensor cores."""
    w = WL.random_case(seed=24, T=16, K=4096, N=8192, S=9, R_max=16)
    dw = DeviceWorkload(w, DEV)
    n0 = L.launch_count()
    y = dw.run(0)
    assert L.launch_count() - n0 == 2
    assert L.last_device_error() == 0
    assert_parity(y, dw.oracle(0), "shrink kernel, tensor-core expand")


def test_shrink_kernel_when_pool_exceeds_one_tile():
    """(S - 1) * R_max > 128: U comes from the shrink kernel ahead of the GEMM."""
    w = WL.random_case(seed=22, T=48, K=512, N=384, S=10, R_max=16)
    dw = DeviceWorkload(w, DEV)
    n0 = L.launch_count()
    y = dw.run(0)
    assert L.launch_count() - n0 == 2
    assert_parity(y, dw.oracle(0), "shrink kernel")


# ------------------------------------------ projections that share x (slices) ----

def _sliced(seed, T, K, d_outs, S, R, ranks=None):
    ws = [WL.random_case(seed=seed + i, T=T, K=K, N=n, S=S, R_max=R, ranks=ranks) for i, n in enumerate(d_outs)]
    ts = [w.targets[0] for w in ws]
    x = ws[0].x.to(DEV)
    ids_np = ws[0].ids.astype(np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    W = torch.cat([t.W for t in ts], 0).to(DEV)
    pools = []
    for t, n in zip(ts, d_outs):
        p = L.Pool(S, R, K, n, device=DEV)
        p.load_padded(t.A, t.B, t.rank, t.alpha)
        pools.append(p)
    plan = L.Plan(T, S, R, K, device=DEV).build(ids)
    torch.cuda.synchronize()
    ref = O.lora_linear_sliced(f64(x), [f64(t.W) for t in ts], [f64(t.A) for t in ts], [f64(t.B) for t in ts],
                               [t.rank for t in ts], [t.alpha for t in ts], ids_np)
    return x, W, pools, plan, ids_np, ref


@pytest.mark.parametrize("d_outs,kernels", [([256, 128, 128], 1), ([256, 136], 1), ([136, 256], 2)])
def test_sliced_decode_fused(d_outs, kernels):
    """QKV-like slices, shrink fused in: one GEMM for every slice when no weight
    tile straddles two slices, else one per slice."""
    x, W, pools, plan, ids_np, ref = _sliced(60, 64, 512, d_outs, S=9, R=16, ranks=[0, 16, 9, 16, 4, 16, 12, 16, 1])
    n0 = L.launch_count()
    y = L.linear_sliced(x, W, d_outs, pools, plan)
    assert L.launch_count() - n0 == kernels
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    assert_parity(y, ref, f"slices {d_outs}")
    if kernels == 1:
        # one launch splits K as the base-only projection of every output does
        yb = L.linear_sliced(x, W, d_outs)
        torch.cuda.synchronize()
        base = np.nonzero(ids_np == 0)[0]
        assert len(base) > 0
        for r in base:
            assert torch.equal(y[int(r)].view(torch.int16), yb[int(r)].view(torch.int16))


def test_sliced_decode_shrink_kernel():
    """(S - 1) * R_max > 128: one shrink kernel and one GEMM per slice."""
    d_outs = [256, 128]
    x, W, pools, plan, ids_np, ref = _sliced(70, 48, 512, d_outs, S=20, R=16)
    n0 = L.launch_count()
    y = L.linear_sliced(x, W, d_outs, pools, plan)
    assert L.launch_count() - n0 == 4
    torch.cuda.synchronize()
    assert_parity(y, ref, "slices, shrink kernel")


def test_sliced_prefill():
    """The wide kernel, one call per slice, each writing its columns of y."""
    d_outs = [256, 128, 136]
    x, W, pools, plan, ids_np, ref = _sliced(80, 300, 256, d_outs, S=12, R=16)
    y = L.linear_sliced(x, W, d_outs, pools, plan)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    assert_parity(y, ref, "slices, prefill")


def test_sliced_argument_errors():
    """Pools that do not match their slice, or too many slices, are refused
    before anything runs."""
    x, W, pools, plan, ids_np, ref = _sliced(90, 16, 256, [128, 256], S=5, R=16)
    n0 = L.launch_count()
    with pytest.raises(L.LoraError):
        L.linear_sliced(x, W, [128, 256], [pools[1], pools[0]], plan)   # d_out of each pool mismatched
    with pytest.raises(L.LoraError):
        L.linear_sliced(x, torch.cat([W] * 3, 0), [128, 256] * 3, pools * 3, plan)   # 6 > LORA_MAX_SLICES
    assert L.launch_count() == n0


# ------------------------------------------------------------ host buffers ----

def test_host_buffers_match_device_call():
    """lora_linear_host (copies in, plan, layer, copy out) gives the device
    call's bits, with and without a plan."""
    w = WL.random_case(seed=95, T=64, K=1024, N=384, S=9, R_max=16)
    dw = DeviceWorkload(w, DEV)
    t = dw.targets[0]
    y_dev_ref = dw.run(0)
    yb_ref = dw.run(0, base_only=True)
    x_h = w.x.contiguous().pin_memory()
    ids_h = torch.from_numpy(w.ids.astype(np.int32)).pin_memory()
    y_h = torch.empty((64, 384), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty((64, 1024), dtype=torch.bfloat16, device=DEV)
    ids_d = torch.empty(64, dtype=torch.int32, device=DEV)
    y_d = torch.empty((64, 384), dtype=torch.bfloat16, device=DEV)
    plan = L.Plan(64, w.S, w.R_max, 1024, device=DEV)
    L.linear_host(x_h, t.W, y_h, x_d, y_d, t.pool, plan, ids_h, ids_d)
    torch.cuda.synchronize()
    assert torch.equal(y_h.view(torch.int16), y_dev_ref.cpu().view(torch.int16))
    L.linear_host(x_h, t.W, y_h, x_d, y_d)
    torch.cuda.synchronize()
    assert torch.equal(y_h.view(torch.int16), yb_ref.cpu().view(torch.int16))


def test_host_buffers_two_streams_without_sync():
    """Steps alternate between two streams, each with its own staging buffers
    and plan, with no synchronisation in between: every step's output is
    right."""
    T, K, N, S, R = 48, 512, 256, 9, 16
    w = WL.random_case(seed=96, T=T, K=K, N=N, S=S, R_max=R)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    rng = np.random.default_rng(97)
    n_steps = 6
    xs = [torch.from_numpy(rng.standard_normal((T, K), dtype=np.float32)).to(torch.bfloat16).pin_memory()
          for _ in range(n_steps)]
    idss = [torch.from_numpy(rng.integers(0, S, size=T).astype(np.int32)).pin_memory() for _ in range(n_steps)]
    ys = [torch.empty((T, N), dtype=torch.bfloat16).pin_memory() for _ in range(n_steps)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    stage = [dict(x=torch.empty((T, K), dtype=torch.bfloat16, device=DEV),
                  ids=torch.empty(T, dtype=torch.int32, device=DEV),
                  y=torch.empty((T, N), dtype=torch.bfloat16, device=DEV),
                  plan=L.Plan(T, S, R, K, device=DEV)) for _ in range(2)]
    torch.cuda.synchronize()
    for k in range(n_steps):
        b, st = stage[k % 2], streams[k % 2]
        L.linear_host(xs[k], W, ys[k], b["x"], b["y"], pool, b["plan"], idss[k], b["ids"], stream=st)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    for k in range(n_steps):
        ref = O.lora_linear(f64(xs[k]), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, idss[k].numpy())
        assert_parity(ys[k], ref, f"step {k}")


# ------------------------------------- plans in CUDA graphs, padded batches ----

def test_graph_replays_with_new_ids_and_inputs():
    """The plan and the layer are captured once in a CUDA graph; each replay
    reads whatever ids and x the same buffers hold, so one graph serves every
    step of a fixed batch size."""
    T, K, N, S, R = 64, 512, 256, 9, 16
    w = WL.random_case(seed=120, T=T, K=K, N=N, S=S, R_max=R)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    x_buf = torch.zeros((T, K), dtype=torch.bfloat16, device=DEV)
    ids_buf = torch.zeros(T, dtype=torch.int32, device=DEV)
    y_buf = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    plan = L.Plan(T, S, R, K, device=DEV)
    plan.build(ids_buf)
    L.linear(x_buf, W, pool, plan, y_buf)               # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.build(ids_buf)
            L.linear(x_buf, W, pool, plan, y_buf)
    torch.cuda.current_stream().wait_stream(s)
    rng = np.random.default_rng(121)
    for k in range(3):
        ids_np = rng.integers(0, S, size=T).astype(np.int32)
        x_new = torch.from_numpy(rng.standard_normal((T, K), dtype=np.float32)).to(torch.bfloat16)
        ids_buf.copy_(torch.from_numpy(ids_np))
        x_buf.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        ref = O.lora_linear(f64(x_new), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, ids_np)
        assert_parity(y_buf, ref, f"replay {k}")


@pytest.mark.parametrize("T_real,T_cap", [(37, 64), (200, 256), (300, 512)])
def test_padded_batch_rows_on_slot0(T_real, T_cap):
    """A batch padded to a fixed capacity with slot-0 rows: the real rows get
    the unpadded layer's result, the zero padding rows get zeros."""
    K, N, S, R = 384, 264, 12, 16
    w = WL.random_case(seed=130 + T_real, T=T_real, K=K, N=N, S=S, R_max=R)
    t = w.targets[0]
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    x = torch.zeros((T_cap, K), dtype=torch.bfloat16, device=DEV)
    x[:T_real] = w.x.to(DEV)
    ids = torch.zeros(T_cap, dtype=torch.int32, device=DEV)
    ids[:T_real] = torch.from_numpy(w.ids.astype(np.int32)).to(DEV)
    plan = L.Plan(T_cap, S, R, K, device=DEV).build(ids)
    y = L.linear(x, W, pool, plan)
    torch.cuda.synchronize()
    ref = O.lora_linear(f64(w.x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, w.ids)
    assert_parity(y[:T_real], ref, f"padded {T_real} -> {T_cap}")
    assert torch.count_nonzero(y[T_real:]) == 0


# ------------------------------------------- selected rows (the LM head) ----

@pytest.mark.parametrize("T_all,T,N,S,R", [(300, 37, 1032, 9, 16), (1000, 300, 264, 12, 16)])
def test_selected_rows(T_all, T, N, S, R):
    """The layer on sampled positions only, each with its own slot; one
    selected index lies outside x and reads a zero row."""
    K = 512
    w = WL.random_case(seed=140 + T, T=T, K=K, N=N, S=S, R_max=R)
    t = w.targets[0]
    rng = np.random.default_rng(141)
    x_all = torch.from_numpy(rng.standard_normal((T_all, K), dtype=np.float32)).to(torch.bfloat16)
    sel = rng.choice(T_all, size=T, replace=False).astype(np.int32)
    sel[3] = T_all + 5                                    # outside x: a zero row
    W = t.W.to(DEV)
    pool = L.Pool(S, R, K, N, device=DEV)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    ids = torch.from_numpy(w.ids.astype(np.int32)).to(DEV)
    plan = L.Plan(T, S, R, K, device=DEV).build(ids)
    y = L.linear_rows(x_all.to(DEV), torch.from_numpy(sel).to(DEV), W, pool, plan)
    torch.cuda.synchronize()
    assert L.last_device_error() == 0
    ref = O.lora_linear_rows(f64(x_all), sel, f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, w.ids)
    assert_parity(y, ref, f"selected rows {T} of {T_all}")
    assert torch.count_nonzero(y[3]) == 0
