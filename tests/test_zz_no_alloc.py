"""lora_linear_static_scratch: the layer for callers that cannot allocate.

Callers that cannot call cudaMalloc (a program that owns all device memory in
its own arena, a C caller without a device allocator, a decode loop that cannot
afford the device-wide synchronization an allocation may cause) run the layer
through this entry point, which keeps the plan and the shrink result in a fixed
array inside the library. Its output must equal the planned path (lora_plan +
lora_linear with a caller-allocated workspace, the same kernels) bit for bit on
consecutive calls that share that array, and match the oracle. This file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from adapter_gemm_gb300 import lora as L
from adapter_gemm_gb300 import workloads as WL
from oracle import lora_oracle as O

from _gpu_common import assert_parity, f64

pytestmark = pytest.mark.gpu


def _static(x, W, pool, ids, y):
    T, d_in = x.shape
    return L._lib().lora_linear_static_scratch(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W.data_ptr()), T, d_in, W.shape[0],
        ctypes.byref(pool.c), ctypes.c_void_p(ids.data_ptr()) if ids.numel() else None,
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(w, dev):
    t = w.targets[0]
    x = w.x.to(dev)
    W = t.W.to(dev)
    pool = L.Pool(w.S, w.R_max, t.d_in, t.d_out, device=dev)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    return t, x, W, pool


def _two_calls_match_planned_path(w, ids_list, dev, oracle_check=True):
    """Consecutive calls share the array: each must equal the planned path
    (the same kernels over a caller-allocated workspace) bit for bit; the
    first is also checked against the oracle."""
    t, x, W, pool = _case(w, dev)
    for k, ids_np in enumerate(ids_list):
        ids = torch.from_numpy(ids_np.astype(np.int32)).to(dev)
        y = torch.empty(w.T, t.d_out, dtype=torch.bfloat16, device=dev)
        assert _static(x, W, pool, ids, y) == 0
        plan = L.Plan(w.T, w.S, w.R_max, t.d_in, device=dev).build(ids)
        ref = L.linear(x, W, pool, plan)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), f"call {k} differs from the planned path"
        if oracle_check and k == 0:
            assert_parity(y, O.lora_linear(f64(w.x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, ids_np),
                          "static scratch vs oracle")
    assert L.last_device_error() == 0


def test_static_scratch_matches_planned_path_on_consecutive_calls():
    from adapter_gemm_gb300 import build
    build.build()
    dev = torch.device("cuda")
    w = WL.q_decode()                        # T=64, 4096 -> 4096, 8 rank-16 adapters (shrink fused in)
    rng = np.random.default_rng(7)
    _two_calls_match_planned_path(w, [w.ids, rng.integers(0, w.S, size=w.T)], dev)


def test_static_scratch_at_its_limits():
    """The largest sizes the array holds (T=256 rows, 64 slots, rank cap 64):
    the shrink runs as its own kernel and U fills most of the array."""
    dev = torch.device("cuda")
    w = WL.random_case(seed=11, T=256, K=512, N=384, S=64, R_max=64)
    rng = np.random.default_rng(12)
    _two_calls_match_planned_path(w, [w.ids, rng.integers(0, w.S, size=w.T)], dev)


def test_static_scratch_empty_batch():
    dev = torch.device("cuda")
    pool = L.Pool(4, 16, 64, 64, device=dev)
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(0, dtype=torch.int32, device=dev)
    y = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    assert _static(x, W, pool, ids, y) == 0
    torch.cuda.synchronize()


def test_static_scratch_rejects_sizes_beyond_its_limit():
    dev = torch.device("cuda")
    pool = L.Pool(65, 16, 64, 64, device=dev)               # more slots than the array holds
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    ids = torch.zeros(8, dtype=torch.int32, device=dev)
    y = torch.empty(8, 64, dtype=torch.bfloat16, device=dev)
    assert L.STATUS[_static(x, W, pool, ids, y)] == "LORA_ESCRATCH"
    pool = L.Pool(4, 16, 64, 64, device=dev)
    x = torch.zeros(300, 64, dtype=torch.bfloat16, device=dev)   # more rows than it holds
    ids = torch.zeros(300, dtype=torch.int32, device=dev)
    y = torch.empty(300, 64, dtype=torch.bfloat16, device=dev)
    assert L.STATUS[_static(x, W, pool, ids, y)] == "LORA_ESCRATCH"
