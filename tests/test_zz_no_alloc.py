"""lora_linear_static_scratch: the layer for callers that cannot allocate.

Callers that cannot call cudaMalloc (a program that owns all device memory in
its own arena, a C caller without a device allocator, a decode loop that cannot
afford the device-wide synchronization an allocation may cause) run the layer
through this entry point, which keeps the plan and the shrink result in a fixed
array inside the library. Its output must match the planned path
(lora_plan + lora_linear with a caller-allocated workspace) on consecutive calls
that share that array. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from adapter_gemm_gb300 import lora as L
from adapter_gemm_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

REL = 2e-2          # |y - ref| <= 2e-2 * (1 + |ref|), as in the parity tests


def _static(x, W, pool, ids, y):
    T, d_in = x.shape
    return L._lib().lora_linear_static_scratch(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W.data_ptr()), T, d_in, W.shape[0],
        ctypes.byref(pool.c), ctypes.c_void_p(ids.data_ptr()) if ids.numel() else None,
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a: torch.Tensor, b: torch.Tensor):
    a64, b64 = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.isfinite(a64).all()
    assert (np.abs(a64 - b64) <= REL * (1 + np.abs(b64))).all(), np.abs(a64 - b64).max()


def test_static_scratch_matches_planned_path_on_consecutive_calls():
    from adapter_gemm_gb300 import build
    build.build()
    dev = torch.device("cuda")
    w = WL.q_decode()                        # T=64, 4096 -> 4096, 8 rank-16 adapters
    t = w.targets[0]
    x = w.x.to(dev)
    W = t.W.to(dev)
    pool = L.Pool(w.S, w.R_max, t.d_in, t.d_out, device=dev)
    pool.load_padded(t.A, t.B, t.rank, t.alpha)
    ids_a = torch.from_numpy(w.ids).to(dev)
    rng = np.random.default_rng(7)
    ids_b = torch.from_numpy(rng.integers(0, w.S, size=w.T).astype(np.int32)).to(dev)
    for ids in (ids_a, ids_b):               # two calls in a row share the array
        y = torch.empty(w.T, t.d_out, dtype=torch.bfloat16, device=dev)
        assert _static(x, W, pool, ids, y) == 0
        plan = L.Plan(w.T, w.S, w.R_max, t.d_in, device=dev).build(ids)
        ref = L.linear(x, W, pool, plan)
        torch.cuda.synchronize()
        _close(y, ref)
    assert L.last_device_error() == 0


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
