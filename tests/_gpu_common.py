"""Helpers shared by the GPU parity tests: move a seeded workload to the device,
run the layer through the C ABI, and compare with the CPU oracle."""
import numpy as np
import torch

from adapter_gemm_gb300 import lora as L
from adapter_gemm_gb300 import workloads as WL
from oracle import lora_oracle as O

# max |y - ref| <= 2e-2 * (1 + |ref|) for bf16 outputs with fp32 accumulation
REL = 2e-2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


class DeviceTarget:
    def __init__(self, t: WL.Target, S: int, R_max: int, dev):
        self.t = t
        self.W = t.W.to(dev).contiguous()
        self.pool = L.Pool(S, R_max, t.d_in, t.d_out, device=dev)
        self.pool.load_padded(t.A, t.B, t.rank, t.alpha)


class DeviceWorkload:
    def __init__(self, w: WL.Workload, dev="cuda"):
        self.w = w
        self.dev = torch.device(dev)
        self.ids = torch.from_numpy(w.ids.astype(np.int32)).to(self.dev)
        self.xs = {}
        self.targets = [DeviceTarget(t, w.S, w.R_max, self.dev) for t in w.targets]
        d_cap = max(t.d_in for t in w.targets)
        self.plan = L.Plan(w.T, w.S, w.R_max, d_cap, device=self.dev)
        self.plan.build(self.ids)

    def x_for(self, i: int) -> torch.Tensor:
        t = self.w.targets[i]
        key = id(WL.input_for(self.w, t))
        if key not in self.xs:
            self.xs[key] = WL.input_for(self.w, t).to(self.dev).contiguous()
        return self.xs[key]

    def run(self, i: int = 0, base_only: bool = False) -> torch.Tensor:
        dt = self.targets[i]
        # a base-only run takes the pool too: it picks the kernel (the choice
        # weighs the pool's ranks), so slot-0 rows compare bitwise
        y = L.linear(self.x_for(i), dt.W, dt.pool, None if base_only else self.plan)
        torch.cuda.synchronize()
        return y

    def oracle(self, i: int = 0, rows=None) -> np.ndarray:
        t = self.w.targets[i]
        x = WL.input_for(self.w, t)
        return O.lora_linear(f64(x), f64(t.W), f64(t.A), f64(t.B), t.rank, t.alpha, self.w.ids, rows=rows)


def assert_parity(y: torch.Tensor, ref: np.ndarray, what: str = ""):
    yy = f64(y)
    assert yy.shape == ref.shape, (yy.shape, ref.shape)
    assert np.isfinite(yy).all(), f"{what}: non-finite output"
    err = np.abs(yy - ref)
    bound = REL * (1.0 + np.abs(ref))
    bad = err > bound
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at "
                             f"({i},{j}) y={yy[i, j]} ref={ref[i, j]} max err {err.max():.3e}")


def sample_rows(ids: np.ndarray, n: int = 96, seed: int = 0) -> np.ndarray:
    """Rows to check at full size: the first and last rows, every segment
    boundary of the sorted order, a row of every slot, plus random rows."""
    T = len(ids)
    rng = np.random.default_rng(seed)
    rows = {0, T - 1}
    for s in np.unique(ids):
        r = np.nonzero(ids == s)[0]
        rows.update([int(r[0]), int(r[-1])])
    rows.update(int(v) for v in rng.choice(T, size=min(T, n), replace=False))
    return np.array(sorted(rows))
