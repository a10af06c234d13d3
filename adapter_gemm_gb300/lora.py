"""Python binding of the C ABI in include/lora_gb300.h (argument marshalling only).

Every step of the layer runs in the CUDA library; this module allocates the
caller-owned buffers with PyTorch (device memory and streams are all PyTorch is
used for), passes raw pointers, and turns status codes into exceptions. There
is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_int32 = ctypes.c_int32
_c_size_t = ctypes.c_size_t

STATUS = {
    0: "LORA_OK", -1: "LORA_EINVAL", -2: "LORA_ESLOT", -3: "LORA_ERANK", -4: "LORA_ESHAPE",
    -5: "LORA_ENONFINITE", -6: "LORA_ECUDA", -7: "LORA_EIDRANGE", -8: "LORA_ESPACE",
    -9: "LORA_ETIMEOUT", -10: "LORA_ESCRATCH",
}
TILE_ROWS = 128


class LoraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({_lib().lora_strerror(status).decode()})")


class lora_pool(ctypes.Structure):
    _fields_ = [("A", _c_void_p), ("B", _c_void_p), ("scale", _c_void_p), ("rank", _c_void_p),
                ("work", _c_void_p), ("S", _c_int32), ("R_max", _c_int32), ("d_in", _c_int32),
                ("d_out", _c_int32)]


class lora_plan_t(ctypes.Structure):
    _fields_ = [("slot_of_token", _c_void_p), ("token_order", _c_void_p), ("counts", _c_void_p),
                ("indptr", _c_void_p), ("active", _c_void_p), ("n_active", _c_void_p),
                ("tiles", _c_void_p), ("n_tiles", _c_void_p), ("n_invalid", _c_void_p),
                ("U", _c_void_p), ("x_sorted", _c_void_p), ("ids", _c_void_p), ("U_hl", _c_void_p),
                ("mt_ptr", _c_void_p), ("mt_seg", _c_void_p), ("T", _c_int32), ("S", _c_int32),
                ("R_max", _c_int32), ("d_in_cap", _c_int32), ("max_tiles", _c_int32)]


_LIB = None

# name -> (restype, argtypes); mirrors the header.
_SIGS = {
    "lora_plan_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "lora_plan_init": (_c_int, [ctypes.POINTER(lora_plan_t), _c_void_p, _c_size_t, _c_int, _c_int, _c_int, _c_int]),
    "lora_pool_init": (_c_int, [ctypes.POINTER(lora_pool), _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "lora_pool_install": (_c_int, [ctypes.POINTER(lora_pool), _c_int, _c_void_p, _c_void_p, ctypes.c_float,
                                   _c_int, _c_void_p]),
    "lora_plan": (_c_int, [_c_void_p, _c_int, ctypes.POINTER(lora_plan_t), _c_void_p]),
    "lora_plan_check": (_c_int, [ctypes.POINTER(lora_plan_t), _c_void_p, ctypes.POINTER(_c_int32)]),
    "lora_linear": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, ctypes.POINTER(lora_pool),
                             ctypes.POINTER(lora_plan_t), _c_void_p, _c_void_p]),
    "lora_linear_path": (_c_int, [_c_int, _c_int, _c_int]),
    "lora_linear_path_for": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "lora_linear_kernel_for": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "lora_linear_rows": (_c_int, [_c_void_p, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                  ctypes.POINTER(lora_pool), ctypes.POINTER(lora_plan_t), _c_void_p, _c_void_p,
                                  _c_void_p]),
    "lora_linear_host": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                  ctypes.POINTER(lora_pool), ctypes.POINTER(lora_plan_t), _c_void_p, _c_void_p,
                                  _c_void_p, _c_void_p]),
    "lora_linear_sliced": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, ctypes.POINTER(_c_int32),
                                    ctypes.POINTER(ctypes.POINTER(lora_pool)), ctypes.POINTER(lora_plan_t),
                                    _c_void_p, _c_void_p]),
    "lora_profile_gemm_events": (_c_int, [_c_void_p, _c_void_p]),
    "lora_linear_static_scratch": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, ctypes.POINTER(lora_pool),
                                            _c_void_p, _c_void_p, _c_void_p]),
    "lora_last_device_error": (_c_int, [ctypes.POINTER(_c_int32)]),
    "lora_strerror": (ctypes.c_char_p, [_c_int]),
    "lora_version": (_c_int, []),
    "lora_launch_count": (ctypes.c_uint64, []),
}


def library_path() -> str:
    return _build.LIB


def _lib():
    """Load the CUDA library (building it in-tree first if it is missing)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


def header_functions() -> list:
    """Names of the functions include/lora_gb300.h declares."""
    with open(os.path.join(_build.INCLUDE, "lora_gb300.h")) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(lora_\w+)\s*\(", text, re.M)))


def _check(status: int, what: str):
    if status != 0:
        raise LoraError(status, what)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return _c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return _c_void_p(t.data_ptr())


def launch_count() -> int:
    """Kernels the library has launched (or captured) so far in this process."""
    return int(_lib().lora_launch_count())


def version() -> int:
    return _lib().lora_version()


def linear_path(T: int, d_in: int, d_out: int, pool: "Pool | None" = None) -> int:
    """Kernel family a call takes: 0 skinny (decode), 1 wide (prefill); with a
    pool, the rank-aware choice for its S and R_max."""
    if pool is not None:
        return _lib().lora_linear_path_for(T, d_in, d_out, pool.S, pool.R_max)
    return _lib().lora_linear_path(T, d_in, d_out)


def kernel_for(T: int, d_in: int, d_out: int, pool: "Pool | None" = None) -> int:
    """Kernel a call runs: 0 skinny (decode), 1 wide (prefill), 2 wide on CTA
    pairs; with a pool, for its S and R_max."""
    S, R = (pool.S, pool.R_max) if pool is not None else (0, 0)
    return _lib().lora_linear_kernel_for(T, d_in, d_out, S, R)


def plan_workspace_bytes(T: int, S: int, R_max: int, d_in_cap: int) -> int:
    return _lib().lora_plan_workspace_bytes(T, S, R_max, d_in_cap)


class Pool:
    """A device slot pool for one adapted linear (A [S,R,d_in], B [S,d_out,R] bf16)."""

    def __init__(self, S: int, R_max: int, d_in: int, d_out: int, device=None, stream=None):
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.A = torch.empty((S, R_max, d_in), dtype=torch.bfloat16, device=dev)
        self.B = torch.empty((S, d_out, R_max), dtype=torch.bfloat16, device=dev)
        self.scale = torch.empty((S,), dtype=torch.float32, device=dev)
        self.rank = torch.empty((S,), dtype=torch.int32, device=dev)
        self.work = torch.empty((4,), dtype=torch.int32, device=dev)
        self.S, self.R_max, self.d_in, self.d_out = S, R_max, d_in, d_out
        self.c = lora_pool()
        _check(_lib().lora_pool_init(ctypes.byref(self.c), _ptr(self.A), _ptr(self.B), _ptr(self.scale),
                                     _ptr(self.rank), _ptr(self.work), S, R_max, d_in, d_out,
                                     _stream(stream)), "lora_pool_init")

    def install(self, slot: int, A: torch.Tensor, B: torch.Tensor, alpha: float, stream=None):
        """Load A [rank, d_in] and B [d_out, rank] (bf16, unscaled) into `slot`."""
        if A.dim() != 2 or B.dim() != 2 or A.shape[1] != self.d_in or B.shape[0] != self.d_out \
                or A.shape[0] != B.shape[1]:
            raise ValueError("install wants A [rank, d_in] and B [d_out, rank]")
        _check(_lib().lora_pool_install(ctypes.byref(self.c), int(slot), _ptr(A, torch.bfloat16, "A"),
                                        _ptr(B, torch.bfloat16, "B"), float(alpha), int(A.shape[0]),
                                        _stream(stream)), "lora_pool_install")

    def load_padded(self, A_pool: torch.Tensor, B_pool: torch.Tensor, ranks, alphas, stream=None):
        """Install every slot s >= 1 with rank > 0 from padded host/device pools."""
        dev = self.A.device
        for s in range(1, self.S):
            r = int(ranks[s])
            if r == 0:
                continue
            a = A_pool[s, :r].to(dev).contiguous()
            b = B_pool[s, :, :r].to(dev).contiguous()
            self.install(s, a, b, float(alphas[s]), stream)


class Plan:
    """The per-step plan and its scratch, in one caller-owned device workspace."""

    def __init__(self, T: int, S: int, R_max: int, d_in_cap: int, device=None):
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        n = plan_workspace_bytes(T, S, R_max, d_in_cap)
        if n == 0 and T >= 0:
            raise LoraError(-1, "lora_plan_workspace_bytes")
        self.workspace = torch.empty((max(n, 256),), dtype=torch.uint8, device=dev)
        self.T, self.S, self.R_max, self.d_in_cap = T, S, R_max, d_in_cap
        self.c = lora_plan_t()
        _check(_lib().lora_plan_init(ctypes.byref(self.c), _ptr(self.workspace), n, T, S, R_max, d_in_cap),
               "lora_plan_init")

    def build(self, ids: torch.Tensor, stream=None):
        """Build the plan from the step's token slot ids ([T] int32 CUDA)."""
        if ids.numel() != self.T:
            raise ValueError("ids length must equal the plan's T")
        self.ids = ids          # the plan records this buffer's address; keep it alive
        _check(_lib().lora_plan(_ptr(ids, torch.int32, "ids") if self.T else None, self.T,
                                ctypes.byref(self.c), _stream(stream)), "lora_plan")
        return self

    def check(self, stream=None) -> int:
        """Synchronise and return how many ids were outside [0, S)."""
        n = _c_int32(0)
        st = _lib().lora_plan_check(ctypes.byref(self.c), _stream(stream), ctypes.byref(n))
        if st not in (0, -7):
            _check(st, "lora_plan_check")
        return int(n.value)

    def _view(self, field: str, count: int, dtype=torch.int32) -> torch.Tensor:
        p = getattr(self.c, field)
        if p is None or count == 0:
            return torch.empty((0,), dtype=dtype, device=self.workspace.device)
        off = p - self.workspace.data_ptr()
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)

    # read-only views of the plan arrays (valid after build, stream-ordered)
    def slot_of_token(self): return self._view("slot_of_token", self.T)
    def token_order(self): return self._view("token_order", self.T)
    def counts(self): return self._view("counts", self.S)
    def indptr(self): return self._view("indptr", self.S + 1)
    def n_active(self): return int(self._view("n_active", 1).item())
    def active(self): return self._view("active", self.S)[: self.n_active()]
    def n_tiles(self): return int(self._view("n_tiles", 1).item())
    def tiles(self): return self._view("tiles", 4 * self.c.max_tiles).view(-1, 4)[: self.n_tiles()]
    def n_invalid(self): return int(self._view("n_invalid", 1).item())
    def U(self): return self._view("U", self.T * self.R_max, torch.float32).view(self.T, self.R_max)


def linear(x: torch.Tensor, W: torch.Tensor, pool: Pool | None = None, plan: Plan | None = None,
           y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = x W^T + per-row adapter correction (plan=None: base projection only,
    on the kernel a call with this pool would take)."""
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError("x [T, d_in] and W [d_out, d_in] expected")
    T, d_in = x.shape
    d_out = W.shape[0]
    if y is None:
        y = torch.empty((T, d_out), dtype=torch.bfloat16, device=x.device)
    if plan is not None and pool is None:
        raise ValueError("a plan needs a pool")
    _check(_lib().lora_linear(_ptr(x, torch.bfloat16, "x"), _ptr(W, torch.bfloat16, "W"), T, d_in, d_out,
                              ctypes.byref(pool.c) if pool is not None else None,
                              ctypes.byref(plan.c) if plan is not None else None,
                              _ptr(y, torch.bfloat16, "y"), _stream(stream)), "lora_linear")
    return y


def linear_rows(x_all: torch.Tensor, rows: torch.Tensor, W: torch.Tensor, pool: Pool | None = None,
                plan: Plan | None = None, x_rows: torch.Tensor | None = None, y: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """The layer on rows `rows` ([T] int32 CUDA) of x_all [T_all, d_in]: y [T,
    d_out], with the plan built for those rows' slots."""
    T_all, d_in = x_all.shape
    T = rows.numel()
    d_out = W.shape[0]
    if x_rows is None:
        x_rows = torch.empty((T, d_in), dtype=torch.bfloat16, device=x_all.device)
    if y is None:
        y = torch.empty((T, d_out), dtype=torch.bfloat16, device=x_all.device)
    if plan is not None and pool is None:
        raise ValueError("a plan needs a pool")
    _check(_lib().lora_linear_rows(_ptr(x_all, torch.bfloat16, "x_all"), T_all, _ptr(rows, torch.int32, "rows"), T,
                                   d_in, d_out, _ptr(W, torch.bfloat16, "W"),
                                   ctypes.byref(pool.c) if pool is not None else None,
                                   ctypes.byref(plan.c) if plan is not None else None,
                                   _ptr(x_rows, torch.bfloat16, "x_rows"), _ptr(y, torch.bfloat16, "y"),
                                   _stream(stream)), "lora_linear_rows")
    return y


def linear_host(x_host: torch.Tensor, W: torch.Tensor, y_host: torch.Tensor, x_dev: torch.Tensor,
                y_dev: torch.Tensor, pool: Pool | None = None, plan: Plan | None = None,
                ids_host: torch.Tensor | None = None, ids_dev: torch.Tensor | None = None, stream=None):
    """The layer on host buffers (pinned CPU tensors x_host [T, d_in], y_host
    [T, d_out], ids_host [T] int32): copies in, plan, layer, copy out, all
    queued on the stream, through the device staging tensors x_dev, ids_dev,
    y_dev."""
    if x_host.device.type != "cpu" or y_host.device.type != "cpu":
        raise ValueError("x_host and y_host must be host tensors")
    T, d_in = x_host.shape
    d_out = W.shape[0]
    if plan is not None:
        if pool is None or ids_host is None or ids_dev is None:
            raise ValueError("a plan needs a pool, ids_host and ids_dev")
        if ids_host.dtype != torch.int32 or not ids_host.is_contiguous():
            raise ValueError("ids_host must be contiguous int32")
        plan.ids = ids_dev
    for nm, t, dt in (("x_host", x_host, torch.bfloat16), ("y_host", y_host, torch.bfloat16)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous {dt}")
    _check(_lib().lora_linear_host(_c_void_p(x_host.data_ptr()),
                                   _c_void_p(ids_host.data_ptr()) if plan is not None else None,
                                   _c_void_p(y_host.data_ptr()), T, d_in, d_out, _ptr(W, torch.bfloat16, "W"),
                                   ctypes.byref(pool.c) if pool is not None else None,
                                   ctypes.byref(plan.c) if plan is not None else None,
                                   _ptr(x_dev, torch.bfloat16, "x_dev"),
                                   _ptr(ids_dev, torch.int32, "ids_dev") if plan is not None else None,
                                   _ptr(y_dev, torch.bfloat16, "y_dev"), _stream(stream)), "lora_linear_host")
    return y_host


def linear_sliced(x: torch.Tensor, W: torch.Tensor, d_outs, pools=None, plan: Plan | None = None,
                  y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Projections that share x: W [sum(d_outs), d_in] stacks the slices'
    weights, pools[i] holds slice i's adapters; y [T, sum(d_outs)] gets each
    slice's outputs in its columns (plan=None: base projection only)."""
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError("x [T, d_in] and W [N, d_in] expected")
    d_outs = [int(d) for d in d_outs]
    if sum(d_outs) != W.shape[0]:
        raise ValueError("the slices' d_out must add up to W's rows")
    T, d_in = x.shape
    if y is None:
        y = torch.empty((T, W.shape[0]), dtype=torch.bfloat16, device=x.device)
    if plan is not None and (pools is None or len(pools) != len(d_outs)):
        raise ValueError("a plan needs one pool per slice")
    n = len(d_outs)
    douts = (_c_int32 * n)(*d_outs)
    pptrs = (ctypes.POINTER(lora_pool) * n)(*[ctypes.pointer(p.c) for p in pools]) if plan is not None else None
    _check(_lib().lora_linear_sliced(_ptr(x, torch.bfloat16, "x"), _ptr(W, torch.bfloat16, "W"), T, d_in, n, douts,
                                     pptrs, ctypes.byref(plan.c) if plan is not None else None,
                                     _ptr(y, torch.bfloat16, "y"), _stream(stream)), "lora_linear_sliced")
    return y


def profile_gemm_events(start=None, stop=None):
    """Record torch.cuda.Event `start`/`stop` around each following GEMM launch
    (None, None: off)."""
    a = _c_void_p(start.cuda_event) if start is not None else None
    b = _c_void_p(stop.cuda_event) if stop is not None else None
    _check(_lib().lora_profile_gemm_events(a, b), "lora_profile_gemm_events")


def last_device_error() -> int:
    """Synchronise; return and clear the kernels' bounded-wait error word."""
    code = _c_int32(0)
    st = _lib().lora_last_device_error(ctypes.byref(code))
    if st not in (0, -9):
        _check(st, "lora_last_device_error")
    return int(code.value)
