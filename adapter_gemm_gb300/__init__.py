"""Multi-LoRA linear layer for GB300 (sm_103a): y = x W^T + (alpha_s/r_s)(x A_s^T) B_s^T.

The compute runs in the CUDA library built from csrc/ (see build.py); `lora`
is the thin binding of its C ABI.
"""
from . import build, lora, workloads  # noqa: F401
from .lora import Plan, Pool, linear, linear_path, LoraError  # noqa: F401
