"""Helpers shared by the GPU parity tests (tests marked ``gpu``)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa

# Tolerances against the fp64 oracle (max absolute error):
SOFTMAX_F32_TOL = 1e-5      # fp32 row softmax
ATTN_F32_O_TOL = 1e-4       # fp32 attention output
ATTN_F32_LSE_TOL = 1e-4     # fp32 attention logsumexp
ATTN_BF16_O_TOL = 2e-2      # bf16 attention output (oracle on the same bf16 inputs)
ATTN_BF16_LSE_TOL = 1e-3    # bf16 attention logsumexp


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fa.lib()   # raises if the library is missing: no fallback exists
    return torch.device("cuda", 0)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.size == 0:
        return 0.0
    assert np.all(np.isfinite(a)), "non-finite GPU output"
    return float(np.max(np.abs(a - b)))


def device_error_clear():
    """The kernels raised no error bit since the last check (and clears it)."""
    code = fa.fa_get_device_error()
    assert code == 0, f"device error word = {code:#x}"
