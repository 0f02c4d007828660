"""Attention forward on HOST buffers (fa_attention_fwd_host) on the GPU.

The host entry point runs, head group by head group, the same kernel as
fa_attention_fwd does on device tensors, so its O and lse must equal those bit
for bit; one case is also compared with the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
import workloads
from gpu_common import (ATTN_BF16_LSE_TOL, ATTN_BF16_O_TOL, device_error_clear, max_abs,
                        require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def host_inputs(shape, seed, pinned):
    Q, K, V = workloads.attention_inputs(shape, seed=seed)
    out = []
    for t in (Q, K, V):
        t = t.contiguous()
        out.append(t.pin_memory() if pinned else t)
    return out


# head counts below, at and above the number of head groups (8), and not
# multiples of it; ragged sequence lengths, long and many short sequences
@pytest.mark.parametrize("B,N,H,d,causal", [
    (2, 300, 3, 128, True),
    (1, 513, 12, 64, False),
    (2, 256, 17, 128, False),
    (1, 1, 1, 64, True),
    (3, 129, 8, 64, True),
    (1, 1100, 32, 128, True),
    (1, 4100, 2, 128, True),
    (1, 4100, 2, 64, False),
    (3, 2000, 4, 128, True),
    (3, 2000, 4, 64, False),
    (12, 1100, 2, 128, True),
    (40, 200, 2, 64, True),
    (100, 64, 1, 128, False),
])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_matches_device(dev, B, N, H, d, causal, pinned):
    Q, K, V = host_inputs((B, N, H, d), seed=B * 1000 + N + H + d, pinned=pinned)
    O_d, lse_d = fa.attention_fwd(Q.to(dev), K.to(dev), V.to(dev), causal=causal)
    torch.cuda.synchronize(dev)
    O_h, lse_h, _ = fa.attention_fwd_host(Q, K, V, causal=causal, device=dev)
    assert torch.equal(O_h.view(torch.int16), O_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())
    device_error_clear()


def test_host_full_size_matches_device(dev):
    """The benchmark's e2e call (causal B=2 H=32 N=4096 d=128, pinned buffers)."""
    w = workloads.WORKLOADS["attn_bf16_causal_b2h32n4096d128"]
    Q, K, V = (t.contiguous().pin_memory() for t in w.inputs())
    O_h, lse_h, _ = fa.attention_fwd_host(Q, K, V, causal=True, device=dev)
    O_d, lse_d = fa.attention_fwd(Q.to(dev), K.to(dev), V.to(dev), causal=True)
    torch.cuda.synchronize(dev)
    assert torch.equal(O_h.view(torch.int16), O_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())
    device_error_clear()


def test_host_against_oracle(dev):
    B, N, H, d = 2, 257, 5, 128
    Q, K, V = host_inputs((B, N, H, d), seed=77, pinned=True)
    O, lse, _ = fa.attention_fwd_host(Q, K, V, causal=True, device=dev)
    Or, lr = oracle.attention_dense(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                    1 / math.sqrt(d), True)
    assert max_abs(O.float().numpy(), Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse.numpy(), lr) <= ATTN_BF16_LSE_TOL
    device_error_clear()


def test_host_repeated_calls_share_a_workspace(dev):
    """Back-to-back calls reuse the workspace and the pipeline's events; each
    result is that call's own."""
    shape = (1, 384, 9, 64)
    ws = None
    for seed in (3, 4, 5):
        Q, K, V = host_inputs(shape, seed=seed, pinned=True)
        O_h, lse_h, ws = fa.attention_fwd_host(Q, K, V, causal=False, workspace=ws, device=dev)
        O_d, lse_d = fa.attention_fwd(Q.to(dev), K.to(dev), V.to(dev), causal=False)
        torch.cuda.synchronize(dev)
        assert torch.equal(O_h.view(torch.int16), O_d.cpu().view(torch.int16))
        assert torch.equal(lse_h, lse_d.cpu())
    device_error_clear()


def test_host_workspace_errors(dev):
    B, N, H, d = 1, 128, 2, 64
    Q, K, V = host_inputs((B, N, H, d), seed=9, pinned=False)
    O = torch.empty_like(Q)
    lse = torch.empty((B, H, N), dtype=torch.float32)
    need = fa.fa_attention_host_workspace_bytes(B, H, N, d)
    assert need > 0
    ws = torch.empty(need + 256, dtype=torch.uint8, device=dev)
    args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), lse.data_ptr(), B, H, N, d,
            0.125, 0)
    assert fa.fa_attention_fwd_host(*args, ws.data_ptr(), need - 1) == -2       # too small
    assert fa.fa_attention_fwd_host(*args, ws.data_ptr() + 16, need) == -4     # misaligned
    assert fa.fa_attention_fwd_host(*args, ws.data_ptr(), need) == 0
    torch.cuda.synchronize(dev)
    assert np.all(np.isfinite(O.float().numpy()))
    device_error_clear()
