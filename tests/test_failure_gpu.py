"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait of the attention kernels is bounded.  A wait that gives up
sets FA_DEVERR_WAIT_TIMEOUT in the device error word and raises the CTA's abort
flag; the other roles then leave their loops, the copies and tensor-core work
already issued are waited for, tensor memory is freed, and the CTA exits.
fa_debug_expire_next_wait makes one launch wait, with a short bound, on a
barrier that nothing arrives at (a flag nothing sets), so that this path runs
for real; the test checks the error word, that the context is still usable
and that the next call on the same stream matches the oracle.
"""
import math
import time

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
import workloads
from gpu_common import ATTN_BF16_LSE_TOL, ATTN_BF16_O_TOL, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


@pytest.mark.parametrize("N,d,causal", [(256, 128, True), (300, 64, False), (1000, 128, True)])
def test_expired_wait_is_reported_and_the_next_call_is_correct(dev, N, d, causal):
    B, H = 2, 3
    Q, K, V = workloads.attention_inputs((B, N, H, d), seed=N + d)
    q, k, v = (t.to(dev) for t in (Q, K, V))
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    assert fa.fa_get_device_error() == 0
    o = torch.full_like(q, 3.0)
    lse = torch.full((B, H, N), 3.0, dtype=torch.float32, device=dev)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            1 / math.sqrt(d), int(causal), None)
    assert fa.fa_debug_expire_next_wait(20_000) == 0          # 20 us
    t0 = time.perf_counter()
    assert fa.fa_attention_fwd(*args) == 0
    torch.cuda.synchronize(dev)
    elapsed = time.perf_counter() - t0
    assert fa.fa_get_device_error() == fa.FA_DEVERR_WAIT_TIMEOUT
    assert fa.fa_get_device_error() == 0                       # read and cleared
    # the aborted launch wrote nothing and ended well before any 2 s bound
    assert bool((o == 3.0).all()) and bool((lse == 3.0).all())
    assert elapsed < 1.5, elapsed
    # the switch was one-shot: the next call on the same stream runs normally
    assert fa.fa_attention_fwd(*args) == 0
    torch.cuda.synchronize(dev)
    assert fa.fa_get_device_error() == 0
    Or, lr = oracle.attention_dense(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                    1 / math.sqrt(d), causal)
    assert max_abs(o.float().cpu().numpy(), Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse.cpu().numpy(), lr) <= ATTN_BF16_LSE_TOL


BWD_TOL = 2.0 ** -6          # the one-pass backward's parity bound (normwise)


def _normwise(g, ref):
    return float(np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-3))


@pytest.mark.parametrize("packed,lens,d,causal", [
    (False, (256, 256), 128, True),       # dense B=2: two or four 64-query steps per CTA
    (False, (300, 300), 64, False),       # dense B=2, d = 64 (zero rows of K^T)
    (False, (1000, 1000), 128, True),     # dense B=2: up to 16 steps, the 3-stage ring wraps
    (True, (1, 129, 700, 0, 64), 128, True),   # packed: ragged, one token, an empty sequence
])
def test_expired_wait_in_one_pass_backward(dev, packed, lens, d, causal):
    """The same switch on the one-pass backward: its tensor-core warp gives up,
    the row warps and the copy warp leave their loops, dK and dV stay
    unwritten, dQ is converted from an accumulator that received nothing
    (zero), and the next call matches the oracle."""
    H = 3
    B, N = len(lens), max(lens)
    cu = workloads.cu_seqlens_of(lens)
    total = int(cu[-1])
    shape = (total, H, d) if packed else (B, N, H, d)
    Q, K, V = workloads.attention_inputs(shape, seed=7 * N + d)
    dO = workloads.attention_inputs(shape, seed=7 * N + d + 1)[0]
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    cu_d = torch.from_numpy(cu).to(dev) if packed else None
    if packed:
        o, lse = fa.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu_d, max_seqlen=N)
        nbytes = fa.fa_attention_bwd_atomic_varlen_workspace_bytes(B, H, N, total, d)
        lse_shape = (H, total)
    else:
        o, lse = fa.attention_fwd(q, k, v, causal=causal)
        nbytes = fa.fa_attention_bwd_atomic_workspace_bytes(B, H, N, d)
        lse_shape = (B, H, N)
    torch.cuda.synchronize(dev)
    assert nbytes > 0 and fa.fa_get_device_error() == 0
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    d_buf = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.full_like(q, 3.0) for _ in range(3))
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), d_buf.data_ptr())

    def call():
        if packed:
            return fa.fa_attention_bwd_atomic_varlen(*ptrs, B, H, N, total, d, 1 / math.sqrt(d),
                                                     int(causal), cu_d.data_ptr(),
                                                     ws.data_ptr(), nbytes)
        return fa.fa_attention_bwd_atomic(*ptrs, B, H, N, d, 1 / math.sqrt(d), int(causal),
                                          ws.data_ptr(), nbytes)

    assert fa.fa_debug_expire_next_wait(20_000) == 0          # 20 us
    t0 = time.perf_counter()
    assert call() == 0
    torch.cuda.synchronize(dev)
    elapsed = time.perf_counter() - t0
    assert fa.fa_get_device_error() == fa.FA_DEVERR_WAIT_TIMEOUT
    assert fa.fa_get_device_error() == 0                       # read and cleared
    assert bool((dk == 3.0).all()) and bool((dv == 3.0).all())
    assert bool((dq == 0.0).all())
    assert elapsed < 1.5, elapsed
    # one-shot: the next call on the same stream runs normally
    assert call() == 0
    torch.cuda.synchronize(dev)
    assert fa.fa_get_device_error() == 0
    args = [t.float().numpy() for t in (Q, K, V, dO)]
    if packed:
        ref = oracle.attention_bwd_packed(*args, cu, 1 / math.sqrt(d), causal)
    else:
        ref = oracle.attention_bwd(*args, 1 / math.sqrt(d), causal)
    for name, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
        e = _normwise(g.float().cpu().numpy(), ref[name])
        assert e <= BWD_TOL, f"{name}: {e}"
