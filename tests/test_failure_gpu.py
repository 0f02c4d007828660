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
