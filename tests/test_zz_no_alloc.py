"""fa_attention_fwd_splitkv_noalloc (split-KV attention on the library's static
scratch array) against fa_attention_fwd_splitkv with caller-owned scratch,
through the C ABI.  Both run the same kernels on the same inputs with the same
split count, so their results must be equal bit for bit; each case is also
checked against the fp64 oracle (bottom-right causal alignment), so a carve-up
of the array that lands the partials in the wrong place fails even where it
stays close to the caller-scratch result.

The file name sorts last so that pytest collects it after every other test:
the static array must give correct results both in a fresh process and after
the other tests have used the library.
"""
import math

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


def inputs(B, H, Nq, Nk, d, causal, seed, dev):
    w = workloads.SplitKVWorkload("t", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, seed=seed)
    return tuple(t.to(dev) for t in w.inputs())


def call_noalloc(q, k, v, causal, splits):
    """One call of the no-allocation entry point; returns (rc, O, lse)."""
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa.fa_set_stream(torch.cuda.current_stream(q.device).cuda_stream)
    rc = fa.fa_attention_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                                             1 / math.sqrt(d), int(causal), splits)
    return rc, o, lse


def assert_oracle(q, k, v, causal, o, lse):
    """Every row of O and lse against the oracle on the same bf16 inputs."""
    d = q.shape[3]
    Or, lr = oracle.attention_qk(q.float().cpu().numpy(), k.float().cpu().numpy(),
                                 v.float().cpu().numpy(), 1 / math.sqrt(d), causal)
    err_o = max_abs(o.float().cpu().numpy(), Or)
    err_l = max_abs(lse.cpu().numpy(), lr)
    print(f"no-alloc {tuple(q.shape)} keys {k.shape[1]}: O err {err_o:.3e}, lse err {err_l:.3e}")
    assert err_o <= ATTN_BF16_O_TOL and err_l <= ATTN_BF16_LSE_TOL


def test_noalloc_two_calls_match_caller_scratch(dev):
    # call 1: the decode-like split-KV workload, split count chosen by the
    # library; call 2, right after it: another shape and split count, so the
    # array still holds call 1's partials where call 2 starts
    cases = [
        (workloads.SPLITKV_WORKLOADS["attn_bf16_splitkv_b1h16nq256nk32768d128_causal"], 0),
        (workloads.SplitKVWorkload("t", B=2, H=4, Nq=300, Nk=3000, d=64, causal=True,
                                   seed=11), 7),
    ]
    data = [(tuple(t.to(dev) for t in w.inputs()), w.causal, s) for w, s in cases]
    results = []
    for (q, k, v), causal, s in data:           # two calls in a row
        rc, o, lse = call_noalloc(q, k, v, causal, s)
        assert rc == 0, fa.strerror(rc)
        results.append((o, lse))
    torch.cuda.synchronize(dev)
    device_error_clear()
    for ((q, k, v), causal, s), (o, lse) in zip(data, results):
        o_ref, lse_ref = fa.attention_fwd_splitkv(q, k, v, causal=causal, num_splits=s)
        torch.cuda.synchronize(dev)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
        assert_oracle(q, k, v, causal, o, lse)


def test_noalloc_scratch_limit(dev):
    # non-causal d = 128, 10 key tiles, 5 splits: 5 * Nq * 129 * 4 bytes of
    # scratch; Nq = 26011 fits in 64 MiB, one more query row does not
    d, Nk, splits = 128, 1280, 5
    fits = fa.FA_NOALLOC_SCRATCH_BYTES // (splits * (d + 1) * 4)
    assert fits == 26011
    q, k, v = inputs(1, 1, fits, Nk, d, False, 21, dev)
    rc, o, lse = call_noalloc(q, k, v, False, splits)
    assert rc == 0, fa.strerror(rc)
    o_ref, lse_ref = fa.attention_fwd_splitkv(q, k, v, causal=False, num_splits=splits)
    torch.cuda.synchronize(dev)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)

    q2 = torch.cat([q, q[:, :1]], dim=1).contiguous()
    o2 = torch.full_like(q2, 7.0)
    lse2 = torch.full((1, 1, fits + 1), 7.0, dtype=torch.float32, device=dev)
    rc = fa.fa_attention_fwd_splitkv_noalloc(q2.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o2.data_ptr(), lse2.data_ptr(), 1, 1, fits + 1,
                                             Nk, d, 1 / math.sqrt(d), 0, splits)
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in fa.strerror(rc)
    torch.cuda.synchronize(dev)
    assert bool((o2 == 7.0).all()) and bool((lse2 == 7.0).all())   # nothing launched
    # one split needs no scratch
    rc, o1, lse1 = call_noalloc(q2, k, v, False, 1)
    assert rc == 0, fa.strerror(rc)
    device_error_clear()


def test_noalloc_argument_errors_match(dev):
    q = torch.zeros((1, 256, 1, 64), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 256), dtype=torch.float32, device=dev)
    p = q.data_ptr()
    # causal with fewer keys than queries, negative split count, bad d
    for args in [(1, 1, 256, 128, 64, 0.125, 1, 1), (1, 1, 256, 256, 64, 0.125, 1, -1),
                 (1, 1, 256, 256, 96, 0.125, 1, 2)]:
        a = fa.fa_attention_fwd_splitkv_noalloc(p, k.data_ptr(), k.data_ptr(), p,
                                                lse.data_ptr(), *args)
        b = fa.fa_attention_fwd_splitkv(p, k.data_ptr(), k.data_ptr(), p, lse.data_ptr(),
                                        *args, None, None)
        assert a == b < 0
    # a malformed call that would also exceed the scratch reports the
    # malformation first, as fa_attention_fwd_splitkv does: a NULL Q, then a
    # misaligned O, at 64 splits of 4096 queries (64 * 4096 * 65 * 4 bytes)
    big = (1, 1, 4096, 8192, 64, 0.125, 0, 64)
    kp = k.data_ptr()
    for qp, op_, want in ((None, p, fa.FA_ERR_NULL_POINTER), (p, p + 2, fa.FA_ERR_MISALIGNED)):
        a = fa.fa_attention_fwd_splitkv_noalloc(qp, kp, kp, op_, lse.data_ptr(), *big)
        b = fa.fa_attention_fwd_splitkv(qp, kp, kp, op_, lse.data_ptr(), *big, p, lse.data_ptr())
        assert a == b == want
