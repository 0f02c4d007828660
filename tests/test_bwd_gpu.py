"""Attention backward (dQ, dK, dV) on the GPU, through the C ABI, against the
fp64 oracle's gradients of sum(dO * O).

The GPU backward takes O and lse from the library's own bf16 forward; the
oracle recomputes everything from the same bf16 Q, K, V, dO in double.

Tolerance (normwise, per gradient tensor): max |g - g_ref| <= BWD_TOL *
max |g_ref|.  The kernels round P and dS to bf16 before the products that
use them and the gradients to bf16 at the end (unit roundoff u = 2^-9 each);
D_i uses the bf16 O.  Each gradient element is a sum of terms rounded with
relative error <= u, so its error is at most ~2u times the sum of the terms'
magnitudes, which for these inputs stays within a few times the largest
gradient magnitude: BWD_TOL = 2^-6 (8u).  Observed: 0.002-0.005 on the small
shapes, <= 0.011 on the full-size rows.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
from gpu_common import device_error_clear, require_gpu

pytestmark = pytest.mark.gpu

BWD_TOL = 2.0 ** -6


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def make_inputs(B, H, N, d, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(4):
        x = rng.standard_normal((B, N, H, d)).astype(np.float32)
        out.append(torch.from_numpy(x).to(torch.bfloat16))
    return out   # Q, K, V, dO (bf16, CPU)


def run_gpu(Q, K, V, dO, causal, dev):
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    o, lse = fa.attention_fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=causal)
    torch.cuda.synchronize(dev)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


def normwise(g, ref):
    return float(np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 128, 64, False),
    (2, 2, 256, 128, True),
    (1, 3, 300, 128, True),      # ragged last tile
    (2, 2, 200, 64, False),      # ragged, batch rows follow each other
    (1, 1, 1, 64, True),         # one token
    (1, 2, 385, 128, False),
    (2, 1, 640, 64, True),
    (1, 2, 192, 128, True),      # last tile exactly one 64-row sub-tile
    (1, 1, 65, 64, True),        # two sub-tiles, one tile
    (1, 2, 1000, 128, True),     # up to 8 key steps of the dQ pass: its ring wraps, ragged end
    (2, 1, 900, 64, False),      # the same at d = 64, non-causal, two sequences
])
def test_bwd_matches_oracle(dev, B, H, N, d, causal):
    Q, K, V, dO = make_inputs(B, H, N, d, seed=N * 7 + d + B)
    dq, dk, dv = run_gpu(Q, K, V, dO, causal, dev)
    ref = oracle.attention_bwd(*(t.float().numpy() for t in (Q, K, V, dO)), 1 / math.sqrt(d),
                               causal)
    errs = {name: normwise(g, ref[name]) for name, g in (("dQ", dq), ("dK", dk), ("dV", dv))}
    print(f"B{B} H{H} N{N} d{d} causal={causal}: normwise errors {errs}")
    for name, e in errs.items():
        assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def test_bwd_full_size_sampled(dev):
    """The benchmark's backward workload (causal B=2 H=32 N=4096 d=128): every
    gradient of sampled query rows and keys of two heads against the oracle."""
    B, H, N, d = 2, 32, 4096, 128
    Q, K, V, dO = make_inputs(B, H, N, d, seed=4242)
    dq, dk, dv = run_gpu(Q, K, V, dO, True, dev)
    Qf, Kf, Vf, dOf = (t.float().numpy() for t in (Q, K, V, dO))
    rng = np.random.default_rng(7)
    for (b, h) in [(0, 3), (1, 30)]:
        qi = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 20)]))
        ki = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 20)]))
        rq, rk, rv = oracle.attention_bwd_head(Qf, Kf, Vf, dOf, 1 / math.sqrt(d), True, b, h,
                                               qi, ki)
        for name, g, ref in (("dQ", dq[b, qi, h], rq), ("dK", dk[b, ki, h], rk),
                             ("dV", dv[b, ki, h], rv)):
            e = normwise(g, ref)
            print(f"full size (b={b}, h={h}) {name}: normwise error {e}")
            assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def run_gpu_packed(Q, K, V, dO, cu, max_len, causal, dev):
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    cu_d = torch.from_numpy(np.asarray(cu, np.int32)).to(dev)
    o, lse = fa.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu_d, max_seqlen=max_len)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, cu_seqlens=cu_d,
                                  max_seqlen=max_len)
    torch.cuda.synchronize(dev)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lens", [[1, 129, 300, 64, 257, 0, 128, 700], [1000, 3]])
def test_bwd_packed_matches_oracle(dev, lens, d, causal):
    """Packed sequences (lengths not multiples of the tiles, an empty one, one
    token, the dQ pass's ring wrapping): every gradient against the oracle's
    per-sequence backward."""
    import workloads
    cu = workloads.cu_seqlens_of(lens)
    total, H = int(cu[-1]), 3
    rng = np.random.default_rng(sum(lens) + d + causal)
    Q, K, V, dO = (torch.from_numpy(rng.standard_normal((total, H, d)).astype(np.float32))
                   .to(torch.bfloat16) for _ in range(4))
    dq, dk, dv = run_gpu_packed(Q, K, V, dO, cu, max(lens), causal, dev)
    ref = oracle.attention_bwd_packed(*(t.float().numpy() for t in (Q, K, V, dO)), cu,
                                      1 / math.sqrt(d), causal)
    errs = {name: normwise(g, ref[name]) for name, g in (("dQ", dq), ("dK", dk), ("dV", dv))}
    print(f"packed {lens} d{d} causal={causal}: normwise errors {errs}")
    for name, e in errs.items():
        assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def test_bwd_packed_equal_lengths_is_the_dense_call(dev):
    """Packed sequences of one length give the dense call's bits (the same
    kernels on the same rows; only the statistics' layout differs)."""
    B, H, N, d = 2, 2, 300, 128
    Q, K, V, dO = make_inputs(B, H, N, d, seed=17)
    dense = run_gpu(Q, K, V, dO, True, dev)
    cu = np.arange(B + 1, dtype=np.int32) * N
    packed = run_gpu_packed(*(t.reshape(B * N, H, d) for t in (Q, K, V, dO)), cu, N, True, dev)
    for x, y in zip(dense, packed):
        assert np.array_equal(x.reshape(B * N, H, d), y)


def test_bwd_packed_length_over_n_is_flagged(dev):
    """A sequence longer than N is flagged in the device error word and not
    computed (no access past the tensors)."""
    H, d = 1, 64
    q = torch.zeros((300, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((H, 300), dtype=torch.float32, device=dev)
    cu = torch.tensor([0, 300], dtype=torch.int32, device=dev)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    p, l = q.data_ptr(), lse.data_ptr()
    rc = fa.fa_attention_bwd_varlen(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, d, 0.125, 1,
                                    cu.data_ptr())
    assert rc == 0
    assert fa.fa_get_device_error() == fa.FA_DEVERR_BAD_SEQLENS
    assert fa.fa_get_device_error() == 0
    assert fa.fa_attention_bwd_varlen(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, d, 0.125, 1,
                                      None) == fa.FA_ERR_NULL_POINTER


def test_bwd_deterministic(dev):
    """No atomics: two runs give identical bits."""
    Q, K, V, dO = make_inputs(2, 2, 512, 128, seed=9)
    a = run_gpu(Q, K, V, dO, True, dev)
    b = run_gpu(Q, K, V, dO, True, dev)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_bad_arguments(dev):
    q = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    p, l = q.data_ptr(), lse.data_ptr()
    assert fa.fa_attention_bwd(p, p, p, p, p, l, p, p, p, l, 1, 1, 128, 96, 0.1, 0) == -3
    assert fa.fa_attention_bwd(p, p, p, p, p, l, p, p, p, None, 1, 1, 128, 64, 0.1, 0) == -1
    assert fa.fa_attention_bwd(p + 2, p, p, p, p, l, p, p, p, l, 1, 1, 128, 64, 0.1, 0) == -4
    assert fa.fa_attention_bwd(p, p, p, p, p, l, p, p, p, l, -1, 1, 128, 64, 0.1, 0) == -2
