"""Attention forward on the GPU (through the C ABI) against the fp64 oracle.

Every case, the full-size workloads included, is compared element by element
on every (token, head) row of O and lse, plus properties that hold at any
size.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
import workloads
from gpu_common import (ATTN_BF16_LSE_TOL, ATTN_BF16_O_TOL, ATTN_F32_LSE_TOL, ATTN_F32_O_TOL,
                        device_error_clear, max_abs, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _to_dev(t, dev):
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(t)
    return t.contiguous().to(dev)


def gpu_dense(Q, K, V, causal, dev, scale=None):
    q, k, v = (_to_dev(t, dev) for t in (Q, K, V))
    O, lse = fa.attention_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize(dev)
    return O.float().cpu().numpy(), lse.cpu().numpy()


def gpu_packed(Q, K, V, cu, max_len, causal, dev, via_readback=False):
    q, k, v = (_to_dev(t, dev) for t in (Q, K, V))
    cu_d = torch.from_numpy(np.asarray(cu, np.int32)).to(dev)
    if via_readback:
        # the spec entry point: total is read back from cu_seqlens[B]
        O = torch.empty_like(q)
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
        fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
        f = fa.fa_attention_fwd if q.dtype == torch.bfloat16 else fa.fa_attention_fwd_f32
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), lse.data_ptr(),
               len(cu) - 1, q.shape[1], int(max_len), q.shape[2], 1 / math.sqrt(q.shape[2]),
               int(causal), cu_d.data_ptr())
        assert rc == 0, fa.strerror(rc)
    else:
        O, lse = fa.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu_d, max_seqlen=max_len)
    torch.cuda.synchronize(dev)
    return O.float().cpu().numpy(), lse.cpu().numpy()


def f32(t):
    return t.float().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float32)


# ---------------------------------------------------------------------------
# fp32 path
# ---------------------------------------------------------------------------

def test_f32_single_head_workload(dev):
    w = workloads.WORKLOADS["attn_f32_b1h1n256d64"]
    Q, K, V = w.inputs()
    O, lse = gpu_dense(Q, K, V, w.causal, dev)
    Or, lr = oracle.attention_dense(Q, K, V, w.scale, w.causal)
    assert max_abs(O, Or) <= ATTN_F32_O_TOL
    assert max_abs(lse, lr) <= ATTN_F32_LSE_TOL
    device_error_clear()


@pytest.mark.parametrize("N,d,causal", [(1, 64, False), (7, 32, True), (129, 64, True),
                                        (300, 128, False), (300, 100, True), (77, 17, False)])
def test_f32_shapes(dev, N, d, causal):
    Q, K, V = workloads.attention_inputs((2, N, 3, d), seed=N * 7 + d, dtype="f32")
    O, lse = gpu_dense(Q, K, V, causal, dev)
    Or, lr = oracle.attention_dense(Q, K, V, 1 / math.sqrt(d), causal)
    assert max_abs(O, Or) <= ATTN_F32_O_TOL
    assert max_abs(lse, lr) <= ATTN_F32_LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
def test_f32_varlen(dev, causal):
    lens = [1, 129, 64, 300, 5]
    cu = workloads.cu_seqlens_of(lens)
    Q, K, V = workloads.attention_inputs((int(cu[-1]), 2, 64), seed=41, dtype="f32")
    O, lse = gpu_packed(Q, K, V, cu, max(lens), causal, dev, via_readback=True)
    Or, lr = oracle.attention_packed(Q, K, V, cu, 1 / 8, causal)
    assert max_abs(O, Or) <= ATTN_F32_O_TOL
    assert max_abs(lse, lr) <= ATTN_F32_LSE_TOL


# ---------------------------------------------------------------------------
# bf16 tensor-core path: small shapes in full
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 256, 300, 513, 1024, 1500])
def test_bf16_dense_shapes(dev, N, d, causal):
    Q, K, V = workloads.attention_inputs((2, N, 3, d), seed=1000 * d + N + causal)
    O, lse = gpu_dense(Q, K, V, causal, dev)
    Or, lr = oracle.attention_dense(f32(Q), f32(K), f32(V), 1 / math.sqrt(d), causal)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_varlen(dev, d, causal):
    lens = [1, 129, 300, 64, 257, 128, 700]
    cu = workloads.cu_seqlens_of(lens)
    Q, K, V = workloads.attention_inputs((int(cu[-1]), 4, d), seed=7 + d, q_std=2.0, k_std=2.0)
    for readback in (False, True):
        O, lse = gpu_packed(Q, K, V, cu, max(lens), causal, dev, via_readback=readback)
        Or, lr = oracle.attention_packed(f32(Q), f32(K), f32(V), cu, 1 / math.sqrt(d), causal)
        assert max_abs(O, Or) <= ATTN_BF16_O_TOL
        assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_varlen_max_len_upper_bound(dev, d):
    """N may exceed every sequence length (an upper bound)."""
    lens = [200, 3]
    cu = workloads.cu_seqlens_of(lens)
    Q, K, V = workloads.attention_inputs((int(cu[-1]), 2, d), seed=99)
    O, lse = gpu_packed(Q, K, V, cu, 1000, True, dev)
    Or, lr = oracle.attention_packed(f32(Q), f32(K), f32(V), cu, 1 / math.sqrt(d), True)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_rising_scores_rescale_every_tile(dev, d, causal):
    """The running maximum grows on every key tile and jumps on the last key."""
    Q, K, V = workloads.rising_scores_inputs(1, 700, 2, d, seed=3 + d)
    O, lse = gpu_dense(Q, K, V, causal, dev)
    Or, lr = oracle.attention_dense(f32(Q), f32(K), f32(V), 1 / math.sqrt(d), causal)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL


def test_bf16_uniform_scores(dev):
    """Q = 0: every visible key has weight 1/n, so O is the mean of the visible V
    rows and lse = ln(n) (causal: n = i + 1)."""
    B, N, H, d = 1, 300, 2, 128
    _, _, V = workloads.attention_inputs((B, N, H, d), seed=11)
    Q = torch.zeros((B, N, H, d), dtype=torch.bfloat16)
    K = V.clone()
    O, lse = gpu_dense(Q, K, V, True, dev)
    Vf = f32(V).astype(np.float64)
    mean = np.cumsum(Vf, axis=1) / np.arange(1, N + 1).reshape(1, N, 1, 1)
    assert max_abs(O, mean) <= ATTN_BF16_O_TOL
    assert max_abs(lse[0], np.log(np.arange(1, N + 1))[None, :].repeat(H, 0)) <= ATTN_BF16_LSE_TOL


def test_bf16_deterministic(dev):
    Q, K, V = workloads.attention_inputs((2, 1000, 4, 128), seed=5)
    q, k, v = (t.to(dev) for t in (Q, K, V))
    o1, l1 = fa.attention_fwd(q, k, v, causal=True)
    o2, l2 = fa.attention_fwd(q, k, v, causal=True)
    torch.cuda.synchronize(dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bf16_bad_arguments(dev):
    q = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    p = q.data_ptr()
    assert fa.fa_attention_fwd(p, p, p, p, lse.data_ptr(), 1, 1, 128, 96, 0.1, 0, None) == -3
    assert fa.fa_attention_fwd(p + 2, p, p, p, lse.data_ptr(), 1, 1, 128, 64, 0.1, 0, None) == -4
    assert fa.fa_attention_fwd(None, p, p, p, lse.data_ptr(), 1, 1, 128, 64, 0.1, 0, None) == -1


def test_bf16_seqlen_longer_than_n_is_flagged(dev):
    """cu_seqlens that contradict N raise the device error bit instead of
    computing out of range."""
    lens = [300]
    cu = torch.tensor([0, 300], dtype=torch.int32, device=dev)
    q = torch.zeros((300, 1, 64), dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 300), dtype=torch.float32, device=dev)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    rc = fa.fa_attention_fwd_varlen(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), 1, 1, 200, 300, 64, 0.125, 1, cu.data_ptr())
    assert rc == 0
    assert fa.fa_get_device_error() == fa.FA_DEVERR_BAD_SEQLENS
    assert fa.fa_get_device_error() == 0
    del lens


# ---------------------------------------------------------------------------
# bf16 tensor-core path: the full-size workloads, every row
# ---------------------------------------------------------------------------

def _check_full(w, dev):
    """Every (token, head) row of O and lse of a full-size workload against the
    oracle, element by element, in the launch configuration the benchmark
    times; then the first and last 130 tokens of every sequence, in every
    head, reported on their own (the rows where tile and sequence edges
    fall)."""
    Q, K, V = w.inputs()
    cu = w.cu_seqlens()
    if w.varlen:
        O, lse = gpu_packed(Q, K, V, cu, w.N, w.causal, dev, via_readback=True)
        Qp, Kp, Vp = Q, K, V
        Op, lsep = O, lse                               # [total, H, d], [H, total]
    else:
        O, lse = gpu_dense(Q, K, V, w.causal, dev)
        Qp, Kp, Vp = (t.reshape(w.total, w.H, w.d) for t in (Q, K, V))
        Op = O.reshape(w.total, w.H, w.d)
        lsep = lse.transpose(1, 0, 2).reshape(w.H, w.total)
    device_error_clear()
    Or, lr = oracle.attention_packed(f32(Qp), f32(Kp), f32(Vp), cu, w.scale, w.causal)
    err_o = np.abs(Op - Or).max(axis=2)                 # [total, H]
    err_l = np.abs(lsep - lr).T                         # [total, H]
    assert np.all(np.isfinite(Op)) and np.all(np.isfinite(lsep))
    edge = np.concatenate([np.r_[cu[b]:min(cu[b] + 130, cu[b + 1])]
                           for b in range(len(cu) - 1)] +
                          [np.r_[max(cu[b + 1] - 130, cu[b]):cu[b + 1]]
                           for b in range(len(cu) - 1)])
    edge = np.unique(edge)
    worst = np.unravel_index(np.argmax(err_o), err_o.shape)
    print(f"{w.name}: compared all {err_o.size} (token, head) rows ({Op.size} O elements); "
          f"max |O err| {err_o.max():.3e} at (token, head) {tuple(int(i) for i in worst)}, "
          f"max |lse err| {err_l.max():.3e}; edge rows ({edge.size} tokens x {w.H} heads): "
          f"O {err_o[edge].max():.3e}, lse {err_l[edge].max():.3e}")
    assert err_o[edge].max() <= ATTN_BF16_O_TOL, f"{w.name}: edge O err {err_o[edge].max():.3e}"
    assert err_l[edge].max() <= ATTN_BF16_LSE_TOL, f"{w.name}: edge lse err {err_l[edge].max():.3e}"
    assert err_o.max() <= ATTN_BF16_O_TOL, f"{w.name}: O err {err_o.max():.3e}"
    assert err_l.max() <= ATTN_BF16_LSE_TOL, f"{w.name}: lse err {err_l.max():.3e}"


def test_bf16_workload_noncausal_d64(dev):
    _check_full(workloads.WORKLOADS["attn_bf16_b8h16n2048d64"], dev)


def test_bf16_workload_causal_d128(dev):
    _check_full(workloads.WORKLOADS["attn_bf16_causal_b2h32n4096d128"], dev)


def test_bf16_workload_varlen_causal_d128(dev):
    _check_full(workloads.WORKLOADS["attn_bf16_varlen8_h16d128_causal"], dev)
