"""Split-KV attention (tensor-core kernel per key split + combine kernel) on the
GPU, through the C ABI, against the fp64 oracle with separate query / key
lengths (bottom-right causal alignment)."""
import math

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
import workloads
from gpu_common import ATTN_BF16_LSE_TOL, ATTN_BF16_O_TOL, device_error_clear, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def inputs(B, H, Nq, Nk, d, seed):
    w = workloads.SplitKVWorkload("t", B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=True, seed=seed)
    return w.inputs()


def run(Q, K, V, causal, splits, dev):
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, lse = fa.attention_fwd_splitkv(q, k, v, causal=causal, num_splits=splits)
    torch.cuda.synchronize(dev)
    return O.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", [
    (2, 2, 128, 128, 64, True, 1),      # square, one split
    (2, 2, 300, 300, 128, True, 3),     # square: the third split is empty, Q0 idle in split 1
    (1, 3, 1, 2049, 128, True, 4),      # one new query against a ragged key length
    (2, 2, 100, 1000, 64, True, 5),     # rows with no visible key inside a split's range
    (1, 2, 200, 1000, 128, True, 8),
    (1, 2, 256, 4096, 128, True, 0),    # split count chosen by the library
    (2, 1, 257, 777, 128, False, 7),
    (1, 2, 130, 1300, 64, False, 64),   # clamped to the 11 key tiles
    (1, 2, 200, 5120, 128, False, 40),  # 40 one-tile splits: two chunks of the combine
    (1, 2, 256, 8192, 128, True, 37),   # splits 32..36 empty (lse -inf) in the second chunk
])
def test_splitkv_matches_oracle(dev, B, H, Nq, Nk, d, causal, splits):
    Q, K, V = inputs(B, H, Nq, Nk, d, seed=Nq * 31 + Nk + d + splits)
    O, lse = run(Q, K, V, causal, splits, dev)
    Or, lr = oracle.attention_qk(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                 1 / math.sqrt(d), causal)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL
    device_error_clear()


def test_splitkv_one_split_equals_main_path(dev):
    """With Nq == Nk and one split the same kernel path runs: bitwise equal."""
    Q, K, V = inputs(2, 3, 700, 700, 128, seed=5)
    q, k, v = (t.to(dev) for t in (Q, K, V))
    o1, l1 = fa.attention_fwd(q, k, v, causal=True)
    o2, l2 = fa.attention_fwd_splitkv(q, k, v, causal=True, num_splits=1)
    torch.cuda.synchronize(dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("splits", [2, 5, 11])
def test_splitkv_splits_agree(dev, splits):
    """Different split counts give the same result within rounding."""
    Q, K, V = inputs(1, 4, 256, 2816, 128, seed=7)
    O1, l1 = run(Q, K, V, True, 1, dev)
    O2, l2 = run(Q, K, V, True, splits, dev)
    assert max_abs(O2, O1) <= ATTN_BF16_O_TOL
    assert max_abs(l2, l1) <= ATTN_BF16_LSE_TOL


def test_splitkv_workload_every_row(dev):
    """The benchmark's split-KV workload, every (query, head) row checked."""
    w = workloads.SPLITKV_WORKLOADS["attn_bf16_splitkv_b1h16nq256nk32768d128_causal"]
    Q, K, V = w.inputs()
    O, lse = run(Q, K, V, w.causal, 0, dev)
    Or, lr = oracle.attention_qk(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                 w.scale, w.causal)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL
    device_error_clear()


def test_splitkv_bad_arguments(dev):
    q = torch.zeros((1, 256, 1, 64), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 256), dtype=torch.float32, device=dev)
    p = q.data_ptr()
    # causal with fewer keys than queries
    assert fa.fa_attention_fwd_splitkv(p, k.data_ptr(), k.data_ptr(), p, lse.data_ptr(),
                                       1, 1, 256, 128, 64, 0.125, 1, 1, None, None) == -2
    # several splits without scratch
    k2 = torch.zeros((1, 1024, 1, 64), dtype=torch.bfloat16, device=dev)
    assert fa.fa_attention_fwd_splitkv(p, k2.data_ptr(), k2.data_ptr(), p, lse.data_ptr(),
                                       1, 1, 256, 1024, 64, 0.125, 1, 4, None, None) == -1
    assert fa.fa_splitkv_num_splits(1, 1, 256, 1024, 96) == -3


# ---------------------------------------------------------------------------
# packed sequences with their own query and key counts (a decode step over
# caches of different lengths)
# ---------------------------------------------------------------------------

def packed_inputs(lens_q, lens_k, H, d, seed):
    rng = np.random.default_rng(seed)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    mk = lambda n: torch.from_numpy(rng.standard_normal((n, H, d), dtype=np.float32)).to(
        torch.bfloat16)
    return mk(tq), mk(tk), mk(tk)


def run_packed(Q, K, V, lens_q, lens_k, causal, splits, dev):
    cq = torch.from_numpy(workloads.cu_seqlens_of(lens_q)).to(dev)
    ck = torch.from_numpy(workloads.cu_seqlens_of(lens_k)).to(dev)
    q, k, v = (t.to(dev) for t in (Q, K, V))
    O, lse = fa.attention_fwd_splitkv_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k),
                                             causal=causal, num_splits=splits)
    torch.cuda.synchronize(dev)
    return O.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [0, 1, 3, 16])
def test_splitkv_packed_matches_oracle(dev, d, causal, splits):
    """Sequences of 1, 7, 0, 300 and 129 new queries against 1000, 7, 50, 3000
    and 129 keys (a query-free sequence, a square one, one whose keys fit one
    tile): every row against the oracle's per-sequence attention."""
    lens_q, lens_k = [1, 7, 0, 300, 129], [1000, 7, 50, 3000, 129]
    Q, K, V = packed_inputs(lens_q, lens_k, 3, d, seed=d + causal + splits)
    O, lse = run_packed(Q, K, V, lens_q, lens_k, causal, splits, dev)
    Or, lr = oracle.attention_qk_packed(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                        workloads.cu_seqlens_of(lens_q),
                                        workloads.cu_seqlens_of(lens_k), 1 / math.sqrt(d), causal)
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse, lr) <= ATTN_BF16_LSE_TOL
    device_error_clear()


def test_splitkv_packed_equal_lengths_is_the_dense_call(dev):
    """Packed sequences of one query and one key count give the dense split-KV
    call's bits at the same split count."""
    B, H, Nq, Nk, d = 3, 2, 200, 1500, 128
    Q, K, V = inputs(B, H, Nq, Nk, d, seed=77)
    Od, ld = run(Q, K, V, True, 4, dev)
    Op, lp = run_packed(Q.reshape(B * Nq, H, d), K.reshape(B * Nk, H, d),
                        V.reshape(B * Nk, H, d), [Nq] * B, [Nk] * B, True, 4, dev)
    assert np.array_equal(Op, Od.reshape(B * Nq, H, d))
    assert np.array_equal(lp, ld.transpose(1, 0, 2).reshape(H, B * Nq))


def test_splitkv_packed_bad_lengths_are_flagged(dev):
    """Causal with fewer keys than queries in one sequence, or a key count over
    the stated maximum, sets the device error bit instead of computing."""
    H, d = 1, 64
    q = torch.zeros((10, H, d), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((20, H, d), dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros((H, 10), dtype=torch.float32, device=dev)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    for lens_q, lens_k, Nk in (([6, 4], [2, 18], 18), ([10], [20], 16)):
        cq = torch.from_numpy(workloads.cu_seqlens_of(lens_q)).to(dev)
        ck = torch.from_numpy(workloads.cu_seqlens_of(lens_k)).to(dev)
        rc = fa.fa_attention_fwd_splitkv_varlen(q.data_ptr(), k.data_ptr(), k.data_ptr(),
                                                o.data_ptr(), lse.data_ptr(), len(lens_q), H,
                                                max(lens_q), Nk, 10, 20, d, 0.125, 1, 1,
                                                cq.data_ptr(), ck.data_ptr(), None, None)
        assert rc == 0
        assert fa.fa_get_device_error() == fa.FA_DEVERR_BAD_SEQLENS
    assert fa.fa_attention_fwd_splitkv_varlen(q.data_ptr(), k.data_ptr(), k.data_ptr(),
                                              o.data_ptr(), lse.data_ptr(), 1, H, 10, 20, 10, 20,
                                              d, 0.125, 1, 1, None, None, None,
                                              None) == fa.FA_ERR_NULL_POINTER


@pytest.mark.parametrize("splits", [1, 3])
def test_splitkv_packed_sequence_without_keys(dev, splits):
    """A non-causal packed sequence with queries but no keys: its rows see no
    key, so O = 0 and lse = -inf (the oracle's reading); the other sequences
    are unaffected."""
    lens_q, lens_k, d = [3, 5, 130], [0, 300, 1000], 128
    Q, K, V = packed_inputs(lens_q, lens_k, 2, d, seed=31 + splits)
    O, lse = run_packed(Q, K, V, lens_q, lens_k, False, splits, dev)
    Or, lr = oracle.attention_qk_packed(Q.float().numpy(), K.float().numpy(), V.float().numpy(),
                                        workloads.cu_seqlens_of(lens_q),
                                        workloads.cu_seqlens_of(lens_k), 1 / math.sqrt(d), False)
    assert np.all(O[:3] == 0.0) and np.all(np.isneginf(lse[:, :3]))
    assert np.array_equal(np.isneginf(lse), np.isneginf(lr))
    assert max_abs(O, Or) <= ATTN_BF16_O_TOL
    assert max_abs(lse[:, 3:], lr[:, 3:]) <= ATTN_BF16_LSE_TOL
    device_error_clear()
