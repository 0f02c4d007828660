"""The one-pass backward (fa_attention_bwd_atomic: dQ summed over the key
tiles by fp32 reduce-adds) on the GPU, through the C ABI, against the fp64
oracle's gradients of sum(dO * O).

Same tolerance as the two-pass backward (tests/test_bwd_gpu.py, BWD_TOL =
2^-6 normwise per gradient tensor): P and dS are rounded to bf16 as there; the
dQ shares are summed in fp32 in another order, which changes nothing at that
scale.
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
    return [torch.from_numpy(rng.standard_normal((B, N, H, d)).astype(np.float32))
            .to(torch.bfloat16) for _ in range(4)]   # Q, K, V, dO (bf16, CPU)


def run_gpu(Q, K, V, dO, causal, dev, deterministic=False):
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    o, lse = fa.attention_fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=causal,
                                  deterministic=deterministic)
    torch.cuda.synchronize(dev)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


def normwise(g, ref, floor=1e-30):
    return float(np.abs(g - ref).max() / max(np.abs(ref).max(), floor))


# An all-zero reference (one token: P = 1, so dS = dP - D is exactly 0) is
# compared against this floor: the kernel's dS is then the rounding
# difference of two fp32 dot products of d terms (~1e-7 here).
ZERO_FLOOR = 1e-3


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 128, 64, False),
    (2, 2, 200, 64, False),      # d = 64: ragged, a tile's last key rows are the next sequence's
    (1, 2, 1000, 64, True),      # d = 64: ring and dS buffers wrap
    (1, 1, 1, 64, True),
    (1, 2, 128, 128, False),
    (2, 2, 256, 128, True),
    (1, 3, 300, 128, True),  # ragged last key tile and query sub-tile
    (2, 2, 200, 128, False), # ragged: a tile's last key rows are the next sequence's
    (3, 1, 170, 128, True),  # the same, causal, three sequences
    (1, 1, 1, 128, True),    # one token
    (1, 2, 385, 128, False),
    (1, 2, 192, 128, True),  # last key tile of one 64-row sub-tile
    (1, 1, 65, 128, True),   # two sub-tiles, one tile
    (1, 2, 1000, 128, True), # 16 sub-steps: the 3-stage ring and both dS buffers wrap
    (2, 1, 900, 128, False),
])
def test_bwd_atomic_matches_oracle(dev, B, H, N, d, causal):
    Q, K, V, dO = make_inputs(B, H, N, d, seed=N * 11 + B)
    dq, dk, dv = run_gpu(Q, K, V, dO, causal, dev)
    ref = oracle.attention_bwd(*(t.float().numpy() for t in (Q, K, V, dO)), 1 / math.sqrt(d),
                               causal)
    errs = {name: normwise(g, ref[name], ZERO_FLOOR)
            for name, g in (("dQ", dq), ("dK", dk), ("dV", dv))}
    print(f"one-pass B{B} H{H} N{N} d{d} causal={causal}: normwise errors {errs}")
    for name, e in errs.items():
        assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def test_bwd_atomic_full_size_sampled(dev):
    """The benchmark's backward workload (causal B=2 H=32 N=4096 d=128):
    gradients of sampled query rows and keys of three heads against the
    oracle."""
    B, H, N, d = 2, 32, 4096, 128
    Q, K, V, dO = make_inputs(B, H, N, d, seed=4243)
    dq, dk, dv = run_gpu(Q, K, V, dO, True, dev)
    Qf, Kf, Vf, dOf = (t.float().numpy() for t in (Q, K, V, dO))
    rng = np.random.default_rng(8)
    for (b, h) in [(0, 0), (0, 17), (1, 31)]:
        qi = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, N - 1], rng.integers(0, N, 20)]))
        ki = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 20)]))
        rq, rk, rv = oracle.attention_bwd_head(Qf, Kf, Vf, dOf, 1 / math.sqrt(d), True, b, h,
                                               qi, ki)
        for name, g, ref in (("dQ", dq[b, qi, h], rq), ("dK", dk[b, ki, h], rk),
                             ("dV", dv[b, ki, h], rv)):
            e = normwise(g, ref)
            print(f"one-pass full size (b={b}, h={h}) {name}: normwise error {e}")
            assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def test_bwd_atomic_dk_dv_reproducible(dev):
    """dK and dV involve no atomic sums: two runs give the same bits; dQ's
    sums may be added in another order, so it is compared within a few fp32
    roundings of its bf16 result."""
    Q, K, V, dO = make_inputs(2, 2, 640, 128, seed=19)
    a = run_gpu(Q, K, V, dO, True, dev)
    b = run_gpu(Q, K, V, dO, True, dev)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert normwise(a[0], b[0]) <= 2.0 ** -8


def test_bwd_atomic_ignores_workspace_contents(dev):
    """The workspace's contents on entry do not matter (the first kernel
    zeroes the accumulator): NaN-filled scratch gives the same gradients as
    the two-pass call within the tolerance."""
    B, H, N, d = 1, 2, 300, 128
    Q, K, V, dO = make_inputs(B, H, N, d, seed=23)
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    nbytes = fa.fa_attention_bwd_atomic_workspace_bytes(B, H, N, d)
    assert nbytes == B * H * 320 * (d + 2) * 4       # N rounded up to 64
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    d_buf = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    rc = fa.fa_attention_bwd_atomic(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), d_buf.data_ptr(), B, H, N, d,
                                    1 / math.sqrt(d), 1, ws.data_ptr(), nbytes)
    assert rc == 0
    torch.cuda.synchronize(dev)
    ref = fa.attention_bwd(q, k, v, o, do, lse, causal=True)
    for g, r in zip((dq, dk, dv), ref):
        g, r = g.float().cpu().numpy(), r.float().cpu().numpy()
        assert np.isfinite(g).all()
        assert normwise(g, r) <= 2.0 ** -7
    device_error_clear()


def test_bwd_atomic_bad_arguments(dev):
    q = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    ws = torch.zeros((128 * 130 + 64,), dtype=torch.float32, device=dev)
    p, l, w = q.data_ptr(), lse.data_ptr(), ws.data_ptr()
    need = fa.fa_attention_bwd_atomic_workspace_bytes(1, 1, 128, 128)
    assert need == 128 * 130 * 4
    assert fa.fa_attention_bwd_atomic_workspace_bytes(1, 1, 128, 96) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_attention_bwd_atomic_workspace_bytes(1, 1, 128, 64) == 128 * 66 * 4
    assert fa.fa_attention_bwd_atomic_workspace_bytes(-1, 1, 128, 128) == fa.FA_ERR_BAD_SIZE
    call = fa.fa_attention_bwd_atomic
    assert call(p, p, p, p, p, l, p, p, p, l, 1, 1, 128, 96, 0.1, 0, w, need) == \
        fa.FA_ERR_UNSUPPORTED
    assert call(p, p, p, p, p, l, p, p, p, l, 1, 1, 128, 128, 0.1, 0, None, need) == \
        fa.FA_ERR_NULL_POINTER
    assert call(p, p, p, p, p, l, p, p, p, l, 1, 1, 128, 128, 0.1, 0, w, need - 4) == \
        fa.FA_ERR_BAD_SIZE
    assert call(p, p, p, p, p, l, p, p, p, l, 1, 1, 128, 128, 0.1, 0, w + 16, need) == \
        fa.FA_ERR_MISALIGNED
    assert call(p, p, p, p, p, l, p, p, p, l, 1, 1, 0, 128, 0.1, 0, None, 0) == 0


def run_gpu_packed(Q, K, V, dO, cu, max_len, causal, dev):
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    cu_d = torch.from_numpy(np.asarray(cu, np.int32)).to(dev)
    o, lse = fa.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu_d, max_seqlen=max_len)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, cu_seqlens=cu_d,
                                  max_seqlen=max_len, deterministic=False)
    torch.cuda.synchronize(dev)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lens", [[1, 129, 300, 64, 257, 0, 128, 700], [1000, 3]])
def test_bwd_atomic_packed_matches_oracle(dev, lens, causal, d):
    """Packed sequences (ragged lengths, an empty one, one token, a long one
    whose ring wraps): every gradient against the oracle's per-sequence
    backward."""
    import workloads
    H = 3
    cu = workloads.cu_seqlens_of(lens)
    total = int(cu[-1])
    rng = np.random.default_rng(sum(lens) + 11 * causal)
    Q, K, V, dO = (torch.from_numpy(rng.standard_normal((total, H, d)).astype(np.float32))
                   .to(torch.bfloat16) for _ in range(4))
    dq, dk, dv = run_gpu_packed(Q, K, V, dO, cu, max(lens), causal, dev)
    ref = oracle.attention_bwd_packed(*(t.float().numpy() for t in (Q, K, V, dO)), cu,
                                      1 / math.sqrt(d), causal)
    errs = {name: normwise(g, ref[name], ZERO_FLOOR)
            for name, g in (("dQ", dq), ("dK", dk), ("dV", dv))}
    print(f"one-pass packed {lens} d{d} causal={causal}: normwise errors {errs}")
    for name, e in errs.items():
        assert e <= BWD_TOL, f"{name}: {e}"
    device_error_clear()


def test_bwd_atomic_packed_equal_lengths_is_the_dense_call(dev):
    """Packed sequences of one length: dK and dV equal the dense one-pass
    call's bits (the same arithmetic on the same rows); dQ's sums may be
    added in another order."""
    B, H, N, d = 2, 2, 300, 128
    Q, K, V, dO = make_inputs(B, H, N, d, seed=29)
    dense = run_gpu(Q, K, V, dO, True, dev)
    cu = np.arange(B + 1, dtype=np.int32) * N
    packed = run_gpu_packed(*(t.reshape(B * N, H, d) for t in (Q, K, V, dO)), cu, N, True, dev)
    dense = [x.reshape(B * N, H, d) for x in dense]
    assert np.array_equal(dense[1], packed[1]) and np.array_equal(dense[2], packed[2])
    assert normwise(packed[0], dense[0]) <= 2.0 ** -8


def test_bwd_atomic_packed_length_over_n_is_flagged(dev):
    """A sequence longer than N is flagged in the device error word and not
    computed (no access past the tensors or the workspace)."""
    H, d = 1, 128
    q = torch.zeros((300, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((H, 300), dtype=torch.float32, device=dev)
    cu = torch.tensor([0, 300], dtype=torch.int32, device=dev)
    nbytes = fa.fa_attention_bwd_atomic_varlen_workspace_bytes(1, H, 200, 300, d)
    assert nbytes == H * (300 + 64) * d * 4 + H * 1 * 256 * 8
    ws = torch.empty((nbytes // 4,), dtype=torch.float32, device=dev)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    p, l, w = q.data_ptr(), lse.data_ptr(), ws.data_ptr()
    call = fa.fa_attention_bwd_atomic_varlen
    assert call(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, d, 0.125, 1, cu.data_ptr(), w,
                nbytes) == 0
    torch.cuda.synchronize(dev)
    assert fa.fa_get_device_error() == fa.FA_DEVERR_BAD_SEQLENS
    assert fa.fa_get_device_error() == 0
    assert call(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, d, 0.125, 1, None, w,
                nbytes) == fa.FA_ERR_NULL_POINTER
    assert call(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, d, 0.125, 1, cu.data_ptr(), w,
                nbytes - 8) == fa.FA_ERR_BAD_SIZE
    assert call(p, p, p, p, p, l, p, p, p, l, 1, H, 200, 300, 96, 0.125, 1, cu.data_ptr(), w,
                nbytes) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_attention_bwd_atomic_varlen_workspace_bytes(1, H, 200, 300, 96) == \
        fa.FA_ERR_UNSUPPORTED


def test_bwd_atomic_full_size_every_element_matches_two_pass(dev):
    """Every gradient element of the benchmark's backward workload (causal
    B=2 H=32 N=4096 d=128, all 64 heads) from the one-pass form against the
    two-pass form.  dK and dV are formed the same way in both (D_i summed in
    the same order: 16 lanes of 8 elements, then the same shuffle tree; the
    same products in the same K-step order), so their bits must be equal.
    dQ is summed in another order (fp32 atomic adds over the key tiles
    against one accumulator per query tile), so it may differ by a few units
    in the last place of its bf16 result: bound 2^-9 of the largest |dQ|
    (observed 5.9e-4).  The oracle checks of both forms fix correctness;
    this one makes a fault confined to some heads or tiles of the full grid
    show."""
    B, H, N, d = 2, 32, 4096, 128
    g = torch.Generator(device=dev).manual_seed(7)
    q, k, v, do = (torch.randn((B, N, H, d), generator=g, device=dev).to(torch.bfloat16)
                   for _ in range(4))
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    one = fa.attention_bwd(q, k, v, o, do, lse, causal=True, deterministic=False)
    two = fa.attention_bwd(q, k, v, o, do, lse, causal=True, deterministic=True)
    torch.cuda.synchronize(dev)
    assert torch.equal(one[1], two[1]), "dK differs from the two-pass form"
    assert torch.equal(one[2], two[2]), "dV differs from the two-pass form"
    a, b = one[0].float(), two[0].float()
    assert torch.isfinite(a).all()
    per_head = (a - b).abs().amax(dim=(1, 3)) / b.abs().amax().item()   # [B, H]
    worst = per_head.max().item()
    print(f"full size, every element, one-pass vs two-pass: dK, dV equal; dQ max {worst:.2e} "
          f"of max |dQ| (per head: min {per_head.min().item():.2e})")
    assert worst <= 2.0 ** -9, f"dQ: {worst}"
