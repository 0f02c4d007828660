"""FP8 attention forward (rotation, blockwise e4m3 quantisation, e4m3 tensor
cores) on the GPU, through the C ABI, against the reference in oracle/fp8.py:
the same rotation and quantisation steps in float64, then the fp64 attention
oracle on the dequantised values.

Tolerances against that reference: the kernels also round P to e4m3 (unit
roundoff u = 2^-4) before P V, which the reference does not, so an element of
O may differ by at most u * max |V| (all rounding errors of a row aligned);
their root mean square over O is bounded by FP8_O_RMSE = 1e-2 (independent
errors, at least a few visible keys per row: ~u / sqrt(3) * rms(V) /
sqrt(keys)).  The row sums use the unrounded p in fp32, so lse keeps the bf16
path's 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
from oracle import fp8
from gpu_common import device_error_clear, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def make(B, H, N, d, seed, outliers=False):
    rng = np.random.default_rng(seed)
    xs = [rng.standard_normal((B, N, H, d)) for _ in range(3)]
    if outliers:
        for x in xs:
            x[rng.random(x.shape) < 0.001] *= 10.0
    qkv = [torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16) for x in xs]
    signs = rng.choice([-1.0, 1.0], size=d).astype(np.float32)
    return qkv, signs


def run(qkv, signs, causal, dev):
    q, k, v = (t.to(dev) for t in qkv)
    s = torch.from_numpy(signs).to(dev)
    o, lse, ws = fa.attention_fwd_fp8(q, k, v, s, causal=causal)
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy(), lse.cpu().numpy(), ws.cpu().numpy()


def layout(B, H, N, d):
    up = lambda x: (x + 255) & ~255
    T = (N + 127) // 128
    elems = B * N * H * d
    qf = 0
    kf = up(qf + elems)
    vt = up(kf + elems)
    sq = up(vt + B * H * d * 128 * T)
    sk = up(sq + B * H * T * 4)
    vamax = up(sk + B * H * T * 4)
    sv = up(vamax + B * H * T * 4)
    return dict(qf=qf, kf=kf, vt=vt, sq=sq, sk=sk, vamax=vamax, sv=sv, T=T)


def e4m3_decode(codes):
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def assert_codes_match(codes, ref, name):
    """The kernel's e4m3 codes against the reference's values: the kernel
    forms x / scale in fp32, the reference in fp64, so a value within rounding
    of an e4m3 half-way point may land on the neighbouring code -- at most
    1e-3 of the codes, each one step (in the code's magnitude) from the
    reference's, with the same sign unless one of them is zero."""
    codes = np.ascontiguousarray(codes)
    got = e4m3_decode(codes)
    diff = got != ref
    print(f"{name}: {diff.mean():.2e} of codes differ")
    assert diff.mean() < 1e-3, name
    g = codes[diff].astype(np.int16)
    r = torch.from_numpy(np.ascontiguousarray(ref[diff])).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy().astype(np.int16)
    mg, mr = g & 0x7F, r & 0x7F
    sign_ok = (((g ^ r) & 0x80) == 0) | (mg == 0) | (mr == 0)
    assert np.all(sign_ok & (np.abs(mg - mr) == 1)), name


# the last case has 960 work items (Q, K, V tiles), several per CTA of the
# persistent quantisation kernel, and a ragged last tile per sequence
@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 256, False), (2, 1, 300, True),
                                          (2, 16, 1200, True)])
def test_fp8_quantisation_matches_reference(dev, B, H, N, causal):
    d = 128
    (Q, K, V), signs = make(B, H, N, d, seed=N + B)
    _, _, ws = run((Q, K, V), signs, causal, dev)
    L = layout(B, H, N, d)
    for name, X, off, soff in (("Q", Q, L["qf"], L["sq"]), ("K", K, L["kf"], L["sk"])):
        Xr = fp8.rotate(X.float().numpy(), signs)
        _, ref_scales = fp8.blockwise_qk(Xr)
        got_scales = ws[soff:soff + B * H * L["T"] * 4].view(np.float32).reshape(B, H, L["T"])
        assert np.allclose(got_scales, ref_scales, rtol=1e-5), name
        codes = ws[off:off + B * N * H * d].reshape(B, N, H, d)
        ref = fp8.e4m3_round(Xr / np.repeat(got_scales, 128, axis=2)[:, :, :N].transpose(0, 2, 1)[..., None])
        assert_codes_match(codes, ref, name)
    # V': one scale per (sequence, head), codes transposed to [B, H, d, n_pad],
    # zero codes past N; the codes decided in float32 on both sides, so they
    # are compared exactly
    ref, ref_sv = fp8.per_head_v_fp32(V.float().numpy())
    got_sv = ws[L["sv"]:L["sv"] + B * H * 4].view(np.float32).reshape(B, H)
    assert np.array_equal(got_sv, ref_sv)
    n_pad = 128 * L["T"]
    codes = ws[L["vt"]:L["vt"] + B * H * d * n_pad].reshape(B, H, d, n_pad)
    assert not np.any(codes[..., N:]), "padding keys must hold zero codes"
    got = e4m3_decode(np.ascontiguousarray(codes[..., :N]))
    assert np.array_equal(got, ref.transpose(0, 2, 3, 1)), "V' codes"


@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 256, False), (2, 2, 512, True), (1, 3, 300, True),
                                          (1, 1, 1, True), (2, 1, 700, False)])
def test_fp8_matches_reference(dev, B, H, N, causal):
    d = 128
    qkv, signs = make(B, H, N, d, seed=7 * N + B)
    O, lse, _ = run(qkv, signs, causal, dev)
    Q, K, V = (t.float().numpy() for t in qkv)
    Or, lr = fp8.fp8_attention(Q, K, V, signs, 1 / math.sqrt(d), causal)
    O_ex, l_ex = oracle.attention_dense(Q, K, V, 1 / math.sqrt(d), causal)
    rmse = float(np.sqrt(np.mean((O - Or) ** 2)))
    mx = float(np.abs(O - Or).max())
    rmse_ex = float(np.sqrt(np.mean((O - O_ex) ** 2)))
    print(f"B{B} H{H} N{N} causal={causal}: vs FP8 reference rmse {rmse:.2e} max {mx:.2e} "
          f"lse {np.abs(lse - lr).max():.2e}; vs exact rmse {rmse_ex:.2e}")
    assert rmse <= FP8_O_RMSE and mx <= 2.0 ** -4 * float(np.abs(V).max())
    assert float(np.abs(lse - lr).max()) <= FP8_LSE_MAX
    device_error_clear()


def test_fp8_full_size_sampled(dev):
    """The benchmark's FP8 launch (causal B=2 H=32 N=4096 d=128): every tile
    scale of Q M and K M against the reference's, and O and lse on sampled
    (token, head) rows against the reference attention on the dequantised
    inputs (the reference row by row: the oracle's per-row attention)."""
    import workloads
    B, H, N, d = 2, 32, 4096, 128
    qkv, signs = make(B, H, N, d, seed=4096)
    O, lse, ws = run(qkv, signs, True, dev)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse))
    Q, K, V = (t.float().numpy() for t in qkv)
    L = layout(B, H, N, d)
    for name, X, soff in (("Q", Q, L["sq"]), ("K", K, L["sk"])):
        _, ref_scales = fp8.blockwise_qk(fp8.rotate(X, signs))
        got = ws[soff:soff + B * H * L["T"] * 4].view(np.float32).reshape(B, H, L["T"])
        assert np.allclose(got, ref_scales, rtol=1e-5), name
    Qd, Kd, Vd = (x.reshape(B * N, H, d).astype(np.float32) for x in fp8.fp8_inputs(Q, K, V, signs))
    must = list(range(0, 130)) + list(range(N - 130, N + 130)) + list(range(B * N - 130, B * N))
    tok, head = workloads.sample_rows(B * N, H, 2000, seed=4097)
    tok = np.concatenate([tok, np.asarray(must, np.int64)])
    head = np.concatenate([head, np.asarray(must, np.int64) % H])
    cu = np.arange(B + 1, dtype=np.int32) * N
    Or, lr = oracle.attention_rows(Qd, Kd, Vd, cu, 1 / math.sqrt(d), True, tok, head)
    Op = O.reshape(B * N, H, d)[tok, head]
    lp = lse.transpose(1, 0, 2).reshape(H, B * N)[head, tok]
    rmse = float(np.sqrt(np.mean((Op - Or) ** 2)))
    mx = float(np.abs(Op - Or).max())
    print(f"full size: rmse {rmse:.2e} max {mx:.2e} lse {np.abs(lp - lr).max():.2e}")
    assert rmse <= FP8_O_RMSE and mx <= 2.0 ** -4 * float(np.abs(V).max())
    assert float(np.abs(lp - lr).max()) <= FP8_LSE_MAX
    device_error_clear()


def test_fp8_outliers_pages_experiment(dev):
    """The pages' outlier test ([FG] §4.6): RMSE against exact attention,
    below per-tensor FP8 (emulated on the CPU from its definition)."""
    B, H, N, d = 1, 2, 512, 128
    qkv, signs = make(B, H, N, d, seed=104, outliers=True)
    O, _, _ = run(qkv, signs, False, dev)
    Q, K, V = (t.float().numpy() for t in qkv)
    O_ex, _ = oracle.attention_dense(Q, K, V, 1 / math.sqrt(d), False)
    Ob, _ = fp8.fp8_attention(Q, K, V, signs, 1 / math.sqrt(d), False, per_tensor_scales=True,
                              rotate_qk=False)
    rmse = float(np.sqrt(np.mean((O - O_ex) ** 2)))
    rmse_b = float(np.sqrt(np.mean((Ob - O_ex) ** 2)))
    print(f"outliers: GPU FP8 rmse {rmse:.3e}; per-tensor FP8 rmse {rmse_b:.3e}")
    assert rmse < 1.5e-2 and rmse < rmse_b


def dequantised_from_workspace(ws, B, H, N, d):
    """Q', K', V' as the kernels quantised them (codes times scales, float32),
    read back from the workspace."""
    L = layout(B, H, N, d)
    T = L["T"]
    e = B * N * H * d

    def tile_scaled(off, soff):
        codes = e4m3_decode(ws[off:off + e]).reshape(B, N, H, d)
        sc = ws[soff:soff + B * H * T * 4].view(np.float32).reshape(B, H, T).astype(np.float64)
        return codes * np.repeat(sc, 128, axis=2)[:, :, :N].transpose(0, 2, 1)[..., None]

    Qd = tile_scaled(L["qf"], L["sq"])
    Kd = tile_scaled(L["kf"], L["sk"])
    vt = ws[L["vt"]:L["vt"] + B * H * d * 128 * T].reshape(B, H, d, 128 * T)
    sv = ws[L["sv"]:L["sv"] + B * H * 4].view(np.float32).reshape(B, H).astype(np.float64)
    Vd = e4m3_decode(np.ascontiguousarray(vt[..., :N])) * sv[:, :, None, None]
    return (Qd.astype(np.float32), Kd.astype(np.float32),
            np.ascontiguousarray(Vd.transpose(0, 3, 1, 2)).astype(np.float32))


def test_fp8_many_heads(dev):
    """More sequence-heads than a grid's y dimension holds (65535): the
    quantisation and attention grids take them along x.  The attention is
    checked on the codes the kernels produced (a few of 34 M codes may be
    the neighbour of the float64 method's, which moves a one-key row's lse
    by ~1e-2; the codes themselves are checked by the quantisation test)."""
    B, H, N, d = 1, 66000, 2, 128
    qkv, signs = make(B, H, N, d, seed=66)
    O, lse, ws = run(qkv, signs, True, dev)
    Qd, Kd, Vd = dequantised_from_workspace(ws, B, H, N, d)
    Or, lr = oracle.attention_dense(Qd, Kd, Vd, 1 / math.sqrt(d), True)
    rmse = float(np.sqrt(np.mean((O - Or) ** 2)))
    V = qkv[2].float().numpy()
    assert rmse <= FP8_O_RMSE and float(np.abs(O - Or).max()) <= 2.0 ** -4 * float(np.abs(V).max())
    assert float(np.abs(lse - lr).max()) <= FP8_LSE_MAX
    device_error_clear()


def test_fp8_bad_arguments(dev):
    assert fa.fa_attention_fp8_workspace_bytes(1, 1, 128, 64) == -3
    q = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    s = torch.ones(128, dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    p = q.data_ptr()
    assert fa.fa_attention_fwd_fp8(p, p, p, p, lse.data_ptr(), 1, 1, 128, 128, 0.1, 0,
                                   s.data_ptr(), ws.data_ptr(), 256) == -2   # too small
    assert fa.fa_attention_fwd_fp8(p, p, p, p, lse.data_ptr(), 1, 1, 128, 64, 0.1, 0,
                                   s.data_ptr(), ws.data_ptr(), 256) == -3


FP8_O_RMSE = 1e-2
FP8_LSE_MAX = 1e-3
