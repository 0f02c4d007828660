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


def layout(B, H, N, d, total=None):
    up = lambda x: (x + 255) & ~255
    T = (N + 127) // 128
    elems = (B * N if total is None else total) * H * d
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
        # the reference's codes come from its own float64 rotation and scales
        Xr = fp8.rotate(X.float().numpy(), signs)
        _, ref_scales = fp8.blockwise_qk(Xr)
        got_scales = ws[soff:soff + B * H * L["T"] * 4].view(np.float32).reshape(B, H, L["T"])
        assert np.allclose(got_scales, ref_scales, rtol=1e-5), name + " scales"
        codes = ws[off:off + B * N * H * d].reshape(B, N, H, d)
        per_row = np.repeat(ref_scales, 128, axis=2)[:, :, :N].transpose(0, 2, 1)[..., None]
        assert_codes_match(codes, fp8.e4m3_round(Xr / per_row), name)
    # V': one scale per (sequence, head), codes transposed to [B, H, d, n_pad],
    # zero codes past N
    n_pad = 128 * L["T"]
    codes = ws[L["vt"]:L["vt"] + B * H * d * n_pad].reshape(B, H, d, n_pad)
    assert not np.any(codes[..., N:]), "padding keys must hold zero codes"
    got_codes = np.ascontiguousarray(codes[..., :N].transpose(0, 3, 1, 2))   # [B, N, H, d]
    got_sv = ws[L["sv"]:L["sv"] + B * H * 4].view(np.float32).reshape(B, H)
    # (1) against the float64 method (scale amax / 448 and the quotient in
    # float64): only neighbouring codes where the quotient falls within
    # float32 rounding of a half-way point
    Vf = V.float().numpy()
    _, sv64 = fp8.per_head_v(Vf)
    assert np.allclose(got_sv, sv64, rtol=1e-7), "sv against the float64 method"
    assert_codes_match(got_codes, fp8.e4m3_round(Vf / sv64[:, None, :, None]), "V (float64)")
    # (2) against the same method with the decision taken in float32, as the
    # kernel takes it: equal, code for code
    ref, ref_sv = fp8.per_head_v_fp32(Vf)
    assert np.array_equal(got_sv, ref_sv)
    assert np.array_equal(e4m3_decode(got_codes), ref), "V' codes (float32 decision)"


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


def check_against_reference(O, lse, qkv, signs, causal, label):
    """O and lse of every (token, head) row against the reference (the float64
    rotation and blockwise quantisation, then the fp64 oracle on the
    dequantised inputs).

    O: RMSE <= FP8_O_RMSE and max <= 2^-4 max|V| (P rounded to e4m3).
    lse: the kernel rotates in fp32 (tensor-core summation order), so at most
    1e-3 of its Q', K' codes (observed ~1e-7) are the neighbour of the
    reference's.  A score moves by at most scale * sum_k |dq'_k k'_k| +
    |q'_k dk'_k| and lse, 1-Lipschitz in the largest score change, as much;
    with every code one step off (a step is at most 2^-3 (1 + 2^-3) of the
    value) that is bound_i = 2^-2 (1 + 2^-3) scale sum_k |q'_ik| max_j |k'_jk|.
    So lse is held to FP8_LSE_MAX on all but 1e-3 of the rows (the bound the
    quantisation test puts on neighbouring codes; observed up to 1.8e-4 of the
    rows when every row has one or two keys) and every row to
    max(bound_i, FP8_LSE_MAX): a grid, tile or scale slip misplaces whole
    tiles or heads and fails one of the three."""
    Q, K, V = (t.float().numpy() for t in qkv)
    B, N, H, d = Q.shape
    scale = 1 / math.sqrt(d)
    Qd, Kd, Vd = fp8.fp8_inputs(Q, K, V, signs)
    Or, lr = oracle.attention_dense(Qd.astype(np.float32), Kd.astype(np.float32),
                                    Vd.astype(np.float32), scale, causal)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse))
    rmse = float(np.sqrt(np.mean((O - Or) ** 2)))
    mx = float(np.abs(O - Or).max())
    err_l = np.abs(lse - lr)                                            # [B, H, N]
    kmax = np.abs(Kd).max(axis=1)                                       # [B, H, d]
    bound = 2.0 ** -2 * (1 + 2.0 ** -3) * scale * np.einsum("bnhk,bhk->bhn", np.abs(Qd), kmax)
    frac_off = float(np.mean(err_l > FP8_LSE_MAX))
    print(f"{label}: all {O.size // d} rows; O rmse {rmse:.2e} max {mx:.2e}; lse max "
          f"{err_l.max():.2e}, {frac_off:.2e} of rows above {FP8_LSE_MAX}")
    assert rmse <= FP8_O_RMSE and mx <= 2.0 ** -4 * float(np.abs(V).max())
    assert frac_off <= 1e-3
    assert np.all(err_l <= np.maximum(bound, FP8_LSE_MAX))


def test_fp8_full_size(dev):
    """The benchmark's FP8 launch (causal B=2 H=32 N=4096 d=128): every tile
    scale of Q M and K M against the reference's, and O and lse of every
    (token, head) row against the reference attention on the dequantised
    inputs."""
    B, H, N, d = 2, 32, 4096, 128
    qkv, signs = make(B, H, N, d, seed=4096)
    O, lse, ws = run(qkv, signs, True, dev)
    device_error_clear()
    L = layout(B, H, N, d)
    for name, X, soff in (("Q", qkv[0], L["sq"]), ("K", qkv[1], L["sk"])):
        _, ref_scales = fp8.blockwise_qk(fp8.rotate(X.float().numpy(), signs))
        got = ws[soff:soff + B * H * L["T"] * 4].view(np.float32).reshape(B, H, L["T"])
        assert np.allclose(got, ref_scales, rtol=1e-5), name
    check_against_reference(O, lse, qkv, signs, True, "full size")


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


def test_fp8_many_heads(dev):
    """More sequence-heads than a grid's y dimension holds (65535): the
    quantisation and attention grids take them along x.  Every row against
    the reference; a one-key row's lse is its single score, which a
    neighbouring Q' or K' code moves by up to ~1e-2 (the bound in
    check_against_reference)."""
    B, H, N, d = 1, 66000, 2, 128
    qkv, signs = make(B, H, N, d, seed=66)
    O, lse, _ = run(qkv, signs, True, dev)
    device_error_clear()
    check_against_reference(O, lse, qkv, signs, True, "many heads")


# ---------------------------------------------------------------------------
# packed sequences
# ---------------------------------------------------------------------------

def make_packed(lens, H, d, seed):
    rng = np.random.default_rng(seed)
    total = int(sum(lens))
    xs = [rng.standard_normal((total, H, d)) for _ in range(3)]
    qkv = [torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16) for x in xs]
    signs = rng.choice([-1.0, 1.0], size=d).astype(np.float32)
    return qkv, signs


def run_packed(qkv, signs, lens, causal, dev):
    import workloads
    q, k, v = (t.to(dev) for t in qkv)
    cu = torch.from_numpy(workloads.cu_seqlens_of(lens)).to(dev)
    o, lse, ws = fa.attention_fwd_fp8(q, k, v, torch.from_numpy(signs).to(dev), causal=causal,
                                      cu_seqlens=cu, max_seqlen=max(lens))
    torch.cuda.synchronize(dev)
    return o.float().cpu().numpy(), lse.cpu().numpy(), ws.cpu().numpy()


PACKED_LENS = [1, 129, 300, 0, 256, 700]    # ragged tiles, an empty sequence, whole tiles


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_packed_quantisation_matches_reference(dev, causal):
    """Each sequence is quantised on its own: its Q', K' tile scales and codes
    (tiles from its first token, a ragged last tile taking its amax over the
    sequence's rows only) and its V' codes and scale against the reference run
    on that sequence alone; no tile writes into another sequence's rows."""
    import workloads
    H, d = 2, 128
    qkv, signs = make_packed(PACKED_LENS, H, d, seed=61 + causal)
    _, _, ws = run_packed(qkv, signs, PACKED_LENS, causal, dev)
    cu = workloads.cu_seqlens_of(PACKED_LENS)
    B, N, total = len(PACKED_LENS), max(PACKED_LENS), int(cu[-1])
    L = layout(B, H, N, d, total)
    T = L["T"]
    for name, X, off, soff in (("Q", qkv[0], L["qf"], L["sq"]), ("K", qkv[1], L["kf"], L["sk"])):
        got_scales = ws[soff:soff + B * H * T * 4].view(np.float32).reshape(B, H, T)
        codes = ws[off:off + total * H * d].reshape(total, H, d)
        for b in range(B):
            s0, s1 = int(cu[b]), int(cu[b + 1])
            if s1 == s0:
                continue
            Xr = fp8.rotate(X[s0:s1].float().numpy()[None], signs)
            _, ref_scales = fp8.blockwise_qk(Xr)
            nt = ref_scales.shape[2]
            assert np.allclose(got_scales[b, :, :nt], ref_scales[0], rtol=1e-5), (name, b)
            per_row = np.repeat(ref_scales, 128, axis=2)[:, :, :s1 - s0].transpose(0, 2, 1)[..., None]
            assert_codes_match(codes[None, s0:s1], fp8.e4m3_round(Xr / per_row), f"{name} seq {b}")
    n_pad = 128 * T
    vt = ws[L["vt"]:L["vt"] + B * H * d * n_pad].reshape(B, H, d, n_pad)
    got_sv = ws[L["sv"]:L["sv"] + B * H * 4].view(np.float32).reshape(B, H)
    for b in range(B):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        ref, ref_sv = fp8.per_head_v_fp32(qkv[2][s0:s1].float().numpy()[None])
        assert np.array_equal(got_sv[b], ref_sv[0]), b
        got = e4m3_decode(np.ascontiguousarray(vt[b, :, :, :s1 - s0]))       # [H, d, L]
        assert np.array_equal(got, ref[0].transpose(1, 2, 0)), f"V' codes seq {b}"
        assert not np.any(vt[b, :, :, s1 - s0:128 * ((s1 - s0 + 127) // 128)]), "padding keys"


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_packed_matches_reference(dev, causal):
    """O and lse of every row of a packed batch against the reference run
    sequence by sequence (the lse bound of check_against_reference, per
    sequence)."""
    import workloads
    H, d = 2, 128
    qkv, signs = make_packed(PACKED_LENS, H, d, seed=71 + causal)
    O, lse, _ = run_packed(qkv, signs, PACKED_LENS, causal, dev)
    device_error_clear()
    cu = workloads.cu_seqlens_of(PACKED_LENS)
    for b in range(len(PACKED_LENS)):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        seq = [t[s0:s1][None] for t in qkv]
        check_against_reference(O[None, s0:s1], lse[None, :, s0:s1], seq, signs, causal,
                                f"packed seq {b} ({s1 - s0} tokens)")


def test_fp8_packed_equal_lengths_is_the_dense_call(dev):
    """Packed sequences of one length give the dense call's bits."""
    B, H, N, d = 2, 3, 300, 128
    (Q, K, V), signs = make(B, H, N, d, seed=81)
    O_d, l_d, _ = run((Q, K, V), signs, True, dev)
    O_p, l_p, _ = run_packed([t.reshape(B * N, H, d) for t in (Q, K, V)], signs, [N] * B, True,
                             dev)
    assert np.array_equal(O_p, O_d.reshape(B * N, H, d))
    assert np.array_equal(l_p, l_d.transpose(1, 0, 2).reshape(H, B * N))


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
