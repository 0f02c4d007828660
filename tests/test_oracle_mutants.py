"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is the committed ``oracle/oracle.c`` with one plausible mistake
(a dropped term, a wrong sign, a wrong index, an off-by-one mask, a transposed
operand).  It is compiled on the CPU into a temporary library and the pins of
``tests/oracle_pins.py`` are run against it; a mutant that passes every pin
would mean the pins cannot see that kind of mistake.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement, occurrence index to replace)
MUTANTS = [
    ("softmax_min_not_max", "        if (xj > m)\n", "        if (xj < m)\n", 0),
    ("softmax_no_shift_in_sum", "        s += exp((double)x[j] - m);", "        s += exp((double)x[j]);", 0),
    ("softmax_no_normalise", "        y[j] = exp((double)x[j] - m) / s;", "        y[j] = exp((double)x[j] - m);", 0),
    ("merge_wrong_sign", "l = exp(m - mn) * l + exp(mb - mn) * lb;", "l = exp(mn - m) * l + exp(mb - mn) * lb;", 0),
    ("merge_keeps_old_max", "            m = mn;\n", "            m = m;\n", 0),
    ("causal_excludes_diagonal", "int64_t nvis = causal ? (i + 1 < L ? i + 1 : L) : L;", "int64_t nvis = causal ? (i < L ? i : L) : L;", 0),
    ("causal_sees_one_future_key", "int64_t nvis = causal ? (i + 1 < L ? i + 1 : L) : L;", "int64_t nvis = causal ? (i + 2 < L ? i + 2 : L) : L;", 0),
    ("scale_dropped", "        s[j] = scale * dot;", "        s[j] = dot;", 0),
    ("key_indexed_by_query", "const float *k = K + ((start + j) * H + h) * d;", "const float *k = K + ((start + i) * H + h) * d;", 0),
    ("value_indexed_by_query", "const float *v = V + ((start + j) * H + h) * d;", "const float *v = V + ((start + i) * H + h) * d;", 0),
    ("query_ignores_head", "const float *q = Q + ((start + i) * H + h) * d;", "const float *q = Q + ((start + i) * H) * d;", 0),
    ("q_and_k_swapped", "dot += (double)q[c] * (double)k[c];", "dot += (double)k[c] * (double)k[c];", 0),
    ("lse_drops_max", "*lse = nvis > 0 ? m + log(l) : -INFINITY;", "*lse = nvis > 0 ? log(l) : -INFINITY;", 0),
    ("lse_log2", "*lse = nvis > 0 ? m + log(l) : -INFINITY;", "*lse = nvis > 0 ? m + log2(l) : -INFINITY;", 0),
    ("p_not_normalised", "double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);", 0),
    ("p_unshifted", "double p = exp(s[j] - m) / l;", "double p = exp(s[j]) / l;", 0),
    ("varlen_start_zero", "            int64_t start = cu_seqlens[b];\n", "            int64_t start = 0;\n", 0),
    ("varlen_length_is_total", "            int64_t L = (int64_t)cu_seqlens[b + 1] - start;\n", "            int64_t L = (int64_t)cu_seqlens[B] - start;\n", 0),
    ("owner_off_by_one", "if ((int64_t)cu_seqlens[mid] <= t)", "if ((int64_t)cu_seqlens[mid] < t)", 0),
    ("online_no_correction", "                l *= corr;\n", "", 0),
    ("online_acc_no_correction", "                    acc[c] *= corr;\n", "", 0),
    ("rows_wrong_lse_slot", "O_rows + r * d, lse_rows + r);", "O_rows + r * d, lse_rows + (r > 0 ? r - 1 : 0));", 0),
    ("qk_top_left_causal", "int64_t nvis = causal ? i + (Nk - Nq) + 1 : Nk;", "int64_t nvis = causal ? i + 1 : Nk;", 0),
    ("qk_offset_sign", "int64_t nvis = causal ? i + (Nk - Nq) + 1 : Nk;", "int64_t nvis = causal ? i + (Nq - Nk) + 1 : Nk;", 0),
    ("qk_key_stride_uses_nq", "const float *k = K + ((b * Nk + j) * H + h) * d;", "const float *k = K + ((b * Nq + j) * H + h) * d;", 0),
    ("qk_sample_head_ignored", "                h = samp_h[r];", "                h = 0;", 0),
    ("bwd_ds_wrong_sign", "dP[i * N + j] = P[i * N + j] * (dP[i * N + j] - Di);", "dP[i * N + j] = P[i * N + j] * (dP[i * N + j] + Di);", 0),
    ("bwd_ds_no_jacobian_term", "dP[i * N + j] = P[i * N + j] * (dP[i * N + j] - Di);", "dP[i * N + j] = P[i * N + j] * dP[i * N + j];", 0),
    ("bwd_dq_scale_dropped", "ROW(dQ, i)[c] = scale * acc;", "ROW(dQ, i)[c] = acc;", 0),
    ("bwd_dk_uses_keys", "acc_k += dP[i * N + j] * (double)ROW(Q, i)[c];", "acc_k += dP[i * N + j] * (double)ROW(K, i)[c];", 0),
    ("bwd_dv_transposed_p", "acc_v += P[i * N + j] * (double)ROW(dO, i)[c];", "acc_v += P[j * N + i] * (double)ROW(dO, i)[c];", 0),
    ("bwd_causal_dk_misses_diagonal", "for (int64_t i = causal ? j : 0; i < N; ++i) {\n                    acc_k", "for (int64_t i = causal ? j + 1 : 0; i < N; ++i) {\n                    acc_k", 0),
    ("bwd_p_uses_max_not_lse", "P[i * N + j] = exp(P[i * N + j] - L);   /* [FG] §2.4 */", "P[i * N + j] = exp(P[i * N + j] - m);   /* [FG] §2.4 */", 0),
    ("bwd_head_ds_wrong_sign", "const double dS = P * (pdot - Dv[i]);\n                for (int64_t c = 0; c < d; ++c)\n                    out", "const double dS = P * (pdot + Dv[i]);\n                for (int64_t c = 0; c < d; ++c)\n                    out", 0),
]


# Mistakes planted in copies of ``oracle/fp8.py`` (the FP8 method's rotation
# and quantisation), run against the FP8 pins.
FP8_MUTANTS = [
    ("fp8_hadamard_block_sign", "H = np.block([[H, H], [H, -H]])", "H = np.block([[H, H], [-H, H]])", 0),
    ("fp8_rotation_unnormalised", "return (s[:, None] * sylvester_hadamard(d)) / math.sqrt(d)",
     "return s[:, None] * sylvester_hadamard(d)", 0),
    ("fp8_rotation_signs_on_columns", "(s[:, None] * sylvester_hadamard(d))",
     "(sylvester_hadamard(d) * s[None, :])", 0),
    ("fp8_e4m3_truncates", "np.round(a / ulp)", "np.floor(a / ulp)", 0),
    ("fp8_e4m3_max_240", "E4M3_MAX = 448.0", "E4M3_MAX = 240.0", 0),
    ("fp8_e4m3_subnormal_binade", "e = np.maximum(ex - 1, -6)", "e = np.maximum(ex - 1, -7)", 0),
    ("fp8_e4m3_two_fraction_bits", "ulp = np.ldexp(1.0, e - 3)", "ulp = np.ldexp(1.0, e - 2)", 0),
    ("fp8_scale_over_256", "amax / E4M3_MAX, 1.0", "amax / 256.0, 1.0", 0),
    ("fp8_tile_64_rows", "TILE_ROWS = 128", "TILE_ROWS = 64", 0),
    ("fp8_block_amax_signed", "sc = _scale_of(np.abs(blk).max(axis=(1, 3)))",
     "sc = _scale_of(blk.max(axis=(1, 3)))", 0),
    ("fp8_v_unquantised", "blockwise_qk(Kr)[0], per_head_v(V)[0]",
     "blockwise_qk(Kr)[0], np.asarray(V, dtype=np.float64)", 0),
    ("fp8_v_per_tensor", "blockwise_qk(Kr)[0], per_head_v(V)[0]",
     "blockwise_qk(Kr)[0], per_tensor(V)[0]", 0),
    ("fp8_q_unrotated", "Qr = rotate(Q, signs) if rotate_qk", "Qr = np.asarray(Q, dtype=np.float64) if rotate_qk", 0),
    ("fp8_k_unrotated", "Kr = rotate(K, signs) if rotate_qk", "Kr = np.asarray(K, dtype=np.float64) if rotate_qk", 0),
]


# Mistakes planted in copies of ``oracle/__init__.py``: the Python layer that
# lays out the C oracle's results and slices packed batches per sequence.
PY_MUTANTS = [
    ("dense_lse_layout", "lse.reshape(H, B, N).transpose(1, 0, 2).copy()", "lse.reshape(B, H, N).copy()", 0),
    ("qk_lse_layout", "lse.reshape(B, Nq, H).transpose(0, 2, 1).copy()", "lse.reshape(B, H, Nq).copy()", 0),
    ("qk_packed_keys_at_query_offsets", "K[None, k0:k1], V[None, k0:k1]", "K[None, q0:q1], V[None, q0:q1]", 0),
    ("qk_packed_values_at_query_offsets", "K[None, k0:k1], V[None, k0:k1]", "K[None, k0:k1], V[None, q0:q1]", 0),
    ("bwd_packed_d_from_lse", 'out["D"][:, s0:s1] = g["D"][0]', 'out["D"][:, s0:s1] = g["lse"][0]', 0),
    ("bwd_packed_v_and_do_swapped", "for X in (Q, K, V, dO)), scale", "for X in (Q, K, dO, V)), scale", 0),
    ("bwd_packed_skips_last_sequence", "    for b in range(cu.size - 1):\n        s0, s1 = int(cu[b]), int(cu[b + 1])\n        if s1 == s0:\n            continue\n        g =",
     "    for b in range(cu.size - 2):\n        s0, s1 = int(cu[b]), int(cu[b + 1])\n        if s1 == s0:\n            continue\n        g =", 0),
]


def _mutate(src, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = src.find(old, idx + 1)
        if idx < 0:
            raise AssertionError(f"mutation target not found: {old!r}")
    return src[:idx] + new + src[idx + len(old):]


_RUNNER = r"""
import sys
sys.path[:0] = [p for p in sys.argv[1].split("|") if p] + [sys.argv[2]]
import oracle, oracle_pins
print("ORACLE_PACKAGE", oracle.__file__)
lib = oracle.load(sys.argv[3])
prefix = sys.argv[4] if len(sys.argv) > 4 else "pin_"
failed = []
for pin in [p for p in oracle_pins.PINS if p.__name__.startswith(prefix)]:
    try:
        pin(lib)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED_PINS", ",".join(failed))
sys.exit(0 if failed else 3)
"""


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    """A mutant is caught when some pin fails, or when it crashes outright
    (a wrong index may run past a buffer); it runs in a child process so a
    crash cannot take the test session down."""
    src = open(SRC, encoding="utf-8").read()
    mutated = _mutate(src, old, new, occ)
    c_path = tmp_path / f"{name}.c"
    c_path.write_text(mutated, encoding="utf-8")
    so = oracle.compile_oracle(str(c_path), str(tmp_path / f"lib{name}.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    tests = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _RUNNER, root, tests, so],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 3, f"mutant {name} passed every pin"


def _run_package_mutant(tmp_path, fname, name, old, new, occ, prefix):
    """A copy of the oracle package whose ``fname`` holds the mistake, first on
    the path of a child process that runs the pins named ``prefix*``."""
    pkg = os.path.dirname(oracle.__file__)
    dst = tmp_path / "oracle"
    dst.mkdir()
    for f in ("__init__.py", "fp8.py", "oracle.c"):
        text = open(os.path.join(pkg, f), encoding="utf-8").read()
        (dst / f).write_text(_mutate(text, old, new, occ) if f == fname else text,
                             encoding="utf-8")
    so = oracle.compile_oracle(SRC, str(tmp_path / "liboracle.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    tests = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _RUNNER, f"{tmp_path}|{root}", tests, so, prefix],
                       capture_output=True, text=True, timeout=300)
    assert f"ORACLE_PACKAGE {dst / '__init__.py'}" in r.stdout, (r.stdout, r.stderr[-2000:])
    assert r.returncode != 3, f"mutant {name} passed every pin named {prefix}*"


@pytest.mark.parametrize("name,old,new,occ", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_mutant_is_caught(tmp_path, name, old, new, occ):
    """The same for the FP8 method's Python steps, against the FP8 pins."""
    _run_package_mutant(tmp_path, "fp8.py", name, old, new, occ, "pin_fp8")


@pytest.mark.parametrize("name,old,new,occ", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_binding_mutant_is_caught(tmp_path, name, old, new, occ):
    """The same for the oracle's Python layer (layouts of the row statistics,
    per-sequence slicing of packed batches), against every pin."""
    _run_package_mutant(tmp_path, "__init__.py", name, old, new, occ, "pin_")
