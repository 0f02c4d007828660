"""fp64 CPU oracle for the row softmax and the attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, OpenMP over rows);
this module only compiles it with gcc and marshals numpy arrays through ctypes.
Which page and section each function follows is stated in ``oracle.c``.

Parity status of the functions below: every one is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle.py`` (worked values printed on
the pages, closed forms, invariants, independent library routines and brute
force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None


def compile_oracle(src_path: str = _SRC, out_path: str = _LIB_PATH) -> str:
    """Compile an oracle source file into a shared library with gcc.

    -O2 without -ffast-math keeps every double operation IEEE (no reassociation,
    no contraction into FMA across statements that would change results in a
    way a reader cannot see; -ffp-contract=off makes that explicit).
    """
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
           "-shared", "-std=c11", src_path, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Build ``_build/liboracle.so`` if it is missing or older than the source."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB_PATH


def _bind(lib):
    c_i64, c_dbl, c_int = ctypes.c_int64, ctypes.c_double, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_softmax_rows.argtypes = [vp, vp, c_i64, c_i64]
    lib.oracle_softmax_rows.restype = None
    lib.oracle_online_softmax_state.argtypes = [vp, c_i64, vp, c_i64, vp, vp]
    lib.oracle_online_softmax_state.restype = None
    lib.oracle_attention_fwd.argtypes = [vp, vp, vp, vp, vp, c_i64, c_i64, c_i64, c_dbl,
                                         c_int, vp]
    lib.oracle_attention_fwd.restype = None
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, c_i64, c_i64, c_i64, c_dbl, c_int, vp,
                                          vp, vp, c_i64, vp, vp]
    lib.oracle_attention_rows.restype = None
    lib.oracle_attention_fwd_online.argtypes = [vp, vp, vp, vp, vp, c_i64, c_i64, c_i64,
                                                c_dbl, c_int, vp, c_i64]
    lib.oracle_attention_fwd_online.restype = None
    lib.oracle_attention_qk.argtypes = [vp, vp, vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_dbl,
                                        c_int, vp, vp, vp, c_i64, vp, vp]
    lib.oracle_attention_qk.restype = None
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, c_i64, c_dbl,
                                         c_int, vp, vp, vp, vp, vp, vp]
    lib.oracle_attention_bwd.restype = None
    lib.oracle_attention_bwd_head.argtypes = [vp, vp, vp, vp, c_i64, c_i64, c_i64, c_i64,
                                              c_dbl, c_int, c_i64, c_i64, vp, c_i64, vp, c_i64,
                                              vp, vp, vp]
    lib.oracle_attention_bwd_head.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = c_int
    lib.oracle_set_num_threads.argtypes = [c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.

    ``path`` loads another build of an oracle source (the mutation tests use
    it); the default is the committed ``oracle.c``.
    """
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _f32(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return np.ascontiguousarray(a)


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    """Thread count of the oracle's parallel loops from now on (for timing)."""
    (lib or load()).oracle_set_num_threads(int(n))


def softmax_rows(x, lib=None) -> np.ndarray:
    """Stable row softmax of a 2-D array (cast to fp32, as the GPU path sees it).

    Returns float64 [rows, N].
    """
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    rows, N = x.shape
    y = np.empty((rows, N), dtype=np.float64)
    (lib or load()).oracle_softmax_rows(_ptr(x), _ptr(y), rows, N)
    return y


def online_softmax_state(x, block_ends, lib=None):
    """(m, l) of a 1-D row consumed block by block with the online merge rule."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    ends = np.ascontiguousarray(np.asarray(block_ends, dtype=np.int64))
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    (lib or load()).oracle_online_softmax_state(_ptr(x), x.size, _ptr(ends), ends.size,
                                                 _ptr(m), _ptr(l))
    return float(m[0]), float(l[0])


def _cu(cu_seqlens) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))


def attention_packed(Q, K, V, cu_seqlens, scale, causal, lib=None, online_tile=None):
    """Exact attention over packed sequences.

    Q, K, V: [total, H, d] (any float dtype; cast to fp32, exact for bf16 values).
    cu_seqlens: [B+1] prefix sums.  Returns (O [total, H, d] f64, lse [H, total] f64).
    ``online_tile`` selects the tiled online recurrence (cross-check only).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    total, H, d = Q.shape
    cu = _cu(cu_seqlens)
    B = cu.size - 1
    if int(cu[-1]) != total:
        raise ValueError("cu_seqlens[-1] must equal the number of packed tokens")
    O = np.zeros((total, H, d), dtype=np.float64)
    lse = np.zeros((H, total), dtype=np.float64)
    lib = lib or load()
    if online_tile is None:
        lib.oracle_attention_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), B, H, d,
                                 float(scale), int(bool(causal)), _ptr(cu))
    else:
        lib.oracle_attention_fwd_online(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), B, H,
                                        d, float(scale), int(bool(causal)), _ptr(cu),
                                        int(online_tile))
    return O, lse


def attention_dense(Q, K, V, scale, causal, lib=None, online_tile=None):
    """Exact attention on a dense batch.

    Q, K, V: [B, N, H, d].  Returns (O [B, N, H, d] f64, lse [B, H, N] f64).
    """
    Q = np.asarray(Q)
    B, N, H, d = Q.shape
    cu = np.arange(B + 1, dtype=np.int32) * N
    O, lse = attention_packed(np.reshape(Q, (B * N, H, d)), np.reshape(K, (B * N, H, d)),
                              np.reshape(V, (B * N, H, d)), cu, scale, causal, lib=lib,
                              online_tile=online_tile)
    return O.reshape(B, N, H, d), lse.reshape(H, B, N).transpose(1, 0, 2).copy()


def attention_rows(Q, K, V, cu_seqlens, scale, causal, tok, head, lib=None):
    """The attention definition on sampled (token, head) pairs of a packed batch.

    Returns (O_rows [n, d] f64, lse_rows [n] f64).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    total, H, d = Q.shape
    cu = _cu(cu_seqlens)
    B = cu.size - 1
    tok = np.ascontiguousarray(np.asarray(tok, dtype=np.int64))
    head = np.ascontiguousarray(np.asarray(head, dtype=np.int64))
    if tok.shape != head.shape:
        raise ValueError("tok and head must have the same shape")
    if tok.size and (tok.min() < 0 or tok.max() >= total or head.min() < 0 or head.max() >= H):
        raise ValueError("sample index out of range")
    n = tok.size
    O = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    (lib or load()).oracle_attention_rows(_ptr(Q), _ptr(K), _ptr(V), B, H, d, float(scale),
                                          int(bool(causal)), _ptr(cu), _ptr(tok), _ptr(head),
                                          n, _ptr(O), _ptr(lse))
    return O, lse


def attention_qk(Q, K, V, scale, causal, samples=None, lib=None):
    """Attention with separate query / key lengths on dense batches.

    Q: [B, Nq, H, d]; K, V: [B, Nk, H, d]; causal is bottom-right aligned
    (query i sees keys j <= i + Nk - Nq).  Without ``samples`` returns
    (O [B, Nq, H, d] f64, lse [B, H, Nq] f64); with ``samples`` = (b, i, h)
    index arrays returns (O_rows [n, d], lse_rows [n]).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Nq, H, d = Q.shape
    Nk = K.shape[1]
    if K.shape != (B, Nk, H, d) or V.shape != K.shape:
        raise ValueError("K and V must be [B, Nk, H, d] with Q's B, H, d")
    lib = lib or load()
    if samples is None:
        n = B * Nq * H
        O = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        lib.oracle_attention_qk(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d, float(scale),
                                int(bool(causal)), None, None, None, n, _ptr(O), _ptr(lse))
        return O.reshape(B, Nq, H, d), lse.reshape(B, Nq, H).transpose(0, 2, 1).copy()
    sb, si, sh = (np.ascontiguousarray(np.asarray(a, dtype=np.int64)) for a in samples)
    if not (sb.shape == si.shape == sh.shape):
        raise ValueError("sample arrays must have one shape")
    if sb.size and (sb.min() < 0 or sb.max() >= B or si.min() < 0 or si.max() >= Nq
                    or sh.min() < 0 or sh.max() >= H):
        raise ValueError("sample index out of range")
    n = sb.size
    O = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    lib.oracle_attention_qk(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d, float(scale),
                            int(bool(causal)), _ptr(sb), _ptr(si), _ptr(sh), n, _ptr(O),
                            _ptr(lse))
    return O, lse


def attention_qk_packed(Q, K, V, cu_seqlens_q, cu_seqlens_k, scale, causal, lib=None):
    """Attention with separate query / key lengths on packed sequences.

    Q: [total_q, H, d]; K, V: [total_k, H, d]; sequence b owns query rows
    cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] ..
    cu_seqlens_k[b+1]-1, and attends to nothing else ("第二十二课…" §三十五).
    causal is bottom-right aligned within each sequence (query i sees keys
    j <= i + Lk - Lq).  Each sequence is attention_qk's dense case with B = 1.
    Returns (O [total_q, H, d] f64, lse [H, total_q] f64).
    """
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    cq, ck = _cu(cu_seqlens_q), _cu(cu_seqlens_k)
    if cq.size != ck.size:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have one length")
    total_q, H, d = Q.shape
    if int(cq[-1]) != total_q or int(ck[-1]) != K.shape[0] or V.shape != K.shape:
        raise ValueError("prefix sums must end at the row counts of Q and K, V")
    O = np.zeros((total_q, H, d))
    lse = np.zeros((H, total_q))
    for b in range(cq.size - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        Ob, lb = attention_qk(Q[None, q0:q1], K[None, k0:k1], V[None, k0:k1], scale, causal,
                              lib=lib)
        O[q0:q1] = Ob[0]
        lse[:, q0:q1] = lb[0]
    return O, lse


def attention_bwd(Q, K, V, dO, scale, causal, lib=None):
    """Gradients of sum(dO * O) for dense Q, K, V, dO [B, N, H, d].

    Returns a dict of float64 arrays: dQ, dK, dV, O [B, N, H, d] and lse, D
    [B, H, N] (the row logsumexp and D_i = sum_j P_ij dP_ij).  Materialises
    N x N per (b, h): small N only.
    """
    Q, K, V, dO = _f32(Q), _f32(K), _f32(V), _f32(dO)
    B, N, H, d = Q.shape
    for t in (K, V, dO):
        if t.shape != Q.shape:
            raise ValueError("Q, K, V, dO must have one shape")
    out = {k: np.zeros((B, N, H, d)) for k in ("dQ", "dK", "dV", "O")}
    out["lse"] = np.zeros((B, H, N))
    out["D"] = np.zeros((B, H, N))
    (lib or load()).oracle_attention_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, d, float(scale), int(bool(causal)),
        _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]), _ptr(out["O"]), _ptr(out["lse"]),
        _ptr(out["D"]))
    return out


def attention_bwd_packed(Q, K, V, dO, cu_seqlens, scale, causal, lib=None):
    """Gradients of sum(dO * O) for packed sequences ("第二十二课…" §三十五:
    a packed batch is a row of sequences, none attending to another).

    Q, K, V, dO: [total, H, d]; cu_seqlens: [B+1] prefix sums.  Each sequence's
    gradients are those of its own attention, so the dense backward runs on
    each sequence's rows.  Returns a dict of float64 arrays: dQ, dK, dV, O
    [total, H, d] and lse, D [H, total] (the packed layout of the row
    statistics).
    """
    Q, K, V, dO = _f32(Q), _f32(K), _f32(V), _f32(dO)
    total, H, d = Q.shape
    for t in (K, V, dO):
        if t.shape != Q.shape:
            raise ValueError("Q, K, V, dO must have one shape")
    cu = _cu(cu_seqlens)
    if int(cu[-1]) != total:
        raise ValueError("cu_seqlens[-1] must equal the number of packed tokens")
    out = {k: np.zeros((total, H, d)) for k in ("dQ", "dK", "dV", "O")}
    out["lse"] = np.zeros((H, total))
    out["D"] = np.zeros((H, total))
    for b in range(cu.size - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        g = attention_bwd(*(X[None, s0:s1] for X in (Q, K, V, dO)), scale, causal, lib=lib)
        for k in ("dQ", "dK", "dV", "O"):
            out[k][s0:s1] = g[k][0]
        out["lse"][:, s0:s1] = g["lse"][0]
        out["D"][:, s0:s1] = g["D"][0]
    return out


def attention_bwd_head(Q, K, V, dO, scale, causal, b, h, q_idx, k_idx, lib=None):
    """dQ of the query rows q_idx and dK, dV of the keys k_idx for one (b, h).

    Returns (dQ_rows [len(q_idx), d], dK_rows, dV_rows [len(k_idx), d]) in float64.
    """
    Q, K, V, dO = _f32(Q), _f32(K), _f32(V), _f32(dO)
    B, N, H, d = Q.shape
    qi = np.ascontiguousarray(np.asarray(q_idx, dtype=np.int64))
    ki = np.ascontiguousarray(np.asarray(k_idx, dtype=np.int64))
    for a in (qi, ki):
        if a.size and (a.min() < 0 or a.max() >= N):
            raise ValueError("row index out of range")
    if not (0 <= b < B and 0 <= h < H):
        raise ValueError("(b, h) out of range")
    dq = np.zeros((qi.size, d))
    dk = np.zeros((ki.size, d))
    dv = np.zeros((ki.size, d))
    (lib or load()).oracle_attention_bwd_head(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, d, float(scale), int(bool(causal)), b, h,
        _ptr(qi), qi.size, _ptr(ki), ki.size, _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


if __name__ == "__main__":  # pragma: no cover - manual rebuild
    print(build(force="--force" in sys.argv))
