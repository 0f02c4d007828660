"""FP8 attention forward, reference side (TEST INFRASTRUCTURE ONLY).

The method of "少搬一趟：FlashAttention 四代进化史" §4.6 (FP8 with blockwise
quantisation and incoherent processing), step by step in float64 on the CPU:

  1. incoherent processing: Q and K are multiplied by the same random
     orthogonal matrix M = diag(signs) H_d / sqrt(d) (random +-1 signs, the
     Sylvester-Hadamard matrix H_d); (QM)(KM)^T = Q M M^T K^T = Q K^T;
  2. blockwise quantisation: one scale per block instead of one per tensor --
     Q and K per (sequence, head, 128-row tile), V per (sequence, head) -- with
     scale = amax(block) / 448 (the largest e4m3 value), values x / scale
     rounded to e4m3 (round to nearest even, saturating at +-448);
  3. attention on the dequantised values (the fp64 oracle).

``per_tensor=True, rotate=False`` gives the baseline the pages compare with
(one scale per tensor, no rotation).  Only tests, the smoke check and the
benchmark's CPU leg use this module; the library does not.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
TILE_ROWS = 128


def sylvester_hadamard(d: int) -> np.ndarray:
    """H_1 = [1]; H_2n = [[H_n, H_n], [H_n, -H_n]] (entries +-1, d a power of 2)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotation_matrix(signs) -> np.ndarray:
    """M = diag(signs) H_d / sqrt(d): orthogonal, M M^T = I."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.size
    return (s[:, None] * sylvester_hadamard(d)) / math.sqrt(d)


def rotate(X, signs) -> np.ndarray:
    """X M over the last axis, in float64."""
    return np.asarray(X, dtype=np.float64) @ rotation_matrix(signs)


def e4m3_round(x) -> np.ndarray:
    """Round float64 values to e4m3 (nearest, ties to even, saturating at
    +-448) in one step from the float64 value.

    e4m3 has 3 fraction bits: in the binade [2^e, 2^(e+1)) the spacing is
    2^(e-3), and below the smallest normal 2^-6 the subnormal spacing is 2^-9;
    so a value is rounded to an integer multiple of its spacing (an exact
    power-of-two scaling in float64; numpy rounds halves to even).  Going
    through float32 first would round twice: a value just above a half-way
    point can become the half-way point and then go to the even neighbour.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(a)                       # a = m 2^ex, m in [0.5, 1): binade ex - 1
    e = np.maximum(ex - 1, -6)
    ulp = np.ldexp(1.0, e - 3)
    q = np.minimum(np.round(a / ulp) * ulp, E4M3_MAX)
    return np.copysign(q, x)


def _scale_of(amax):
    amax = np.asarray(amax, dtype=np.float64)
    return np.where(amax > 0, amax / E4M3_MAX, 1.0)


def blockwise_qk(X):
    """Quantise a [B, N, H, d] tensor per (b, h, 128-row tile).

    Returns (dequantised float64 [B, N, H, d], scales [B, H, n_tiles])."""
    X = np.asarray(X, dtype=np.float64)
    B, N, H, d = X.shape
    nt = (N + TILE_ROWS - 1) // TILE_ROWS
    out = np.empty_like(X)
    scales = np.empty((B, H, nt))
    for t in range(nt):
        blk = X[:, t * TILE_ROWS:(t + 1) * TILE_ROWS]             # [B, rows, H, d]
        sc = _scale_of(np.abs(blk).max(axis=(1, 3)))              # [B, H]
        scales[:, :, t] = sc
        s4 = sc[:, None, :, None]
        out[:, t * TILE_ROWS:(t + 1) * TILE_ROWS] = e4m3_round(blk / s4) * s4
    return out, scales


def per_head_v(V):
    """Quantise V [B, N, H, d] with one scale per (b, h).  Returns (deq, scales [B, H])."""
    V = np.asarray(V, dtype=np.float64)
    sc = _scale_of(np.abs(V).max(axis=(1, 3)))
    s4 = sc[:, None, :, None]
    return e4m3_round(V / s4) * s4, sc


def per_head_v_fp32(V):
    """V's e4m3 codes with the rounding decision taken in float32, as the GPU
    takes it (the pages fix no precision): sv = amax / 448 and 1 / sv rounded
    to float32, x = v * (1 / sv) rounded to float32, then one rounding to e4m3.
    A code is an integer decided by floating point, so both sides decide it in
    the same precision.  Returns (codes as float64 values [B, N, H, d],
    sv [B, H] float32)."""
    V32 = np.asarray(V, dtype=np.float32)
    amax = np.abs(V32).max(axis=(1, 3))
    sv = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / sv).astype(np.float32)
    x = (V32 * inv[:, None, :, None]).astype(np.float32)
    return e4m3_round(x.astype(np.float64)), sv


def per_tensor(X):
    X = np.asarray(X, dtype=np.float64)
    sc = float(_scale_of(np.abs(X).max()))
    return e4m3_round(X / sc) * sc, sc


def fp8_inputs(Q, K, V, signs, per_tensor_scales=False, rotate_qk=True):
    """The dequantised (Q', K', V') the FP8 method multiplies, in float64."""
    Qr = rotate(Q, signs) if rotate_qk else np.asarray(Q, dtype=np.float64)
    Kr = rotate(K, signs) if rotate_qk else np.asarray(K, dtype=np.float64)
    if per_tensor_scales:
        return per_tensor(Qr)[0], per_tensor(Kr)[0], per_tensor(V)[0]
    return blockwise_qk(Qr)[0], blockwise_qk(Kr)[0], per_head_v(V)[0]


def fp8_attention(Q, K, V, signs, scale, causal, per_tensor_scales=False, rotate_qk=True,
                  lib=None):
    """Attention (fp64 oracle) on the FP8 method's dequantised inputs.

    Returns (O [B, N, H, d], lse [B, H, N]) in float64."""
    from . import attention_dense
    Qd, Kd, Vd = fp8_inputs(Q, K, V, signs, per_tensor_scales, rotate_qk)
    # the C oracle takes float32 inputs: the dequantised values are e4m3 codes
    # times a scale, rounded here to float32 (relative 6e-8, far below e4m3's
    # 2^-4)
    return attention_dense(Qd.astype(np.float32), Kd.astype(np.float32),
                           Vd.astype(np.float32), scale, causal, lib=lib)


def fp8_attention_packed(Q, K, V, cu_seqlens, signs, scale, causal, lib=None):
    """The FP8 method on packed sequences: each sequence is quantised on its
    own (Q and K tiles of 128 rows from the sequence's first token, one V scale
    per (sequence, head)) and attends only to itself.

    Q, K, V: [total, H, d]; cu_seqlens: [B+1].  Returns (O [total, H, d],
    lse [H, total]) in float64."""
    Q, K, V = (np.asarray(X) for X in (Q, K, V))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total, H, d = Q.shape
    O = np.zeros((total, H, d))
    lse = np.zeros((H, total))
    for b in range(cu.size - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        Ob, lb = fp8_attention(Q[None, s0:s1], K[None, s0:s1], V[None, s0:s1], signs, scale,
                               causal, lib=lib)
        O[s0:s1] = Ob[0]
        lse[:, s0:s1] = lb[0]
    return O, lse

