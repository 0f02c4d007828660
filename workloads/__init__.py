"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds only random-number draws, rounding to the storage dtype and
the shapes of the workloads; none of the method's arithmetic.  Both the CUDA
path and the fp64 oracle take their inputs from here, never from each other.

Recipe (the pages print no seeds or distributions beyond the shapes):
  * numpy ``default_rng(seed)``; float32 standard normals scaled by the stated
    standard deviation;
  * bf16 inputs are those float32 draws rounded to nearest-even bf16 by torch;
  * row softmax: x ~ N(0, 3^2); every row whose index is a multiple of 64 gets
    +1000 added to every entry (the overflow case of the stable-softmax
    lesson: 1000, 999, 998 overflow a naive exp);
  * packed variable-length batches: lengths drawn uniformly from [lo, hi]
    (both inclusive) and not rounded to tile multiples.

Named workloads (``WORKLOADS``) follow the five configurations the library is
measured on: single-head fp32 attention, the fp32 row softmax at five row
lengths, non-causal bf16 d=64, causal bf16 d=128, and causal varlen bf16
d=128 with Q, K ~ N(0, 2^2).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 1000


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal_f32(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def to_bf16(x: np.ndarray):
    """Round a float32 array to bf16 (nearest-even); returns a CPU torch tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def softmax_rows_input(rows: int, N: int, seed: int, std: float = 3.0,
                       shift_every: int = 64, shift: float = 1000.0) -> np.ndarray:
    """fp32 [rows, N]; N(0, std^2) entries, rows r % shift_every == 0 shifted by +shift."""
    x = normal_f32(rng_for(seed), (rows, N), std)
    if shift_every:
        x[::shift_every] += np.float32(shift)
    return x


def varlen_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Sequence lengths uniform in [lo, hi] (inclusive)."""
    return rng_for(seed).integers(lo, hi + 1, size=n_seqs).astype(np.int64)


def cu_seqlens_of(lengths) -> np.ndarray:
    """Prefix sums [0, L0, L0+L1, ...] as int32 (the packed-sequence index)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(lengths.size + 1, dtype=np.int64)
    np.cumsum(lengths, out=cu[1:])
    if cu[-1] > np.iinfo(np.int32).max:
        raise ValueError("packed length exceeds int32")
    return cu.astype(np.int32)


def attention_inputs(shape, seed: int, dtype: str = "bf16", q_std: float = 1.0,
                     k_std: float = 1.0, v_std: float = 1.0):
    """Q, K, V of the given shape, drawn in that order from one generator.

    dtype "f32" returns numpy float32 arrays; "bf16" returns CPU torch bf16
    tensors (the values the GPU sees; ``.float()`` is exact for the oracle).
    """
    rng = rng_for(seed)
    q = normal_f32(rng, shape, q_std)
    k = normal_f32(rng, shape, k_std)
    v = normal_f32(rng, shape, v_std)
    if dtype == "f32":
        return q, k, v
    if dtype == "bf16":
        return to_bf16(q), to_bf16(k), to_bf16(v)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    B: int
    H: int
    N: int                  # sequence length (dense) or longest sequence (varlen)
    d: int
    causal: bool
    dtype: str              # "f32" or "bf16"
    seed: int
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    lengths: tuple = field(default=())   # varlen only

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def varlen(self) -> bool:
        return len(self.lengths) > 0

    @property
    def total(self) -> int:
        return int(sum(self.lengths)) if self.varlen else self.B * self.N

    def cu_seqlens(self) -> np.ndarray:
        if self.varlen:
            return cu_seqlens_of(self.lengths)
        return cu_seqlens_of([self.N] * self.B)

    def flops(self) -> float:
        """Algorithmic flops: 4*N^2*d per (sequence, head), halved when causal."""
        lens = self.lengths if self.varlen else [self.N] * self.B
        f = sum(4.0 * self.H * L * L * self.d for L in lens)
        return f / 2 if self.causal else f

    def inputs(self):
        """Dense: [B, N, H, d]; varlen: packed [total, H, d]."""
        shape = (self.total, self.H, self.d) if self.varlen else (self.B, self.N, self.H, self.d)
        return attention_inputs(shape, self.seed, self.dtype, self.q_std, self.k_std,
                                self.v_std)


def _varlen_workload(name, n_seqs, lo, hi, H, d, seed, causal=True, q_std=2.0, k_std=2.0):
    lens = tuple(int(x) for x in varlen_lengths(n_seqs, lo, hi, seed))
    return AttentionWorkload(name=name, B=n_seqs, H=H, N=max(lens), d=d, causal=causal,
                             dtype="bf16", seed=seed, q_std=q_std, k_std=k_std, v_std=1.0,
                             lengths=lens)


@dataclass(frozen=True)
class SplitKVWorkload:
    """Nq queries against Nk keys per (sequence, head); causal is bottom-right
    aligned (query i sees keys j <= i + Nk - Nq)."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    dtype: str = "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def visible_keys(self):
        """Visible keys of each query position (array of Nq)."""
        i = np.arange(self.Nq, dtype=np.int64)
        if not self.causal:
            return np.full(self.Nq, self.Nk, dtype=np.int64)
        return np.minimum(i + (self.Nk - self.Nq) + 1, self.Nk)

    def flops(self) -> float:
        """Algorithmic flops: 4 * d per (query, visible key), summed."""
        return float(4.0 * self.d * self.B * self.H * self.visible_keys().sum())

    def inputs(self):
        """Q [B, Nq, H, d]; K, V [B, Nk, H, d]; N(0, 1) drawn in that order."""
        rng = rng_for(self.seed)
        q = normal_f32(rng, (self.B, self.Nq, self.H, self.d))
        k = normal_f32(rng, (self.B, self.Nk, self.H, self.d))
        v = normal_f32(rng, (self.B, self.Nk, self.H, self.d))
        return to_bf16(q), to_bf16(k), to_bf16(v)


SPLITKV_WORKLOADS = {
    # a block of 256 new queries against a 32K-token context, 16 heads: only 16
    # (sequence, head, query block) items without key splits
    "attn_bf16_splitkv_b1h16nq256nk32768d128_causal": SplitKVWorkload(
        "attn_bf16_splitkv_b1h16nq256nk32768d128_causal", B=1, H=16, Nq=256, Nk=32768, d=128,
        causal=True, seed=SEED_BASE + 6),
}


SOFTMAX_ROWS = 4096
SOFTMAX_NS = (32, 128, 1024, 4096, 32768)
SOFTMAX_SEED = SEED_BASE + 2

WORKLOADS = {
    "attn_f32_b1h1n256d64": AttentionWorkload(
        "attn_f32_b1h1n256d64", B=1, H=1, N=256, d=64, causal=False, dtype="f32",
        seed=SEED_BASE + 1),
    "attn_bf16_b8h16n2048d64": AttentionWorkload(
        "attn_bf16_b8h16n2048d64", B=8, H=16, N=2048, d=64, causal=False, dtype="bf16",
        seed=SEED_BASE + 3),
    "attn_bf16_causal_b2h32n4096d128": AttentionWorkload(
        "attn_bf16_causal_b2h32n4096d128", B=2, H=32, N=4096, d=128, causal=True,
        dtype="bf16", seed=SEED_BASE + 4),
    "attn_bf16_varlen8_h16d128_causal": _varlen_workload(
        "attn_bf16_varlen8_h16d128_causal", n_seqs=8, lo=512, hi=16384, H=16, d=128,
        seed=SEED_BASE + 5),
}


def softmax_workload(N: int, rows: int = SOFTMAX_ROWS, seed: int = SOFTMAX_SEED) -> np.ndarray:
    """The row-softmax input for one row length (a distinct stream per N)."""
    return softmax_rows_input(rows, N, seed * 100003 + N)


def rising_scores_inputs(B: int, N: int, H: int, d: int, seed: int, growth: float = 0.05):
    """Q, K, V (bf16, [B, N, H, d]) whose scores rise along the key index.

    Every query is a fixed direction u (plus small noise) and key j is
    (growth * j) * u plus noise, so each query's largest score sits at the last
    key it can see and its running maximum grows on every key tile: the
    rescale path runs on every tile.  The last key of each sequence is
    additionally scaled up by 4 so the final tile carries a large jump.
    """
    rng = rng_for(seed)
    u = normal_f32(rng, (1, 1, H, d))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    q = (u * np.float32(4.0) + normal_f32(rng, (B, N, H, d), 0.05)).astype(np.float32)
    steps = (np.arange(N, dtype=np.float32) * np.float32(growth)).reshape(1, N, 1, 1)
    k = (u * steps + normal_f32(rng, (B, N, H, d), 0.05)).astype(np.float32)
    k[:, -1] *= np.float32(4.0)
    v = normal_f32(rng, (B, N, H, d))
    return to_bf16(q), to_bf16(k), to_bf16(v)


def sample_rows(total: int, H: int, n: int, seed: int, must_tokens=()):
    """(token, head) pairs to check one by one: n random pairs plus every head of
    the listed tokens."""
    rng = rng_for(seed)
    tok = rng.integers(0, total, size=n)
    head = rng.integers(0, H, size=n)
    extra = np.asarray(list(must_tokens), dtype=np.int64)
    if extra.size:
        tok = np.concatenate([tok, np.repeat(extra, H)])
        head = np.concatenate([head, np.tile(np.arange(H), extra.size)])
    return tok.astype(np.int64), head.astype(np.int64)
