"""Seeded synthetic inputs for the attention forward, shared by the CUDA path's tests and bench
and by the oracle's tests.

This module draws random numbers and rounds them to the storage type; it holds none of the
attention arithmetic. Tensors are returned as numpy uint16 bit patterns in the [B, N, H, d]
layout, so that the CUDA path (after a byte copy to the device) and the oracle (which decodes
the same bits exactly) see identical inputs.

Recipe
------
* Q, K, V entries are iid N(0, 1) from numpy's PCG64 generator: seed s for Q, s + 1 for K,
  s + 2 for V (s = 1000 * workload index for the named workloads below).
* Optional stress transform, applied before rounding: Q multiplied by ``q_scale``; for each
  (b, h) a set of ``round(k_outlier_frac * N)`` distinct token positions, drawn with seed
  s + 3, has its K rows multiplied by ``k_outlier_scale``.
* Rounding to the storage type is round-to-nearest-even: fp16 through numpy's float16 cast;
  bf16 by rounding the float64 value to float32 and then the float32 bits to their upper
  16 bits. (The two-step bf16 rounding can differ from a one-step rounding in rare ties; that
  is irrelevant here because both sides consume the rounded bits.)
* The softmax scale is fp32(1 / sqrt(d)).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-forward problem: sizes, storage type, mask and input recipe."""
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16" or "fp16"
    causal: bool
    seed: int
    q_scale: float = 1.0
    k_outlier_frac: float = 0.0
    k_outlier_scale: float = 1.0
    Nk: int = 0           # keys (and values); 0 means N. Queries are then the last N positions.
    window: tuple = (-1, -1)   # sliding window (left, right); negative = unbounded
    seqlens_k: tuple = ()      # per-batch key lengths (padding mask); empty = all keys

    @property
    def scale(self) -> float:
        return softmax_scale(self.d)

    @property
    def n_keys(self) -> int:
        return self.Nk or self.N

    @property
    def masked(self) -> bool:
        """A padding or sliding-window mask besides (or instead of) the causal one."""
        return self.window != (-1, -1) or bool(self.seqlens_k)

    def describe(self) -> str:
        extra = ""
        if self.q_scale != 1.0 or self.k_outlier_frac:
            extra = ", Q x%g, %g%% of K rows x%g" % (self.q_scale, 100 * self.k_outlier_frac,
                                                      self.k_outlier_scale)
        if self.window != (-1, -1):
            extra += ", window (left, right) = (%d, %d)" % self.window
        if self.seqlens_k:
            extra += ", key lengths %s" % (list(self.seqlens_k),)
        n = ("N=%d" % self.N) if not self.Nk else ("Nq=%d Nk=%d" % (self.N, self.Nk))
        return "B=%d H=%d %s d=%d %s %s%s" % (self.B, self.H, n, self.d, self.dtype,
                                              "causal" if self.causal else "non-causal", extra)


# The five workloads (the second one in both mask modes). Sizes, types and input statistics
# follow the workloads stated for this attention forward; seeds are 1000 * index.
WORKLOADS = {
    "tiny_n256_d64": Workload("tiny_n256_d64", 1, 1, 256, 64, "bf16", False, 1000),
    "n1k_d64": Workload("n1k_d64", 4, 16, 1024, 64, "bf16", False, 2000),
    "n1k_d64_causal": Workload("n1k_d64_causal", 4, 16, 1024, 64, "bf16", True, 2000),
    "n8k_d128_causal": Workload("n8k_d128_causal", 2, 16, 8192, 128, "bf16", True, 3000),
    "n32k_d128_causal": Workload("n32k_d128_causal", 1, 8, 32768, 128, "bf16", True, 4000),
    "n2000_d128_fp16_stress": Workload("n2000_d128_fp16_stress", 16, 32, 2000, 128, "fp16",
                                       False, 5000, q_scale=8.0, k_outlier_frac=0.01,
                                       k_outlier_scale=10.0),
    # The shapes of the pages' fused-vs-standard comparison (d = 128 at N = 1K and 8K; batch and
    # heads are not stated there, 2 x 16 is used).
    "n1k_d128": Workload("n1k_d128", 2, 16, 1024, 128, "bf16", False, 6000),
    "n8k_d128": Workload("n8k_d128", 2, 16, 8192, 128, "bf16", False, 7000),
    # One decoding step against a long sequence (the FlashDecoding case the pages mention for
    # N > 32K): 1 query per (b, h) attends to 65536 cached keys.
    "decode_nk64k_d128": Workload("decode_nk64k_d128", 4, 32, 1, 128, "bf16", True, 8000,
                                  Nk=65536),
    # The extra masks at the headline shape: a causal sliding window of 1024 keys (the query and
    # the 1023 before it), and key padding with the second sequence 5000 keys long.
    "n8k_d128_window1k": Workload("n8k_d128_window1k", 2, 16, 8192, 128, "bf16", True, 9000,
                                  window=(1023, -1)),
    "n8k_d128_padded": Workload("n8k_d128_padded", 2, 16, 8192, 128, "bf16", False, 10000,
                                seqlens_k=(8192, 5000)),
}


def softmax_scale(d: int) -> float:
    """fp32(1/sqrt(d)) as a Python float (exactly the fp32 value)."""
    return float(np.float32(1.0 / math.sqrt(d)))


def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round a real array to bf16/fp16 (nearest-even) and return the uint16 bit patterns."""
    x = np.asarray(x)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        f32 = x.astype(np.float32)
        u = f32.view(np.uint32).astype(np.uint64)
        # round-to-nearest-even on the 16 dropped bits; NaN is not produced by this generator
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return u.astype(np.uint16)
    raise ValueError("dtype must be 'bf16' or 'fp16'")


def normal(shape, seed: int) -> np.ndarray:
    """iid N(0, 1) float64 values from PCG64(seed)."""
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def make_qkv(B: int, H: int, N: int, d: int, dtype: str, seed: int, q_scale: float = 1.0,
             k_outlier_frac: float = 0.0, k_outlier_scale: float = 1.0, Nk: int | None = None):
    """Q [B, N, H, d] and K, V [B, Nk, H, d] (Nk defaults to N) as uint16 bit arrays following
    the recipe above."""
    Nk = N if not Nk else Nk
    q = normal((B, N, H, d), seed)
    shape = (B, Nk, H, d)
    if q_scale != 1.0:
        q *= q_scale
    qb = round_to_bits(q, dtype)
    del q
    k = normal(shape, seed + 1)
    n_out = int(round(k_outlier_frac * Nk))
    if n_out > 0 and k_outlier_scale != 1.0:
        rng = np.random.Generator(np.random.PCG64(seed + 3))
        for b in range(B):
            for h in range(H):
                pos = rng.choice(Nk, size=n_out, replace=False)
                k[b, pos, h, :] *= k_outlier_scale
    kb = round_to_bits(k, dtype)
    del k
    vb = round_to_bits(normal(shape, seed + 2), dtype)
    return qb, kb, vb


def make_workload(w: Workload):
    """Q, K, V bit arrays for a named workload."""
    return make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.q_scale, w.k_outlier_frac,
                    w.k_outlier_scale, Nk=w.Nk or None)


def sample_rows(B: int, H: int, N: int, per_head: int, seed: int) -> np.ndarray:
    """(b, h, i) triples for sampled parity checks: every (b, h) with rows 0, 1, N-1 and the
    last row of each 128-row tile boundary neighbourhood, plus ``per_head`` seeded rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    fixed = sorted({0, min(1, N - 1), N - 1, min(127, N - 1), min(128, N - 1)})
    for b in range(B):
        for h in range(H):
            rows = set(fixed)
            rows.update(int(r) for r in rng.integers(0, N, size=per_head))
            out.extend((b, h, r) for r in sorted(rows))
    return np.array(out, dtype=np.int64)
