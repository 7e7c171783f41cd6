"""Seeded synthetic inputs for the attention forward pass.

This module only draws random inputs and describes workload shapes; it holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle
can be fed from it without sharing any of the method.

Recipe (the same on every machine):

* ``torch.Generator("cpu").manual_seed(seed)``; Q, then K, then V drawn with
  ``torch.randn`` in float32 in that order, each of the full tensor shape;
* Q and K multiplied by ``qk_mult`` (2 for the sharp-softmax workload; an
  exact power-of-two scaling) before the cast;
* then cast to the storage dtype (bfloat16 rounds to nearest even);
* variable-length batches draw their lengths with
  ``numpy.random.default_rng(len_seed).integers(lo, hi + 1, num_seqs)``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def default_scale(D: int) -> float:
    """``float32(1 / sqrt(D))`` as a Python float (0.125 exactly for D=64)."""
    return float(np.float32(1.0 / math.sqrt(D)))


@dataclass(frozen=True)
class Workload:
    """One attention forward problem.

    Dense workloads have ``B, H, N, D`` and layout ``[B, H, N, D]``.
    Variable-length workloads have ``lengths`` (one per sequence) and layout
    ``[total, H, D]`` with ``cu_seqlens`` prefix offsets; ``B``/``N`` are then
    unused.  ``window=(wl, wr)`` (dense only) restricts query i to the keys
    ``i - wl .. i + wr``, -1 leaving a side unbounded.
    """

    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str
    causal: bool
    seed: int
    qk_mult: float = 1.0
    lengths: tuple = field(default=())
    window: tuple = field(default=())

    @property
    def varlen(self) -> bool:
        return len(self.lengths) > 0

    @property
    def scale(self) -> float:
        return default_scale(self.D)

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    @property
    def total(self) -> int:
        return int(sum(self.lengths)) if self.varlen else self.B * self.N

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lengths)) if self.varlen else self.N

    def visible_range(self, rows, n: int):
        """First and last key position (lo, hi) that each query row of a
        sequence of n attends to under the workload's mask; hi < lo when
        none."""
        rows = np.asarray(rows, dtype=np.int64)
        lo = np.zeros_like(rows)
        hi = np.full_like(rows, n - 1)
        if self.causal:
            hi = np.minimum(hi, rows)
        if self.window:
            wl, wr = self.window
            if wl >= 0:
                lo = np.maximum(lo, rows - wl)
            if wr >= 0:
                hi = np.minimum(hi, rows + wr)
        return lo, hi

    def visible_keys(self, rows, n: int) -> np.ndarray:
        """Number of keys each query row attends to under the mask."""
        lo, hi = self.visible_range(rows, n)
        return np.maximum(hi - lo + 1, 0)

    def flops(self) -> float:
        """Algorithmic FLOPs: two (n x n x d) contractions at 2 flops per
        multiply-add, i.e. 4 n^2 d per head, halved under the causal mask
        (the benchmark's stated convention).  Under a band window: 4 d per
        (query, key) pair that the band keeps."""
        if self.window:
            pairs = float(self.visible_keys(np.arange(self.N), self.N).sum())
            return 4.0 * self.B * self.H * self.D * pairs
        f = 0.5 if self.causal else 1.0
        if self.varlen:
            return sum(4.0 * self.H * n * n * self.D * f for n in self.lengths)
        return 4.0 * self.B * self.H * self.N * self.N * self.D * f

    def min_bytes(self, out_bytes: int) -> int:
        """Algorithmic HBM bytes: read Q, K, V once, write O and L once."""
        s_in = 4 if self.dtype == "f32" else 2
        tok = self.total * self.H
        return tok * self.D * (3 * s_in + out_bytes) + tok * 4


def make_inputs(w: Workload):
    """Return ``(q, k, v)`` CPU tensors in the workload's storage dtype."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    if w.varlen:
        shape = (w.total, w.H, w.D)
    else:
        shape = (w.B, w.H, w.N, w.D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.qk_mult != 1.0:
        q = q * w.qk_mult
        k = k * w.qk_mult
    dt = _TORCH_DTYPE[w.dtype]
    return q.to(dt), k.to(dt), v.to(dt)


def make_inputs_device(w: Workload, device, count: int = 3) -> list:
    """``count`` tensors of the workload's shape (q, k, v, then any extra such
    as dO), drawn on ``device`` from a generator there seeded with the
    workload's seed, in the storage dtype.

    For sizes whose CPU generation would take minutes (tensors past 2^31
    elements).  The values differ from :func:`make_inputs` (another
    generator); a test copies the slices the oracle needs to the host."""
    g = torch.Generator(device).manual_seed(w.seed)
    shape = (w.total, w.H, w.D) if w.varlen else (w.B, w.H, w.N, w.D)
    dt = _TORCH_DTYPE[w.dtype]
    out = [torch.randn(shape, generator=g, device=device, dtype=dt) for _ in range(count)]
    if w.qk_mult != 1.0:
        out[0].mul_(w.qk_mult)
        out[1].mul_(w.qk_mult)
    return out


def varlen_lengths(num_seqs: int, lo: int, hi: int, len_seed: int) -> tuple:
    """Sequence lengths uniform in ``[lo, hi]`` (inclusive) from a seed."""
    rng = np.random.default_rng(len_seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, num_seqs))


# The five benchmark-defining workloads.
C1 = Workload("B1_H1_N256_D64_f32", 1, 1, 256, 64, "f32", False, 0)
C2 = Workload("B4_H8_N1024_D64_bf16", 4, 8, 1024, 64, "bf16", False, 1)
C3 = Workload("B2_H16_N4096_D128_bf16_causal", 2, 16, 4096, 128, "bf16",
              True, 2)
C4 = Workload("B1_H32_N8192_D64_bf16_causal_qk2", 1, 32, 8192, 64, "bf16",
              True, 3, qk_mult=2.0)
C5 = Workload("varlen16_H16_D128_bf16_causal", 0, 16, 0, 128, "bf16", True,
              4, lengths=varlen_lengths(16, 128, 4096, 4))

# Few (batch, head) units and a long sequence: 64 causal 256-row blocks per
# head x 2 heads = 128 work items for 152 SMs, the case split keys are for.
SPLIT_LONG = Workload("B1_H2_N16384_D128_bf16_causal", 1, 2, 16384, 128, "bf16", True, 5)

# The local band |i - j| <= 64 that the exactness demo contrasts with exact
# attention, at the shape of C3.
BAND64 = Workload("B2_H16_N4096_D128_bf16_band64", 2, 16, 4096, 128, "bf16", False, 6,
                  window=(64, 64))
# A causal sliding window of 4096 keys over a 32K-token context.
SLIDING4K = Workload("B1_H16_N32768_D128_bf16_sliding4096", 1, 16, 32768, 128, "bf16", False, 7,
                     window=(4096, 0))

WORKLOADS = {w.name: w for w in (C1, C2, C3, C4, C5, SPLIT_LONG, BAND64, SLIDING4K)}
