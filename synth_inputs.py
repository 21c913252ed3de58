"""Seeded synthetic inputs for the fused output-projection + cross-entropy path.

This module only draws random numbers and lays them out; it holds none of the
loss arithmetic. Both the fp64 oracle (through the tests) and the CUDA path
(through the tests and the benchmark) consume exactly these arrays.

Workloads (shapes from the pages, values synthetic because the corpora the pages
train on are not available here):

* ``tiny``       N=256, d=64, V=1000, fp32; 26 of 256 positions (10%) ignored,
                 picked by a seeded permutation; uniform targets.
* ``gpt1b``      N=4096 (1 x 4096 ctx), d=2048, V=50304 (the tied vocab of the
                 1.11B run on the "6GB显卡预训练11亿参数模型" page, section
                 "让预训练成为可能的5项技术组合"), bf16, Zipf(1.1) targets, the
                 trailing 614 positions (15%) padded.
* ``llama8b``    N=8x2048, d=4096, V=128256, bf16, per-sequence valid length
                 ~ N(850, 300) clipped to [64, 2048] (the batch-8 x 2048 /
                 mean-length-850 example of the "为什么26万词表会卡死16GB显卡"
                 page, section 1), Zipf(1.1) targets.
* ``vocab256k``  N=8x2048, d=4096, V=262144, bf16, Zipf(1.05), trailing 819 of
                 every 2048 positions (40%) padded, logit std ~4.
* ``smallvocab`` N=8x4096, d=2048, V=32000, bf16, per-sequence valid length
                 uniform in [1, 4096], uniform targets, W scale 5 (peaky softmax).

Recipe: H ~ N(0, 1); W ~ N(0, 1/d) * w_scale; bf16 values are the
round-to-nearest-even bf16 of an fp32 draw. Every array has its own PCG64
stream derived from (seed, tag[, block]) so arrays can be drawn independently
and in parallel with results that do not depend on the thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

IGNORE_INDEX = -100

_TAG_H, _TAG_W, _TAG_T, _TAG_PAD = 1, 2, 3, 4
_BLOCK_ROWS = 1024


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    d: int
    V: int
    dtype: str                 # "fp32" or "bf16"
    w_scale: float
    targets: tuple             # ("uniform",) or ("zipf", s)
    padding: tuple             # see _valid_mask
    seqs: int = 1
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 64, 1000, "fp32", 3.0, ("uniform",), ("random_frac", 0.10)),
    "gpt1b": Workload("gpt1b", 4096, 2048, 50304, "bf16", 3.0, ("zipf", 1.1),
                      ("trailing_frac", 0.15), seqs=1),
    "llama8b": Workload("llama8b", 16384, 4096, 128256, "bf16", 3.0, ("zipf", 1.1),
                        ("normal_len", 850.0, 300.0, 64, 2048), seqs=8),
    "vocab256k": Workload("vocab256k", 16384, 4096, 262144, "bf16", 4.0, ("zipf", 1.05),
                          ("trailing_frac", 0.40), seqs=8),
    "smallvocab": Workload("smallvocab", 32768, 2048, 32000, "bf16", 5.0, ("uniform",),
                           ("uniform_len", 1, 4096), seqs=8),
}


def _gen(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *tags])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_matrix(seed: int, tag: int, rows: int, cols: int, scale: float, bf16: bool,
                   threads: int | None = None) -> np.ndarray:
    """rows x cols of N(0,1)*scale, drawn in blocks of _BLOCK_ROWS rows, each block
    from its own stream, so the result does not depend on the thread count."""
    out = np.empty((rows, cols), dtype=np.uint16 if bf16 else np.float32)
    nblk = (rows + _BLOCK_ROWS - 1) // _BLOCK_ROWS

    def fill(b: int) -> None:
        r0, r1 = b * _BLOCK_ROWS, min(rows, (b + 1) * _BLOCK_ROWS)
        x = _gen(seed, tag, b).standard_normal((r1 - r0, cols), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[r0:r1] = f32_to_bf16_bits(x) if bf16 else x

    threads = threads or min(16, os.cpu_count() or 1)
    if nblk == 1 or threads == 1:
        for b in range(nblk):
            fill(b)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def _valid_mask(w: Workload) -> np.ndarray:
    N, kind = w.N, w.padding[0]
    valid = np.ones(N, dtype=bool)
    g = _gen(w.seed, _TAG_PAD)
    if kind == "none":
        return valid
    if kind == "all":
        valid[:] = False
        return valid
    if kind == "random_frac":
        n_pad = int(round(w.padding[1] * N))
        valid[g.permutation(N)[:n_pad]] = False
        return valid
    if N % w.seqs:
        raise ValueError("N must be a multiple of the sequence count")
    L = N // w.seqs
    if kind == "trailing_frac":
        n_pad = int(round(w.padding[1] * L))
        lengths = np.full(w.seqs, L - n_pad)
    elif kind == "normal_len":
        mu, sigma, lo, hi = w.padding[1:]
        lengths = np.clip(np.rint(g.normal(mu, sigma, w.seqs)), lo, min(hi, L)).astype(np.int64)
    elif kind == "uniform_len":
        lo, hi = w.padding[1:]
        lengths = g.integers(lo, min(hi, L) + 1, w.seqs)
    else:
        raise ValueError(f"unknown padding recipe {kind!r}")
    for b in range(w.seqs):
        valid[b * L + int(lengths[b]): (b + 1) * L] = False
    return valid


def _targets(w: Workload) -> np.ndarray:
    g = _gen(w.seed, _TAG_T)
    if w.targets[0] == "uniform":
        t = g.integers(0, w.V, w.N, dtype=np.int64)
    elif w.targets[0] == "zipf":
        # truncated Zipf on ranks 1..V, P(r) proportional to r^-s, drawn by
        # inverse CDF; token id = rank - 1
        s = float(w.targets[1])
        cdf = np.cumsum(np.arange(1, w.V + 1, dtype=np.float64) ** (-s))
        cdf /= cdf[-1]
        t = np.minimum(np.searchsorted(cdf, g.random(w.N), side="right"), w.V - 1).astype(np.int64)
    else:
        raise ValueError(f"unknown target recipe {w.targets[0]!r}")
    t[~_valid_mask(w)] = IGNORE_INDEX
    return t


@dataclass
class Inputs:
    workload: Workload
    H: np.ndarray        # [N, d] float32, or uint16 bf16 bits
    W: np.ndarray        # [V, d] float32, or uint16 bf16 bits
    targets: np.ndarray  # [N] int64, IGNORE_INDEX on padded positions

    @property
    def bf16(self) -> bool:
        return self.workload.dtype == "bf16"

    def H_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.H) if self.bf16 else self.H

    def W_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.W) if self.bf16 else self.W


def make_targets(w: Workload) -> np.ndarray:
    return _targets(w)


def make_inputs(w: Workload | str, **overrides) -> Inputs:
    """Draw (H, W, targets) for a workload (by name or object); keyword overrides
    replace workload fields (e.g. a smaller N for a parity case)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if overrides:
        w = w.with_(**overrides)
    bf16 = w.dtype == "bf16"
    H = _normal_matrix(w.seed, _TAG_H, w.N, w.d, 1.0, bf16)
    W = _normal_matrix(w.seed, _TAG_W, w.V, w.d, w.w_scale / np.sqrt(w.d), bf16)
    return Inputs(w, H, W, _targets(w))
