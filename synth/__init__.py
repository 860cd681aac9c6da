"""Seeded synthetic inputs for the fine-grained FP8 path.

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic (no scaling, no FP8 rounding, no GEMM), so both the
CPU oracle and the CUDA path can be fed from it.  Every generator is numpy
``Generator(PCG64)`` seeded per workload, with one independent substream per
role (A, B, outliers, routing) from ``SeedSequence(seed).spawn``; large
tensors are drawn in fixed blocks of rows, each from its own child substream,
so the values do not depend on how many threads fill them.  Values are drawn
in fp32, outlier multipliers are applied in fp32, and the result is rounded
once to bf16 (round to nearest even).  bf16 tensors are returned as their
uint16 bit patterns.

Workloads (sizes of the training-step GEMMs of a large MoE transformer layer):

* tiny end-to-end: A[256,512] ~ N(0,1) with 4 columns x50, B[512,256] ~ N(0,1)
* quantizers: activation [8192,7168] ~ N(0,1) with 1% of channels x100,
  weight [7168,18432] ~ N(0, 0.02^2)
* forward GEMM: A[8192,7168] ~ N(0,1), W[7168,18432] ~ N(0, 0.02^2)
* weight-gradient GEMM: dY[8192,18432], X[8192,7168] ~ N(0, 1e-3^2) with
  per-element Bernoulli(0.001) outliers x1000
* MoE grouped GEMM: 32 experts W_g[7168,2048] ~ N(0, 0.02^2); 16384 tokens x 8
  picks routed i.i.d. with p_g proportional to (g+1)^-1.1 (Zipf, s = 1.1);
  per-expert row counts padded to multiples of 128; activations ~ N(0,1), pad
  rows zero.
"""
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "f32_from_bf16_bits", "normal_bf16",
    "tiny_end_to_end", "activation", "weight", "wgrad_tensor", "moe_routing",
    "moe_inputs", "MoEInputs",
]


def bf16_bits_from_f32(f) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); uint16 bit patterns.
    Inputs are finite."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _bf16_fast(f) -> np.ndarray:
    """Same rounding as bf16_bits_from_f32, through torch's (multithreaded)
    float32 -> bfloat16 cast, which also rounds to nearest even."""
    try:
        import torch
    except ImportError:
        return bf16_bits_from_f32(f)
    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_from_bf16_bits(h) -> np.ndarray:
    """Exact float32 values of bf16 bit patterns."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _seqs(seed: int, n: int = 4):
    return np.random.SeedSequence(seed).spawn(n)


def _streams(seed: int, n: int = 4):
    return [np.random.Generator(np.random.PCG64(s)) for s in _seqs(seed, n)]


BLOCK_ROWS = 1024


def _fill_blocks(out, seq, fill, threads=None):
    """Fill out[r0:r1] for every block of BLOCK_ROWS rows with
    fill(Generator(child_seq[b]), r0, r1); blocks run on a thread pool (numpy's
    generators release the GIL), each with its own child substream."""
    rows = out.shape[0]
    n_blocks = -(-rows // BLOCK_ROWS)
    children = seq.spawn(n_blocks)

    def job(b):
        r0 = b * BLOCK_ROWS
        r1 = min(rows, r0 + BLOCK_ROWS)
        out[r0:r1] = fill(np.random.Generator(np.random.PCG64(children[b])), r0, r1)
    threads = threads or min(32, os.cpu_count() or 1)
    if threads <= 1 or n_blocks <= 1:
        for b in range(n_blocks):
            job(b)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(job, range(n_blocks)))
    return out


def normal_bf16(seq, shape, sigma=1.0, out=None) -> np.ndarray:
    """N(0, sigma^2) fp32 draws rounded to bf16, generated in row blocks.
    `seq` is a numpy SeedSequence; `out` (optional) receives the values."""
    shape = tuple(int(d) for d in shape)
    if out is None:
        out = np.empty(shape, np.uint16)

    def fill(rng, r0, r1):
        f = rng.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if sigma != 1.0:
            f *= np.float32(sigma)
        return _bf16_fast(f)
    return _fill_blocks(out, seq, fill)


def tiny_end_to_end(seed: int = 1, M: int = 256, K: int = 512, N: int = 256,
                    n_outlier_cols: int = 4, outlier_mult: float = 50.0):
    """A[M,K] ~ N(0,1) with `n_outlier_cols` seeded columns scaled x50, and
    B[K,N] ~ N(0,1).  Returns (A_bits, B_bits, outlier_cols)."""
    ra, rb, ro, _ = _streams(seed)
    a = ra.standard_normal((M, K), dtype=np.float32)
    cols = np.sort(ro.choice(K, n_outlier_cols, replace=False))
    a[:, cols] *= np.float32(outlier_mult)
    b = rb.standard_normal((K, N), dtype=np.float32)
    return bf16_bits_from_f32(a), bf16_bits_from_f32(b), cols


def activation(seed: int, M: int, K: int, outlier_frac: float = 0.01,
               outlier_mult: float = 100.0):
    """Activation [M,K] ~ N(0,1) with round(outlier_frac*K) seeded channels
    scaled by `outlier_mult`.  Returns (bits, outlier_channels)."""
    sa, _, so, _ = _seqs(seed)
    ro = np.random.Generator(np.random.PCG64(so))
    n_out = int(round(outlier_frac * K))
    cols = np.sort(ro.choice(K, n_out, replace=False)) if n_out else np.zeros(0, np.int64)
    out = np.empty((M, K), np.uint16)

    def fill(rng, r0, r1):
        f = rng.standard_normal((r1 - r0, K), dtype=np.float32)
        if n_out:
            f[:, cols] *= np.float32(outlier_mult)
        return _bf16_fast(f)
    return _fill_blocks(out, sa, fill), cols


def weight(seed: int, K: int, N: int, sigma: float = 0.02):
    """Weight [K,N] (K input channels, N output channels) ~ N(0, sigma^2)."""
    _, sb, _, _ = _seqs(seed)
    return normal_bf16(sb, (K, N), sigma)


def wgrad_tensor(seed: int, stream: int, rows: int, cols: int, sigma: float = 1e-3,
                 outlier_p: float = 1e-3, outlier_mult: float = 1000.0):
    """[rows, cols] ~ N(0, sigma^2) with i.i.d. Bernoulli(outlier_p) elements
    scaled by `outlier_mult`.  `stream` selects an independent substream (0 for
    the activation X, 1 for the output gradient dY)."""
    seq = _seqs(seed, 4)[stream]
    out = np.empty((rows, cols), np.uint16)

    def fill(rng, r0, r1):
        f = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        f *= np.float32(sigma)
        mask = rng.random((r1 - r0, cols), dtype=np.float32) < np.float32(outlier_p)
        f[mask] *= np.float32(outlier_mult)
        return _bf16_fast(f)
    return _fill_blocks(out, seq, fill)


def moe_routing(seed: int, G: int = 32, tokens: int = 16384, topk: int = 8,
                zipf_s: float = 1.1, pad: int = 128):
    """Per-expert routed row counts ~ Multinomial(tokens*topk, p_g ∝ (g+1)^-s),
    then each padded up to a multiple of `pad`.  Returns (counts, offsets) with
    offsets int32 [G+1] over the padded counts."""
    _, _, _, rr = _streams(seed)
    p = (np.arange(1, G + 1, dtype=np.float64)) ** (-zipf_s)
    p /= p.sum()
    counts = rr.multinomial(tokens * topk, p).astype(np.int64)
    padded = (counts + pad - 1) // pad * pad
    offsets = np.zeros(G + 1, np.int64)
    offsets[1:] = np.cumsum(padded)
    return counts, offsets.astype(np.int32)


@dataclass
class MoEInputs:
    x: np.ndarray         # bf16 bits [M_total, K]; pad rows are zero
    w: np.ndarray         # bf16 bits [G, K, N]
    counts: np.ndarray    # routed rows per expert (before padding)
    offsets: np.ndarray   # int32 [G+1], padded row ranges
    routed_rows: int


def moe_inputs(seed: int = 5, G: int = 32, K: int = 7168, N: int = 2048,
               tokens: int = 16384, topk: int = 8, zipf_s: float = 1.1,
               sigma_w: float = 0.02, with_weights: bool = True) -> MoEInputs:
    counts, offsets = moe_routing(seed, G, tokens, topk, zipf_s)
    sa, sb, _, _ = _seqs(seed)
    M_total = int(offsets[-1])
    x = np.zeros((M_total, K), np.uint16)
    xseq = sa.spawn(G)
    for g in range(G):
        r0 = int(offsets[g])
        n = int(counts[g])
        if n:
            normal_bf16(xseq[g], (n, K), 1.0, out=x[r0:r0 + n])
    w = normal_bf16(sb, (G * K, N), sigma_w).reshape(G, K, N) if with_weights else None
    return MoEInputs(x=x, w=w, counts=counts, offsets=offsets,
                     routed_rows=int(counts.sum()))


def swiglu_inputs(seed: int, M: int, F: int, sigma: float = 1.7):
    """Cached gate and up projections of an MLP, side by side as one bf16
    [M, 2F] tensor (gate = columns [0, F), up = [F, 2F)), each ~ N(0, sigma^2):
    an N(0, 1) activation times N(0, 0.02^2) weights over 7168 input channels
    has sigma = 0.02 * sqrt(7168) = 1.7."""
    seq = _seqs(seed, 4)[2]
    return normal_bf16(seq, (M, 2 * F), sigma=sigma)
