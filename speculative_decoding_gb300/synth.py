"""Seeded synthetic inputs for the XPress Jacobi pass.

This module only draws random data: it holds none of the pass's arithmetic
(no argmax, no matmul, no mixer), so both the CUDA path and the CPU oracle can
be fed from it.  Trained weights and real hidden states are not available, so
the distributions below stand in for them (all from one seed per workload):

  E[V, D]            bf16  ~ N(0, 0.02)               token embedding
  W_lat[D, R]        bf16  ~ N(0, 1/sqrt(D))          [in, out]
  Wg, Wu[R, H]       bf16  ~ N(0, 1/sqrt(R))
  Wd[H, R]           bf16  ~ N(0, 1/sqrt(H))
  W2[R, V]           bf16  ~ N(0, 1/sqrt(R))
  L[B, B, R]         fp32  lower-triangular ~ U(0, 1), each (b, r) row
                           normalised to sum 1 over j <= b (the folded mixer)
  hcache[N, B, R]    bf16  ~ N(0, 1)
  base[N*(B-1), V]   bf16  ~ N(0, 3)
  bias[N*(B-1), V]   bf16  ~ N(0, 1)                 (standalone add-argmax)
  am1[N], blk[N, B]  int64 ~ U[0, V)

N(0, s) names the standard deviation s.  bf16 tensors are returned as numpy
``uint16`` bit patterns (converted from fp32 with torch's round-to-nearest-even
cast); tokens as ``int64``; L as ``float32``.

Normals come from numpy's Philox generator in fixed chunks, one child seed per
chunk, so the values do not depend on the number of threads used.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

_CHUNK = 1 << 22


@dataclass(frozen=True)
class PassShape:
    """One workload of the pass: N blocks of B slots, vocab V, embedding width
    D, latent rank R, MLP hidden H, and its seed."""

    name: str
    N: int
    B: int
    V: int
    D: int
    R: int
    H: int
    seed: int

    @property
    def rows(self) -> int:
        return self.N * (self.B - 1)


# Workloads, named by what they are.
TINY = PassShape("tiny N=2 B=4 V=1000 D=64 R=32 H=64", 2, 4, 1000, 64, 32, 64, seed=0)
SERVE = PassShape("pass N=32 B=16 V=152064 D=3584 R=512 H=1536", 32, 16, 152064, 3584, 512, 1536, seed=2)
FLOOR = PassShape("pass N=1 B=16 V=152064 D=3584 R=512 H=1536", 1, 16, 152064, 3584, 512, 1536, seed=3)
FIXPOINT = PassShape("fixpoint N=64 B=16 V=152064 D=3584 R=512 H=1536", 64, 16, 152064, 3584, 512, 1536, seed=4)

ARGMAX_ROWS, ARGMAX_V, ARGMAX_SEED = 480, 152064, 1   # rows = 32 * 15


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_f32(seed: int, stream: int, n: int, std: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    kids = np.random.SeedSequence([seed, stream]).spawn(nchunks)
    s = np.float32(std)

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        if hi > lo:
            g = np.random.Generator(np.random.Philox(kids[i]))
            g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
            out[lo:hi] *= s

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 numpy -> bf16 bit patterns (uint16), torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(seed: int, stream: int, shape, std: float) -> np.ndarray:
    n = int(np.prod(shape))
    return to_bf16_bits(_normal_f32(seed, stream, n, std)).reshape(shape)


def tokens(seed: int, stream: int, shape, V: int) -> np.ndarray:
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream])))
    return g.integers(0, V, size=shape, dtype=np.int64)


def mixer(seed: int, B: int, R: int) -> np.ndarray:
    """L[b, j, r]: U(0,1) for j <= b, 0 above the diagonal, each (b, r) row
    scaled to sum 1 over j."""
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 7])))
    u = g.random((B, B, R), dtype=np.float64)
    tri = np.tril(np.ones((B, B)))[:, :, None]
    u = u * tri
    u = u / u.sum(axis=1, keepdims=True)
    return u.astype(np.float32)


# stream ids, fixed per tensor
_S = dict(E=1, W_lat=2, Wg=3, Wu=4, Wd=5, W2=6, hcache=8, base=9, bias=10, am1=11, blk=12)


def pass_inputs(shape: PassShape, with_embedding: bool = True) -> dict:
    """All inputs of one pass.  ``with_embedding=False`` skips E (the largest
    tensor) for callers that build it elsewhere."""
    s, N, B, V, D, R, H = shape.seed, shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    out = dict(
        W_lat=normal_bf16(s, _S["W_lat"], (D, R), 1.0 / math.sqrt(D)),
        L=mixer(s, B, R),
        Wg=normal_bf16(s, _S["Wg"], (R, H), 1.0 / math.sqrt(R)),
        Wu=normal_bf16(s, _S["Wu"], (R, H), 1.0 / math.sqrt(R)),
        Wd=normal_bf16(s, _S["Wd"], (H, R), 1.0 / math.sqrt(H)),
        W2=normal_bf16(s, _S["W2"], (R, V), 1.0 / math.sqrt(R)),
        hcache=normal_bf16(s, _S["hcache"], (N, B, R), 1.0),
        base=normal_bf16(s, _S["base"], (N * (B - 1), V), 3.0),
        am1=tokens(s, _S["am1"], (N,), V),
        blk=tokens(s, _S["blk"], (N, B), V),
    )
    if with_embedding:
        out["E"] = normal_bf16(s, _S["E"], (V, D), 0.02)
    return out


def pass_activations(shape: PassShape) -> dict:
    """The per-pass inputs of ``pass_inputs`` (hcache, base, am1, blk: the same
    values, same streams) without the weights, for runs that reuse the weights
    of another workload of the same model dimensions."""
    s, N, B, V, R = shape.seed, shape.N, shape.B, shape.V, shape.R
    return dict(hcache=normal_bf16(s, _S["hcache"], (N, B, R), 1.0),
                base=normal_bf16(s, _S["base"], (N * (B - 1), V), 3.0),
                am1=tokens(s, _S["am1"], (N,), V), blk=tokens(s, _S["blk"], (N, B), V))


def exact_mixer(B: int, R: int) -> np.ndarray:
    """A folded mixer of powers of two: row b of channel r puts 1 (b = 0),
    1/2 1/2 (b = 1), 1/2 1/4 1/4 (b = 2) or 1/2 1/4 1/8 1/8 (b >= 3) on
    the distinct slots j = (r + k) mod (b+1), k = 0, 1, ...; zero elsewhere.
    Rows sum to 1 exactly and differ from channel to channel."""
    L = np.zeros((B, B, R), np.float32)
    for b in range(B):
        w = {0: [1.0], 1: [0.5, 0.5], 2: [0.5, 0.25, 0.25]}.get(b, [0.5, 0.25, 0.125, 0.125])
        for r in range(R):
            for k, wt in enumerate(w):
                L[b, (r + k) % (b + 1), r] = wt
    return L


def exact_pass_inputs(shape: PassShape) -> dict:
    """Pass inputs on which every sum of the method is exact in fp32 (so any
    correct summation order gives the same bits): E holds integers in [-3, 3]
    over 4 and W_lat integers in [-2, 2] over 4, so x = hcache + e @ W_lat is
    a multiple of 1/16 (hcache: integers in [-4, 4] over 4); the mixer is
    exact_mixer, so u is a multiple of 2^-7; Wg = 0, so m = 0 and
    lat = bf16(u), again a multiple of 2^-7; W2 holds integers in [-2, 2] over
    16, so every partial sum of lat @ W2 is a multiple of 2^-11 (exact while
    below 2^13).  Magnitudes stay far inside those bounds for the shapes the
    tests use.  base ~ N(0, 0.5) (the bias then moves tokens); am1 and blk
    ~ U[0, V)."""
    N, B, V, D, R, H, seed = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H, shape.seed
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 31])))

    def q(a):
        return to_bf16_bits(np.asarray(a, np.float32))

    return dict(E=q(g.integers(-3, 4, (V, D)) / 4.0), W_lat=q(g.integers(-2, 3, (D, R)) / 4.0),
                hcache=q(g.integers(-4, 5, (N, B, R)) / 4.0), L=exact_mixer(B, R),
                Wg=np.zeros((R, H), np.uint16), Wu=q(g.integers(-2, 3, (R, H)) / 4.0),
                Wd=q(g.integers(-2, 3, (H, R)) / 4.0), W2=q(g.integers(-2, 3, (R, V)) / 16.0),
                base=normal_bf16(seed, _S["base"], (N * (B - 1), V), 0.5),
                am1=g.integers(0, V, N).astype(np.int64), blk=g.integers(0, V, (N, B)).astype(np.int64))


def plant_ties(base: np.ndarray, bias: np.ndarray, frac: float, seed: int, min_rows: int = 1):
    """Plant duplicated row maxima, in place.

    For round(frac * rows) rows (at least ``min_rows`` when frac > 0), 2 to 4
    random positions get base = a value above max(base[row]) + max(bias[row]) + 1
    and bias = 0, so those positions hold the row's strict maximum and tie with
    each other; the lowest of them is the expected answer by construction.
    Returns {row: sorted positions}."""
    rows, V = base.shape
    k = int(round(frac * rows))
    if frac > 0:
        k = max(k, min_rows)
    k = min(k, rows)
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 99])))
    chosen = sorted(g.choice(rows, size=k, replace=False).tolist()) if k else []
    planted = {}
    for r in chosen:
        bmax = float(np.max(_f32(base[r]))) + float(np.max(_f32(bias[r]))) + 1.0
        top = to_bf16_bits(np.array([bmax], np.float32))[0]
        if _f32(np.array([top]))[0] <= bmax - 1.0:   # cannot happen for these ranges
            raise AssertionError("planted value does not exceed the row")
        cnt = int(g.integers(2, 5))
        pos = np.sort(g.choice(V, size=min(cnt, V), replace=False))
        base[r, pos] = top
        bias[r, pos] = 0
        planted[r] = pos.tolist()
    return planted


def _f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def argmax_inputs(rows: int, V: int, N: int, B: int, seed: int, tie_frac: float):
    """Standalone add-argmax inputs: base ~N(0,3), bias ~N(0,1), [rows, V]
    row-contiguous, plus a block buffer and the planted-tie rows."""
    base = normal_bf16(seed, _S["base"], (rows, V), 3.0)
    bias = normal_bf16(seed, _S["bias"], (rows, V), 1.0)
    planted = plant_ties(base, bias, tie_frac, seed)
    blk = tokens(seed, _S["blk"], (N, B), V)
    return dict(base=base, bias=bias, blk=blk, planted=planted)
