"""Seeded synthetic inputs for the causal LLA forward pass.

This module holds only input generation: it draws q, k, v with the shapes,
dtypes and value distributions of the workloads below and rounds them to the
compute dtype.  It contains none of the method's arithmetic, so both the CUDA
path and the float64 oracle can be fed from it.

Random numbers come from numpy's PCG64 generator (platform independent); bf16
rounding is torch's round-to-nearest-even conversion.

Workloads (all causal, [B, H, n, d] row-major):

* ``tiny_fp32``        B=1,  H=1,  n=64,    d=16,  fp32; q,k,v ~ N(0,1)/sqrt(d);
                        tau=1/sqrt(d), lambda=0.1, CG to rel. residual 1e-7 (cap 64).
* ``piecewise_fp32``   B=64, H=1,  n=1024,  d=32,  fp32; synthetic stand-in for the
                        test-time piecewise regression of the reading notes (section 4.1):
                        k, q uniform on the unit sphere, 16 unit centroids split space by
                        nearest centroid, v_j = A_s k_j + c_s with A_s ~ N(0, 1/d),
                        c_s ~ N(0, 1); tau=4, lambda=1e-2, CG to 1e-7 (cap 64).
* ``lm_bf16``          B=8,  H=16, n=4096,  d=128, bf16; q,k,v ~ N(0,1), q and k
                        RMS-normalised per row in fp32 (eps 1e-6) before rounding;
                        tau=1/sqrt(128), lambda=1, fixed 16 CG iterations.
* ``long_bf16``        B=1,  H=8,  n=32768, d=128, bf16; generated as ``lm_bf16``.
* ``illcond_bf16``     B=4,  H=8,  n=8192,  d=64,  bf16; generated as ``lm_bf16``;
                        tau=1/8, lambda in {1e-3, 1e-1, 1e6}, CG to 1e-4 (cap 64).
* ``decode_bf16``      B=64, H=16, n=4096,  d=128, bf16; generated as ``lm_bf16``; a decode step:
                        the caches are k, v and the new query is q's last row (64 sequences,
                        one token each, against 4096 cached positions).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "workload"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dtype: str          # "fp32" or "bf16"
    gen: str            # "gauss", "piecewise" or "gauss_rmsnorm"
    tau: float
    lam: float
    cg_max_iters: int
    cg_tol: float
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 64, 16, "fp32", "gauss", 0.25, 0.1, 64, 1e-7),
    "piecewise_fp32": Workload("piecewise_fp32", 64, 1, 1024, 32, "fp32", "piecewise", 4.0, 1e-2, 64, 1e-7),
    "lm_bf16": Workload("lm_bf16", 8, 16, 4096, 128, "bf16", "gauss_rmsnorm", 1.0 / math.sqrt(128.0), 1.0, 16, 0.0),
    "long_bf16": Workload("long_bf16", 1, 8, 32768, 128, "bf16", "gauss_rmsnorm", 1.0 / math.sqrt(128.0), 1.0, 16, 0.0),
    "illcond_bf16": Workload("illcond_bf16", 4, 8, 8192, 64, "bf16", "gauss_rmsnorm", 0.125, 1e-1, 64, 1e-4),
    # decode step: B sequences x H heads, each a cache of n rows (the query is row n-1)
    "decode_bf16": Workload("decode_bf16", 64, 16, 4096, 128, "bf16", "gauss_rmsnorm", 1.0 / math.sqrt(128.0), 1.0, 16,
                            0.0),
}


def workload(name, **overrides):
    """The named workload, with any field overridden (e.g. a smaller n for tests)."""
    return WORKLOADS[name].with_(**overrides)


def _unit_sphere(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rmsnorm_rows(x):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + np.float32(1e-6))


def make_inputs(w: Workload):
    """Draw (q, k, v) as CPU torch tensors of shape [B, H, n, d] in w's dtype.

    Draw order is fixed per generator so a given (workload, seed) is reproducible.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    shape = (w.B, w.H, w.n, w.d)
    if w.gen == "gauss":
        s = np.float32(1.0 / math.sqrt(w.d))
        q = rng.standard_normal(shape, dtype=np.float32) * s
        k = rng.standard_normal(shape, dtype=np.float32) * s
        v = rng.standard_normal(shape, dtype=np.float32) * s
    elif w.gen == "gauss_rmsnorm":
        q = rng.standard_normal(shape, dtype=np.float32)
        k = rng.standard_normal(shape, dtype=np.float32)
        v = rng.standard_normal(shape, dtype=np.float32)
        q = _rmsnorm_rows(q)
        k = _rmsnorm_rows(k)
    elif w.gen == "piecewise":
        S = 16
        centroids = _unit_sphere(rng, (S, w.d))
        A = rng.standard_normal((S, w.d, w.d), dtype=np.float32) * np.float32(1.0 / math.sqrt(w.d))
        c = rng.standard_normal((S, w.d), dtype=np.float32)
        k = _unit_sphere(rng, shape)
        q = _unit_sphere(rng, shape)
        seg = np.argmax(k @ centroids.T, axis=-1)           # nearest unit centroid; ties -> lowest index
        v = np.empty(shape, dtype=np.float32)
        for s_ in range(S):
            sel = seg == s_
            v[sel] = k[sel] @ A[s_].T + c[s_]
    else:
        raise ValueError(f"unknown generator {w.gen!r}")
    td = w.torch_dtype
    return (torch.from_numpy(np.ascontiguousarray(q)).to(td),
            torch.from_numpy(np.ascontiguousarray(k)).to(td),
            torch.from_numpy(np.ascontiguousarray(v)).to(td))


def make_probe(w: Workload, seed_offset=1000):
    """Parallax probe [B, H, n, d] fp32 (CPU torch), drawn after (q, k, v) from its own stream.

    The page computes rho = RMSNorm(W_R x) from the layer input; without trained weights the
    stand-in is an RMS-normalised Gaussian row divided by sqrt(d), so (k_j - kbar).rho is of
    order one for the unit-RMS keys of the LM workloads (the correction is of the size of the
    softmax output, neither negligible nor dominant).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed + seed_offset))
    r = _rmsnorm_rows(rng.standard_normal((w.B, w.H, w.n, w.d), dtype=np.float32))
    return torch.from_numpy(np.ascontiguousarray(r * np.float32(1.0 / math.sqrt(w.d))))


def sample_rows(w: Workload, count, seed=1, tile=128):
    """Stratified (b, h, i) rows for sampled parity checks at full size.

    Always includes the first 16 positions, both sides of every multiple of
    ``tile`` up to 512, and the last position, then seeded uniform rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed_i = sorted({i for i in list(range(min(16, w.n)))
                      + [t + o for t in range(tile, min(w.n, 513), tile) for o in (-1, 0)]
                      + [w.n - 1] if 0 <= i < w.n})
    rows = []
    for j, i in enumerate(fixed_i):
        rows.append((j % w.B, (j // w.B) % w.H, i))
    while len(rows) < count:
        rows.append((int(rng.integers(w.B)), int(rng.integers(w.H)), int(rng.integers(w.n))))
    return rows


def make_cotangent(w: Workload, seed_offset=2000):
    """Output cotangent dL/dout [B, H, n, d] (CPU torch, w's dtype) from its own stream: a unit
    Gaussian per entry, the gradient a loss that is a random linear function of the output sends."""
    rng = np.random.Generator(np.random.PCG64(w.seed + seed_offset))
    g = rng.standard_normal((w.B, w.H, w.n, w.d), dtype=np.float32)
    return torch.from_numpy(np.ascontiguousarray(g)).to(w.torch_dtype)
