"""Seeded synthetic inputs for the fused residual-Add + LayerNorm operation.

This module holds no arithmetic of the method itself: it only draws X, R,
gamma and beta with the distributions a workload states and rounds them to
the workload's I/O dtype.  Both the oracle tests and the GPU path take their
inputs from here, so the same seed gives the same bytes on both sides.

Recipe (every workload, in this fixed order of child streams of
``numpy.random.SeedSequence(seed)``):
  0. X ~ N(x_loc, x_scale), drawn in fp32
  1. R ~ N(r_loc, r_scale), drawn in fp32
  2. gamma = 1 + 0.1 * N(0, 1), fp32 [H]
  3. beta  = 0.1 * N(0, 1), fp32 [H]
  4. constant rows: round(frac * rows) rows chosen without replacement; each
     gets X_row = c (one N(x_loc, x_scale) draw) and R_row = 0
  5. outliers: round(frac * rows * H) positions of X chosen without
     replacement, each set to +-mag with a fair random sign
(Softmax workloads draw no R: its stream is spawned but left unused.)
X and R are then rounded to the I/O dtype with round-to-nearest-even (torch's
float -> half / bfloat16 conversion).  Outputs are host (CPU) torch tensors.
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import Workload

TORCH_DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


def _normal_f32(g: np.random.Generator, n: int, loc: float, scale: float) -> np.ndarray:
    v = g.standard_normal(n, dtype=np.float32)
    if scale != 1.0:
        v *= np.float32(scale)
    if loc != 0.0:
        v += np.float32(loc)
    return v


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw one batch of inputs for workload ``w``.

    Returns a dict with host tensors ``x``, ``r`` ([rows, H], I/O dtype),
    ``gamma``, ``beta`` ([H], fp32), the float ``eps``, and the index arrays
    ``const_rows`` (sorted row ids) and ``outlier_pos`` (sorted flat ids).
    """
    ss = np.random.SeedSequence(seed)
    gx, gr, gg, gb, gc, go = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(6)]
    rows, H = w.rows, w.H
    n = rows * H

    x = _normal_f32(gx, n, *w.x_dist)
    r = _normal_f32(gr, n, *w.r_dist) if w.op != "softmax" else None
    gamma = (np.float32(1.0) + np.float32(0.1) * gg.standard_normal(H, dtype=np.float32)).astype(np.float32)
    beta = (np.float32(0.1) * gb.standard_normal(H, dtype=np.float32)).astype(np.float32)

    const_rows = np.zeros(0, dtype=np.int64)
    if w.n_const_rows:
        const_rows = np.sort(gc.choice(rows, size=w.n_const_rows, replace=False)).astype(np.int64)
        consts = _normal_f32(gc, w.n_const_rows, *w.x_dist)
        x2 = x.reshape(rows, H)
        r2 = r.reshape(rows, H)
        x2[const_rows, :] = consts[:, None]
        r2[const_rows, :] = 0.0

    outlier_pos = np.zeros(0, dtype=np.int64)
    if w.n_outliers:
        outlier_pos = np.sort(go.choice(n, size=w.n_outliers, replace=False)).astype(np.int64)
        signs = go.integers(0, 2, size=w.n_outliers).astype(np.float32) * 2.0 - 1.0
        x[outlier_pos] = signs * np.float32(w.outlier_mag)

    td = TORCH_DTYPES[w.dtype]
    xt = torch.from_numpy(x).view(rows, H).to(td)
    rt = torch.from_numpy(r).view(rows, H).to(td).contiguous() if r is not None else None
    return {
        "x": xt.contiguous(),
        "r": rt,
        "gamma": torch.from_numpy(gamma),
        "beta": torch.from_numpy(beta),
        "eps": float(w.eps),
        "const_rows": const_rows,
        "outlier_pos": outlier_pos,
    }


def make_affine(H: int, seed: int = 0) -> tuple:
    """gamma, beta for an ad-hoc row length (same recipe as make_inputs)."""
    ss = np.random.SeedSequence([seed, H])
    gg, gb = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(2)]
    gamma = (np.float32(1.0) + np.float32(0.1) * gg.standard_normal(H, dtype=np.float32)).astype(np.float32)
    beta = (np.float32(0.1) * gb.standard_normal(H, dtype=np.float32)).astype(np.float32)
    return torch.from_numpy(gamma), torch.from_numpy(beta)


def make_grad(w: Workload, seed: int = 0, scale: float = 1.0):
    """Upstream gradient dY ~ N(0, scale) for workload w, rounded to its dtype
    (child stream 6 of SeedSequence(seed); streams 0-5 are make_inputs')."""
    ss = np.random.SeedSequence(seed)
    gd = np.random.Generator(np.random.PCG64(ss.spawn(7)[6]))
    v = _normal_f32(gd, w.rows * w.H, 0.0, scale)
    return torch.from_numpy(v).view(w.rows, w.H).to(TORCH_DTYPES[w.dtype]).contiguous()
