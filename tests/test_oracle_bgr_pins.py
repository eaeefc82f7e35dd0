"""Pins for the oracle's bias + GELU + residual chain (CPU only).

Y = GELU(X + bias) + R with the exact GELU v * Phi(v) = v/2 (1 + erf(v/sqrt 2))
("算子融合的收益量化", the BiasAdd -> GELU -> Residual diagram).  Pins:
an erf summed as a 50-digit Taylor series (independent of libm), the odd
identity GELU(v) - GELU(-v) = v, the residual and bias entering linearly and
per column, torch's exact GELU in float64, and the diagram's own numbers.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, localcontext

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TD = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


def _erf_series(z: float) -> Decimal:
    with localcontext() as ctx:
        ctx.prec = 50
        zd = Decimal(z)
        term, total, n = zd, zd, 0
        while True:
            n += 1
            term = -term * zd * zd / n
            add = term / (2 * n + 1)
            total += add
            if abs(add) < Decimal(10) ** -45:
                break
        pi = Decimal("3.14159265358979323846264338327950288419716939937510")
        return 2 * total / pi.sqrt()


def _gelu_series(v: float) -> float:
    with localcontext() as ctx:
        ctx.prec = 50
        z = Decimal(v) / Decimal(2).sqrt()
        return float(Decimal(v) / 2 * (1 + _erf_series(float(z))))


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_matches_series_gelu(dtype):
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(3, 40, generator=g) * 1.5).to(TD[dtype])
    r = (torch.randn(3, 40, generator=g) * 0.5).to(TD[dtype])
    bias = 0.1 * torch.randn(40, generator=g)
    y = oracle.oracle_bias_gelu_residual(x, r, bias, dtype)
    xd, rd = x.double().numpy(), r.double().numpy()
    bd = bias.double().numpy()
    for i in range(3):
        for j in range(40):
            ref = _gelu_series(float(xd[i, j] + bd[j])) + rd[i, j]
            assert abs(y[i, j] - ref) <= 1e-14 * (1 + abs(ref))


def test_odd_identity_and_zero():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(4, 100, generator=g) * 3
    z = torch.zeros(4, 100)
    b = torch.zeros(100)
    yp = oracle.oracle_bias_gelu_residual(x, z, b, "fp32")
    ym = oracle.oracle_bias_gelu_residual(-x, z, b, "fp32")
    assert np.allclose(yp - ym, x.double().numpy(), rtol=1e-14, atol=1e-15)
    y0 = oracle.oracle_bias_gelu_residual(z, x, b, "fp32")          # GELU(0) = 0
    assert np.array_equal(y0, x.double().numpy())


def test_asymptotes():
    x = torch.tensor([[10.0, -10.0, 40.0, -40.0]])
    y = oracle.oracle_bias_gelu_residual(x, torch.zeros(1, 4), torch.zeros(4), "fp32")[0]
    assert y[0] == pytest.approx(10.0, rel=1e-15) and abs(y[1]) < 1e-20
    assert y[2] == 40.0 and y[3] == 0.0          # erf saturates to +-1 in fp64


def test_residual_and_bias_enter_linearly_per_column():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(5, 64, generator=g)
    r = torch.randn(5, 64, generator=g)
    bias = torch.randn(64, generator=g)
    y = oracle.oracle_bias_gelu_residual(x, r, bias, "fp32")
    y0 = oracle.oracle_bias_gelu_residual(x, torch.zeros(5, 64), bias, "fp32")
    assert np.allclose(y - y0, r.double().numpy(), rtol=0, atol=1e-15 * 8)
    # bias j shifts column j only: X = 0 gives GELU(bias_j) in every row
    yb = oracle.oracle_bias_gelu_residual(torch.zeros(5, 64), torch.zeros(5, 64), bias, "fp32")
    col = np.array([0.5 * b * (1 + math.erf(b / math.sqrt(2))) for b in bias.double().tolist()])
    assert np.allclose(yb, np.broadcast_to(col, (5, 64)), rtol=1e-15, atol=0)


@pytest.mark.parametrize("name", synth.BGR_NAMES)
def test_matches_torch_gelu_float64(name):
    w = synth.with_rows(synth.get(name), 16)
    d = synth.make_inputs(w, seed=0)
    y = oracle.oracle_bias_gelu_residual(d["x"], d["r"], d["beta"], w.dtype)
    ref = (torch.nn.functional.gelu(d["x"].double() + d["beta"].double(), approximate="none")
           + d["r"].double()).numpy()
    assert np.all(np.abs(y - ref) <= 1e-14 * (1 + np.abs(ref)))


def test_diagram_numbers_and_the_corrected_accounting():
    gold = json.load(open(os.path.join(GOLDEN, "pages_bgr_diagram.json")))
    t = gold["tensor_MB"]
    printed = gold["unfused_as_printed"]
    assert printed["bias_add_MB"] + printed["gelu_MB"] + printed["residual_MB"] == printed["total_MB"]
    assert printed["total_MB"] == 3 * 2 * t                     # the page's own sum
    assert gold["fused_as_printed"]["total_MB"] == 2 * t
    assert round(100 * (1 - 2 * t / (6 * t)), 1) == gold["cut_as_printed_percent"]
    # the workload that stands in for the diagram moves 3 tensors fused ...
    w = synth.get("bgr_pages_1024x4096_fp16")
    MB = 1 << 20
    assert w.rows * w.H * w.elem_bytes == t * MB
    assert w.algorithmic_bytes() - 4 * w.H == 3 * t * MB          # 24 MB, not 16
    # ... against 7 tensor passes unfused (56 MB, not 48): R is a second input
    assert (2 + 2 + 3) * t == 56


def test_round_intermediates_is_the_stored_chain():
    # the chain mode equals rounding by hand between the steps (oracle_round)
    g = torch.Generator().manual_seed(9)
    x = torch.randn(4, 32, generator=g).to(torch.bfloat16)
    r = torch.randn(4, 32, generator=g).to(torch.bfloat16)
    bias = 0.3 * torch.randn(32, generator=g)
    y = oracle.oracle_bias_gelu_residual(x, r, bias, "bf16", round_intermediates=True)
    v = oracle.oracle_round(x.double().numpy() + bias.double().numpy(), "bf16")
    gl = oracle.oracle_round(np.vectorize(lambda t: 0.5 * t * (1 + math.erf(t / math.sqrt(2))))(v), "bf16")
    assert np.array_equal(y, gl + r.double().numpy())
    assert not np.array_equal(y, oracle.oracle_bias_gelu_residual(x, r, bias, "bf16"))
