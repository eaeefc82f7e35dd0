"""Pins for the oracle's Add+LayerNorm backward (CPU only).

The pages give no backward; the oracle takes the textbook derivative of the
forward definition.  Pins that would catch a dropped term, a wrong sign or a
transposed operand: torch autograd in float64 through layer_norm(x + r),
central finite differences of the oracle's own forward, exact invariants on
rows whose statistics are exact in fp32, and the optional A-gradient entering
linearly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth


def _stats(a64, eps):
    mean = a64.mean(axis=1)
    var = ((a64 - mean[:, None]) ** 2).mean(axis=1)
    return mean, 1.0 / np.sqrt(var + eps)


@pytest.mark.parametrize("H", [1, 2, 7, 64, 1000])
def test_matches_torch_autograd_float64(H):
    g = torch.Generator().manual_seed(H)
    rows, eps = 6, 1e-5
    x = torch.randn(rows, H, generator=g) * 2 + 0.5
    r = torch.randn(rows, H, generator=g)
    a32 = (x + r)                                   # the stored A (fp32)
    gamma = 1 + 0.1 * torch.randn(H, generator=g)
    beta = 0.1 * torch.randn(H, generator=g)
    dy = torch.randn(rows, H, generator=g)
    # autograd through the float64 forward of the same A
    a = a32.double().requires_grad_(True)
    gm = gamma.double().requires_grad_(True)
    bt = beta.double().requires_grad_(True)
    y = torch.nn.functional.layer_norm(a, (H,), gm, bt, eps=eps)
    (y * dy.double()).sum().backward()
    mean, rstd = _stats(a32.double().numpy(), eps)
    o = oracle.oracle_add_layernorm_bwd(dy, a32, mean.astype(np.float32), rstd.astype(np.float32),
                                        gamma, "fp32")
    scale = 1 + np.abs(a.grad.numpy())
    # mean/rstd are handed over in fp32, so agreement is to ~1e-6, not 1e-15
    assert np.all(np.abs(o["dx"] - a.grad.numpy()) <= 2e-5 * scale)
    assert np.allclose(o["dgamma"], gm.grad.numpy(), rtol=2e-5, atol=2e-5)
    assert np.allclose(o["dbeta"], bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_matches_finite_differences_of_the_oracle_forward():
    g = torch.Generator().manual_seed(5)
    rows, H, eps = 3, 9, 1e-3
    x = torch.randn(rows, H, generator=g, dtype=torch.float64).float()
    r = torch.zeros(rows, H)
    gamma = 1 + 0.2 * torch.randn(H, generator=g)
    beta = torch.zeros(H)
    dy = torch.randn(rows, H, generator=g)
    fwd = oracle.oracle_add_layernorm(x, r, gamma, beta, eps, "fp32")
    o = oracle.oracle_add_layernorm_bwd(dy, x, fwd["mean"].astype(np.float32),
                                        fwd["rstd"].astype(np.float32), gamma, "fp32")
    h = 1e-3
    num = np.zeros((rows, H))
    for i in range(rows):
        for j in range(H):
            xp, xm = x.clone(), x.clone()
            xp[i, j] += h
            xm[i, j] -= h
            fp = oracle.oracle_add_layernorm(xp, r, gamma, beta, eps, "fp32")["y"]
            fm = oracle.oracle_add_layernorm(xm, r, gamma, beta, eps, "fp32")["y"]
            num[i, j] = ((fp - fm) * dy.double().numpy()).sum() / (
                float(xp[i, j]) - float(xm[i, j]))
    assert np.allclose(o["dx"], num, rtol=2e-3, atol=2e-4)


def test_exact_invariants_when_statistics_are_exact():
    # rows [0,0,2,2] and [-1,-1,1,1]*2+1: mean, var exact, eps = 0 -> rstd exact
    a = torch.tensor([[0.0, 0.0, 2.0, 2.0], [-1.0, 3.0, -1.0, 3.0]])
    mean = np.array([1.0, 1.0], dtype=np.float32)
    rstd = np.array([1.0, 0.5], dtype=np.float32)
    g = torch.Generator().manual_seed(6)
    dy = torch.randn(2, 4, generator=g)
    gamma = 1 + 0.3 * torch.randn(4, generator=g)
    o = oracle.oracle_add_layernorm_bwd(dy, a, mean, rstd, gamma, "fp32")
    xhat = (a.double().numpy() - mean[:, None]) * rstd[:, None]
    assert np.allclose(o["dx"].sum(axis=1), 0.0, atol=1e-15)          # orthogonal to shifts
    assert np.allclose((o["dx"] * xhat).sum(axis=1), 0.0, atol=1e-15)  # and to xhat (eps = 0)
    assert np.allclose(o["dbeta"], dy.double().numpy().sum(axis=0), rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_incoming_a_gradient_adds_and_rows_are_independent(dtype):
    w = synth.with_rows(synth.get("cancel_65536x1000_bf16"), 5)
    d = synth.make_inputs(w, seed=1)
    td = synth.TORCH_DTYPES[dtype]
    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], "bf16")
    a = torch.from_numpy(fwd["a"]).to(td)
    dy = synth.make_grad(w, seed=1).to(td)
    dres = synth.make_grad(w, seed=2).to(td)
    m, rs = fwd["mean"].astype(np.float32), fwd["rstd"].astype(np.float32)
    o0 = oracle.oracle_add_layernorm_bwd(dy, a, m, rs, d["gamma"], dtype)
    o1 = oracle.oracle_add_layernorm_bwd(dy, a, m, rs, d["gamma"], dtype, dres=dres)
    assert np.allclose(o1["dx"] - o0["dx"], dres.double().numpy(), rtol=0, atol=1e-12)
    assert np.array_equal(o0["dgamma"], o1["dgamma"])
    for i in range(5):
        oi = oracle.oracle_add_layernorm_bwd(dy[i:i + 1], a[i:i + 1], m[i:i + 1], rs[i:i + 1],
                                             d["gamma"], dtype)
        assert np.array_equal(oi["dx"][0], o0["dx"][i])
