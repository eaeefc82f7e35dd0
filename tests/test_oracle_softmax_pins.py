"""Pins for the oracle's row softmax (CPU only).

The oracle follows fused_softmax of "算子融合与Kernel合并" 4.3: a max pass, an
exp-sum pass of exp(x - max), a divide pass, in fp64.  Each pin would fail on
a plausible mistake:

* a dropped max subtraction -> overflow at |x| ~ 1e3 (extreme-value pins)
* a wrong normaliser, index or stride -> 60-digit decimal brute force, sum = 1
* a wrong decode -> brute force on all three dtypes (decoded by numpy/torch)
* a library cross-check: torch.softmax in float64
"""
from __future__ import annotations

import math
from decimal import Decimal, localcontext

import numpy as np
import pytest
import torch

import oracle
import synth

TD = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


def _decode_lib(t):
    if t.dtype == torch.float16:
        return t.numpy().astype(np.float64)
    return t.to(torch.float64).numpy()


def _brute(x):
    """exp in 60-digit decimal arithmetic of the exactly decoded inputs."""
    xs = _decode_lib(x)
    out = np.empty_like(xs)
    with localcontext() as ctx:
        ctx.prec = 60
        for i, row in enumerate(xs):
            d = [Decimal(float(v)) for v in row]
            mx = max(d)
            e = [(v - mx).exp() for v in d]
            s = sum(e, Decimal(0))
            out[i] = [float(v / s) for v in e]
    return out


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 2, 3, 8, 16, 33])
@pytest.mark.parametrize("scale", [1.0, 8.0])
def test_softmax_matches_decimal_brute_force(dtype, H, scale):
    g = torch.Generator().manual_seed(H)
    x = (torch.randn(3, H, generator=g) * scale + 5.0).to(TD[dtype])
    o = oracle.oracle_softmax(x, dtype)
    ref = _brute(x)
    assert np.all(np.abs(o["y"] - ref) <= 1e-14 * ref + 1e-300)


def test_constant_row_is_uniform_and_single_entry_is_one():
    x = torch.full((2, 1000), 3.25)
    o = oracle.oracle_softmax(x, "fp32")
    assert np.allclose(o["y"], 1e-3, rtol=1e-15, atol=0)
    assert np.all(o["max"] == 3.25) and np.allclose(o["sum"], 1000.0, rtol=1e-15)
    one = oracle.oracle_softmax(torch.tensor([[-7.5], [1e4]]), "fp32")
    assert np.all(one["y"] == 1.0)


def test_two_values_give_the_logistic():
    a, b = 2.0, -1.5
    o = oracle.oracle_softmax(torch.tensor([[a, b]]), "fp32")
    p = 1.0 / (1.0 + math.exp(b - a))
    assert math.isclose(o["y"][0, 0], p, rel_tol=1e-15)
    assert math.isclose(o["y"][0, 1], 1 - p, rel_tol=1e-14)


def test_extreme_values_neither_overflow_nor_lose_the_winner():
    x = torch.tensor([[1e4, 1e4 - 1.0, -1e4], [0.0, -1000.0, -2000.0]])
    o = oracle.oracle_softmax(x, "fp32")
    assert np.all(np.isfinite(o["y"]))
    e = math.exp(-1.0)
    assert math.isclose(o["y"][0, 0], 1 / (1 + e), rel_tol=1e-15)
    assert o["y"][0, 2] == 0.0                       # exp(-2e4) underflows to 0
    assert o["y"][1, 0] == 1.0 and o["y"][1, 1] == 0.0


def test_rows_sum_to_one_and_are_shift_invariant():
    g = torch.Generator().manual_seed(3)
    x = torch.round(torch.randn(16, 777, generator=g) * 64) / 64   # exact under + 100
    o1 = oracle.oracle_softmax(x, "fp32")
    o2 = oracle.oracle_softmax(x + 100.0, "fp32")
    assert np.allclose(o1["y"].sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(o1["y"], o2["y"], rtol=1e-13, atol=0)
    assert np.allclose(o2["max"] - o1["max"], 100.0, rtol=0, atol=0)


def test_permutation_equivariance_and_monotonicity():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(4, 64, generator=g).to(torch.bfloat16)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(5))
    o1 = oracle.oracle_softmax(x, "bf16")
    o2 = oracle.oracle_softmax(x[:, perm].contiguous(), "bf16")
    assert np.allclose(o1["y"][:, perm.numpy()], o2["y"], rtol=1e-14, atol=0)
    xd = _decode_lib(x)
    for i in range(4):
        order = np.argsort(xd[i], kind="stable")
        assert np.all(np.diff(o1["y"][i][order]) >= 0)


def test_rows_are_independent():
    g = torch.Generator().manual_seed(6)
    x = torch.randn(5, 129, generator=g).to(torch.float16)
    whole = oracle.oracle_softmax(x, "fp16")
    for i in range(5):
        assert np.array_equal(whole["y"][i], oracle.oracle_softmax(x[i:i + 1], "fp16")["y"][0])


@pytest.mark.parametrize("name", synth.SOFTMAX_NAMES)
def test_softmax_matches_torch_float64(name):
    w = synth.with_rows(synth.get(name), 24)
    d = synth.make_inputs(w, seed=0)
    o = oracle.oracle_softmax(d["x"], w.dtype)
    ref = torch.softmax(d["x"].double(), dim=-1).numpy()
    assert np.all(np.abs(o["y"] - ref) <= 1e-13 * ref + 1e-300)


def test_softmax_bad_arguments():
    with pytest.raises(ValueError):
        oracle.oracle_softmax(np.zeros((2, 0), dtype=np.float32), "fp32")
