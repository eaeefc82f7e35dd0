"""Pins that tie the fp64 oracle to things other than itself (CPU only).

The oracle is the plain two-pass LayerNorm of "算子融合与Kernel合并" 4.2
(fused_layernorm) applied to the residual sum A = X + R of "算子融合的收益量化"
section 1.  Each pin below would fail on a plausible mistake in it:

* format decode / rounding  -> exhaustive comparison with numpy / torch
* dropped or wrong term, /(H-1) instead of /H, eps outside the sqrt,
  gamma and beta swapped, a wrong row stride -> exact rational brute force
* cancellation (mean >> std) -> brute force at mean 1e4 and the shift invariant
* any formula slip -> closed forms (constant row, H = 1, H = 2, unit affine)
* a library cross-check: torch.nn.functional.layer_norm in float64
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TD = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


# ----------------------------------------------------------------- decoding
def test_decode_fp16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.oracle_decode(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_all_patterns_match_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = oracle.oracle_decode(t, "bf16")
    ref = t.to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_fp32_is_identity():
    v = np.random.default_rng(1).standard_normal(4096).astype(np.float32) * 1e3
    assert np.array_equal(oracle.oracle_decode(v, "fp32"), v.astype(np.float64))


# ----------------------------------------------------------------- rounding
def _random_doubles(n, lo_exp, hi_exp, seed):
    g = np.random.default_rng(seed)
    mant = g.uniform(1.0, 2.0, n)
    ex = g.integers(lo_exp, hi_exp, n)
    sign = np.where(g.integers(0, 2, n) == 0, -1.0, 1.0)
    return sign * np.ldexp(mant, ex)


def test_round_fp16_matches_numpy_direct_conversion():
    # numpy converts float64 -> float16 in one correctly rounded step
    v = _random_doubles(200000, -27, 17, 2)
    got = oracle.oracle_round(v, "fp16")
    ref = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, ref)


def test_round_fp32_matches_numpy():
    v = _random_doubles(200000, -150, 129, 3)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float32).astype(np.float64)
    got = oracle.oracle_round(v, "fp32")
    assert np.array_equal(got, ref)


def test_round_bf16_matches_torch_on_float32_values():
    # torch rounds float32 -> bfloat16 to nearest-even in one step; restrict the
    # inputs to float32 values so that no double rounding is involved.
    v = _random_doubles(200000, -134, 128, 4).astype(np.float32).astype(np.float64)
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.oracle_round(v, "bf16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype,p", [("fp16", 11), ("bf16", 8), ("fp32", 24)])
def test_round_ties_go_to_even(dtype, p):
    u = 2.0 ** (1 - p)                      # ulp of 1.0
    assert oracle.oracle_round([1 + u / 2], dtype)[0] == 1.0          # tie, even below
    assert oracle.oracle_round([1 + 1.5 * u], dtype)[0] == 1 + 2 * u  # tie, even above
    assert oracle.oracle_round([-(1 + u / 2)], dtype)[0] == -1.0


def test_round_overflow_and_subnormal_fp16():
    mx = 65504.0
    assert oracle.oracle_round([mx + 15.99], "fp16")[0] == mx       # below the midpoint
    assert math.isinf(oracle.oracle_round([mx + 16.0], "fp16")[0])  # midpoint: ties to even -> inf
    assert oracle.oracle_round([2.0 ** -25], "fp16")[0] == 0.0      # half the smallest subnormal
    assert oracle.oracle_round([3 * 2.0 ** -25], "fp16")[0] == 2.0 ** -23


# ---------------------------------------------------- exact rational brute force
def _decode_lib(t: torch.Tensor) -> list:
    """Decode with numpy/torch (not the oracle) to Python floats."""
    if t.dtype == torch.float16:
        return t.numpy().astype(np.float64).ravel().tolist()
    return t.to(torch.float64).numpy().ravel().tolist()


def _dec(fr: Fraction) -> Decimal:
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def _brute(x: torch.Tensor, r: torch.Tensor, gamma, beta, eps: float, round_A_dtype=None):
    """Exact mean and variance in rationals, the square root in 60-digit
    decimals.  Returns float y, mean, rstd."""
    rows, H = x.shape
    xs, rs = _decode_lib(x), _decode_lib(r)
    g = [Fraction(float(v)) for v in gamma.tolist()]
    b = [Fraction(float(v)) for v in beta.tolist()]
    y = np.empty((rows, H))
    mean = np.empty(rows)
    rstd = np.empty(rows)
    with localcontext() as ctx:
        ctx.prec = 60
        for i in range(rows):
            A = [Fraction(xs[i * H + j]) + Fraction(rs[i * H + j]) for j in range(H)]
            if round_A_dtype is not None:
                A = [Fraction(float(torch.tensor(float(v), dtype=torch.float64)
                                    .to(TD[round_A_dtype]).to(torch.float64))) for v in A]
            mu = sum(A, Fraction(0)) / H
            var = sum(((a - mu) ** 2 for a in A), Fraction(0)) / H
            std = (_dec(var) + _dec(Fraction(eps))).sqrt()
            rs_i = Decimal(1) / std
            mean[i] = float(mu)
            rstd[i] = float(rs_i)
            for j in range(H):
                y[i, j] = float(_dec(g[j] * (A[j] - mu)) * rs_i + _dec(b[j]))
    return y, mean, rstd


def _rand_case(rows, H, dtype, loc=0.0, scale=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, H, generator=g) * scale + loc).to(TD[dtype])
    r = torch.randn(rows, H, generator=g).to(TD[dtype])
    gamma = 1 + 0.1 * torch.randn(H, generator=g)
    beta = 0.1 * torch.randn(H, generator=g)
    return x, r, gamma, beta


def _assert_close_to_brute(o, y, mean, rstd):
    scale = 1 + np.abs(mean)[:, None] * rstd[:, None]
    assert np.all(np.abs(o["y"] - y) <= 1e-12 * (1 + np.abs(y)) * scale)
    assert np.all(np.abs(o["mean"] - mean) <= 1e-14 * (np.abs(mean) + 1 / rstd) * 16)
    assert np.all(np.abs(o["rstd"] - rstd) <= 1e-13 * rstd)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 2, 3, 5, 8, 16])
def test_oracle_matches_rational_brute_force(dtype, H):
    x, r, gamma, beta = _rand_case(4, H, dtype, seed=H)
    eps = 1e-5
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, eps, dtype)
    y, mean, rstd = _brute(x, r, gamma, beta, eps)
    _assert_close_to_brute(o, y, mean, rstd)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_oracle_matches_brute_force_under_cancellation(dtype):
    # mean far above std: the regime where sum/sum-of-squares fails
    loc = {"fp32": 1e4, "fp16": 1e3, "bf16": 100.0}[dtype]
    x, r, gamma, beta = _rand_case(3, 16, dtype, loc=loc, seed=7)
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, dtype)
    y, mean, rstd = _brute(x, r, gamma, beta, 1e-5)
    _assert_close_to_brute(o, y, mean, rstd)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_round_A_mode_matches_brute_force(dtype):
    x, r, gamma, beta = _rand_case(3, 16, dtype, loc=3.0, seed=11)
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, dtype, round_A=True)
    y, mean, rstd = _brute(x, r, gamma, beta, 1e-5, round_A_dtype=dtype)
    _assert_close_to_brute(o, y, mean, rstd)


def test_rows_are_independent_and_strided_correctly():
    # distinct rows computed together equal each row computed alone
    x, r, gamma, beta = _rand_case(6, 33, "bf16", loc=2.0, seed=5)
    whole = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, "bf16")
    for i in range(6):
        one = oracle.oracle_add_layernorm(x[i:i + 1], r[i:i + 1], gamma, beta, 1e-5, "bf16")
        for k in ("y", "a", "mean", "rstd"):
            assert np.array_equal(whole[k][i], one[k][0])


# ------------------------------------------------------------- closed forms
def test_constant_row_gives_beta_mean_c_rstd_inv_sqrt_eps():
    H, eps = 1000, 1e-5
    c = 101.0
    x = torch.full((2, H), c, dtype=torch.bfloat16)
    r = torch.zeros((2, H), dtype=torch.bfloat16)
    gamma = 1 + 0.1 * torch.randn(H, generator=torch.Generator().manual_seed(3))
    beta = 0.1 * torch.randn(H, generator=torch.Generator().manual_seed(4))
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, eps, "bf16")
    assert np.array_equal(o["y"], np.broadcast_to(beta.double().numpy(), (2, H)))
    assert np.all(o["mean"] == c)
    assert np.allclose(o["rstd"], eps ** -0.5, rtol=1e-15, atol=0)
    assert np.all(o["a"] == c)


def test_constant_row_with_eps_zero_is_zero_over_zero():
    # eps = 0 leaves the definition's (A - mean) / sqrt(var + eps) = 0 / 0 on
    # a constant row: NaN outputs, rstd = +inf, the mean still exact; other
    # rows of the same call are unaffected
    H = 64
    x = torch.full((2, H), 3.0)
    x[1] = torch.arange(H, dtype=torch.float32)
    r = torch.zeros((2, H))
    o = oracle.oracle_add_layernorm(x, r, torch.ones(H), torch.zeros(H), 0.0, "fp32")
    assert np.all(np.isnan(o["y"][0])) and o["rstd"][0] == np.inf and o["mean"][0] == 3.0
    assert np.all(np.isfinite(o["y"][1]))
    assert math.isclose(o["rstd"][1], 1 / math.sqrt((H * H - 1) / 12), rel_tol=1e-14)


def test_h_equals_one_gives_beta():
    x = torch.tensor([[3.5], [-2.0], [7.25]])
    r = torch.tensor([[1.0], [0.5], [-0.25]])
    gamma, beta = torch.tensor([1.7]), torch.tensor([0.3])
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, "fp32")
    assert np.all(o["y"] == np.float64(np.float32(0.3)))
    assert np.array_equal(o["mean"], np.array([4.5, -1.5, 7.0]))


def test_h_equals_two_closed_form():
    a, b = 3.0, 0.5                     # A row = [a, b] with R = 0
    x = torch.tensor([[a, b]])
    r = torch.zeros(1, 2)
    gamma = torch.tensor([1.5, 0.75])
    beta = torch.tensor([0.25, -0.5])
    eps = 1e-3
    o = oracle.oracle_add_layernorm(x, r, gamma, beta, eps, "fp32")
    d = (a - b) / 2
    g0, g1 = float(gamma[0]), float(gamma[1])
    b0, b1 = float(beta[0]), float(beta[1])
    assert o["mean"][0] == (a + b) / 2
    assert math.isclose(o["rstd"][0], 1 / math.sqrt(d * d + eps), rel_tol=1e-15)
    assert math.isclose(o["y"][0, 0], g0 * d / math.sqrt(d * d + eps) + b0, rel_tol=1e-15)
    assert math.isclose(o["y"][0, 1], -g1 * d / math.sqrt(d * d + eps) + b1, rel_tol=1e-15)


def test_worked_row_1234():
    # A = [1,2,3,4], unit affine, eps = 0: mean 2.5, var 1.25
    x = torch.tensor([[1.0, 2.0, 3.0, 4.0]])
    o = oracle.oracle_add_layernorm(x, torch.zeros(1, 4), torch.ones(4), torch.zeros(4), 0.0, "fp32")
    s = math.sqrt(1.25)
    assert o["mean"][0] == 2.5
    assert np.allclose(o["y"][0], [-1.5 / s, -0.5 / s, 0.5 / s, 1.5 / s], rtol=1e-15, atol=0)


@pytest.mark.parametrize("eps", [1e-5, 1e-12, 0.5])
def test_unit_affine_gives_zero_mean_and_variance_var_over_var_plus_eps(eps):
    x, r, _, _ = _rand_case(8, 257, "fp32", loc=1.0, scale=2.0, seed=9)
    H = 257
    o = oracle.oracle_add_layernorm(x, r, torch.ones(H), torch.zeros(H), eps, "fp32")
    y = o["y"]
    a = x.double().numpy() + r.double().numpy()
    var = a.var(axis=1)
    assert np.all(np.abs(y.mean(axis=1)) < 1e-12)
    assert np.allclose(y.var(axis=1), var / (var + eps), rtol=1e-12, atol=0)


# ---------------------------------------------------------------- invariants
def test_shift_invariance_t100():
    # X on a 1/64 grid keeps X + 100 exact in fp32, so the two inputs describe
    # the same row up to a shift: LayerNorm must not see it
    g = torch.Generator().manual_seed(21)
    x = torch.round(torch.randn(8, 512, generator=g) * 64) / 64
    r = torch.round(torch.randn(8, 512, generator=g) * 64) / 64
    gamma = 1 + 0.1 * torch.randn(512, generator=g)
    beta = 0.1 * torch.randn(512, generator=g)
    o1 = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, "fp32")
    o2 = oracle.oracle_add_layernorm(x + 100, r, gamma, beta, 1e-5, "fp32")
    assert np.allclose(o1["y"], o2["y"], rtol=0, atol=1e-12)
    assert np.allclose(o2["mean"] - o1["mean"], 100.0, rtol=0, atol=1e-12)
    assert np.allclose(o1["rstd"], o2["rstd"], rtol=1e-12, atol=0)


def test_scale_invariance_with_eps_scaled():
    x, r, gamma, beta = _rand_case(4, 300, "fp32", seed=22)
    s = 4.0                                   # power of two: exact scaling
    o1 = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-3, "fp32")
    o2 = oracle.oracle_add_layernorm(x * s, r * s, gamma, beta, 1e-3 * s * s, "fp32")
    assert np.allclose(o1["y"], o2["y"], rtol=0, atol=1e-13)
    assert np.allclose(o2["rstd"] * s, o1["rstd"], rtol=1e-14, atol=0)


def test_permutation_equivariance():
    x, r, gamma, beta = _rand_case(3, 64, "bf16", seed=23)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(1))
    o1 = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, "bf16")
    o2 = oracle.oracle_add_layernorm(x[:, perm].contiguous(), r[:, perm].contiguous(),
                                     gamma[perm], beta[perm], 1e-5, "bf16")
    assert np.allclose(o1["y"][:, perm.numpy()], o2["y"], rtol=0, atol=1e-13)
    assert np.allclose(o1["mean"], o2["mean"], rtol=1e-14, atol=0)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_unfused_chain_equals_fused(dtype):
    x, r, gamma, beta = _rand_case(5, 129, dtype, loc=1.0, seed=24)
    fused = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, dtype)
    a = oracle.oracle_add(x, r, dtype)
    chain = oracle.oracle_layernorm(a, gamma, beta, 1e-5)
    for k in ("y", "mean", "rstd"):
        assert np.array_equal(fused[k], chain[k])
    # the chain that stores A in the dtype: same definition on the rounded sum
    fused_r = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, dtype, round_A=True)
    chain_r = oracle.oracle_layernorm(oracle.oracle_round(a, dtype), gamma, beta, 1e-5)
    for k in ("y", "mean", "rstd"):
        assert np.array_equal(fused_r[k], chain_r[k])


def test_a_output_is_rounded_sum_and_matches_torch_rounding():
    for dtype in ("fp32", "fp16", "bf16"):
        x, r, gamma, beta = _rand_case(16, 1000, dtype, loc=100.0, seed=25)
        o = oracle.oracle_add_layernorm(x, r, gamma, beta, 1e-5, dtype)
        # x + r is exact in float32 for these 16-bit inputs, so torch's one-step
        # float32 -> dtype rounding is the correctly rounded sum
        ref = (x.float() + r.float()).to(TD[dtype]).double().numpy()
        assert np.array_equal(o["a"], ref)


# ------------------------------------------------- library cross-check (torch)
@pytest.mark.parametrize("name", synth.PRIMARY + synth.TAILS)
def test_oracle_matches_torch_layer_norm_fp64(name):
    w = synth.with_rows(synth.get(name), 48)
    d = synth.make_inputs(w, seed=0)
    o = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype)
    a = d["x"].double() + d["r"].double()
    ref = torch.nn.functional.layer_norm(a, (w.H,), d["gamma"].double(), d["beta"].double(),
                                         eps=d["eps"]).numpy()
    rstd = o["rstd"][:, None]
    scale = 1 + np.abs(o["mean"][:, None]) * rstd
    assert np.all(np.abs(o["y"] - ref) <= 1e-12 * (1 + np.abs(ref)) * scale)


def test_bad_arguments_are_rejected():
    with pytest.raises(ValueError):
        oracle.oracle_layernorm(np.zeros((2, 3)), np.ones(3), np.zeros(3), -1.0)
    with pytest.raises(ValueError):
        oracle.oracle_layernorm(np.zeros((2, 3)), np.ones(3), np.zeros(3), float("nan"))


# ------------------------------------------------------------ pages' numbers
def test_traffic_model_reproduces_pages_accounting():
    gold = json.load(open(os.path.join(GOLDEN, "pages_traffic.json")))
    w = synth.get("pages_2048x4096_fp16")
    B, S, H = gold["shape_BSH"]
    assert (w.rows, w.H) == (B * S, H) and w.dtype == gold["dtype"]
    MB = 1 << 20
    tensor = w.rows * w.H * w.elem_bytes
    assert tensor == gold["tensor_bytes"] == gold["tensor_MB_as_printed"] * MB
    affine = 8 * w.H                         # gamma, beta: not in the page's totals
    assert w.algorithmic_bytes() - affine == gold["fused"]["total_MB"] * MB
    assert w.unfused_algorithmic_bytes() - affine == gold["unfused"]["total_MB"] * MB
    add_only = 3 * tensor
    assert add_only == gold["unfused"]["residual_add_MB"] * MB
    cut = 1 - gold["fused"]["total_MB"] / gold["unfused"]["total_MB"]
    assert round(100 * cut) == gold["fused_traffic_cut_percent"]
