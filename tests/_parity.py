"""Tolerances and comparison helpers for GPU-vs-oracle parity tests.

Bounds, all against the fp64 oracle:
  Y fp32           |dy| <= 1e-5 * (1 + |y|)
  Y fp16 / bf16    |dy| <= max(4e-3 / 3e-2, ulp_dtype(|y|))
                   The stated absolute bounds lie below the format's own
                   rounding step at large |y| (bf16 spacing is 0.0625 on
                   [8, 16)), so a faithfully rounded value -- within one unit
                   in the last place of the exact result -- also passes.
  A (resid_out)    bit-exact: the exact sum rounded to nearest-even in dtype
  mean             |dmean| <= 1e-5 * (|mean| + sqrt(var + eps))
                   (relative to the row's scale: a row mean near 0 would make
                   a plain relative bound meaningless)
  rstd             |drstd| <= 1e-5 * rstd
"""
from __future__ import annotations

import numpy as np
import torch

Y_TOL = {"fp32": 1e-5, "fp16": 4e-3, "bf16": 3e-2}
PRECISION = {"fp32": 24, "fp16": 11, "bf16": 8}
MIN_NORMAL_EXP = {"fp32": -126, "fp16": -14, "bf16": -126}
STAT_TOL = 1e-5


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` values at |v| (subnormal spacing below the normals)."""
    p = PRECISION[dtype]
    lo = MIN_NORMAL_EXP[dtype]
    m, e = np.frexp(np.abs(np.asarray(v, dtype=np.float64)))   # |v| = m 2^e, 1/2 <= m < 1
    e = np.where(m > 0, e - 1, lo)                              # floor(log2 |v|)
    return np.ldexp(1.0, (np.maximum(e, lo) - p + 1).astype(np.int64))


def to_f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def y_violations(y_gpu, y_ref: np.ndarray, dtype: str) -> np.ndarray:
    """Boolean mask of Y elements outside the bound."""
    yg = to_f64(y_gpu)
    err = np.abs(yg - y_ref)
    if dtype == "fp32":
        bound = Y_TOL["fp32"] * (1 + np.abs(y_ref))
    else:
        bound = np.maximum(Y_TOL[dtype], ulp(y_ref, dtype))
    return ~(err <= bound)


def assert_y(y_gpu, y_ref, dtype, what=""):
    bad = y_violations(y_gpu, y_ref, dtype)
    if bad.any():
        yg = to_f64(y_gpu)
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} Y elements out of bound; first "
            + ", ".join(f"{tuple(i)} gpu={yg[tuple(i)]!r} ref={y_ref[tuple(i)]!r}" for i in idx))


# ------------------------------------------------ correctly rounded outputs
# A 16-bit output within one unit in the last place of the exact value passes
# the bounds above, so a kernel that rounded every value one unit the same
# way would pass them too.  The fraction of outputs equal to the exact value
# rounded to nearest-even in the dtype exposes that: fp32 arithmetic leaves a
# misrounding only where the exact value lies within a few fp32 units of a
# rounding midpoint (a fraction of about 2^-13 * k for fp16, 2^-16 * k for
# bf16, k the few fp32 roundings on the way), while a systematic one-unit
# bias would misround about half of all outputs.
CR_MIN = 0.995          # LayerNorm and bias + GELU + residual outputs
CR_MIN_SOFTMAX = 0.98   # the hardware exponential's error grows with |x - max|
CR_MIN_ELEMENTS = 4096  # below this the fraction says little
CR_LOG = []             # (what, elements, fraction, above, below) for the summary


class Rounding:
    """Counts, over one or more chunks of outputs, how many equal the exact
    value rounded to nearest-even in the dtype, and how many lie above or
    below it."""

    def __init__(self, dtype: str, what: str = ""):
        self.dtype, self.what = dtype, what
        self.n = self.correct = self.above = self.below = 0

    def add(self, y_gpu, y_exact: np.ndarray):
        import oracle
        if self.dtype == "fp32":
            return
        yg = to_f64(y_gpu)
        rn = oracle.oracle_round(y_exact, self.dtype)
        ok = np.isfinite(rn)
        yg, rn = yg[ok], rn[ok]
        self.n += yg.size
        self.correct += int((yg == rn).sum())
        self.above += int((yg > rn).sum())
        self.below += int((yg < rn).sum())

    @property
    def fraction(self) -> float:
        return self.correct / self.n if self.n else 1.0

    def check(self, minimum: float = CR_MIN):
        if self.dtype == "fp32" or self.n == 0:
            return
        CR_LOG.append((self.what, self.n, self.fraction, self.above, self.below))
        if self.n >= CR_MIN_ELEMENTS and self.fraction < minimum:
            raise AssertionError(
                f"{self.what}: only {self.fraction:.5f} of {self.n} {self.dtype} outputs are the "
                f"correctly rounded exact value ({self.above} above, {self.below} below; "
                f"minimum {minimum})")


def assert_correctly_rounded(y_gpu, y_exact, dtype, what="", minimum: float = CR_MIN):
    r = Rounding(dtype, what)
    r.add(y_gpu, y_exact)
    r.check(minimum)
    return r


def assert_a(a_gpu, a_ref, what=""):
    ag = to_f64(a_gpu)
    same = (ag == a_ref) | (np.isnan(ag) & np.isnan(a_ref))
    if not same.all():
        idx = np.argwhere(~same)[:5]
        raise AssertionError(
            f"{what}: {int((~same).sum())} A elements differ from the rounded sum; first "
            + ", ".join(f"{tuple(i)} gpu={ag[tuple(i)]!r} ref={a_ref[tuple(i)]!r}" for i in idx))


def assert_stats(mean_gpu, rstd_gpu, mean_ref, rstd_ref, what=""):
    mg, rg = to_f64(mean_gpu), to_f64(rstd_gpu)
    scale = np.abs(mean_ref) + 1.0 / rstd_ref
    badm = ~(np.abs(mg - mean_ref) <= STAT_TOL * scale)
    badr = ~(np.abs(rg - rstd_ref) <= STAT_TOL * rstd_ref)
    if badm.any() or badr.any():
        i = int(np.argmax(badm | badr))
        raise AssertionError(
            f"{what}: {int(badm.sum())} mean / {int(badr.sum())} rstd out of bound; row {i}: "
            f"mean gpu={mg[i]!r} ref={mean_ref[i]!r}, rstd gpu={rg[i]!r} ref={rstd_ref[i]!r}")


def softmax_violations(y_gpu, y_ref: np.ndarray, dtype: str) -> np.ndarray:
    """Softmax bound: fp32 |dy| <= 1e-5 |y| + 1e-12 (fp32 arithmetic and the
    hardware exponential give a relative error well under 1e-5 wherever y
    exceeds 1e-30); fp16 / bf16 within one unit in the last place of the
    exact value plus that relative term (a faithful rounding)."""
    yg = to_f64(y_gpu)
    err = np.abs(yg - y_ref)
    bound = 1e-5 * np.abs(y_ref) + (1e-12 if dtype == "fp32" else ulp(y_ref, dtype))
    return ~(err <= bound)


def assert_softmax(y_gpu, y_ref, dtype, what=""):
    bad = softmax_violations(y_gpu, y_ref, dtype)
    if bad.any():
        yg = to_f64(y_gpu)
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} softmax outputs out of bound; first "
            + ", ".join(f"{tuple(i)} gpu={yg[tuple(i)]!r} ref={y_ref[tuple(i)]!r}" for i in idx))


def bgr_violations(y_gpu, y_ref, v_ref, r_ref, dtype: str, chain: bool = False) -> np.ndarray:
    """Bias + GELU + residual bound, from the fp32 arithmetic and the erf
    approximation (absolute error below 1.5e-7, so GELU is within about
    1e-7 |v|): |dy| <= 1e-6 (1 + |x + bias| + |r|), plus one unit in the last place
    of the exact value for 16-bit outputs.  The unfused chain (chain=True)
    rounds X + bias and GELU of it to the dtype between kernels and may land a
    unit away at each step: four units of the dtype at that scale."""
    yg = to_f64(y_gpu)
    scale = 1.0 + np.abs(v_ref) + np.abs(r_ref)
    if dtype == "fp32":
        bound = 1e-6 * scale
    elif chain:
        bound = 4 * ulp(scale, dtype)
    else:
        bound = 1e-6 * scale + ulp(y_ref, dtype)
    return ~(np.abs(yg - y_ref) <= bound)


def assert_bwd(out, ref, inputs, dtype, what=""):
    """Backward bounds, from the fp32 arithmetic: dA element (i, j) within
    1e-5 * rstd_i * (|g_ij| + mean_k |g_ik| + |xhat_ij| mean_k |g_ik xhat_ik|)
    + 1e-6 |dA_in_ij| (+ one ulp of the exact value for 16-bit outputs);
    dgamma_j within 1e-5 sum_i |dY_ij xhat_ij|, dbeta_j within 1e-5 sum_i |dY_ij|
    (+ 1e-30)."""
    dy, a, mean, rstd, gamma, dres = inputs
    dyd = to_f64(dy)
    xh = (to_f64(a) - np.asarray(mean, np.float64)[:, None]) * np.asarray(rstd, np.float64)[:, None]
    g = dyd * to_f64(gamma)[None, :]
    scale = np.asarray(rstd, np.float64)[:, None] * (
        np.abs(g) + np.abs(g).mean(axis=1, keepdims=True)
        + np.abs(xh) * np.abs(g * xh).mean(axis=1, keepdims=True))
    bound = 1e-5 * scale + 1e-30
    if dres is not None:
        bound = bound + 1e-6 * np.abs(to_f64(dres))
    if dtype != "fp32":
        bound = bound + ulp(ref["dx"], dtype)
    dx = to_f64(out[0])
    bad = ~(np.abs(dx - ref["dx"]) <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} dx out of bound; first {i}: "
                             f"gpu={dx[i]!r} ref={ref['dx'][i]!r} bound={bound[i]!r}")
    for k, s in (("dgamma", np.abs(dyd * xh).sum(axis=0)), ("dbeta", np.abs(dyd).sum(axis=0))):
        got = to_f64(out[1] if k == "dgamma" else out[2])
        badk = ~(np.abs(got - ref[k]) <= 1e-5 * s + 1e-30)
        if badk.any():
            j = int(np.argwhere(badk)[0][0])
            raise AssertionError(f"{what}: {int(badk.sum())} {k} out of bound; first {j}: "
                                 f"gpu={got[j]!r} ref={ref[k][j]!r}")


def over_row_chunks(rows: int, H: int, fn, elements: int = 4 << 20, workers: int = 8) -> list:
    """fn(lo, hi) on consecutive row chunks of about `elements` values each,
    in a pool of threads (the C oracle and numpy's large-array loops release
    the GIL); returns the results in row order and re-raises the first
    failure."""
    from concurrent.futures import ThreadPoolExecutor
    step = max(1, elements // max(1, H))
    bounds = [(lo, min(rows, lo + step)) for lo in range(0, rows, step)]
    with ThreadPoolExecutor(max_workers=max(1, min(workers, len(bounds)))) as ex:
        futs = [ex.submit(fn, lo, hi) for lo, hi in bounds]
        return [f.result() for f in futs]
