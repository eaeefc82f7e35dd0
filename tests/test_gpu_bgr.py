"""GPU parity of the fused bias + GELU + residual kernel (and of the
three-kernel chain it replaces) against the fp64 oracle on the same seeded
inputs: vector and element paths, ragged and misaligned buffers, in place,
and every row of the full-size workloads, with the correctly rounded
fraction of 16-bit outputs held to a minimum."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import Rounding, assert_correctly_rounded, bgr_violations, over_row_chunks

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()


def check(d, dtype, y, what, chain=False, rows=None):
    x, r, b = d["x"], d["r"], d["beta"]
    if rows is not None:
        x, r, y = x[rows], r[rows], y[rows]
    ref = oracle.oracle_bias_gelu_residual(x, r, b, dtype, round_intermediates=chain)
    v = x.double().numpy() + b.double().numpy()
    bad = bgr_violations(y, ref, v, r.double().numpy(), dtype, chain=chain)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} outputs out of bound; first {i}: "
                             f"gpu={y.double().numpy()[i]!r} ref={ref[i]!r}")
    return ref


@pytest.mark.parametrize("name", synth.BGR_NAMES)
def test_small(name):
    w = synth.with_rows(synth.get(name), 37)
    d = synth.make_inputs(w, seed=1)
    x, r, b = d["x"].cuda(), d["r"].cuda(), d["beta"].cuda()
    y = mba.bias_gelu_residual(x, r, b)
    torch.cuda.synchronize()
    ref = check(d, w.dtype, y.cpu(), name)
    assert_correctly_rounded(y.cpu(), ref, w.dtype, name)
    yu = mba.bias_gelu_residual_unfused(x, r, b)
    torch.cuda.synchronize()
    check(d, w.dtype, yu.cpu(), name + " unfused", chain=True)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 3, 8, 1000, 1024, 4097])
def test_shapes_misaligned_and_in_place(dtype, H):
    w = synth.custom(9, H, dtype, r_dist=(0.0, 0.5), op="bias_gelu_residual")
    d = synth.make_inputs(w, seed=H)
    td = synth.TORCH_DTYPES[dtype]
    x, r, b = d["x"].cuda(), d["r"].cuda(), d["beta"].cuda()
    y = mba.bias_gelu_residual(x, r, b)
    torch.cuda.synchronize()
    check(d, dtype, y.cpu(), f"9x{H}")
    n = 9 * H
    xb = torch.empty(n + 8, dtype=td, device="cuda")
    xm = xb[1:1 + n].view(9, H)
    xm.copy_(x)
    ym = torch.empty_like(xm)
    mba.bias_gelu_residual_fwd(xm, r, b, ym)
    torch.cuda.synchronize()
    check(d, dtype, ym.cpu(), f"9x{H} misaligned")
    xi = x.clone()
    mba.bias_gelu_residual_fwd(xi, r, b, xi)            # y = x in place
    ri = r.clone()
    mba.bias_gelu_residual_fwd(x, ri, b, ri)            # y = r in place
    torch.cuda.synchronize()
    check(d, dtype, xi.cpu(), f"9x{H} y=x")
    check(d, dtype, ri.cpu(), f"9x{H} y=r")


@pytest.mark.slow
@pytest.mark.parametrize("name", synth.BGR_NAMES)
def test_full_size_every_row(name):
    w = synth.get(name)
    d = synth.make_inputs(w, seed=0)
    y = mba.bias_gelu_residual(d["x"].cuda(), d["r"].cuda(), d["beta"].cuda()).cpu()
    what = f"{name} full size"

    def one(lo, hi):
        rows = slice(lo, hi)
        ref = check(d, w.dtype, y, f"{what} rows [{lo}, {hi})", rows=rows)
        rnd = Rounding(w.dtype)
        rnd.add(y[rows], ref)
        return rnd

    total = Rounding(w.dtype, what)
    for r in over_row_chunks(w.rows, w.H, one):
        for k in ("n", "correct", "above", "below"):
            setattr(total, k, getattr(total, k) + getattr(r, k))
    total.check()
