"""Seeded random shapes through every operation's automatic dispatch, against
the oracle: row lengths drawn across all the dispatch boundaries (warp /
CTA kernels, full and ragged chunks, aligned and misaligned rows, the
longest rows), all three dtypes, and row counts that leave partial CTA waves.
The draw is fixed (seed 2026), so a failure names a reproducible case."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import assert_bwd, assert_softmax
from test_gpu_bgr import check as check_bgr
from test_gpu_parity import check as check_fwd

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")
TD = synth.TORCH_DTYPES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()
    yield


def _draw(n, seed, hmax16=32768, hmax32=16384):
    rng = np.random.default_rng(seed)
    edges = [1, 8, 32, 255, 256, 1000, 1024, 1025, 2048, 4096, 8192, 16384, 32768]
    out = []
    for _ in range(n):
        dtype = ["fp32", "fp16", "bf16"][rng.integers(3)]
        hmax = hmax32 if dtype == "fp32" else hmax16
        e = edges[rng.integers(len(edges))]
        H = int(min(hmax, max(1, e + rng.integers(-9, 10))))
        if rng.random() < 0.5:                      # keep it 16-byte aligned half the time
            vec = 4 if dtype == "fp32" else 8
            H = max(vec, H // vec * vec)
        rows = int(rng.integers(1, 40))
        out.append((rows, H, dtype))
    return out


FWD = _draw(40, 2026)
SMX = _draw(30, 2027)
BGR = _draw(30, 2028)
BWD = _draw(30, 2029, hmax16=16384, hmax32=8192)


@pytest.mark.parametrize("rows,H,dtype", FWD)
def test_forward(rows, H, dtype):
    w = synth.custom(rows, H, dtype, x_dist=(1.0, 2.0), want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=H + rows)
    x, r = d["x"].cuda(), d["r"].cuda()
    g, b = d["gamma"].cuda(), d["beta"].cuda()
    y, a = torch.empty_like(x), torch.empty_like(x)
    m, s = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    mba.add_layernorm_fwd(x, r, g, b, y, a, m, s, eps=d["eps"])
    torch.cuda.synchronize()
    out = {"y": y.cpu(), "a": a.cpu(), "mean": m.cpu(), "rstd": s.cpu(),
           "path": mba.addln_last_path()}
    check_fwd(w, d, out, f"{rows}x{H} {dtype} {out['path']}")


@pytest.mark.parametrize("rows,H,dtype", SMX)
def test_softmax(rows, H, dtype):
    w = synth.custom(rows, H, dtype, x_dist=(0.0, 3.0), op="softmax")
    d = synth.make_inputs(w, seed=H + rows)
    x = d["x"].cuda()
    y = torch.empty_like(x)
    mba.softmax_fwd(x, y)
    torch.cuda.synchronize()
    ref = oracle.oracle_softmax(d["x"], dtype)["y"]
    assert_softmax(y.cpu(), ref, dtype, f"{rows}x{H} {dtype} {mba.addln_last_path()}")


@pytest.mark.parametrize("rows,H,dtype", BGR)
def test_bias_gelu_residual(rows, H, dtype):
    w = synth.custom(rows, H, dtype, r_dist=(0.0, 0.5), op="bias_gelu_residual")
    d = synth.make_inputs(w, seed=H + rows)
    y = mba.bias_gelu_residual(d["x"].cuda(), d["r"].cuda(), d["beta"].cuda())
    torch.cuda.synchronize()
    check_bgr(d, dtype, y.cpu(), f"{rows}x{H} {dtype}")


@pytest.mark.parametrize("rows,H,dtype", BWD)
def test_backward(rows, H, dtype):
    w = synth.custom(rows, H, dtype, x_dist=(1.0, 2.0), want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=H + rows)
    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], dtype)
    a = torch.from_numpy(fwd["a"]).to(TD[dtype])
    mean = torch.from_numpy(fwd["mean"].astype(np.float32))
    rstd = torch.from_numpy(fwd["rstd"].astype(np.float32))
    dy = synth.make_grad(w, seed=H)
    case = (dy, a, mean, rstd, d["gamma"], None)
    dx, dg, db = mba.add_layernorm_backward(dy.cuda(), a.cuda(), mean.cuda(), rstd.cuda(),
                                            d["gamma"].cuda())
    torch.cuda.synchronize()
    ref = oracle.oracle_add_layernorm_bwd(dy, a, mean, rstd, d["gamma"], dtype)
    assert_bwd((dx.cpu(), dg.cpu(), db.cpu()), ref, case, dtype,
               f"{rows}x{H} {dtype} {mba.addln_last_path()}")
