"""GPU parity of the Add+LayerNorm backward (add_layernorm_bwd through the C
ABI) against the fp64 oracle.  The forward quantities the backward consumes
(A, mean, rstd) come from the oracle's forward on the CPU, so both sides get
the same inputs and none of them comes from the CUDA path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import assert_bwd

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")
TD = synth.TORCH_DTYPES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()
    mba.addln_set_force_path(0)
    yield
    mba.addln_set_force_path(0)


def make_case(w, seed=0, with_dres=False):
    d = synth.make_inputs(w, seed=seed)
    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype)
    a = torch.from_numpy(fwd["a"]).to(TD[w.dtype])                # exact: already in the dtype
    mean = torch.from_numpy(fwd["mean"].astype(np.float32))
    rstd = torch.from_numpy(fwd["rstd"].astype(np.float32))
    dy = synth.make_grad(w, seed=seed)
    dres = synth.make_grad(w, seed=seed + 101, scale=0.5) if with_dres else None
    return dy, a, mean, rstd, d["gamma"], dres


def run(case, path=0):
    dy, a, mean, rstd, gamma, dres = [t.cuda() if t is not None else None for t in case]
    prev = mba.addln_set_force_path(path)
    try:
        dx, dg, db = mba.add_layernorm_backward(dy, a, mean, rstd, gamma, dres=dres)
        name = mba.addln_last_path()
        torch.cuda.synchronize()
    finally:
        mba.addln_set_force_path(prev)
    assert mba.addln_get_device_error() == 0
    return (dx.cpu(), dg.cpu(), db.cpu()), name


def check(case, dtype, out, what):
    dy, a, mean, rstd, gamma, dres = case
    ref = oracle.oracle_add_layernorm_bwd(dy, a, mean, rstd, gamma, dtype, dres=dres)
    assert_bwd(out, ref, case, dtype, what)


@pytest.mark.parametrize("name", synth.PRIMARY + synth.TAILS)
@pytest.mark.parametrize("path", [0, 4])
def test_small(name, path):
    w = synth.with_rows(synth.get(name), 203)
    case = make_case(w, seed=1)
    out, p = run(case, path)
    check(case, w.dtype, out, f"{name} {p}")


@pytest.mark.parametrize("name", ["tiny_64x768_fp32", "pages_2048x4096_fp16",
                                  "cancel_65536x1000_bf16"])
def test_incoming_a_gradient(name):
    w = synth.with_rows(synth.get(name), 77)
    case = make_case(w, seed=2, with_dres=True)
    out, p = run(case)
    check(case, w.dtype, out, f"{name} dres {p}")


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 8, 33, 1000, 1024, 1025, 1032, 2056, 4096, 4104, 8192, 12288])
def test_shapes(dtype, H):
    w = synth.custom(37, H, dtype, x_dist=(2.0, 1.5), want_resid=True, want_stats=True)
    case = make_case(w, seed=H)
    out, p = run(case)
    check(case, dtype, out, f"37x{H} {dtype} {p}")


# rows enough that every CTA (warp, for H <= 1024) walks several rows, so the
# ring wraps (slot back to 0, mbarrier phase flipped) at every depth
RING_ROWS = {"tiny_64x768_fp32": 64, "cancel_65536x1000_bf16": 8000,
             "pages_2048x4096_fp16": 2048, "large_32768x8192_bf16": 912}


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
@pytest.mark.parametrize("name", sorted(RING_ROWS))
def test_ring_depths(name, stages):
    # the staging ring's depth changes only the launch, never the grid (so the
    # workspace size is the same for every depth)
    w = synth.with_rows(synth.get(name), RING_ROWS[name])
    case = make_case(w, seed=5)
    prev = mba.addln_set_cta_shape(0, stages)
    try:
        out, p = run(case)
    finally:
        mba.addln_set_cta_shape(prev, 0)
    check(case, w.dtype, out, f"{name} ring {stages} {p}")


def test_deterministic_and_in_place():
    w = synth.with_rows(synth.get("large_32768x8192_bf16"), 300)
    case = make_case(w, seed=3)
    o1, _ = run(case)
    o2, _ = run(case)
    assert all(torch.equal(u, v) for u, v in zip(o1, o2))
    dy, a, mean, rstd, gamma, _ = [t.cuda() if t is not None else None for t in case]
    dx = dy.clone()
    dg = torch.empty(w.H, device="cuda")
    db = torch.empty(w.H, device="cuda")
    mba.add_layernorm_bwd(dx, a, mean, rstd, gamma, dx, dg, db)     # dx written over dY
    torch.cuda.synchronize()
    assert torch.equal(dx.cpu(), o1[0]) and torch.equal(dg.cpu(), o1[1])


def test_workspace_errors_and_zero_rows():
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 64)
    dy, a, mean, rstd, gamma, _ = [t.cuda() if t is not None else None for t in make_case(w)]
    dx = torch.empty_like(dy)
    dg = torch.empty(w.H, device="cuda")
    db = torch.empty(w.H, device="cuda")
    need = mba.add_layernorm_bwd_workspace_size(64, w.H, mba.FP16)
    assert need > 0
    # the size covers every plan the pointers may pick (vector or element
    # path); one partial of [2][H] floats is less than any plan needs
    small = torch.empty(8 * w.H, dtype=torch.uint8, device="cuda")
    with pytest.raises(mba.AddLNError) as e:
        mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx, dg, db, workspace=small)
    assert e.value.code == mba.binding.ERR_WORKSPACE
    enough = torch.zeros(need, dtype=torch.uint8, device="cuda")
    mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx, dg, db, workspace=enough)
    # no dgamma / dbeta: no workspace needed
    mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx)
    dg.fill_(7.0)
    db.fill_(7.0)
    e0 = torch.empty(0, w.H, dtype=torch.float16, device="cuda")
    z = torch.empty(0, device="cuda")
    mba.add_layernorm_bwd(e0, e0, z, z, gamma, e0, dg, db)
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["pages_2048x4096_fp16", "cancel_65536x1000_bf16"])
def test_full_size(name):
    w = synth.get(name)
    case = make_case(w, seed=0)
    out, p = run(case)
    check(case, w.dtype, out, f"{name} full size {p}")


def test_wait_timeout_sets_device_error_and_recovers():
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 32)
    case = make_case(w, seed=4)
    dy, a, mean, rstd, gamma, _ = [t.cuda() if t is not None else None for t in case]
    dx = torch.empty_like(dy)
    prev = mba.addln_set_wait_limit_ns(0)
    try:
        mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx)
        assert mba.addln_get_device_error() == mba.binding.ERR_DEVICE_TIMEOUT
    finally:
        mba.addln_set_wait_limit_ns(prev)
    assert mba.addln_get_device_error() == 0
    out, p = run(case)
    check(case, w.dtype, out, "after timeout")


@pytest.mark.parametrize("rows,H,dtype,min_g,max_g", [
    (16384, 64, "fp32", 1025, None),   # more than 1024 partials: two rounds of loads a thread
    (4096, 768, "bf16", 513, 1024),    # two column quads a block, one round
    (2048, 4096, "fp16", 257, 512),    # four quads a block
    (512, 8192, "bf16", 1, 256),       # eight quads a block
])
def test_column_sum_widths(rows, H, dtype, min_g, max_g):
    # the column-sum kernel picks its block width from the number of
    # partials G (= workspace bytes / 8H); each case sits in one band of G
    w = synth.custom(rows, H, dtype)
    g_count = mba.add_layernorm_bwd_workspace_size(rows, H, mba.binding.DTYPE_CODE[TD[dtype]]) // (8 * H)
    assert g_count >= min_g and (max_g is None or g_count <= max_g), g_count
    case = make_case(w, seed=rows + H)
    out, p = run(case)
    check(case, w.dtype, out, f"{rows}x{H} {dtype} G={g_count} {p}")


def test_workspace_reused_across_calls_and_shapes():
    # one workspace, large enough for the largest shape, serves calls of
    # several shapes in a row, each result matching the oracle
    shapes = [("pages_2048x4096_fp16", 700), ("bert_base_4096x768_fp16", 900),
              ("large_32768x8192_bf16", 200), ("pages_2048x4096_fp16", 33)]
    need = max(mba.add_layernorm_bwd_workspace_size(r, synth.get(n).H,
                                                    mba.binding.DTYPE_CODE[TD[synth.get(n).dtype]])
               for n, r in shapes)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for name, rows in shapes * 2:
        w = synth.with_rows(synth.get(name), rows)
        case = make_case(w, seed=rows)
        dy, a, mean, rstd, gamma, _ = [t.cuda() if t is not None else None for t in case]
        dx = torch.empty_like(dy)
        dg = torch.empty(w.H, device="cuda")
        db = torch.empty(w.H, device="cuda")
        mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx, dg, db, workspace=ws)
        torch.cuda.synchronize()
        assert mba.addln_get_device_error() == 0
        check(case, w.dtype, (dx.cpu(), dg.cpu(), db.cpu()), f"{name} {rows} shared workspace")
