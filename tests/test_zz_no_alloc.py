"""add_layernorm_bwd_noalloc: the backward for callers that cannot allocate
device memory (a plugin that is handed only tensor pointers, a loop where
cudaMalloc / cudaFree are ruled out because they block and synchronise).

It runs the same kernels as add_layernorm_bwd, with the library's built-in
scratch buffer as the workspace, so its outputs must equal that entry point's
bit for bit, and both must lie within the backward's bounds of the fp64
oracle.  Two calls in a row share the buffer (the second sees whatever the
first left there).  Also: the incoming-gradient path, and the path without
column sums (which needs no buffer at all).
This file is collected last, so a run that stops at the first failure has
run every other test first; it also passes alone in a fresh process."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import assert_bwd

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()


def _case(name, rows, seed, with_dres=False):
    w = synth.with_rows(synth.get(name), rows)
    d = synth.make_inputs(w, seed=seed)
    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype)
    td = synth.TORCH_DTYPES[w.dtype]
    host = {"dy": synth.make_grad(w, seed=seed), "a": torch.from_numpy(fwd["a"]).to(td),
            "mean": torch.from_numpy(fwd["mean"].astype(np.float32)),
            "rstd": torch.from_numpy(fwd["rstd"].astype(np.float32)), "gamma": d["gamma"],
            "dres": synth.make_grad(w, seed=seed + 101, scale=0.5) if with_dres else None}
    return w, host, {k: (v.cuda() if v is not None else None) for k, v in host.items()}


def _noalloc_via_c_abi(g, dx, dg, db):
    lib = mba.lib()
    rows, H = g["dy"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    return lib.add_layernorm_bwd_noalloc(p(g["dy"]), p(g["a"]), p(g["mean"]), p(g["rstd"]),
                                         p(g["gamma"]), p(g["dres"]), p(dx), p(dg), p(db), rows, H,
                                         mba.binding.DTYPE_CODE[g["dy"].dtype],
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _with_workspace(g, cols=True):
    dx = torch.empty_like(g["dy"])
    H = g["dy"].shape[1]
    dg = torch.empty(H, device="cuda") if cols else None
    db = torch.empty(H, device="cuda") if cols else None
    mba.add_layernorm_bwd(g["dy"], g["a"], g["mean"], g["rstd"], g["gamma"], dx, dg, db,
                          dres=g["dres"])
    return dx, dg, db


def _against_oracle(w, host, out, what):
    ref = oracle.oracle_add_layernorm_bwd(host["dy"], host["a"], host["mean"], host["rstd"],
                                          host["gamma"], w.dtype, dres=host["dres"])
    inputs = (host["dy"], host["a"], host["mean"].numpy(), host["rstd"].numpy(), host["gamma"],
              host["dres"])
    assert_bwd(tuple(t.cpu() for t in out), ref, inputs, w.dtype, what)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # a wide case first, then a narrower one: the second call runs over the
    # partials the first one left in the shared buffer
    for name, rows, seed in (("large_32768x8192_bf16", 600, 1), ("cancel_65536x1000_bf16", 900, 2)):
        w, host, g = _case(name, rows, seed)
        need = mba.add_layernorm_bwd_workspace_size(rows, w.H, mba.binding.DTYPE_CODE[g["dy"].dtype])
        assert 0 < need <= mba.binding.NOALLOC_SCRATCH_BYTES   # the shared buffer is used
        ref = _with_workspace(g)
        dx = torch.empty_like(g["dy"])
        dg = torch.empty(w.H, device="cuda")
        db = torch.empty(w.H, device="cuda")
        rc = _noalloc_via_c_abi(g, dx, dg, db)
        assert rc == 0, mba.addln_strerror(rc)
        torch.cuda.synchronize()
        assert mba.addln_get_device_error() == 0
        for u, v in zip((dx, dg, db), ref):
            assert torch.equal(u, v), f"{name}: no-alloc result differs from the workspace call"
        _against_oracle(w, host, (dx, dg, db), f"no-alloc {name}")


def test_noalloc_incoming_gradient_and_no_column_sums():
    w, host, g = _case("pages_2048x4096_fp16", 300, 3, with_dres=True)
    # with dres, dgamma and dbeta
    ref = _with_workspace(g)
    dx, dg, db = torch.empty_like(g["dy"]), torch.empty(w.H, device="cuda"), torch.empty(w.H, device="cuda")
    assert _noalloc_via_c_abi(g, dx, dg, db) == 0
    torch.cuda.synchronize()
    assert all(torch.equal(u, v) for u, v in zip((dx, dg, db), ref))
    _against_oracle(w, host, (dx, dg, db), "no-alloc with dres")
    # dX only: no workspace at all, the same dX
    dx2 = torch.empty_like(g["dy"])
    assert _noalloc_via_c_abi(g, dx2, None, None) == 0
    torch.cuda.synchronize()
    assert mba.addln_get_device_error() == 0
    assert torch.equal(dx2, ref[0])
