"""add_layernorm_bwd_noalloc: the backward for callers that cannot allocate
device memory (a plugin that is handed only tensor pointers, a loop where
cudaMalloc / cudaFree are ruled out because they block and synchronise).
It must give what add_layernorm_bwd gives with a workspace of its own, on two
calls in a row that share the library's built-in scratch buffer (the second
call sees whatever the first left there).  This file is collected last, so a
run that stops at the first failure has run every other test first; it also
passes alone in a fresh process."""
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


def _case(name, rows, seed):
    w = synth.with_rows(synth.get(name), rows)
    d = synth.make_inputs(w, seed=seed)
    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype)
    a = torch.from_numpy(fwd["a"]).to(synth.TORCH_DTYPES[w.dtype]).cuda()
    mean = torch.from_numpy(fwd["mean"].astype(np.float32)).cuda()
    rstd = torch.from_numpy(fwd["rstd"].astype(np.float32)).cuda()
    dy = synth.make_grad(w, seed=seed).cuda()
    return w, dy, a, mean, rstd, d["gamma"].cuda()


def _noalloc_via_c_abi(dy, a, mean, rstd, gamma, dx, dg, db):
    lib = mba.lib()
    rows, H = dy.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.add_layernorm_bwd_noalloc(p(dy), p(a), p(mean), p(rstd), p(gamma), None, p(dx),
                                       p(dg), p(db), rows, H, mba.binding.DTYPE_CODE[dy.dtype],
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, mba.addln_strerror(rc)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # a wide case first, then a narrower one: the second call runs over the
    # partials the first one left in the shared buffer
    for name, rows, seed in (("large_32768x8192_bf16", 600, 1), ("cancel_65536x1000_bf16", 900, 2)):
        w, dy, a, mean, rstd, gamma = _case(name, rows, seed)
        need = mba.add_layernorm_bwd_workspace_size(rows, w.H, mba.binding.DTYPE_CODE[dy.dtype])
        assert 0 < need <= mba.binding.NOALLOC_SCRATCH_BYTES   # the shared buffer is used
        dx_ref = torch.empty_like(dy)
        dg_ref = torch.empty(w.H, device="cuda")
        db_ref = torch.empty(w.H, device="cuda")
        mba.add_layernorm_bwd(dy, a, mean, rstd, gamma, dx_ref, dg_ref, db_ref)
        dx = torch.empty_like(dy)
        dg = torch.empty(w.H, device="cuda")
        db = torch.empty(w.H, device="cuda")
        _noalloc_via_c_abi(dy, a, mean, rstd, gamma, dx, dg, db)
        torch.cuda.synchronize()
        ref = {"dx": dx_ref.cpu().double().numpy(), "dgamma": dg_ref.cpu().double().numpy(),
               "dbeta": db_ref.cpu().double().numpy()}
        inputs = (dy.cpu(), a.cpu(), mean.cpu().numpy(), rstd.cpu().numpy(), gamma.cpu(), None)
        assert_bwd((dx.cpu(), dg.cpu(), db.cpu()), ref, inputs, w.dtype, f"no-alloc {name}")
