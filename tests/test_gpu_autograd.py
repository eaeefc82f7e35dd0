"""GPU parity of the autograd wrapper (AddLayerNormFunction): the forward
output and the gradients of x, r, gamma and beta after y.backward(dY),
against the fp64 oracle's forward and backward on the same seeded inputs.
The oracle's backward takes the oracle's own A, mean and rstd, so no oracle
input comes from the CUDA path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import assert_bwd, assert_y

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


@pytest.mark.parametrize("name,rows", [("tiny_64x768_fp32", 64), ("bert_base_4096x768_fp16", 300),
                                       ("pages_2048x4096_fp16", 96), ("cancel_65536x1000_bf16", 200),
                                       ("tail_4096x999_bf16", 50)])
def test_gradients_match_the_oracle(name, rows):
    w = synth.with_rows(synth.get(name), rows)
    d = synth.make_inputs(w, seed=31 + rows)
    dy = synth.make_grad(w, seed=32 + rows)
    x = d["x"].cuda().requires_grad_(True)
    r = d["r"].cuda().requires_grad_(True)
    g = d["gamma"].cuda().requires_grad_(True)
    b = d["beta"].cuda().requires_grad_(True)
    y = mba.add_layernorm_train(x, r, g, b, eps=d["eps"])
    y.backward(dy.cuda())
    torch.cuda.synchronize()
    assert mba.addln_get_device_error() == 0

    fwd = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype)
    assert_y(y.detach().cpu(), fwd["y"], w.dtype, f"{name} autograd forward")
    a = torch.from_numpy(fwd["a"]).to(TD[w.dtype])
    mean = torch.from_numpy(fwd["mean"].astype(np.float32))
    rstd = torch.from_numpy(fwd["rstd"].astype(np.float32))
    case = (dy, a, mean, rstd, d["gamma"], None)
    ref = oracle.oracle_add_layernorm_bwd(dy, a, mean, rstd, d["gamma"], w.dtype)
    out = (x.grad.cpu(), g.grad.cpu(), b.grad.cpu())
    assert_bwd(out, ref, case, w.dtype, f"{name} autograd backward")
    assert torch.equal(x.grad, r.grad)


def test_only_some_inputs_need_gradients():
    # gamma and beta frozen: the backward skips the column sums; x frozen:
    # only r gets a gradient
    w = synth.with_rows(synth.get("bert_base_4096x768_fp16"), 40)
    d = synth.make_inputs(w, seed=33)
    dy = synth.make_grad(w, seed=34).cuda()
    x = d["x"].cuda().requires_grad_(True)
    r = d["r"].cuda()
    g, b = d["gamma"].cuda(), d["beta"].cuda()
    mba.add_layernorm_train(x, r, g, b, eps=d["eps"]).backward(dy)
    x2 = d["x"].cuda()
    r2 = d["r"].cuda().requires_grad_(True)
    g2 = d["gamma"].cuda().requires_grad_(True)
    mba.add_layernorm_train(x2, r2, g2, b, eps=d["eps"]).backward(dy)
    torch.cuda.synchronize()
    assert x.grad is not None and r2.grad is not None and g2.grad is not None
    assert torch.equal(x.grad, r2.grad)


def test_module_trains():
    # the module's parameters get gradients and an optimizer step moves them;
    # its output equals the function's with the same parameters
    w = synth.with_rows(synth.get("bert_base_4096x768_fp16"), 64)
    d = synth.make_inputs(w, seed=35)
    m = mba.FusedAddLayerNorm(w.H, eps=d["eps"], device="cuda")
    with torch.no_grad():
        m.weight.copy_(d["gamma"].cuda())
        m.bias.copy_(d["beta"].cuda())
    x, r = d["x"].cuda(), d["r"].cuda()
    y = m(x, r)
    assert torch.equal(y, mba.add_layernorm(x, r, m.weight.detach(), m.bias.detach(), eps=d["eps"])[0])
    opt = torch.optim.SGD(m.parameters(), lr=0.1)
    before = m.weight.detach().clone()
    y.float().square().mean().backward()
    opt.step()
    torch.cuda.synchronize()
    assert m.weight.grad is not None and m.bias.grad is not None
    assert not torch.equal(before, m.weight.detach())
