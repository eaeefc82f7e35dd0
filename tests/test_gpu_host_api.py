"""add_layernorm_fwd_host (host buffers in and out, the traffic inside the
call): the same results as add_layernorm_fwd on device buffers, bit for bit,
in both of its modes (mapped: page-locked buffers read and written in place by
the kernel; pipelined: chunked copies, with a ragged last chunk), every output
combination, misaligned rows and in-place use; which mode each call takes; and
the oracle on one case."""
from __future__ import annotations

import pytest
import torch

import synth
from test_gpu_parity import check

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()
    yield


def device_reference(d, want_a, want_stats):
    x, r = d["x"].cuda(), d["r"].cuda()
    g, b = d["gamma"].cuda(), d["beta"].cuda()
    y = torch.empty_like(x)
    a = torch.empty_like(x) if want_a else None
    m = torch.empty(x.shape[0], device="cuda") if want_stats else None
    s = torch.empty(x.shape[0], device="cuda") if want_stats else None
    mba.add_layernorm_fwd(x, r, g, b, y, a, m, s, eps=d["eps"])
    torch.cuda.synchronize()
    return [t.cpu() if t is not None else None for t in (y, a, m, s)]


def host_call(d, want_a, want_stats, pin=True, in_place=False):
    prep = (lambda t: t.clone().pin_memory()) if pin else (lambda t: t.clone())
    hx, hr, hg, hb = prep(d["x"]), prep(d["r"]), prep(d["gamma"]), prep(d["beta"])
    hy = hx if in_place else prep(torch.empty_like(d["x"]))
    ha = prep(torch.empty_like(d["x"])) if want_a else None
    hm = prep(torch.empty(d["x"].shape[0])) if want_stats else None
    hs = prep(torch.empty(d["x"].shape[0])) if want_stats else None
    mba.add_layernorm_fwd_host(hx, hr, hg, hb, hy, ha, hm, hs, eps=d["eps"])
    torch.cuda.synchronize()
    return [hy, ha, hm, hs]


CASES = [
    ("pages_2048x4096_fp16", 2048),     # four 512-row chunks
    ("pages_2048x4096_fp16", 1000),     # 512 + 488
    ("cancel_65536x1000_bf16", 5000),   # 2097 + 2097 + 806
    ("large_32768x8192_bf16", 300),     # 256 + 44
    ("tiny_64x768_fp32", 64),           # one chunk
    ("tail_4096x1001_bf16", 777),       # misaligned rows: element kernels on device
]


def device_reaches_host_memory():
    """cudaDevAttrPageableMemoryAccess of the current device, through the CUDA
    runtime this process already loaded (None when it cannot be asked)."""
    import ctypes
    try:
        paths = sorted({ln.split()[-1] for ln in open("/proc/self/maps") if "libcudart.so" in ln})
        rt = ctypes.CDLL(paths[0])
    except (OSError, IndexError):
        return None
    dev, v = ctypes.c_int(0), ctypes.c_int(0)
    if rt.cudaGetDevice(ctypes.byref(dev)) != 0:
        return None
    if rt.cudaDeviceGetAttribute(ctypes.byref(v), 88, dev) != 0:  # PageableMemoryAccess
        return None
    return v.value != 0


@pytest.mark.parametrize("name,rows", CASES)
@pytest.mark.parametrize("want_a,want_stats", [(False, False), (True, True)])
@pytest.mark.parametrize("pin", [True, False])
def test_matches_device_entry_point_bitwise(name, rows, want_a, want_stats, pin):
    w = synth.with_rows(synth.get(name), rows)
    d = synth.make_inputs(w, seed=21)
    ref = device_reference(d, want_a, want_stats)
    got = host_call(d, want_a, want_stats, pin=pin)
    for u, v in zip(got, ref):
        assert (u is None) == (v is None)
        if u is not None:
            assert torch.equal(u, v)


def test_pageable_memory_and_in_place():
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 1500)
    d = synth.make_inputs(w, seed=22)
    ref = device_reference(d, False, False)
    assert torch.equal(host_call(d, False, False, pin=False)[0], ref[0])
    assert torch.equal(host_call(d, False, False, in_place=True)[0], ref[0])


def test_mode_reports_the_path_taken():
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 600)
    d = synth.make_inputs(w, seed=25)
    ref = device_reference(d, True, True)
    host_call(d, True, True, pin=False)
    assert mba.add_layernorm_fwd_host_last_mode() == mba.binding.HOST_PIPELINED
    got = host_call(d, True, True, pin=True)
    reach = device_reaches_host_memory()
    mode = mba.add_layernorm_fwd_host_last_mode()
    if reach is not None:
        assert mode == (mba.binding.HOST_MAPPED if reach else mba.binding.HOST_PIPELINED)
    if mode == mba.binding.HOST_MAPPED:
        # rows in host memory are read by 16-byte loads, never by bulk copies
        assert mba.addln_last_path().startswith("cta_vec"), mba.addln_last_path()
    assert all(torch.equal(u, v) for u, v in zip(got, ref))
    # page-locked rows that are not 16-byte aligned never go mapped
    n = w.rows * w.H
    bx = torch.empty(n + 8, dtype=d["x"].dtype).pin_memory()
    by = torch.empty(n + 8, dtype=d["x"].dtype).pin_memory()
    hx = bx[1:1 + n].view(w.rows, w.H)
    hx.copy_(d["x"])
    hy = by[1:1 + n].view(w.rows, w.H)
    mba.add_layernorm_fwd_host(hx, d["r"].pin_memory(), d["gamma"], d["beta"], hy, eps=d["eps"])
    torch.cuda.synchronize()
    assert mba.add_layernorm_fwd_host_last_mode() == mba.binding.HOST_PIPELINED
    assert torch.equal(hy, ref[0])


def test_mapped_mode_captures_into_a_graph():
    # mapped mode queues kernels only (gamma and beta mapped too), so a call
    # can be captured and replayed; replays follow the inputs' current values
    if device_reaches_host_memory() is not True:
        pytest.skip("the device cannot reach host memory: no mapped mode")
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 1000)
    d = synth.make_inputs(w, seed=26)
    d2 = synth.make_inputs(w, seed=27)
    hx, hr, hg, hb = [d[k].clone().pin_memory() for k in ("x", "r", "gamma", "beta")]
    hy, ha = torch.empty_like(hx).pin_memory(), torch.empty_like(hx).pin_memory()
    hm, hs = torch.empty(w.rows).pin_memory(), torch.empty(w.rows).pin_memory()
    ws = torch.empty(mba.add_layernorm_fwd_host_workspace_size(w.rows, w.H, mba.FP16, True, True),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    call = lambda: mba.add_layernorm_fwd_host(hx, hr, hg, hb, hy, ha, hm, hs, eps=d["eps"],
                                              workspace=ws, stream=s)
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    assert mba.add_layernorm_fwd_host_last_mode() == mba.binding.HOST_MAPPED
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for t in (hy, ha, hm, hs):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(u, v) for u, v in zip((hy, ha, hm, hs), device_reference(d, True, True)))
    for k, t in (("x", hx), ("r", hr)):
        t.copy_(d2[k])
    g.replay()
    torch.cuda.synchronize()
    d2["gamma"], d2["beta"] = d["gamma"], d["beta"]
    assert all(torch.equal(u, v) for u, v in zip((hy, ha, hm, hs), device_reference(d2, True, True)))


def test_mean_without_rstd():
    w = synth.with_rows(synth.get("cancel_65536x1000_bf16"), 3000)
    d = synth.make_inputs(w, seed=23)
    ref = device_reference(d, False, True)
    hx, hr = d["x"].pin_memory(), d["r"].pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hm = torch.empty(w.rows).pin_memory()
    mba.add_layernorm_fwd_host(hx, hr, d["gamma"], d["beta"], hy, mean=hm, eps=d["eps"])
    torch.cuda.synchronize()
    assert torch.equal(hy, ref[0]) and torch.equal(hm, ref[2])


def test_against_the_oracle():
    w = synth.with_rows(synth.get("cancel_65536x1000_bf16"), 3000)
    d = synth.make_inputs(w, seed=24)
    hy, ha, hm, hs = host_call(d, True, True)
    out = {"y": hy, "a": ha, "mean": hm, "rstd": hs, "path": "host"}
    check(w, d, out, "host entry point")


def test_two_host_threads_at_once():
    # the copy streams are shared per device: calls from two threads queue
    # behind one another there, each on its own stream, with correct results
    import threading
    cases = []
    for k, (name, rows) in enumerate([("pages_2048x4096_fp16", 1700), ("cancel_65536x1000_bf16", 6000)]):
        w = synth.with_rows(synth.get(name), rows)
        d = synth.make_inputs(w, seed=30 + k)
        cases.append((d, device_reference(d, True, True)))
    results = [None, None]
    errors = []

    def worker(i):
        try:
            d, _ = cases[i]
            s = torch.cuda.Stream()
            outs = []
            for _ in range(3):
                with torch.cuda.stream(s):
                    hx, hr = d["x"].pin_memory(), d["r"].pin_memory()
                    hy = torch.empty_like(hx).pin_memory()
                    ha = torch.empty_like(hx).pin_memory()
                    hm = torch.empty(hx.shape[0]).pin_memory()
                    hs = torch.empty(hx.shape[0]).pin_memory()
                    mba.add_layernorm_fwd_host(hx, hr, d["gamma"], d["beta"], hy, ha, hm, hs,
                                               eps=d["eps"], stream=s)
                    s.synchronize()
                    outs.append((hy, ha, hm, hs))
            results[i] = outs
        except Exception as e:   # reported below
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for i in range(2):
        ref = cases[i][1]
        for outs in results[i]:
            for u, v in zip(outs, ref):
                assert torch.equal(u, v)


def _host_draw(n, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        dtype = ["fp32", "fp16", "bf16"][rng.integers(3)]
        H = int(rng.choice([7, 64, 768, 1000, 1001, 2048, 4096, 5000, 8192]))
        rows = int(rng.integers(1, 3000))
        flags = int(rng.integers(4))
        out.append((rows, H, dtype, bool(flags & 1), bool(flags & 2)))
    return out


@pytest.mark.parametrize("rows,H,dtype,want_a,want_stats", _host_draw(12, 2030))
def test_random_shapes_match_device_entry_point(rows, H, dtype, want_a, want_stats):
    w = synth.custom(rows, H, dtype, x_dist=(1.0, 2.0))
    d = synth.make_inputs(w, seed=rows + H)
    ref = device_reference(d, want_a, want_stats)
    got = host_call(d, want_a, want_stats)
    for u, v in zip(got, ref):
        assert (u is None) == (v is None)
        if u is not None:
            assert torch.equal(u, v)
