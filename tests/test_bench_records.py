"""bench.py reports the ncu traffic figure of its dominant kernel only while
that figure was taken on the current forward kernel sources, in steady state
(consecutive launches, so each pays the write-back of the outputs earlier
launches left dirty in L2): the record's source hash, kernel name and capture
kind must all match, else the line carries null.  Also the harness's choice
of buffer sets."""
from __future__ import annotations

import os
import shutil

import pytest

import bench


def _write(root, kernel, digest, n=123456, capture="steady-state"):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "traffic_wl.txt"), "w") as f:
        f.write("# comment: lines starting with # are skipped\n")
        f.write(f"kernel: {kernel}\nkernel_source_hash: {digest}\ncapture: {capture}\n")
        f.write("launches_averaged: 6\n")
        f.write(f"dram_bytes_read: {n - 6}\ndram_bytes_write: 6\ndram_bytes_per_launch: {n}\n")


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the forward kernel sources under a temporary root."""
    src = os.path.join(bench.ROOT, "memory_bound_add_gb300", "csrc")
    dst = tmp_path / "memory_bound_add_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.FORWARD_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_reported_only_for_the_current_sources(tree):
    digest = bench.kernel_source_hash()
    _write(str(tree), "cta_tma_t128_nv4", digest)
    assert bench.profiled_traffic("wl", "cta_tma_t128_nv4")["bytes"] == 123456
    # a single cold launch under-counts the writes: not reported
    _write(str(tree), "cta_tma_t128_nv4", digest, capture="cold-single-launch")
    assert bench.profiled_traffic("wl", "cta_tma_t128_nv4") is None
    _write(str(tree), "cta_tma_t128_nv4", digest)
    # another kernel path: not this figure
    assert bench.profiled_traffic("wl", "warp_vec_nv3") is None
    # a forward source changes: the record is stale
    p = tree / "memory_bound_add_gb300" / "csrc" / bench.FORWARD_SOURCES[0]
    p.write_text(p.read_text() + "\n// changed\n")
    assert bench.kernel_source_hash() != digest
    assert bench.profiled_traffic("wl", "cta_tma_t128_nv4") is None
    # no record at all
    assert bench.profiled_traffic("other", "cta_tma_t128_nv4") is None


def test_committed_record_names_the_bench_default_kernel():
    # the committed record is for the default workload's dominant kernel;
    # whether its hash still matches is reported, not asserted (a kernel
    # change makes it stale until the next capture, and the bench then
    # prints null)
    path = os.path.join(bench.ROOT, "profiles", "traffic_pages_2048x4096_fp16.txt")
    kv = dict(line.split(":", 1) for line in open(path) if ":" in line and not line.startswith("#"))
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    assert kv["kernel"] == "cta_tma_t128_nv4"
    assert int(kv["dram_bytes_per_launch"]) == int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
    print("committed traffic record matches current sources:",
          kv["kernel_source_hash"] == bench.kernel_source_hash())


def test_buffer_sets_continue_the_rotation_across_replays():
    # the set count divides the steps a replay launches when it can, so
    # replay r + 1 picks up the rotation where replay r left it
    assert bench.pick_sets(20, 9, 50, 10 ** 9) == (10, False)
    assert bench.pick_sets(20, 2, 2 * 10 ** 9, 10 ** 11) == (2, False)
    assert bench.pick_sets(23, 9, 50, 10 ** 9) == (23, False)
    # no divisor fits the memory budget: the minimum count and an L2 flush
    assert bench.pick_sets(23, 2, 2 * 10 ** 9, 10 ** 10) == (2, True)
    for K, need in ((20, 9), (40, 3), (7, 7)):
        n, flush = bench.pick_sets(K, need, 1, 10 ** 9)
        assert not flush and K % n == 0 and n >= need
