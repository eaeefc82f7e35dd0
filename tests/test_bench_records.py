"""bench.py reports the ncu traffic figure of its dominant kernel only while
that figure was taken on the current forward kernel sources: the record's
source hash and kernel name must both match, else the line carries null."""
from __future__ import annotations

import os
import shutil

import pytest

import bench


def _write(root, kernel, digest, n=123456):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "traffic_wl.txt"), "w") as f:
        f.write("# comment: lines starting with # are skipped\n")
        f.write(f"kernel: {kernel}\nkernel_source_hash: {digest}\n")
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
    assert bench.profiled_traffic("wl", "cta_tma_t128_nv4") == 123456
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
