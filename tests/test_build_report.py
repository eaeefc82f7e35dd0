"""Register spills, from the assembler's own report (CPU only: nvcc
cross-compiles for sm_103a without a GPU).

Every kernel instantiation in the library is compiled with ptxas's verbose
report and must show a zero-byte stack frame and no spill stores or loads:
the register caps the kernels carry (__maxnreg__, __launch_bounds__) are set
for occupancy, and a spill would put local-memory traffic on the path these
kernels exist to keep at the HBM roofline."""
from __future__ import annotations

import pytest


@pytest.fixture(scope="module")
def report():
    from memory_bound_add_gb300.build import ptxas_report
    return ptxas_report()


def test_every_kernel_compiles_without_spills(report):
    kernels = {k: v for k, v in report.items() if "registers" in v}
    assert len(kernels) > 100                      # every template instantiation is there
    bad = {k: v for k, v in report.items()
           if v.get("spill_stores", 0) or v.get("spill_loads", 0) or v.get("stack", 0)}
    assert not bad, f"{len(bad)} functions spill or use a stack frame: {sorted(bad)[:5]}"


def test_row_kernels_stay_under_their_register_caps(report):
    # the register-resident CTA kernels are capped at 128 (four CTAs to an SM)
    # or 136; the warp-per-row backward at 168; nothing needs more than 168
    for name, v in report.items():
        if "registers" in v:
            assert v["registers"] <= 168, (name, v["registers"])
