"""fp64 CPU oracle for the fused residual-Add + LayerNorm row operation.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never imports, loads or calls it, and it
shares no code with that path.

The arithmetic lives in ``addln_oracle.c`` (plain C, fp64, two-pass); this
module only marshals host tensors to it.  Every pin that ties it to the
source pages and to mathematics independent of itself is in
``tests/test_oracle_pins.py``; none of its functions is "parity unpinned".
"""
from .oracle import (
    oracle_decode,
    oracle_round,
    oracle_add,
    oracle_layernorm,
    oracle_add_layernorm,
    oracle_softmax,
    oracle_bias_gelu_residual,
    oracle_add_layernorm_bwd,
    load,
)
