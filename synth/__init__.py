"""Seeded synthetic inputs and the workload table (no method arithmetic)."""
from .configs import WORKLOADS, PRIMARY, TAILS, SOFTMAX_NAMES, BGR_NAMES, Workload, get, with_rows, custom, DTYPE_CODES, DTYPE_BYTES
from .gen import make_inputs, make_affine, make_grad, TORCH_DTYPES
