"""Workload table for the fused residual-Add + LayerNorm row operation.

Each entry is a synthetic stand-in for a workload the source pages discuss.
Sizes, dtypes, value distributions and which outputs are written are fixed
here once; the generator (``synth.gen``), the oracle tests, the GPU parity
tests and ``bench.py`` all select a workload by name.

Distribution notation: ``(loc, scale)`` is a normal with mean ``loc`` and
standard deviation ``scale`` (numpy ``normal(loc, scale)`` convention).

Sources (page title, section):
  * "算子融合的收益量化" (fusion gains quantified), section 1: the
    [B,S,H] = [1,2048,4096] fp16 Residual-Add + LayerNorm subgraph.
  * "算子融合与Kernel合并" (operator fusion and kernel merging), section 4.2:
    the LayerNorm definition with eps = 1e-5 as default.
  * "CUDA算子融合优化" (CUDA operator fusion), section 4.1: BERT-base
    inference (hidden size 768) as the fused model.
"""
from __future__ import annotations

from dataclasses import dataclass, field

# dtype codes shared by the C-ABI and the oracle's ABI (an interface, so both
# sides spell it the same way; neither side's arithmetic is shared).
DTYPE_CODES = {"fp32": 0, "fp16": 1, "bf16": 2}
DTYPE_BYTES = {"fp32": 4, "fp16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    H: int
    dtype: str
    eps: float
    x_dist: tuple = (0.0, 1.0)
    r_dist: tuple = (0.0, 1.0)
    want_resid: bool = False      # write A = X + R
    want_stats: bool = False      # write mean[rows] and rstd[rows]
    const_row_frac: float = 0.0   # fraction of rows with X = c (one draw), R = 0
    outlier_frac: float = 0.0     # fraction of X elements replaced by +-outlier_mag
    outlier_mag: float = 50.0
    note: str = ""
    shape_bsh: tuple = field(default=None)
    op: str = "add_layernorm"     # "softmax": row softmax of X (R, gamma, beta unused)
    #                                 "bias_gelu_residual": GELU(X + bias) + R (bias = beta draw)

    @property
    def n_const_rows(self) -> int:
        return int(round(self.const_row_frac * self.rows))

    @property
    def n_outliers(self) -> int:
        return int(round(self.outlier_frac * self.rows * self.H))

    @property
    def elem_bytes(self) -> int:
        return DTYPE_BYTES[self.dtype]

    def algorithmic_bytes(self) -> int:
        """Minimal HBM bytes of one fused call over the whole batch.

        Softmax: read X once, write Y once.

        Read X and R once, write Y once (plus A when requested), 8 bytes of
        fp32 statistics per row when requested, and gamma/beta (fp32 [H]) once.
        This is the fused-kernel accounting of "算子融合的收益量化" section 1
        extended by the optional outputs and the affine parameters.
        """
        s = self.elem_bytes
        if self.op == "softmax":
            return 2 * self.rows * self.H * s
        if self.op == "bias_gelu_residual":
            return 3 * self.rows * self.H * s + 4 * self.H
        per_row = 2 * self.H * s + self.H * s * (1 + int(self.want_resid)) + 8 * int(self.want_stats)
        return self.rows * per_row + 8 * self.H

    def unfused_algorithmic_bytes(self) -> int:
        """Minimal bytes of the two-kernel chain: add (2 reads, 1 write of A),
        then LayerNorm (1 read of A, 1 write of Y), per "算子融合的收益量化"
        section 1.  A is part of the chain, so it is counted once written and
        once read whether or not the caller wants it."""
        s = self.elem_bytes
        add = 3 * self.rows * self.H * s
        ln = 2 * self.rows * self.H * s + 8 * self.rows * int(self.want_stats) + 8 * self.H
        return add + ln


_G = "gamma ~ 1+0.1*N(0,1), beta ~ 0.1*N(0,1) (fp32)"

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_64x768_fp32", 64, 768, "fp32", 1e-5,
                 want_resid=True, want_stats=True,
                 note="tiny correctness case; Y, A, mean, rstd written; " + _G),
        Workload("bert_base_4096x768_fp16", 4096, 768, "fp16", 1e-12,
                 note="batch 32 x seq 128, BERT-base hidden size; Y only; " + _G,
                 shape_bsh=(32, 128, 768)),
        Workload("pages_2048x4096_fp16", 2048, 4096, "fp16", 1e-5, r_dist=(0.0, 0.5),
                 note="the pages' [1,2048,4096] fp16 Add+LayerNorm subgraph; Y only; " + _G,
                 shape_bsh=(1, 2048, 4096)),
        Workload("cancel_65536x1000_bf16", 65536, 1000, "bf16", 1e-5, x_dist=(100.0, 1.0),
                 want_resid=True, want_stats=True, const_row_frac=0.01,
                 note="row mean >> std, 1% constant rows, H not a multiple of 8*32; " + _G),
        Workload("large_32768x8192_bf16", 32768, 8192, "bf16", 1e-5, r_dist=(0.0, 0.5),
                 want_resid=True, outlier_frac=0.001,
                 note="[8,4096,8192], 0.1% of X at +-50; Y and A written; " + _G,
                 shape_bsh=(8, 4096, 8192)),
        # Extra tails: H that is not a whole number of 16-byte vectors, so rows
        # start at misaligned addresses; distributions of the cancellation case.
        Workload("tail_4096x999_bf16", 4096, 999, "bf16", 1e-5, x_dist=(100.0, 1.0),
                 want_resid=True, want_stats=True, note="odd H, misaligned rows"),
        Workload("tail_4096x1001_bf16", 4096, 1001, "bf16", 1e-5, x_dist=(100.0, 1.0),
                 want_resid=True, want_stats=True, note="odd H, misaligned rows"),
        Workload("tail_4096x1002_fp32", 4096, 1002, "fp32", 1e-5, x_dist=(100.0, 1.0),
                 want_resid=True, want_stats=True, note="H not a multiple of 4 fp32"),
    ]
}

# Row softmax ("算子融合与Kernel合并" 4.3): the same reduce-elementwise pattern
# on one input.  The pages give no sizes; these stand in for attention scores
# (32 heads x 1024 queries over 1024 keys) and language-model logits over a
# 32000-entry vocabulary, plus a small ragged fp32 case.
SOFTMAX = [
    Workload("softmax_tiny_64x1000_fp32", 64, 1000, "fp32", 0.0, x_dist=(0.0, 3.0), op="softmax",
             note="small fp32 case, H not a multiple of 32 vectors"),
    Workload("softmax_attention_32768x1024_fp16", 32768, 1024, "fp16", 0.0, x_dist=(0.0, 2.0),
             op="softmax", note="attention scores, 32 heads x 1024 queries x 1024 keys"),
    Workload("softmax_vocab_4096x32000_bf16", 4096, 32000, "bf16", 0.0, x_dist=(0.0, 4.0),
             op="softmax", note="logits of 4096 tokens over a 32000-entry vocabulary"),
]
WORKLOADS.update({w.name: w for w in SOFTMAX})
SOFTMAX_NAMES = [w.name for w in SOFTMAX]

# Bias + GELU + residual ("算子融合的收益量化", the three-kernel diagram): the
# diagram's 8 MB tensors ([1, 1024, 4096] fp16), and a large bf16 case.  The
# bias is the beta draw (fp32 [H]); X ~ N(0, 1), R ~ N(0, 0.5).
BGR = [
    Workload("bgr_pages_1024x4096_fp16", 1024, 4096, "fp16", 0.0, r_dist=(0.0, 0.5),
             op="bias_gelu_residual", note="the diagram's 8 MB tensors", shape_bsh=(1, 1024, 4096)),
    Workload("bgr_large_32768x8192_bf16", 32768, 8192, "bf16", 0.0, r_dist=(0.0, 0.5),
             op="bias_gelu_residual", note="512 MB tensors", shape_bsh=(8, 4096, 8192)),
    Workload("bgr_tail_1000x1001_fp32", 1000, 1001, "fp32", 0.0, r_dist=(0.0, 0.5),
             op="bias_gelu_residual", note="odd H: element path"),
]
WORKLOADS.update({w.name: w for w in BGR})
BGR_NAMES = [w.name for w in BGR]

# The five workloads of the method's scope, in order; the rest are extra tails.
PRIMARY = [
    "tiny_64x768_fp32",
    "bert_base_4096x768_fp16",
    "pages_2048x4096_fp16",
    "cancel_65536x1000_bf16",
    "large_32768x8192_bf16",
]
TAILS = ["tail_4096x999_bf16", "tail_4096x1001_bf16", "tail_4096x1002_fp32"]


def get(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def with_rows(w: Workload, rows: int) -> Workload:
    """The same workload with a different row count (for small CPU cases)."""
    from dataclasses import replace
    return replace(w, name=f"{w.name}@rows{rows}", rows=rows)


def custom(rows: int, H: int, dtype: str, eps: float = 1e-5, **kw) -> Workload:
    """An ad-hoc workload (edge-case sweeps) with the tiny case's distributions."""
    return Workload(f"custom_{rows}x{H}_{dtype}", rows, H, dtype, eps, **kw)
