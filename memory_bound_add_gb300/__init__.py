"""GB300 (sm_103a) fused residual-Add + LayerNorm.

The compute lives in ``_build/libaddln.so`` (hand-written CUDA kernels behind
the C ABI of ``include/addln.h``); ``binding`` marshals PyTorch tensors to it.
"""
from .binding import (  # noqa: F401
    AddLNError,
    add_layernorm_fwd,
    add_layernorm_fwd_host,
    add_layernorm_fwd_host_last_mode,
    add_layernorm_fwd_host_workspace_size,
    add_fwd,
    layernorm_fwd,
    add_layernorm,
    add_then_layernorm,
    softmax_fwd,
    softmax,
    bias_gelu_residual_fwd,
    bias_add_fwd,
    gelu_fwd,
    bias_gelu_residual,
    bias_gelu_residual_unfused,
    add_layernorm_bwd,
    add_layernorm_bwd_workspace_size,
    bwd_workspace,
    add_layernorm_backward,
    add_layernorm_bwd_noalloc,
    addln_get_device_error,
    addln_set_force_path,
    addln_set_wait_limit_ns,
    addln_set_grid_cap,
    addln_set_pdl,
    addln_set_cta_shape,
    addln_set_warp_rows,
    addln_last_path,
    addln_max_hidden,
    addln_strerror,
    lib,
    FP32, FP16, BF16,
    PATH_AUTO, PATH_WARP_VEC, PATH_CTA_TMA, PATH_CTA_VEC, PATH_SCALAR,
)
from .autograd import AddLayerNormFunction, FusedAddLayerNorm, add_layernorm_train  # noqa: F401
