"""GB300-native row-normalization layers: DyT, LayerNorm and Llama-style
RMSNorm, forward and backward, as hand-written CUDA kernels for sm_103a
behind a C ABI (include/gbnorm.h, libgbnorm.so).

    from normalization_layers_fwd_gb300 import dyt_fwd, dyt_bwd, ...   # C-ABI names
    from normalization_layers_fwd_gb300.functional import rms_norm      # autograd
"""
from ._lib import (  # noqa: F401
    GBN_BF16,
    GBN_F32,
    GBN_OP_DYT,
    GBN_OP_LAYERNORM,
    GBN_OP_RMSNORM,
    GbnError,
    dyt_bwd,
    dyt_fwd,
    layernorm_bwd,
    layernorm_fwd,
    load,
    rmsnorm_bwd,
    rmsnorm_fwd,
)
