"""GB300-native row-normalization layers: DyT, LayerNorm and Llama-style
RMSNorm, forward and backward, as hand-written CUDA kernels for sm_103a
behind a C ABI (include/gbnorm.h, libgbnorm.so).

    from normalization_layers_fwd_gb300 import dyt_fwd, dyt_bwd, ...   # C-ABI names
    from normalization_layers_fwd_gb300.functional import rms_norm      # autograd

The Python functions take CUDA tensors of any leading shape.  A strided
input whose rows fold into at most three levels (a head-major view, a
row-padded slice) is passed to the C ABI's *_rows entry points with its
gbn_rows layout and read in place; outputs are contiguous.
"""
from ._lib import (  # noqa: F401
    GBN_BF16,
    GBN_F16,
    GBN_F32,
    GBN_OP_DYT,
    GBN_OP_LAYERNORM,
    GBN_OP_RMSNORM,
    GBN_RMS_CAST_FIRST,
    GBN_RMS_GEMMA,
    GBN_RMS_WEIGHT_FIRST,
    GBN_STATIC_WS_BYTES,
    GbnError,
    dyt_bwd,
    dyt_fwd,
    fold_rows,
    gbn_rows,
    layernorm_bwd,
    layernorm_fwd,
    load,
    read_faults,
    rmsnorm_bwd,
    rmsnorm_bwd_static_ws,
    rmsnorm_fwd,
    row_layout,
    workspace,
)
