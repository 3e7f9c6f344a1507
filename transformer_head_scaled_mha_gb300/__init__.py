"""GB300 (sm_103a) multi-head scaled dot-product attention forward.

``mha_fwd`` computes softmax(Q K^T * scale) V per (batch, head) on hand-written
CUDA kernels: a tcgen05/TMA/TMEM kernel for long sequences, a packed
tensor-core kernel for sentence-length sequences, and an fp32 CUDA-core
kernel.  Masks: causal, key padding, query padding (see include/mha.h).
``mha_fwd_ex`` adds shared key/value heads (grouped- and multi-query
attention) and the [B, L, H, d] layout; ``mha_sublayer_fwd`` runs the whole
multi-head sublayer (projections with biases on ``mha_linear_fwd``'s tensor-core
kernel, attention, output projection).
"""
from .mha import (MHA_DTYPE_BF16, MHA_DTYPE_F32, MHA_ERR_CUDA, MHA_ERR_INVALID_ARGUMENT,
                  MHA_ERR_TIMEOUT, MHA_ERR_UNSUPPORTED, MHA_MASK_CAUSAL, MHA_MASK_KEY_PADDING,
                  MHA_LAYOUT_BHSD, MHA_LAYOUT_BSHD, MHA_MASK_CAUSAL_TAIL, MHA_MASK_NONE,
                  MHA_MASK_QUERY_PADDING, MHA_OK, PATH_NAMES, LIB_PATH, MhaError,
                  lib, mha_debug_set_wait, mha_debug_status, mha_fwd, mha_fwd_lse, mha_fwd_ex, mha_fwd_path, mha_fwd_path_ex,
                  mha_linear_fwd,
                  mha_sublayer_fwd, mha_sublayer_fwd_static, mha_sublayer_workspace_size,
                  mha_bwd, mha_bwd_workspace_size, mha_status_string, mha_version)

__all__ = ["mha_fwd", "mha_fwd_ex", "mha_fwd_lse", "mha_linear_fwd", "mha_sublayer_fwd", "mha_bwd",
           "mha_bwd_workspace_size",
           "mha_sublayer_fwd_static",
           "mha_sublayer_workspace_size", "mha_fwd_path", "mha_fwd_path_ex", "mha_status_string", "mha_debug_status",
           "mha_debug_set_wait", "mha_version",
           "MhaError", "lib", "LIB_PATH", "PATH_NAMES", "MHA_OK", "MHA_ERR_INVALID_ARGUMENT",
           "MHA_ERR_UNSUPPORTED", "MHA_ERR_CUDA", "MHA_ERR_TIMEOUT", "MHA_DTYPE_F32",
           "MHA_DTYPE_BF16", "MHA_MASK_NONE", "MHA_MASK_CAUSAL", "MHA_MASK_KEY_PADDING",
           "MHA_MASK_QUERY_PADDING", "MHA_MASK_CAUSAL_TAIL", "MHA_LAYOUT_BHSD",
           "MHA_LAYOUT_BSHD"]
