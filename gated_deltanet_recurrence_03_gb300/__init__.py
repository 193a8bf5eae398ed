"""Gated DeltaNet state recurrence on GB300 (sm_103a).

The compute runs in libgdn.so (hand-written CUDA: a tcgen05/TMA chunked prefill, a
token-serial CUDA-core prefill and a one-pass decode step) behind the C ABI of
``include/gdn.h``.  This package is the thin PyTorch binding of that ABI.
"""
from ._lib import GdnError, GDN_BF16, GDN_F32, GDN_NORMALIZE_QK  # noqa: F401
from .api import (backward_workspace_size, check_device_status, gdn_causal_conv1d_bwd, gdn_causal_conv1d_fwd,  # noqa: F401
                  gdn_causal_conv1d_fwd_qkv, gdn_causal_conv1d_step, gdn_causal_conv1d_step_qkv, gdn_chunk_fwd,
                  gdn_output_gate_bwd, gdn_output_gate_fwd,
                  gdn_recurrent_bwd, gdn_recurrent_step, version, workspace_size)

__all__ = ["gdn_chunk_fwd", "gdn_recurrent_step", "gdn_recurrent_bwd", "gdn_causal_conv1d_fwd",
           "gdn_causal_conv1d_step", "gdn_output_gate_fwd", "gdn_output_gate_bwd", "gdn_causal_conv1d_bwd", "gdn_causal_conv1d_fwd_qkv", "gdn_causal_conv1d_step_qkv", "workspace_size", "backward_workspace_size", "check_device_status", "version",
           "GdnError"]
