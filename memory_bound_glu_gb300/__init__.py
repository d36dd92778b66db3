"""GB300-native dual-weight GLU GEMV (decode-step gated-MLP segment).

    out = SiLU(h @ gate_w.T) * (h @ up_w.T)

computed by hand-written sm_103a kernels behind the C ABI of libmbglu.so
(include/mbglu.h); this package is the thin Python binding.
"""
from .binding import (BLOCK_M, EXPORTS, LIB_PATH, MAX_M, MODE_FUSED, MODE_HF, POLICY_PDL, POLICY_PREFETCH, POLICY_SERIAL,
                      DualWeightGlu, MbgluError, WORKSPACE_BYTES, add_rmsnorm_glu, column_shard, get_launch_policy, glu_backward,
                      glu_gemv, last_backward_path, last_variant, lib, gdn_gates, new_workspace, read_device_error, set_launch_policy,
                      silu_mul)

__all__ = ["glu_gemv", "column_shard", "glu_backward", "DualWeightGlu", "add_rmsnorm_glu", "silu_mul", "gdn_gates", "MbgluError", "lib", "last_variant", "last_backward_path", "read_device_error",
           "set_launch_policy", "get_launch_policy", "POLICY_SERIAL", "POLICY_PDL", "POLICY_PREFETCH",
           "MODE_FUSED", "MODE_HF", "MAX_M", "BLOCK_M", "EXPORTS", "LIB_PATH", "WORKSPACE_BYTES", "new_workspace"]
