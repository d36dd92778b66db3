"""GB300-native dual-weight GLU GEMV (decode-step gated-MLP segment).

    out = SiLU(h @ gate_w.T) * (h @ up_w.T)

computed by hand-written sm_103a kernels behind the C ABI of libmbglu.so
(include/mbglu.h); this package is the thin Python binding.
"""
from .binding import (EXPORTS, LIB_PATH, MAX_M, MODE_FUSED, MODE_HF, MbgluError, add_rmsnorm_glu, glu_gemv,
                      last_variant, lib, read_device_error)

__all__ = ["glu_gemv", "add_rmsnorm_glu", "MbgluError", "lib", "last_variant", "read_device_error",
           "MODE_FUSED", "MODE_HF", "MAX_M", "EXPORTS", "LIB_PATH"]
