"""GB300 (sm_103a) bit-quantized decode GEMV.

The decode linear y = W x + b with per-row INT4, Q4_0 or int8/group-32
weights and per-token INT8 activations, computed by hand-written CUDA kernels
behind the C ABI in include/w4a8.h.  `_lib` is the thin ctypes binding (same
names as the C entry points); `linear.QuantLinear` prepares and calls one
(possibly shard-fused) linear.
"""
from . import _lib
from ._lib import (W4_FLAG_PDL, W4Error, a8_quantize, clear_device_error, device_error, i8g32_gemv,
                   i8g32_linear, i8g32_quantize, i8g32_repack, i8g32_repacked_bytes, q4_0_gemv, q4_0_linear,
                   q4_0_quantize, q4_0_repack, q4_0_repacked_bytes, w4_concat_f32, w4_quantize_rows, w4_repack,
                   w4_repacked_bytes, w4a8_gemv, w4a8_linear)
from .linear import LinearChain, QuantLinear

__all__ = [
    "W4_FLAG_PDL", "W4Error", "LinearChain", "QuantLinear", "a8_quantize", "clear_device_error", "device_error",
    "i8g32_gemv", "i8g32_linear", "i8g32_quantize", "i8g32_repack", "i8g32_repacked_bytes", "q4_0_gemv",
    "q4_0_linear", "q4_0_quantize", "q4_0_repack", "q4_0_repacked_bytes", "w4_concat_f32", "w4_quantize_rows",
    "w4_repack", "w4_repacked_bytes", "w4a8_gemv", "w4a8_linear",
]
