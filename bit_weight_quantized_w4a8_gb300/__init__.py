"""GB300 (sm_103a) weight-quantized decode linear: W4A8 (row-wise or
group-wise INT4 scales) and W8A16; the MLP's gated product between the
gate/up and down projections; and the IndexSoftmax integer softmax.

The compute lives in libw4a8.so (CUDA kernels behind the C ABI of
include/w4a8.h); this package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    EXPORTS, LAUNCH_PDL, LIB_PATH, PLAN_FIELDS, W4A8_MAX_M, W8A16_MAX_M, W4A8Error,
    act_quantize_i8, lib, w4_quantize_weights, w4a8_device_error, w4a8_gemv,
    w4a8_last_error, w4a8_linear, w4a8_linear_grouped, w4a8_linear_noalloc, w4a8_plan_info, w4a8_set_tuning, w4a8_workspace_bytes,
    w8_quantize_weights, w8a16_gemv, w8a16_workspace_bytes,
    GROUP_PLAN_FIELDS, w4g_quantize_weights, w4g_scale_stride, w4a8g_gemv, w4a8g_linear,
    w4a8g_linear_grouped, w4a8g_plan_info, w4a8g_workspace_bytes,
    ISX_DEFAULT_B, ISX_DEFAULT_C, index_softmax_c_int, index_softmax_lut, index_softmax_u8,
    w4_interleave_rows, w4a8_gate_up_silu, w4a8_gate_up_silu_workspace_bytes, w4a8_silu_mul,
)
from .build import build  # noqa: F401
