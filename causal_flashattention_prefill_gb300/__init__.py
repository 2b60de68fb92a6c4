"""GB300 (sm_103a) causal prefill attention.

``zyfa_*`` are the C ABI entry points (ctypes, argument marshalling only).
``flash_attn_func`` (with its qkv-packed, kv-packed and equal-length varlen
forms) and ``fp8_quantize`` are the torch-level conveniences with the calling
conventions of the ZYFA README ("Usage", "Differences from flash-attn"); every
step of the attention itself runs in the CUDA library.
"""

from ._lib import (  # noqa: F401
    LIB_PATH,
    ZYFA_BF16,
    ZYFA_BHSD,
    ZYFA_BSHD,
    ZYFA_ERR_ALIGN,
    ZYFA_ERR_ARG,
    ZYFA_ERR_DEVICE,
    ZYFA_ERR_DEVICE_TIMEOUT,
    ZYFA_ERR_LAUNCH,
    ZYFA_ERR_UNSUPPORTED,
    ZYFA_F32,
    ZYFA_FP8_E4M3,
    ZYFA_OK,
    ZYFA_OPT_BLOCK_SCALE,
    ZYFA_OPT_DYNAMIC_SCHEDULE,
    ZYFA_OPT_ROUNDED_P,
    ZYFA_OPT_SERIALIZE_PV,
    load,
    zyfa_device_status,
    zyfa_fp8_quantize,
    zyfa_fp8_quantize_noalloc,
    zyfa_fp8_quantize_rotated,
    zyfa_fp8_quantize_workspace_bytes,
    zyfa_fwd,
    zyfa_fwd_scaled,
    zyfa_set_option,
    zyfa_status_string,
    zyfa_validate,
    zyfa_version,
)
from .api import (  # noqa: F401
    ZyfaError,
    attention,
    flash_attn_func,
    flash_attn_kvpacked_func,
    flash_attn_qkvpacked_func,
    flash_attn_varlen_func,
    fp8_quantize,
    fp8_quantize_rotated,
    hadamard_signs,
)
