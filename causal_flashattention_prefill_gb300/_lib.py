"""ctypes binding of the C ABI in ``include/zyfa.h`` (argument marshalling only).

Every function here has the name and argument order of its C counterpart and
returns the C status code.  Pointers are plain integers (device addresses);
``stream`` is a ``cudaStream_t`` as an integer (0 = default stream).  Loading
fails loudly when the library has not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libzyfa_gb300.so")

ZYFA_OK = 0
ZYFA_ERR_ARG = -1
ZYFA_ERR_UNSUPPORTED = -2
ZYFA_ERR_ALIGN = -3
ZYFA_ERR_LAUNCH = -4
ZYFA_ERR_DEVICE = -5
ZYFA_ERR_DEVICE_TIMEOUT = -6

ZYFA_BF16 = 0
ZYFA_FP8_E4M3 = 1
ZYFA_F32 = 2
ZYFA_BSHD = 0
ZYFA_BHSD = 1
ZYFA_OPT_SERIALIZE_PV = 1
ZYFA_OPT_ROUNDED_P = 2
ZYFA_OPT_BLOCK_SCALE = 3
ZYFA_OPT_DYNAMIC_SCHEDULE = 4

# name -> (restype, argtypes); the C ABI of include/zyfa.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_FWD_ARGS = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]
SIGNATURES = {
    "zyfa_fwd": (_I, _FWD_ARGS + [_I, _P]),
    "zyfa_fwd_scaled": (_I, _FWD_ARGS + [_F, _I, _P]),
    "zyfa_validate": (_I, _FWD_ARGS + [_F, _I]),
    "zyfa_status_string": (ctypes.c_char_p, [_I]),
    "zyfa_device_status": (_I, [ctypes.POINTER(_I), _I]),
    "zyfa_set_option": (_I, [_I, _I]),
    "zyfa_version": (_I, []),
    "zyfa_fp8_quantize": (_I, [_P, ctypes.c_longlong, _I, _P, _P, _P, _P]),
    "zyfa_fp8_quantize_workspace_bytes": (ctypes.c_longlong, []),
    "zyfa_fp8_quantize_noalloc": (_I, [_P, ctypes.c_longlong, _I, _P, _P, _P]),
    "zyfa_fp8_quantize_rotated": (_I, [_P, ctypes.c_longlong, _I, _I, _P, _P, _P, _P, _P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library once and declares every C signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built; run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def zyfa_fwd(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
             v_descale, layout, stream) -> int:
    return load().zyfa_fwd(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale,
                           k_descale, v_descale, layout, stream)


def zyfa_fwd_scaled(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
                    v_descale, softmax_scale, layout, stream) -> int:
    return load().zyfa_fwd_scaled(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype,
                                  q_descale, k_descale, v_descale, softmax_scale, layout,
                                  stream)


def zyfa_validate(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
                  v_descale, softmax_scale, layout) -> int:
    return load().zyfa_validate(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale,
                                k_descale, v_descale, softmax_scale, layout)


def zyfa_status_string(status: int) -> str:
    return load().zyfa_status_string(status).decode()


def zyfa_device_status(reset: bool = False):
    """Returns (status, value) of the device status word."""
    v = ctypes.c_int(0)
    st = load().zyfa_device_status(ctypes.byref(v), 1 if reset else 0)
    return st, v.value


def zyfa_set_option(option: int, value: int) -> int:
    return load().zyfa_set_option(option, value)


def zyfa_version() -> int:
    return load().zyfa_version()


def zyfa_fp8_quantize(x, n, x_dtype, x8, descale, workspace, stream) -> int:
    return load().zyfa_fp8_quantize(x, n, x_dtype, x8, descale, workspace, stream)


def zyfa_fp8_quantize_workspace_bytes() -> int:
    return load().zyfa_fp8_quantize_workspace_bytes()


def zyfa_fp8_quantize_noalloc(x, n, x_dtype, x8, descale, stream) -> int:
    return load().zyfa_fp8_quantize_noalloc(x, n, x_dtype, x8, descale, stream)


def zyfa_fp8_quantize_rotated(x, n_rows, d, x_dtype, signs, x8, descale, workspace,
                              stream) -> int:
    return load().zyfa_fp8_quantize_rotated(x, n_rows, d, x_dtype, signs, x8, descale,
                                            workspace, stream)
