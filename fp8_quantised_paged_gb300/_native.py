"""ctypes binding of ``libfp8pa.so`` (the C ABI in ``include/fp8pa.h``).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or does not
load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8pa.so")

# Keep in step with include/fp8pa.h.
OK = 0
ERR_NULL_POINTER, ERR_BAD_ENUM, ERR_BAD_SHAPE, ERR_UNSUPPORTED = -1, -2, -3, -4
ERR_WORKSPACE, ERR_ALIGNMENT, ERR_CUDA = -5, -6, -7
DEVERR_SLOT_RANGE, DEVERR_BLOCK_RANGE, DEVERR_SEQ_LEN, DEVERR_TIMEOUT = 1, 2, 4, 8
E4M3, E5M2, INT8 = 0, 1, 2
SCALE_TOKEN_HEAD, SCALE_CHANNEL_STATIC, SCALE_TOKEN_GROUP, SCALE_MX_BLOCK = 0, 1, 2, 3
SCALE_SEGMENT = 4
SEGMENT_TOKENS = 1024
OUT_BF16, OUT_F32 = 0, 1

# Every symbol the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "fp8pa_kv_append_quant": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _I,
                                   _P]),
    "fp8pa_kv_append_quant_segment": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                           _P, _I, _I, _P]),
    "fp8pa_kv_channel_scales": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "fp8pa_kv_channel_absmax_update": (_I, [_P, _I, _I, _I, _P, _P]),
    "fp8pa_kv_scales_from_absmax": (_I, [_P, _I, _I, _P, _P]),
    "fp8pa_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I]),
    "fp8pa_multiquery_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "fp8pa_paged_decode_attention": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                                          _I, _I, _I, ctypes.c_float, _I, _P, _I, _P,
                                          ctypes.c_size_t, _P]),
    "fp8pa_paged_multiquery_attention": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                              _I, _I, _I, _I, _I, ctypes.c_float, _I, _P, _I, _P,
                                              ctypes.c_size_t, _P]),
    "fp8pa_decode_step": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                               _I, _I, _I, _I, _I, ctypes.c_float, _I, _P, _I, _P,
                               ctypes.c_size_t, _P]),
    "fp8pa_paged_decode_attention_static_ws": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I,
                                                    _I, _I, _I, _I, _I, _I, ctypes.c_float, _I,
                                                    _P, _I, _P]),
    "fp8pa_get_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "fp8pa_selftest_bounded_wait": (_I, [ctypes.c_longlong, _P]),
    "fp8pa_set_decode_workers": (_I, [_I]),
    "fp8pa_set_split_events": (_I, [_P, _P]),
    "fp8pa_error_string": (ctypes.c_char_p, [_I]),
    "fp8pa_version": (_I, []),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "fp8_quantised_paged_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class Fp8paError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {lib.fp8pa_error_string(code).decode()} ({code})")
        self.code = code


def check(code: int, where: str) -> None:
    if code != OK:
        raise Fp8paError(code, where)
