"""ctypes view of libfa.so: one Python callable per entry point of include/fa.h."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa.so")

(FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_LAUNCH, FA_ERR_TIMEOUT,
 FA_ERR_SCRATCH_LIMIT, FA_ERR_OUT_OF_PAGES) = range(8)
FA_BWD_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
FA_DEVERR_SELFTEST_CODE = 0x10FF
FA_OPT_RESCALE_TAU, FA_OPT_POLY_EXP, FA_OPT_WAIT_TIMEOUT_MS = 1, 2, 3
FA_POLY_EXP_DEFAULT = 16  # the library's default share of exponentials on the cubic: one column pair in 16

# every symbol include/fa.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
SIGNATURES = {
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_decode_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "fa_bwd_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_bwd_varlen_workspace_bytes": (_S, [_I, _I, _I]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_masked": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_masked_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P] + [_I] * 10 + [_F, _P]),
    "fa_bwd_masked": (_I, [_P] * 10 + [_I] * 8 + [_F, _P]),
    "fa_bwd_masked_varlen": (_I, [_P] * 12 + [_I] * 10 + [_F, _P]),
    "fa_fp8_quantize": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_fp8": (_I, [_P] * 8 + [_I] * 9 + [_F, _P]),
    "fa_pool_create": (_P, [_I, _I, _I, _I]),
    "fa_pool_destroy": (None, [_P]),
    "fa_pool_free_pages": (_I, [_P]),
    "fa_pool_refcount": (_I, [_P, _I]),
    "fa_pool_add_seq": (_I, [_P, ctypes.POINTER(_I)]),
    "fa_pool_fork": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "fa_pool_release": (_I, [_P, _I]),
    "fa_pool_reserve_append": (_I, [_P, _P, _I, _P, _P, _P]),
    "fa_pool_export": (_I, [_P, _P, _P]),
    "fa_paged_append": (_I, [_P] * 7 + [_I] * 5 + [_P]),
    "fa_decode_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "fa_decode_window": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "fa_decode_paged_window": (_I, [_P] * 7 + [_I] * 10 + [_P, _F, _P]),
    "fa_decode_num_splits": (_I, [_I, _I, _I, _I]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _F, _P]),
    "fa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "fa_device_error": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "fa_selftest_wait_timeout": (_I, [ctypes.c_double, _P]),
    "fa_selftest_exp2": (_I, [_P, _P, _I, _I, _P]),
    "fa_set_option": (_I, [_I, ctypes.c_double]),
}

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libfa.so (once).  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing; build it with exact_attention_94_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FaError(status, where)
