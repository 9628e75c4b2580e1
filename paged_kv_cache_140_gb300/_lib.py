"""ctypes view of the C ABI in include/pa.h (libpagedattn.so).

Loading never compiles anything and never falls back: if the shared library
is missing, importing the API raises with the command that builds it.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_WORKSPACE, PA_ERR_DEVICE_BOUNDS = range(6)
PA_F16, PA_BF16, PA_F32, PA_FP8_E4M3 = 0, 1, 2, 3

FLAG_BAD_SLOT = 0x1
FLAG_BAD_BLOCK_ID = 0x2
FLAG_BAD_CONTEXT_LEN = 0x4
FLAG_BAD_COPY_PAIR = 0x8
FLAG_TIMEOUT = 0x10

# Every symbol include/pa.h declares, with (restype, argtypes).
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pa_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _I, _F, _F, _P, _P]),
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_decode_workspace_init": (_I, [_P, _SZ, _P]),
    "pa_decode_partition_size": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "pa_decode": (_I, [_P, _I, _P, _I, _P, _P, _I, _F, _F, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I64, _F,
                       _I, _P, _SZ, _P, _P]),
    "pa_decode_append": (_I, [_P, _I, _P, _I, _P, _P, _P, _P, _I, _F, _F, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                              _I64, _F, _I, _P, _SZ, _P, _P]),
    "pa_decode_noalloc": (_I, [_P, _I, _P, _I, _P, _P, _I, _F, _F, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I64,
                               _F, _I, _P, _P]),
    "pa_prefill": (_I, [_P, _I, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I64, _I, _I, _I, _I, _I, _I64, _F, _P,
                        _P]),
    "pa_copy_blocks": (_I, [_P, _P, _P, _I64, _I64, _I, _I, _I, _I, _P, _P]),
    "pa_copy_blocks_layers": (_I, [_P, _I, _P, _I64, _I64, _I, _I, _I, _I, _P, _P]),
    "pa_swap_blocks": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _I, _P, _P]),
    "pa_check_err_flag": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int), _P]),
    "pa_status_string": (ctypes.c_char_p, [_I]),
    "pa_version": (_I, []),
}

_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libpagedattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()' or "
            "python -m paged_kv_cache_140_gb300._build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, where)
