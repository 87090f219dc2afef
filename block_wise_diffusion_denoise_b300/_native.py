"""ctypes declarations of the C ABI in ``include/tt_denoise.h`` (libtt_denoise.so).

This module only loads the shared library and declares argument types; it never
touches a GPU by itself.  If the library has not been built, ``lib()`` raises
``NativeLibraryMissing``: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtt_denoise.so")

TT_OK, TT_ERR_INVALID_ARG, TT_ERR_UNSUPPORTED, TT_ERR_CAPACITY, TT_ERR_CUDA, \
    TT_ERR_DEVICE_TIMEOUT, TT_ERR_BOUNDS = range(7)
TT_BF16, TT_FP32 = 0, 1
UNMASK_NOALLOC_SCRATCH_BYTES = 256 * 1024   # TT_UNMASK_NOALLOC_SCRATCH_BYTES

STATUS_NAMES = {
    TT_OK: "TT_OK", TT_ERR_INVALID_ARG: "TT_ERR_INVALID_ARG", TT_ERR_UNSUPPORTED: "TT_ERR_UNSUPPORTED",
    TT_ERR_CAPACITY: "TT_ERR_CAPACITY", TT_ERR_CUDA: "TT_ERR_CUDA",
    TT_ERR_DEVICE_TIMEOUT: "TT_ERR_DEVICE_TIMEOUT", TT_ERR_BOUNDS: "TT_ERR_BOUNDS",
}

# Every symbol the header declares, in declaration order.
EXPORTED = ("tt_status_string", "tt_version", "tt_denoise_attn_workspace_size", "tt_denoise_attn",
            "tt_context_block_attn", "tt_unmask_workspace_size", "tt_unmask", "tt_unmask_noalloc",
            "tt_linear_schedule_mask", "tt_masked_nll_workspace_size", "tt_masked_nll", "tt_kv_append",
            "tt_block_step_workspace_size", "tt_block_step", "tt_get_device_error", "tt_check_wait_timeout")


class NativeLibraryMissing(ImportError):
    pass


class TTError(RuntimeError):
    """A non-zero tt_status returned by the library (or read from the device error word)."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)} "
                         f"({lib().tt_status_string(self.status).decode()})")


class tt_kv_cache(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p),
        ("ctx_len", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGNATURES = {
    "tt_status_string": (ctypes.c_char_p, [_I]),
    "tt_version": (_I, []),
    "tt_denoise_attn_workspace_size": (_I, [_I, _I, _I, _I, _I, _I, _PSZ]),
    "tt_denoise_attn": (_I, [ctypes.POINTER(tt_kv_cache), _P, _P, _P, _P, _P, _I, _I, _I, _F, _I, _P, _SZ,
                             _P, _P]),
    "tt_context_block_attn": (_I, [ctypes.POINTER(tt_kv_cache), _P, _P, _P, _P, _P, _I, _I, _I, _F, _I, _P,
                                   _SZ, _P, _P]),
    "tt_unmask_workspace_size": (_I, [_I, _I, _I, _I, _PSZ]),
    "tt_unmask": (_I, [_P, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tt_unmask_noalloc": (_I, [_P, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "tt_linear_schedule_mask": (_I, [_P, _P, _P, _I, _I, ctypes.c_int32, _P, _P, _P, _P]),
    "tt_masked_nll_workspace_size": (_I, [_I, _I, _I, _I, _PSZ]),
    "tt_masked_nll": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tt_kv_append": (_I, [ctypes.POINTER(tt_kv_cache), _I, _PP, _PP, _P, _I, _I, _P, _P]),
    "tt_block_step_workspace_size": (_I, [_I, _I, _I, _I, _I, _I, _I, _PSZ]),
    "tt_block_step": (_I, [ctypes.POINTER(tt_kv_cache), _I, _PP, _PP, _PP, _PP, _P, _I, _I, _I, _I, _F, _I,
                           _I, _F, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tt_get_device_error": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "tt_check_wait_timeout": (_I, [ctypes.c_uint32, _P, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises NativeLibraryMissing if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise NativeLibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m block_wise_diffusion_denoise_b300.build` "
                "(there is no fallback implementation)")
        so = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(so, name)
            fn.restype = res
            fn.argtypes = args
        _lib = so
    return _lib


def check(status: int, where: str) -> None:
    if status != TT_OK:
        raise TTError(status, where)


def ptr_array(ptrs) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(ptrs))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr
