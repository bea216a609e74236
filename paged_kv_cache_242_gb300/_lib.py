"""ctypes loader for libpkv.so (the C ABI declared in include/pkv.h).

Loading fails loudly: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIBRARY

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_WORKSPACE_TOO_SMALL", 4: "PKV_ERR_CUDA"}
PKV_FP16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
MAX_LAYERS = 128

DEVERR_BAD_SLOT = 1
DEVERR_BAD_BLOCK_ID = 2
DEVERR_BAD_SEQ_LEN = 4
DEVERR_BAD_PAIR = 8
DEVERR_TIMEOUT = 16


class PKVError(RuntimeError):
    """A libpkv call returned a non-OK status, or the library is missing."""

    def __init__(self, message: str, status: int | None = None):
        super().__init__(message)
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int)]


_lib = None


def _declare(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    i32p = ctypes.c_void_p  # device pointer to the int32 error flag
    lib.pkv_kv_write.argtypes = [vp, vp, vp, i32, vp, vp, CacheDesc, i32p, vp]
    lib.pkv_kv_write.restype = ctypes.c_int
    lib.pkv_decode_partition_size.argtypes = [i32, i32, i32]
    lib.pkv_decode_partition_size.restype = i32
    lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pkv_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.pkv_paged_decode_attention.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, CacheDesc,
                                               ctypes.c_float, i32, vp, ctypes.c_size_t, vp, i32p,
                                               vp]
    lib.pkv_paged_decode_attention.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [vp, vp, CacheDesc, vp, i32, i32p, vp]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_paged_prefill_attention.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32,
                                                CacheDesc, ctypes.c_float, vp, i32p, vp]
    lib.pkv_paged_prefill_attention.restype = ctypes.c_int
    ptrs = ctypes.POINTER(ctypes.c_void_p)  # host array of device pointers
    lib.pkv_swap_blocks.argtypes = [vp, vp, i32, vp, vp, i32, CacheDesc, vp, i32, i32p, vp]
    lib.pkv_swap_blocks.restype = ctypes.c_int
    lib.pkv_kv_write_layers.argtypes = [ptrs, ptrs, vp, i32, ptrs, ptrs, i32, CacheDesc, i32p, vp]
    lib.pkv_kv_write_layers.restype = ctypes.c_int
    lib.pkv_copy_blocks_layers.argtypes = [ptrs, ptrs, i32, CacheDesc, vp, i32, i32p, vp]
    lib.pkv_copy_blocks_layers.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.pkv_kv_write_fp8.argtypes = [vp, vp, ctypes.c_int, vp, i32, vp, vp, CacheDesc, f32, f32,
                                     i32p, vp]
    lib.pkv_kv_write_fp8.restype = ctypes.c_int
    lib.pkv_paged_decode_attention_fp8.argtypes = [vp, ctypes.c_int, vp, vp, vp, i32, vp, i32, i32,
                                                   i32, CacheDesc, f32, f32, f32, vp,
                                                   ctypes.c_size_t, vp, i32p, vp]
    lib.pkv_paged_decode_attention_fp8.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_abi_version.argtypes = []
    lib.pkv_abi_version.restype = i32
    return lib


def library_path() -> str:
    return LIBRARY


def load():
    """Load libpkv.so once; raise PKVError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise PKVError(f"{LIBRARY} is missing: build it with "
                           "`python -m paged_kv_cache_242_gb300.build` (there is no fallback)")
        _lib = _declare(ctypes.CDLL(LIBRARY))
    return _lib


def check(status: int, what: str) -> None:
    if status != PKV_OK:
        name = STATUS_NAMES.get(status, str(status))
        raise PKVError(f"{what} failed: {name}", status)
