"""ctypes loader for libbsm.so (the C ABI of include/bsm.h).

The library is loaded on first use.  There is no fallback: if the shared
library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# BSM_LIBRARY may point at another build of the same library.
LIB_PATH = os.environ.get("BSM_LIBRARY") or os.path.join(HERE, "libbsm.so")

BSM_OK = 0
BSM_ERR_INVALID_ARG = -1
BSM_ERR_UNSUPPORTED = -2
BSM_ERR_CUDA = -3
BSM_ERR_DEVICE_TIMEOUT = -4

STATUS_NAMES = {
    BSM_OK: "BSM_OK",
    BSM_ERR_INVALID_ARG: "BSM_ERR_INVALID_ARG",
    BSM_ERR_UNSUPPORTED: "BSM_ERR_UNSUPPORTED",
    BSM_ERR_CUDA: "BSM_ERR_CUDA",
    BSM_ERR_DEVICE_TIMEOUT: "BSM_ERR_DEVICE_TIMEOUT",
}


ABI_VERSION = 302  # the struct layouts below


class MaskSpec(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("window", ctypes.c_int32),
                ("dense_bits", ctypes.c_void_p),
                ("dense_row_words", ctypes.c_int64)]


class MaskInfoStruct(ctypes.Structure):
    _fields_ = [
        ("flags", ctypes.c_uint32),
        ("window", ctypes.c_int32),
        ("num_tables", ctypes.c_int32),
        ("Sq", ctypes.c_int32),
        ("Skv", ctypes.c_int32),
        ("block_q", ctypes.c_int32),
        ("block_kv", ctypes.c_int32),
        ("nq", ctypes.c_int32),
        ("nk", ctypes.c_int32),
        ("block_mask", ctypes.c_void_p),
        ("data_next", ctypes.c_void_p),
        ("row_ptr", ctypes.c_void_p),
        ("kv_idx", ctypes.c_void_p),
        ("kv_cls", ctypes.c_void_p),
        ("seg_range", ctypes.c_void_p),
        ("seg_flags", ctypes.c_void_p),
        ("num_super", ctypes.c_int32),
        ("super_order", ctypes.c_void_p),
        ("dense_bits", ctypes.c_void_p),
        ("dense_row_words", ctypes.c_int64),
    ]


I64x3 = ctypes.c_int64 * 3


class TensorView(ctypes.Structure):
    """bsm_tensor: device data pointer and batch/head/sequence strides."""
    _fields_ = [("data", ctypes.c_void_p), ("strides", ctypes.c_int64 * 3)]

_lock = threading.Lock()
_lib = None


def _declare(lib):
    c = ctypes
    lib.bsm_mask_info_bytes.restype = c.c_size_t
    lib.bsm_mask_info_bytes.argtypes = [c.POINTER(MaskSpec), c.c_int32,
                                        c.c_int32, c.c_int32, c.c_int32,
                                        c.c_int32]
    lib.bsm_build_mask_info.restype = c.c_int
    lib.bsm_build_mask_info.argtypes = [
        c.POINTER(MaskSpec), c.c_void_p, c.c_void_p, c.c_int32, c.c_int32,
        c.c_int32, c.c_int32, c.c_int32, c.c_void_p, c.c_size_t,
        c.POINTER(MaskInfoStruct), c.c_void_p]
    lib.bsm_splash_fwd.restype = c.c_int
    lib.bsm_splash_fwd.argtypes = [
        c.c_void_p, c.c_void_p, c.c_void_p, I64x3, I64x3, I64x3, I64x3,
        c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
        c.POINTER(MaskInfoStruct), c.c_void_p, c.c_void_p, c.c_float,
        c.c_int32, c.c_void_p, c.c_void_p, c.c_void_p, c.c_size_t,
        c.c_void_p]
    lib.bsm_splash_fwd_host_bytes.restype = c.c_size_t
    lib.bsm_splash_fwd_host_bytes.argtypes = [
        c.POINTER(MaskSpec), c.c_int32, c.c_int32, c.c_int32, c.c_int32,
        c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32]
    lib.bsm_splash_fwd_host.restype = c.c_int
    lib.bsm_splash_fwd_host.argtypes = [
        c.POINTER(MaskSpec), c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
        c.c_void_p, c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
        c.c_int32, c.c_int32, c.c_int32, c.c_float, c.c_int32, c.c_void_p,
        c.c_void_p, c.c_void_p, c.c_size_t, c.c_int32, c.c_void_p]
    lib.bsm_splash_fwd_noalloc.restype = c.c_int
    lib.bsm_splash_fwd_noalloc.argtypes = [
        c.c_void_p, c.c_void_p, c.c_void_p, I64x3, I64x3, I64x3, I64x3,
        c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
        c.POINTER(MaskInfoStruct), c.c_void_p, c.c_void_p, c.c_float,
        c.c_int32, c.c_void_p, c.c_void_p, c.c_void_p]
    lib.bsm_splash_fwd_workspace_bytes.restype = c.c_size_t
    lib.bsm_splash_fwd_workspace_bytes.argtypes = []
    lib.bsm_splash_bwd_workspace_bytes.restype = c.c_size_t
    lib.bsm_splash_bwd_workspace_bytes.argtypes = [c.c_int32, c.c_int32,
                                                   c.c_int32, c.c_int32]
    tv = c.POINTER(TensorView)
    lib.bsm_splash_bwd.restype = c.c_int
    lib.bsm_splash_bwd.argtypes = [
        tv, tv, tv, tv, c.c_void_p, tv, c.c_int32, c.c_int32, c.c_int32,
        c.c_int32, c.c_int32, c.c_int32, c.POINTER(MaskInfoStruct),
        c.c_void_p, c.c_void_p, c.c_float, c.c_int32, tv, tv, tv, c.c_void_p,
        c.c_size_t, c.c_void_p]
    lib.bsm_pack_dense_mask.restype = c.c_int
    lib.bsm_pack_dense_mask.argtypes = [c.c_void_p, c.c_int64, c.c_int32,
                                        c.c_int32, c.c_void_p, c.c_int32,
                                        c.c_void_p]
    lib.bsm_device_status.restype = c.c_int
    lib.bsm_device_status.argtypes = [c.c_void_p, c.POINTER(c.c_int32)]
    lib.bsm_selftest_wait_timeout.restype = c.c_int
    lib.bsm_selftest_wait_timeout.argtypes = [c.c_int64, c.c_void_p]
    lib.bsm_debug_set_trace.restype = c.c_int
    lib.bsm_debug_set_trace.argtypes = [c.c_void_p, c.c_size_t]
    lib.bsm_debug_fwd_grid.restype = c.c_int32
    lib.bsm_debug_fwd_grid.argtypes = [c.c_int32, c.c_int32, c.c_int32]
    lib.bsm_last_error.restype = c.c_char_p
    lib.bsm_last_error.argtypes = []
    lib.bsm_version.restype = c.c_int32
    lib.bsm_version.argtypes = []
    return lib


def lib():
    """The loaded library; raises if libbsm.so has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built: run "
                    "`python -m block_sparse_masked_build_gb300.build` "
                    "(there is no CPU fallback)")
            loaded = _declare(ctypes.CDLL(LIB_PATH))
            version = loaded.bsm_version()
            if version != ABI_VERSION:
                raise RuntimeError(
                    f"{LIB_PATH} has ABI version {version}, this binding "
                    f"expects {ABI_VERSION}: rebuild the library")
            _lib = loaded
    return _lib


def last_error() -> str:
    return lib().bsm_last_error().decode("utf-8", "replace")
