"""ctypes view of the C ABI declared in ``include/gbattn.h``.

Loads ``_build/libgbattn.so`` (built by :mod:`scaled_dot_product_03_gb300.build`)
and fails loudly when it is missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgbattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
                3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_TIMEOUT"}
ATTN_F16, ATTN_BF16, ATTN_F32 = 0, 1, 2
ATTN_LAYOUT_DENSE4D, ATTN_LAYOUT_THD = 0, 1

# Every symbol include/gbattn.h declares.
EXPORTS = ("attn_fwd", "attn_bwd_workspace_size", "attn_bwd", "attn_merge_lse",
           "attn_last_error_string", "attn_check_device_error", "attn_set_watchdog_ns",
           "attn_watchdog_selftest", "attn_profile_begin", "attn_profile_read",
           "attn_bwd_noalloc", "attn_bwd_dlse", "attn_merge_lse_bwd",
           "attn_thd_partitioned_indices", "attn_thd_accumulate", "attn_thd_store")
KERNEL_KINDS = {0: "fwd", 1: "bwd_preprocess", 2: "bwd_dkdv", 3: "bwd_dq", 4: "merge",
                5: "simt_fwd", 6: "simt_bwd_dq", 7: "simt_bwd_dkdv", 8: "bwd_fused",
                9: "bwd_dq_convert", 10: "merge_bwd", 11: "bwd_dkv_reduce", 12: "thd_rows"}
NOALLOC_SCRATCH_BYTES = 64 << 20  # GBATTN_NOALLOC_SCRATCH_BYTES


class AttnTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride", ctypes.c_int64 * 4)]


class AttnParams(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("layout", ctypes.c_int), ("B", ctypes.c_int),
                ("Sq", ctypes.c_int), ("Skv", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_kv", ctypes.c_void_p),
                ("max_seqlen_q", ctypes.c_int), ("max_seqlen_kv", ctypes.c_int),
                ("scale", ctypes.c_float), ("window_left", ctypes.c_int),
                ("window_right", ctypes.c_int), ("deterministic", ctypes.c_int),
                ("cu_seqlens_q_padded", ctypes.c_void_p), ("cu_seqlens_kv_padded", ctypes.c_void_p)]


class AttnError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                "libgbattn.so is not built (%s); run scaled_dot_product_03_gb300.build.build()"
                % path)
        lib = ctypes.CDLL(path)
        P, T, S = ctypes.POINTER(AttnParams), AttnTensor, ctypes.c_void_p
        i32, f32p = ctypes.c_int, ctypes.c_void_p
        lib.attn_fwd.argtypes = [P, T, T, T, T, f32p, S]
        lib.attn_fwd.restype = i32
        lib.attn_bwd_workspace_size.argtypes = [P]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd.argtypes = [P, T, T, T, T, T, f32p, T, T, T, ctypes.c_void_p,
                                 ctypes.c_size_t, S]
        lib.attn_bwd.restype = i32
        lib.attn_merge_lse.argtypes = [i32, i32, i32, i32, i32, T, f32p, T, f32p, T, f32p, S]
        lib.attn_merge_lse.restype = i32
        lib.attn_bwd_dlse.argtypes = [P, T, T, T, T, T, f32p, f32p, T, T, T, ctypes.c_void_p,
                                      ctypes.c_size_t, S]
        lib.attn_bwd_dlse.restype = i32
        lib.attn_merge_lse_bwd.argtypes = [i32, i32, i32, i32, i32, T, f32p, T, f32p, T, f32p,
                                           T, f32p, T, f32p, S]
        lib.attn_merge_lse_bwd.restype = i32
        lib.attn_thd_partitioned_indices.argtypes = [ctypes.c_void_p, i32, i32, i32, i32,
                                                     ctypes.c_void_p, S]
        lib.attn_thd_partitioned_indices.restype = i32
        lib.attn_thd_accumulate.argtypes = [i32, i32, i32, i32, T, f32p, i32, ctypes.c_void_p,
                                            ctypes.c_void_p, i32, S]
        lib.attn_thd_accumulate.restype = i32
        lib.attn_thd_store.argtypes = [i32, i32, i32, i32, f32p, T, ctypes.c_void_p, ctypes.c_void_p, i32, S]
        lib.attn_thd_store.restype = i32
        lib.attn_last_error_string.argtypes = []
        lib.attn_last_error_string.restype = ctypes.c_char_p
        lib.attn_check_device_error.argtypes = [S]
        lib.attn_check_device_error.restype = i32
        lib.attn_set_watchdog_ns.argtypes = [ctypes.c_uint64]
        lib.attn_set_watchdog_ns.restype = ctypes.c_uint64
        lib.attn_watchdog_selftest.argtypes = [S]
        lib.attn_watchdog_selftest.restype = i32
        lib.attn_profile_begin.argtypes = [i32]
        lib.attn_profile_begin.restype = i32
        lib.attn_profile_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i32]
        lib.attn_profile_read.restype = i32
        lib.attn_bwd_noalloc.argtypes = [P, T, T, T, T, T, f32p, T, T, T, S]
        lib.attn_bwd_noalloc.restype = i32
        _lib = lib
        return lib


def check(status: int):
    if status != ATTN_OK:
        msg = load().attn_last_error_string()
        raise AttnError(status, msg.decode() if msg else "")
