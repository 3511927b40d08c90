"""ctypes view of libmla.so (the C ABI declared in include/mla.h).

Loading never falls back to anything: if the shared library is missing or does
not export a declared symbol, the caller gets an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_BAD_BLOCK_ID = 3
MLA_ERR_CUDA = 4
MLA_ERR_WORKSPACE = 5
MLA_ERR_TIMEOUT = 6
MLA_ERR_TOO_LARGE = 7
NOALLOC_SCRATCH_BYTES = 32 << 20

KV_BF16 = 0
KV_FP8_E4M3 = 1
OUT_FP32 = 0
OUT_BF16 = 1
PART_CONTEXT = 1
PART_EXTEND = 2
PART_ALL = 3

c_void_p = ctypes.c_void_p
c_int = ctypes.c_int
c_float = ctypes.c_float
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
i32p = ctypes.POINTER(ctypes.c_int32)
u32p = ctypes.POINTER(ctypes.c_uint32)


class Segment(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int32), ("start", ctypes.c_int32), ("len", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("rope_offset", ctypes.c_int64)]


SEGMENT_DTYPE = np.dtype([("req", "<i4"), ("start", "<i4"), ("len", "<i4"), ("reserved", "<i4"),
                          ("rope_offset", "<i8")])
assert SEGMENT_DTYPE.itemsize == ctypes.sizeof(Segment) == 24
segp = ctypes.POINTER(Segment)

# name -> (restype, argtypes); must match include/mla.h
SIGNATURES = {
    "mla_prefill_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int]),
    "mla_prefill_min_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int]),
    "mla_prefill_ctx": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                c_int, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mla_prefill_ctx_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                        i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                        c_int, c_void_p, c_int, c_void_p, c_void_p]),
    "mla_prefill_ctx_fp8w": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                     i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                     c_float, c_int, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mla_kv_b_proj_absmax": (c_int, [c_void_p, c_int, c_void_p, c_void_p]),
    "mla_kv_b_proj_to_e4m3": (c_int, [c_void_p, c_int, c_float, c_void_p, c_void_p]),
    "mla_prefill_absorbed_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int]),
    "mla_prefill_ctx_absorbed": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                         i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                         c_int, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mla_prefill_auto_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int]),
    "mla_prefill_ctx_auto": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                     i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                     c_int, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "mla_prefill_absorbed_fp8_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int]),
    "mla_prefill_ctx_absorbed_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                             i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float,
                                             c_float, c_int, c_void_p, c_int, c_void_p, c_void_p, c_size_t,
                                             c_void_p]),
    "mla_prefill_reuse_workspace_size": (c_size_t, [c_int, i32p, i32p, c_int, segp, c_int, c_int, c_int, i32p, c_int,
                                                    c_void_p]),
    "mla_prefill_reuse": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_int, c_void_p, c_int,
                                  i32p, i32p, c_int, c_int, segp, c_int, c_int, c_void_p, c_float, c_float,
                                  c_int, i32p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                  c_void_p, c_size_t, c_void_p]),
    "mla_get_device_error": (c_int, [c_void_p, c_void_p]),
    "mla_merge_states": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int,
                                 c_void_p]),
    "mla_rope_relocate": (c_int, [c_void_p, c_void_p, c_int64, c_float, c_void_p, c_int, c_int, c_int, c_int,
                                  c_void_p]),
    "mla_gather_latent": (c_int, [c_void_p, c_int, c_float, c_int, c_void_p, c_int, c_int, c_int, c_void_p,
                                  c_void_p, c_void_p]),
    "mla_block_hash": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "mla_block_compare": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "mla_status_string": (ctypes.c_char_p, [c_int]),
    "mla_last_cuda_error": (ctypes.c_char_p, []),
    "mla_launch_count": (ctypes.c_uint64, []),
    "mla_abi_version": (c_int, []),
    "mla_set_kernel_events": (None, [c_void_p, c_void_p]),
    "mla_set_trace": (None, [c_void_p, c_size_t]),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmla.so (once) and binds every declared signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libmla.so not built ({path}); run `python -m mla_prefix_cache_gb300.build` "
                               "or __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)  # AttributeError if the symbol is missing
            fn.restype = res
            fn.argtypes = args
        if lib.mla_abi_version() != 1:
            raise RuntimeError("libmla ABI version mismatch")
        _lib = lib
        return lib


def status_string(st: int) -> str:
    return load().mla_status_string(int(st)).decode()


class MLAError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = int(status)
        detail = load().mla_last_cuda_error().decode() if status == MLA_ERR_CUDA else ""
        super().__init__(f"{call} -> {status_string(status)}{(': ' + detail) if detail else ''}")


def check(call: str, status: int) -> None:
    if status != MLA_OK:
        raise MLAError(call, status)


def i32_host(a) -> tuple:
    """(ctypes pointer, keep-alive array) of a host int32 vector."""
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr.ctypes.data_as(i32p), arr


def segments_host(segments) -> tuple:
    """(ctypes pointer or None, count, keep-alive) from an [S,4] (req, start, len, rope_offset) array."""
    if segments is None:
        return None, 0, None
    s = np.asarray(segments, dtype=np.int64).reshape(-1, 4)
    arr = np.zeros(s.shape[0], dtype=SEGMENT_DTYPE)
    arr["req"], arr["start"], arr["len"], arr["rope_offset"] = s[:, 0], s[:, 1], s[:, 2], s[:, 3]
    if arr.shape[0] == 0:
        return ctypes.cast(arr.ctypes.data, segp), 0, arr
    return arr.ctypes.data_as(segp), int(arr.shape[0]), arr
