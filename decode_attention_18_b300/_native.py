"""ctypes declarations of the C ABI in include/decattn.h.

Loading is lazy: the library is opened on the first call. A missing library
raises at that point; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdecattn.so")

# every symbol the header declares
SYMBOLS = (
    "decattn_status_string",
    "gqa_decode_workspace_size",
    "gqa_decode",
    "mla_absorb_q",
    "mla_decode_workspace_size",
    "mla_decode",
    "mla_out_proj",
    "decattn_check_errors",
    "decattn_set_wait_limit_ns",
    "decattn_set_forced_splits",
    "decattn_last_num_splits",
    "decattn_test_force_timeout",
    "gqa_decode_no_alloc",
    "gqa_decode_dv_workspace_size",
    "gqa_decode_dv",
    "mla_decompress_kv",
    "attn_merge_lse",
    "gqa_decode_fp8_workspace_size",
    "gqa_decode_fp8",
    "decattn_set_grouped_kernel",
)


class DecAttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status) if _lib is not None else f"status {status}"
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")


class KV(ctypes.Structure):
    _fields_ = [
        ("paged", ctypes.c_int),
        ("capacity", ctypes.c_int),
        ("block_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
    ]


_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
SZ = ctypes.c_size_t


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"native library {LIB_PATH} is not built; run decode_attention_18_b300.build")
    lib = ctypes.CDLL(LIB_PATH)
    lib.decattn_status_string.restype = ctypes.c_char_p
    lib.decattn_status_string.argtypes = [I]
    lib.gqa_decode_workspace_size.restype = SZ
    lib.gqa_decode_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.gqa_decode.restype = I
    lib.gqa_decode.argtypes = [P, P, P, KV, P, I, I, I, I, I, I, F, P, P, P, SZ, P]
    lib.mla_absorb_q.restype = I
    lib.mla_absorb_q.argtypes = [P, P, P, P, I, I, I, I, I, F, P]
    lib.mla_decode_workspace_size.restype = SZ
    lib.mla_decode_workspace_size.argtypes = [I, I, I, I, I]
    lib.mla_decode.restype = I
    lib.mla_decode.argtypes = [P, P, P, P, KV, P, I, I, I, I, I, I, F, P, P, P, SZ, P]
    lib.mla_out_proj.restype = I
    lib.mla_out_proj.argtypes = [P, P, P, P, I, I, I, I, I, F, P]
    lib.decattn_check_errors.restype = I
    lib.decattn_check_errors.argtypes = [P]
    lib.decattn_set_wait_limit_ns.restype = None
    lib.decattn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.decattn_set_forced_splits.restype = None
    lib.decattn_set_forced_splits.argtypes = [I]
    lib.decattn_last_num_splits.restype = I
    lib.decattn_last_num_splits.argtypes = []
    lib.decattn_test_force_timeout.restype = None
    lib.decattn_test_force_timeout.argtypes = [I]
    lib.gqa_decode_no_alloc.restype = I
    lib.gqa_decode_no_alloc.argtypes = [P, P, P, KV, P, I, I, I, I, I, I, F, P, P, P]
    lib.gqa_decode_dv_workspace_size.restype = SZ
    lib.gqa_decode_dv_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.gqa_decode_dv.restype = I
    lib.gqa_decode_dv.argtypes = [P, P, P, KV, P, I, I, I, I, I, I, I, F, P, P, P, SZ, P]
    lib.mla_decompress_kv.restype = I
    lib.mla_decompress_kv.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    lib.attn_merge_lse.restype = I
    lib.attn_merge_lse.argtypes = [P, P, P, P, I, I, P, P, P]
    lib.gqa_decode_fp8_workspace_size.restype = SZ
    lib.gqa_decode_fp8_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.gqa_decode_fp8.restype = I
    lib.gqa_decode_fp8.argtypes = [P, P, P, KV, P, I, I, I, I, I, I, F, F, F, P, P, P, SZ, P]
    lib.decattn_set_grouped_kernel.restype = None
    lib.decattn_set_grouped_kernel.argtypes = [I]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().decattn_status_string(int(status)).decode()


def check(status: int, what: str = ""):
    if status != 0:
        raise DecAttnError(status, what)
