"""CPU-only checks of the boundary: the native library builds and loads, it
exports every entry point include/decattn.h declares, and host-side argument
checks refuse bad input without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decattn.h")


@pytest.fixture(scope="module")
def lib():
    from decode_attention_18_b300 import build, _native

    build.build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_][a-z0-9_ ]*[\s\*]+([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M | re.I)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("gqa_decode", "mla_absorb_q", "mla_decode", "mla_out_proj"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from decode_attention_18_b300 import _native

    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(_native.SYMBOLS) == set(names)


def test_status_strings(lib):
    for code in range(6):
        s = lib.decattn_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.decattn_status_string(0) == b"ok"


def test_python_binding_refuses_host_tensors():
    import decode_attention_18_b300 as da

    q = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        da.gqa_decode(q, q, q, sl, max_seqlen=1)


def test_no_cpu_fallback_in_product_path():
    # the package must not import the checker anywhere
    pkg = os.path.join(ROOT, "decode_attention_18_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"(?:import|from)\s+(\w+)", src), f


def test_invalid_arguments_rejected_without_launch(lib):
    from decode_attention_18_b300._native import KV

    kv = KV(0, 16, None, 0, 0, 0)
    null = ctypes.c_void_p(0)
    # null pointers and bad head counts are refused before any CUDA call
    assert lib.gqa_decode(null, null, null, kv, null, 16, 1, 1, 8, 3, 128, 1.0, null, null, null, 0, null) == 1
    assert lib.gqa_decode(null, null, null, kv, null, 16, 1, 0, 8, 8, 128, 1.0, null, null, null, 0, null) == 1
    assert lib.gqa_decode(null, null, null, kv, null, 16, 1, 1025, 8, 8, 128, 1.0, null, null, null, 0, null) == 1
    assert lib.mla_decode(null, null, null, null, kv, null, 16, 1, 1, 8, 512, 64, 1.0, null, null, null, 0,
                          null) == 1
    assert lib.mla_absorb_q(null, null, null, null, 1, 1, 8, 128, 512, 1.0, null) == 1
    assert lib.mla_out_proj(null, null, null, null, 1, 1, 8, 512, 128, 1.0, null) == 1
    # b = 0 is a no-op
    assert lib.gqa_decode(null, null, null, kv, null, 0, 0, 1, 8, 8, 128, 1.0, null, null, null, 0, null) == 0


def test_new_entry_points_refuse_bad_arguments_without_launch(lib):
    from decode_attention_18_b300._native import KV

    kv = KV(0, 16, None, 0, 0, 0)
    null = ctypes.c_void_p(0)
    # grouped-head with its own value width: null pointers, bad head counts, s out of range
    assert lib.gqa_decode_dv(null, null, null, kv, null, 16, 1, 1, 8, 8, 192, 128, 1.0, null, null, null, 0,
                             null) == 1
    assert lib.gqa_decode_dv(null, null, null, kv, null, 16, 1, 1, 8, 3, 192, 128, 1.0, null, null, null, 0,
                             null) == 1
    assert lib.gqa_decode_dv(null, null, null, kv, null, 16, 1, 1025, 8, 8, 192, 128, 1.0, null, null, null, 0,
                             null) == 1
    assert lib.gqa_decode_dv(null, null, null, kv, null, 0, 0, 1, 8, 8, 192, 128, 1.0, null, null, null, 0,
                             null) == 0  # b = 0: nothing to do
    # FP8 cache: null pointers; scales that are not finite and positive
    for ks in (1.0, 0.0, -1.0, float("inf"), float("nan")):
        assert lib.gqa_decode_fp8(null, null, null, kv, null, 16, 1, 1, 8, 8, 128, 1.0, ks, 1.0, null, null, null,
                                  0, null) == 1
    # decompression: negative rows, null pointers; zero rows is a no-op
    assert lib.mla_decompress_kv(null, null, null, null, -1, 8, 128, 512, 64, null, null, null) == 1
    assert lib.mla_decompress_kv(null, null, null, null, 64, 8, 128, 512, 64, null, null, null) == 1
    assert lib.mla_decompress_kv(null, null, null, null, 0, 8, 128, 512, 64, null, null, null) == 0
    # LSE merge: a width that is not a multiple of 8, null pointers; zero rows is a no-op
    assert lib.attn_merge_lse(null, null, null, null, 4, 12, null, null, null) == 1
    assert lib.attn_merge_lse(null, null, null, null, 4, 128, null, null, null) == 1
    assert lib.attn_merge_lse(null, null, null, null, 0, 128, null, null, null) == 0


def test_workspace_queries_refuse_bad_shapes(lib):
    assert lib.gqa_decode_dv_workspace_size(1, 1, 8, 3, 192, 128, 64) == 0  # Hq % Hkv != 0
    assert lib.gqa_decode_fp8_workspace_size(0, 1, 8, 8, 128, 64) == 0     # b = 0
    assert lib.mla_decode_workspace_size(1, 0, 8, 512, 64) == 0             # s = 0
