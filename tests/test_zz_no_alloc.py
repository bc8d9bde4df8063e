"""gqa_decode_no_alloc: grouped-head decode for callers that cannot allocate
device memory (an engine whose allocator already holds the GPU's memory, a
plug-in host without a device allocator, a loop that cannot afford
cudaMalloc's synchronisation). It keeps the split partials in a fixed array
inside the library instead of a caller workspace.

Called through the C ABI (ctypes) and compared with gqa_decode, which takes a
caller workspace, on two calls in a row: the second call runs on different
inputs with fewer context chunks, so partials left in the shared array by
the first call must not leak into its result. A shape whose split plan needs
more than the fixed array is refused before anything is launched.

This file is named so that pytest collects it last."""
import ctypes
import math

import pytest
import torch

from tests.helpers import assert_lse_close, assert_out_close, f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SCRATCH_BYTES = 16 << 20  # DECATTN_NO_ALLOC_SCRATCH_BYTES in include/decattn.h
ERR_WORKSPACE = 3


@pytest.fixture(scope="module")
def lib():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import _native

    da.set_forced_splits(0)
    return _native.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _inputs(b, hq, hkv, d, s, seqlens, seed):
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(b, hq, hkv, d, s, seqlens, seed=seed, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    return q, cache, sl


def _call_no_alloc(lib, q, cache, sl, max_seqlen):
    from decode_attention_18_b300._native import KV

    b, hq, s, d = (int(x) for x in q.shape)
    hkv = int(cache.k.shape[2])
    out = torch.empty_like(q)
    lse = torch.empty((b, hq, s), dtype=torch.float32, device=DEV)
    kv = KV(0, int(cache.k.shape[1]), None, 0, 0, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gqa_decode_no_alloc(_p(q), _p(cache.k), _p(cache.v), kv, _p(sl), max_seqlen, b, s, hq, hkv, d,
                                 1.0 / math.sqrt(d), _p(out), _p(lse), stream)
    return rc, out, lse


def _call_with_workspace(q, cache, sl, max_seqlen):
    import decode_attention_18_b300 as da

    return da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max_seqlen)


def test_matches_gqa_decode_on_two_calls_in_a_row(lib):
    import decode_attention_18_b300 as da

    cases = [
        # (b, Hq, Hkv, d, s, seqlens, seed): both need several context chunks
        (3, 16, 2, 128, 2, [3000, 1500, 257], 11),
        (2, 16, 2, 128, 2, [700, 90], 12),
    ]
    for b, hq, hkv, d, s, seqlens, seed in cases:
        L = max(seqlens)
        need = lib.gqa_decode_workspace_size(b, s, hq, hkv, d, L)
        assert 0 < need <= SCRATCH_BYTES  # the fixed array is really used
        q, cache, sl = _inputs(b, hq, hkv, d, s, seqlens, seed)
        ref_out, ref_lse = _call_with_workspace(q, cache, sl, L)
        rc, out, lse = _call_no_alloc(lib, q, cache, sl, L)
        assert rc == 0, lib.decattn_status_string(rc)
        torch.cuda.synchronize()
        assert da.check_errors() == 0
        assert_out_close(f64(out), f64(ref_out), f"no-alloc vs gqa_decode {seqlens}")
        assert_lse_close(f64(lse), f64(ref_lse), f"no-alloc vs gqa_decode {seqlens} lse")


def test_refuses_shapes_beyond_the_fixed_array(lib):
    # b=64, Hq=256, Hkv=8 (32 query rows per KV head), d=256 at 64k context: the
    # split partials need more than 16 MiB, so the call returns DECATTN_ERR_WORKSPACE
    # and launches nothing (the small tensors below are never touched).
    b, hq, hkv, d, s, L = 64, 256, 8, 256, 1, 65536
    assert lib.gqa_decode_workspace_size(b, s, hq, hkv, d, L) > SCRATCH_BYTES
    q = torch.zeros((1, hq, s, d), dtype=torch.bfloat16, device=DEV)
    kv_t = torch.zeros((1, 1, hkv, d), dtype=torch.bfloat16, device=DEV)
    sl = torch.zeros((b,), dtype=torch.int32, device=DEV)
    out = torch.zeros_like(q)
    from decode_attention_18_b300._native import KV

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gqa_decode_no_alloc(_p(q), _p(kv_t), _p(kv_t), KV(0, L, None, 0, 0, 0), _p(sl), L, b, s, hq, hkv, d,
                                 1.0, _p(out), ctypes.c_void_p(0), stream)
    assert rc == ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0)
