"""Parity of grouped-head decode over an FP8 (E4M3) cache against the fp64
oracle (oracle.gqa_fp8_ref: gqa_ref on k_scale * K8 and v_scale * V8), through
the C ABI. Both kernels widen each cache tile exactly (to f16 for 128- and
256-wide rows, where the MMAs run in f16; to bf16 at d = 64), so the usual
output and LSE tolerances apply. The checker reads the cache bytes itself (a
paged pool through the oracle's gather_paged)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import assert_lse_close, assert_out_close, f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da

    da.set_forced_splits(0)
    yield
    da.set_forced_splits(0)


def make(b, hq, hkv, d, s, seqlens, paged=False, seed=0):
    from decode_attention_18_b300 import workloads as W

    return W.make_gqa_fp8(b, hq, hkv, d, s, seqlens, paged=paged, seed=seed, device=DEV)


def byte_rows(t, cache, i, kv_head=None):
    """Cache bytes [L, Hkv, d] of sequence i in logical order (uint8, checker side)."""
    L = cache.seqlens[i]
    if not cache.paged:
        x = t[i, :L]
        return (x if kv_head is None else x[:, kv_head:kv_head + 1]).cpu().numpy()
    if L == 0:  # an empty sequence owns no page
        x = t[0, :0]
        return (x if kv_head is None else x[:, kv_head:kv_head + 1]).cpu().numpy()
    table = cache.block_table[i].cpu().numpy()
    n = (L + 63) // 64
    pages = {int(table[j]): t[int(table[j])].cpu().numpy() for j in range(n)}
    rows = A.gather_paged(pages, table, L, 64)
    return rows if kv_head is None else rows[:, kv_head:kv_head + 1]


def run(q, cache, ks, vs, seqlens, d):
    import decode_attention_18_b300 as da

    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode_fp8(q, cache.k, cache.v, sl, k_scale=ks, v_scale=vs, max_seqlen=max(seqlens),
                                 block_table=cache.block_table if cache.paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    return out, lse


def check(q, cache, ks, vs, out, lse, seqlens, d, what):
    b = q.shape[0]
    k8 = [byte_rows(cache.k, cache, i) for i in range(b)]
    v8 = [byte_rows(cache.v, cache, i) for i in range(b)]
    ro, rl = A.gqa_fp8_ref(f64(q), k8, v8, seqlens, 1 / math.sqrt(d), ks, vs)
    assert_out_close(f64(out), ro, what)
    assert_lse_close(f64(lse), rl, what + " lse")


@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens,paged", [
    (2, 8, 2, 128, 1, [200, 77], False),     # GQA, ragged, several tiles + tail
    (2, 8, 8, 64, 1, [130, 64], True),       # MHA, paged
    (1, 24, 1, 256, 1, [333], True),         # MQA d = 256 (24 rows per KV head: two m-tiles)
    (2, 16, 2, 128, 4, [300, 97], False),    # causal s = 4, 32 rows per KV head
    (3, 8, 1, 64, 2, [0, 2, 65], False),     # an empty sequence and one holding only the new tokens
    (2, 24, 4, 256, 1, [1500, 700], True),   # longer contexts: split / balanced schedule
])
def test_fp8_vs_oracle(b, hq, hkv, d, s, seqlens, paged):
    q, cache, ks, vs = make(b, hq, hkv, d, s, seqlens, paged=paged, seed=d + s)
    out, lse = run(q, cache, ks, vs, seqlens, d)
    check(q, cache, ks, vs, out, lse, seqlens, d, f"fp8 {b},{hq},{hkv},{d},{s}")


@pytest.mark.parametrize("nsplit", [1, 3])
def test_fp8_forced_splits(nsplit):
    import decode_attention_18_b300 as da

    seqlens = [900, 333]
    q, cache, ks, vs = make(2, 8, 2, 128, 1, seqlens, seed=77)
    da.set_forced_splits(nsplit)
    try:
        out, lse = run(q, cache, ks, vs, seqlens, 128)
        assert da.last_num_splits() == nsplit
    finally:
        da.set_forced_splits(0)
    check(q, cache, ks, vs, out, lse, seqlens, 128, f"fp8 splits {nsplit}")


def test_fp8_nan_bytes_past_the_end_are_never_used():
    seqlens = [150, 70]
    q, cache, ks, vs = make(2, 8, 2, 128, 1, seqlens, seed=5)
    out0, lse0 = run(q, cache, ks, vs, seqlens, 128)
    for i, L in enumerate(seqlens):
        cache.k[i, L:] = 0x7F  # E4M3 NaN
        cache.v[i, L:] = 0xFF
    out1, lse1 = run(q, cache, ks, vs, seqlens, 128)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_fp8_paged_equals_contiguous_bitwise():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [300, 77, 129]
    q, cache, ks, vs = make(3, 8, 2, 128, 1, seqlens, paged=True, seed=9)
    out_p, lse_p = run(q, cache, ks, vs, seqlens, 128)
    cap = max(seqlens)
    k = torch.zeros((3, cap, 2, 128), dtype=torch.uint8, device=DEV)
    v = torch.zeros_like(k)
    for i, L in enumerate(seqlens):
        k[i, :L] = torch.from_numpy(byte_rows(cache.k, cache, i)).to(DEV)
        v[i, :L] = torch.from_numpy(byte_rows(cache.v, cache, i)).to(DEV)
    contig = W.KVCache(k, v, seqlens, False, cap)
    out_c, lse_c = run(q, contig, ks, vs, seqlens, 128)
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)


def test_fp8_argument_errors():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300._native import DecAttnError

    q, cache, ks, vs = make(1, 4, 4, 64, 1, [64], seed=1)
    sl = torch.tensor([64], dtype=torch.int32, device=DEV)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(DecAttnError) as e:
            da.gqa_decode_fp8(q, cache.k, cache.v, sl, k_scale=bad, v_scale=vs, max_seqlen=64)
        assert e.value.status == 1
    q2 = torch.zeros((1, 4, 1, 96), dtype=torch.bfloat16, device=DEV)
    k2 = torch.zeros((1, 64, 4, 96), dtype=torch.uint8, device=DEV)
    with pytest.raises(DecAttnError) as e:  # no compiled instance for d = 96
        da.gqa_decode_fp8(q2, k2, k2, sl, k_scale=ks, v_scale=vs, max_seqlen=64)
    assert e.value.status == 2


def test_fp8_full_size_gqa_64_8_sampled():
    # the grouped-head headline shape (b = 32, Hq = 64, Hkv = 8, d = 128, 4096 keys) in FP8
    seqlens = [4096] * 32
    q, cache, ks, vs = make(32, 64, 8, 128, 1, seqlens, seed=0)
    out, lse = run(q, cache, ks, vs, seqlens, 128)
    rng = np.random.default_rng(3)
    G = 8
    for i, g in zip(rng.integers(0, 32, 4), rng.integers(0, 8, 4)):
        heads = slice(g * G, (g + 1) * G)
        k8 = byte_rows(cache.k, cache, i, kv_head=g)
        v8 = byte_rows(cache.v, cache, i, kv_head=g)
        ro, rl = A.gqa_fp8_ref(f64(q[i:i + 1, heads]), [k8], [v8], [4096], 1 / math.sqrt(128), ks, vs)
        assert_out_close(f64(out[i:i + 1, heads]), ro, f"seq {i} kv head {g}")
        assert_lse_close(f64(lse[i:i + 1, heads]), rl, f"seq {i} kv head {g} lse")


@pytest.mark.parametrize("hq,hkv,d,s,seqlens,paged,nsplit", [
    (24, 1, 256, 1, [1500, 333, 0, 64], True, 0),   # ragged MQA with an empty sequence: balanced pieces
    (16, 2, 128, 4, [700, 65], False, 0),           # 32 rows per KV head, causal s = 4
    (8, 8, 128, 16, [300, 129], True, 0),           # 16 rows per KV head, paged
    (24, 1, 256, 1, [1000, 700], False, 3),         # forced chunks: fixed split and its combine
])
def test_fp8_tensor_core_kernel(hq, hkv, d, s, seqlens, paged, nsplit):
    # the tensor-core kernel over an FP8 cache: E4M3 tiles land by TMA, two warps widen
    # them to f16, and the score and P V MMAs run in f16
    import decode_attention_18_b300 as da

    b = len(seqlens)
    q, cache, ks, vs = make(b, hq, hkv, d, s, seqlens, paged=paged, seed=7 + d + s)
    da.set_grouped_kernel(2)
    da.set_forced_splits(nsplit)
    try:
        out, lse = run(q, cache, ks, vs, seqlens, d)
    finally:
        da.set_grouped_kernel(0)
        da.set_forced_splits(0)
    check(q, cache, ks, vs, out, lse, seqlens, d, f"fp8 tensor-core hq{hq} hkv{hkv} d{d} s{s} n{nsplit}")


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_tensor_core_nan_past_the_end(paged):
    # E4M3 NaN bytes (0x7f) in every cache row past each sequence's end: never read into a result
    import decode_attention_18_b300 as da

    seqlens = [333, 130]
    q, cache, ks, vs = make(2, 24, 1, 256, 1, seqlens, paged=paged, seed=31)
    for t in (cache.k, cache.v):
        for i, L in enumerate(seqlens):
            if paged:
                n = (L + 63) // 64
                last = int(cache.block_table[i, n - 1])
                if L % 64:
                    t[last, L % 64:] = 0x7F
            else:
                t[i, L:] = 0x7F
    da.set_grouped_kernel(2)
    try:
        out, lse = run(q, cache, ks, vs, seqlens, 256)
    finally:
        da.set_grouped_kernel(0)
    assert torch.isfinite(out.float()).all()
    check(q, cache, ks, vs, out, lse, seqlens, 256, f"fp8 tensor-core poisoned paged={paged}")
