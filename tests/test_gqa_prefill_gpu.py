"""Parity of the tensor-core grouped-head kernel (chosen automatically for KV heads
with many query rows: prefill-sized s, or large groups; forced here) against the
fp64 oracle, through the C ABI.
Row blocks of 128 rows span head boundaries when s < 128 (row = head_in_group * s +
token), so the causal window differs from row to row inside a block."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import assert_lse_close, assert_out_close, f64, gqa_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da

    da.set_forced_splits(0)
    da.set_grouped_kernel(2)  # the tensor-core kernel for every shape here, whatever the grid size
    yield
    da.set_grouped_kernel(0)
    da.set_forced_splits(0)


def run(b, hq, hkv, d, s, seqlens, paged=False, seed=0, poison=False, nsplit=0):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, seed=seed, device=DEV)
    if poison:  # rows past each sequence's end hold NaN: never read
        if paged:
            table = cache.block_table.cpu().numpy()
            for i, L in enumerate(seqlens):
                n = (L + 63) // 64
                if n and L % 64:
                    last = int(table[i, n - 1])
                    cache.k[last, L % 64:] = float("nan")
                    cache.v[last, L % 64:] = float("nan")
        else:
            for i, L in enumerate(seqlens):
                cache.k[i, L:] = float("nan")
                cache.v[i, L:] = float("nan")
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    da.set_forced_splits(nsplit)
    try:
        out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(max(seqlens), 1),
                                 block_table=cache.block_table if paged else None)
        torch.cuda.synchronize()
        if nsplit:  # chunks are whole 64-key pages: ceil(L / n) rounded up to 64
            L = max(seqlens)
            chunk = -(-(-(-L // nsplit)) // 64) * 64
            assert da.last_num_splits() == -(-L // chunk)
    finally:
        da.set_forced_splits(0)
    assert da.check_errors() == 0
    return q, cache, out, lse


def check(q, cache, out, lse, seqlens, d, what):
    b = q.shape[0]
    ks = [gqa_rows(cache, i, "k") for i in range(b)]
    vs = [gqa_rows(cache, i, "v") for i in range(b)]
    ro, rl = A.gqa_ref(f64(q), ks, vs, seqlens, 1 / math.sqrt(d))
    assert_out_close(f64(out), ro, what)
    assert_lse_close(f64(lse), rl, what + " lse")


@pytest.mark.parametrize("b,hq,hkv,s,seqlens,paged", [
    (2, 8, 2, 32, [300, 95], False),         # 128 rows per KV head: 4 heads x 32 tokens in one block
    (2, 8, 8, 1, [500, 64], False),          # one row per KV head (decode): 127 idle rows per block
    (1, 4, 4, 100, [450], False),            # MHA, 100 rows: a block with a ragged end
    (3, 2, 1, 64, [64, 500, 0], True),       # one sequence all new tokens, one empty; paged
    (2, 16, 1, 16, [257, 1000], True),       # 256 rows: two blocks, each spanning 8 heads
    (1, 1, 1, 300, [700], False),            # three blocks of one head, causal across them
])
def test_prefill_vs_oracle(b, hq, hkv, s, seqlens, paged):
    q, cache, out, lse = run(b, hq, hkv, 128, s, seqlens, paged=paged, seed=s + b)
    check(q, cache, out, lse, seqlens, 128, f"prefill b{b} hq{hq} hkv{hkv} s{s}")


@pytest.mark.parametrize("nsplit", [1, 3, 7])
def test_prefill_context_split(nsplit):
    # the context cut into chunks (one CTA each), partials merged by the combine kernel;
    # chunks past a row block's causal window carry LSE = -inf
    seqlens = [700, 300]
    q, cache, out, lse = run(2, 8, 2, 128, 32, seqlens, seed=17, nsplit=nsplit)
    check(q, cache, out, lse, seqlens, 128, f"prefill split {nsplit}")


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_mqa_d256(paged):
    # 24 query heads on one KV head, d = 256 (the ragged MQA geometry, shorter contexts)
    seqlens = [1500, 700, 64]
    q, cache, out, lse = run(3, 24, 1, 256, 1, seqlens, paged=paged, seed=23)
    check(q, cache, out, lse, seqlens, 256, f"prefill MQA d256 paged={paged}")


@pytest.mark.parametrize("hq,hkv,d,s,seqlens", [
    (8, 2, 128, 32, [900, 300]),      # 128 rows per KV head
    (24, 1, 256, 1, [2000, 333]),     # 24-row MQA, d = 256
])
def test_both_grouped_kernels_agree(hq, hkv, d, s, seqlens):
    # automatic choice, the split-KV kernels and the tensor-core kernel: the same result
    # within rounding on the same inputs
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(2, hq, hkv, d, s, seqlens, seed=29, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    res = {}
    for mode in (0, 1, 2):
        da.set_grouped_kernel(mode)
        res[mode] = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens))
    da.set_grouped_kernel(2)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    for mode in (0, 1):
        assert_out_close(f64(res[mode][0]), f64(res[2][0]), f"mode {mode} vs 2", max_abs=1e-2, mean_abs=1e-3)
        np.testing.assert_allclose(f64(res[mode][1]), f64(res[2][1]), atol=2e-4, rtol=0)


def test_prefill_sharp_softmax():
    # queries x 8: peaked rows, where the reference maximum moves and O is rescaled
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [600, 300]
    q, cache = W.make_gqa(2, 4, 2, 128, 40, seqlens, seed=9, device=DEV, q_std=8.0)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=600)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    check(q, cache, out, lse, seqlens, 128, "prefill sharp")


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_nan_past_the_end(paged):
    seqlens = [333, 130]
    q, cache, out, lse = run(2, 8, 2, 128, 32, seqlens, paged=paged, seed=7, poison=True)
    assert torch.isfinite(out).all()
    check(q, cache, out, lse, seqlens, 128, f"prefill poisoned paged={paged}")


def test_prefill_paged_equals_contiguous_bitwise():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [300, 77, 129]
    q, cache, out_p, lse_p = run(3, 8, 2, 128, 32, seqlens, paged=True, seed=21)
    cap = max(seqlens)
    k = torch.zeros((3, cap, 2, 128), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros_like(k)
    for i, L in enumerate(seqlens):
        k[i, :L] = torch.from_numpy(gqa_rows(cache, i, "k")).to(DEV, torch.bfloat16)
        v[i, :L] = torch.from_numpy(gqa_rows(cache, i, "v")).to(DEV, torch.bfloat16)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out_c, lse_c = da.gqa_decode(q, k, v, sl, max_seqlen=cap)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)


def test_prefill_forced_timeout():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [400, 200]
    q, cache = W.make_gqa(2, 8, 2, 128, 32, seqlens, seed=5, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    assert da.check_errors() == 0
    da.test_force_timeout(True)
    try:
        da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=400)
        rc = da.check_errors()
    finally:
        da.test_force_timeout(False)
    assert rc == 5  # DECATTN_ERR_TIMEOUT
    out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=400)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    check(q, cache, out, lse, seqlens, 128, "after timeout")


def test_prefill_balanced_pieces_ragged():
    # fewer work items than SMs: each item is cut into near-equal pieces planned on the
    # device from the actual lengths (empty, one-key and sub-tile sequences included), the
    # pieces of an item merged by the balanced combine; the plan depends on the lengths only
    import decode_attention_18_b300 as da

    seqlens = [5000, 0, 64, 1, 3100, 777]
    q, cache, out, lse = run(6, 24, 1, 256, 1, seqlens, paged=True, seed=41)
    assert da.last_num_splits() == 0
    check(q, cache, out, lse, seqlens, 256, "prefill balanced ragged")
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out2, lse2 = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens), block_table=cache.block_table)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_prefill_many_items_fixed_chunks():
    # at least as many work items (sequence, KV head, row block) as SMs: chunks planned from
    # max_seqlen instead of the balanced pieces
    import decode_attention_18_b300 as da

    seqlens = [(i * 331) % 900 + 70 for i in range(40)]
    q, cache, out, lse = run(40, 16, 4, 128, 8, seqlens, seed=43)  # 32 rows per KV head, 160 items
    assert da.last_num_splits() >= 1
    check(q, cache, out, lse, seqlens, 128, "prefill fixed chunks, 160 items")
