"""Parity of the grouped-head decode kernels (split + combine, contiguous and
paged) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import gqa_rows, as_device_bf16, assert_lse_close, assert_out_close, f64

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


def run(b, hq, hkv, d, s, seqlens, paged=False, capacity=None, q_std=1.0, seed=0, heads_subset=None):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, capacity=capacity, seed=seed, device=DEV,
                          q_std=q_std)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens),
                             block_table=cache.block_table if paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    return q, cache, out, lse


def check_all(q, cache, out, lse, seqlens, d, what):
    b = q.shape[0]
    ks = [gqa_rows(cache, i, "k") for i in range(b)]
    vs = [gqa_rows(cache, i, "v") for i in range(b)]
    ro, rl = A.gqa_ref(f64(q), ks, vs, seqlens, 1 / math.sqrt(d))
    assert_out_close(f64(out), ro, what)
    assert_lse_close(f64(lse), rl, what)


def check_sampled(q, cache, out, lse, seqlens, d, seqs, kv_heads):
    """Oracle on selected (sequence, KV head) pairs only: the G query heads of
    each KV head against that head's keys and values."""
    hq = q.shape[1]
    hkv = cache.k.shape[2]
    G = hq // hkv
    for i in seqs:
        for g in kv_heads:
            heads = slice(g * G, (g + 1) * G)
            K = gqa_rows(cache, i, "k", kv_head=g)
            V = gqa_rows(cache, i, "v", kv_head=g)
            ro, rl = A.gqa_ref(f64(q[i:i + 1, heads]), [K], [V], [seqlens[i]], 1 / math.sqrt(d))
            assert_out_close(f64(out[i:i + 1, heads]), ro, f"seq {i} kv head {g}")
            assert_lse_close(f64(lse[i:i + 1, heads]), rl, f"seq {i} kv head {g}")


@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens", [
    (2, 8, 2, 128, 1, [200, 77]),          # GQA, ragged, several tiles + tail
    (2, 8, 8, 64, 1, [130, 64]),           # MHA
    (2, 8, 1, 128, 1, [65, 63]),           # MQA
    (3, 6, 2, 256, 1, [1, 129, 300]),      # d = 256
    (2, 24, 4, 256, 1, [500, 333]),        # 24 / 4 / 256 geometry
    (2, 24, 1, 256, 1, [257, 190]),        # MQA with 24 rows (two row blocks)
    (2, 8, 2, 128, 3, [100, 50]),          # MTP s = 3, causal
    (1, 16, 2, 64, 32, [300]),             # s = 32: 256 rows per KV head
    (2, 64, 8, 128, 2, [4096, 1000]),      # 64 / 8 geometry, s = 2
    (5, 8, 2, 128, 1, [0, 1, 63, 64, 65]),  # empty and page-boundary lengths
])
def test_contiguous_vs_oracle(b, hq, hkv, d, s, seqlens):
    q, cache, out, lse = run(b, hq, hkv, d, s, seqlens, capacity=max(seqlens) + 7)
    check_all(q, cache, out, lse, seqlens, d, f"b{b} hq{hq} hkv{hkv} d{d} s{s}")


@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens", [
    (3, 8, 2, 128, 1, [200, 77, 64]),
    (2, 24, 24, 256, 1, [700, 129]),
    (2, 24, 1, 256, 2, [1000, 65]),
    (4, 8, 4, 64, 1, [0, 1, 191, 192]),
])
def test_paged_vs_oracle(b, hq, hkv, d, s, seqlens):
    q, cache, out, lse = run(b, hq, hkv, d, s, seqlens, paged=True, seed=5)
    check_all(q, cache, out, lse, seqlens, d, f"paged b{b} hq{hq} hkv{hkv} d{d} s{s}")


def test_sharp_softmax():
    # queries x 8: peaked softmax and near-unit outputs
    seqlens = [300, 1000]
    q, cache, out, lse = run(2, 8, 2, 128, 1, seqlens, q_std=8.0, seed=7)
    check_all(q, cache, out, lse, seqlens, 128, "sharp")
    assert np.sqrt(np.mean(f64(out) ** 2)) > 0.2


def test_paged_equals_contiguous_bitwise():
    import decode_attention_18_b300 as da

    seqlens = [517, 64, 1000]
    q, cache, out, lse = run(3, 16, 4, 128, 1, seqlens, paged=True, seed=11)
    cap = max(seqlens)
    kc = torch.zeros((3, cap, 4, 128), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    for i, L in enumerate(seqlens):
        kc[i, :L] = as_device_bf16(gqa_rows(cache, i, "k"), kc)
        vc[i, :L] = as_device_bf16(gqa_rows(cache, i, "v"), vc)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out2, lse2 = da.gqa_decode(q, kc, vc, sl, max_seqlen=cap)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("nsplit", [1, 2, 7])
def test_split_invariance(nsplit):
    import decode_attention_18_b300 as da

    seqlens = [1500, 800]
    q, cache, out, lse = run(2, 8, 2, 128, 1, seqlens, seed=13)
    da.set_forced_splits(nsplit)
    try:
        sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
        out2, lse2 = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens))
        torch.cuda.synchronize()
        L = max(seqlens)
        chunk = -(-(-(-L // nsplit)) // 64) * 64  # chunks are whole 64-key pages
        assert da.last_num_splits() == -(-L // chunk)
    finally:
        da.set_forced_splits(0)
    a, b2 = f64(out), f64(out2)
    rr = np.sqrt(np.mean((a - b2) ** 2)) / np.sqrt(np.mean(a ** 2))
    assert rr <= 1e-2
    assert np.abs(f64(lse) - f64(lse2)).max() <= 1e-4
    check_all(q, cache, out2, lse2, seqlens, 128, f"nsplit {nsplit}")


# ---------------------------------------------------------------------------
# Balanced schedule: whenever the planner splits the context (and no split count is
# forced) every CTA takes an equal run of key tiles over all (sequence, KV head, row
# block) items laid end to end, cutting items anywhere; cut items are merged by the
# combine kernel, whole ones are written directly.


@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens", [
    # many items of mixed length, empty sequences, more items than CTAs take whole
    (40, 8, 2, 64, 1, [(i * 977) % 3001 if i % 7 else 0 for i in range(40)]),
    # MQA with 16 query rows per KV head (8 heads x MTP s=2), ragged
    (5, 8, 1, 256, 2, [5000, 0, 2, 777, 4097]),
    # one long sequence among short ones
    (6, 16, 4, 128, 1, [20000, 64, 65, 3, 0, 129]),
])
def test_balanced_schedule_vs_oracle(b, hq, hkv, d, s, seqlens):
    import decode_attention_18_b300 as da

    q, cache, out, lse = run(b, hq, hkv, d, s, seqlens, paged=True, seed=17)
    assert da.last_num_splits() > 1  # the planner split the context: balanced schedule
    check_all(q, cache, out, lse, seqlens, d, f"balanced b{b} hq{hq} hkv{hkv} d{d} s{s}")
    # deterministic: the schedule depends on the lengths only
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out2, lse2 = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens), block_table=cache.block_table)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_balanced_schedule_loose_bound():
    # max_seqlen far above the actual lengths: the grid and workspace follow the bound,
    # the split of the work follows the lengths
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [300, 5, 1200]
    q, cache = W.make_gqa(3, 8, 2, 128, 1, seqlens, capacity=40000, seed=19, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=40000)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    check_all(q, cache, out, lse, seqlens, 128, "loose bound")


def test_full_size_gqa_64_8_sampled():
    # b=32, Hq=64, Hkv=8, d=128, t=4096: the grouped-head workload at full size
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS["gqa_64_8"]
    seqlens = wl.seqlens()
    q, cache, out, lse = run(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, seed=wl.seed)
    check_sampled(q, cache, out, lse, seqlens, wl.d, seqs=[0, 13, 31], kv_heads=[0, 3, 7])


@pytest.mark.parametrize("hkv", [24, 4, 1])
def test_full_size_paged_ragged_sampled(hkv):
    # b=8, Hq=24, d=256, L ~ U[16384, 32768], 64-token pages in random order
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS[f"gqa_paged_hkv{hkv}"]
    seqlens = wl.seqlens()
    q, cache, out, lse = run(wl.b, wl.heads, wl.hkv, wl.d, wl.s, seqlens, paged=True, seed=wl.seed)
    check_sampled(q, cache, out, lse, seqlens, wl.d, seqs=[0, 7], kv_heads=sorted({0, hkv - 1}))


# ---------------------------------------------------------------------------
# KV heads shared by more than 16 query rows (two m-tiles per CTA, several row blocks)

@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens", [
    (2, 32, 1, 128, 1, [700, 129]),         # MQA, 32 rows, d = 128
    (2, 24, 1, 256, 1, [64, 65]),           # MQA 24 rows, tile boundary
    (2, 8, 1, 256, 3, [300, 40]),           # 24 rows from s = 3 (causal among the new tokens)
    (1, 24, 1, 128, 4, [333]),              # 96 rows: three row blocks
    (6, 24, 2, 256, 1, [0, 1, 63, 64, 65, 1000]),  # empty and page-boundary lengths, 2 KV heads
])
def test_many_rows_per_kv_head_vs_oracle(b, hq, hkv, d, s, seqlens):
    q, cache, out, lse = run(b, hq, hkv, d, s, seqlens, capacity=max(seqlens) + 3, seed=17)
    check_all(q, cache, out, lse, seqlens, d, f"rows b{b} hq{hq} hkv{hkv} d{d} s{s}")
    if 0 in seqlens:
        i = seqlens.index(0)
        assert torch.all(out[i] == 0) and torch.all(torch.isneginf(lse[i]))


def test_many_rows_sharp_and_paged_bitwise():
    import decode_attention_18_b300 as da

    seqlens = [517, 64, 1000]
    q, cache, out, lse = run(3, 24, 1, 256, 1, seqlens, paged=True, seed=19, q_std=8.0)
    check_all(q, cache, out, lse, seqlens, 256, "24-row MQA paged sharp")
    cap = max(seqlens)
    kc = torch.zeros((3, cap, 1, 256), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    for i, L in enumerate(seqlens):
        kc[i, :L] = as_device_bf16(gqa_rows(cache, i, "k"), kc)
        vc[i, :L] = as_device_bf16(gqa_rows(cache, i, "v"), vc)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out2, lse2 = da.gqa_decode(q, kc, vc, sl, max_seqlen=cap)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("nsplit", [1, 3, 8])
def test_many_rows_split_invariance(nsplit):
    import decode_attention_18_b300 as da

    seqlens = [2000, 900]
    q, cache, out, lse = run(2, 24, 1, 256, 1, seqlens, seed=23)
    da.set_forced_splits(nsplit)
    try:
        sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
        out2, lse2 = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens))
        torch.cuda.synchronize()
    finally:
        da.set_forced_splits(0)
    a, b2 = f64(out), f64(out2)
    assert np.sqrt(np.mean((a - b2) ** 2)) / np.sqrt(np.mean(a ** 2)) <= 1e-2
    assert np.abs(f64(lse) - f64(lse2)).max() <= 1e-4
    check_all(q, cache, out2, lse2, seqlens, 256, f"24-row MQA nsplit {nsplit}")


def test_multi_wave_split_grid_then_combine():
    # 24 sequences x 8 KV heads x 7 chunks = 1344 CTAs (several waves), each launched as
    # a programmatic dependent, then the combine over all their partials
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [3000 - 97 * i for i in range(24)]
    q, cache = W.make_gqa(24, 64, 8, 128, 1, seqlens, paged=True, seed=12, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    da.set_forced_splits(7)
    try:
        out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens), block_table=cache.block_table)
        torch.cuda.synchronize()
        assert da.last_num_splits() == 7
    finally:
        da.set_forced_splits(0)
    assert da.check_errors() == 0
    check_sampled(q, cache, out, lse, seqlens, 128, seqs=[0, 11, 23], kv_heads=[0, 5, 7])


def _poison_past_end(tensors, seqlens, paged, block_table):
    """Write NaN into every cache row past each sequence's end (rows a kernel may load
    with a tile but must never let into a result)."""
    for t in tensors:
        for i, L in enumerate(seqlens):
            if not paged:
                t[i, L:] = float("nan")
            elif L % 64:
                t[int(block_table[i, (L - 1) // 64])][L % 64:] = float("nan")


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("nsplit", [0, 3])
@pytest.mark.parametrize("hq,d", [(16, 128), (16, 256), (96, 256)])  # d = 256 with one and two m-tiles
def test_nan_past_the_end_is_never_read(paged, nsplit, hq, d):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [130, 1, 64, 97, 200]
    q, cache = W.make_gqa(5, hq, 4, d, 1, seqlens, paged=paged, capacity=None if paged else 260, seed=13,
                          device=DEV)
    _poison_past_end((cache.k, cache.v), seqlens, paged, cache.block_table)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    da.set_forced_splits(nsplit)
    try:
        out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens),
                                 block_table=cache.block_table if paged else None)
        torch.cuda.synchronize()
    finally:
        da.set_forced_splits(0)
    assert da.check_errors() == 0
    assert torch.isfinite(out.float()).all()
    check_all(q, cache, out, lse, seqlens, d, f"nan past end paged={paged} splits={nsplit} d={d}")
