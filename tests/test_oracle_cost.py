"""Pins of the analytic counter against the numbers the pages print
(tests/golden/pages_numbers.json, each entry cited)."""
import json
import os

import pytest

from oracle import cost

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))
GIB = 1 << 30
KIB = 1 << 10


def test_ridge_points():
    for row in GOLD["ridge_points"]["rows"]:
        r = cost.ridge_point(row["peak_tflops"] * 1e12, row["bw_tbs"] * 1e12)
        assert round(r) == row["ridge"], row


def test_flashattention_ai():
    g = GOLD["fa_ai"]
    sh = g["shape"]
    assert 2 * sh["d"] + sh["p"] == g["flops_per_bhst_over_2"]
    for row in g["rows"]:
        f = cost.fa_flops(1, sh["h"], row["s"], sh["t"], sh["d"], sh["p"])
        by = cost.fa_bytes(1, sh["h"], row["s"], sh["t"], sh["d"], sh["p"])
        ai = cost.arithmetic_intensity(f, by)
        assert round(ai) == row["ai"], (row, ai)
    # s = 1024: s t / (s + t) exactly
    ai = cost.fa_flops(1, 128, 1024, 4096, 128, 64) / cost.fa_bytes(1, 128, 1024, 4096, 128, 64)
    assert ai == pytest.approx(1024 * 4096 / 5120, rel=1e-15)


def test_flashmla_ai_and_ratio():
    g = GOLD["mla_ai"]
    sh = g["shape"]
    assert 2 * sh["k"] + sh["p"] == g["flops_per_bhst_over_2"]
    for row in g["rows"]:
        for b in (1, 32, 64):  # batch cancels
            ai = cost.mla_flops(b, sh["h"], row["s"], sh["t"], sh["k"], sh["p"]) / \
                cost.mla_bytes(b, sh["h"], row["s"], sh["t"], sh["k"], sh["p"])
            assert round(ai) == row["ai"], (b, ai)
    ratio = cost.mla_flops(1, 128, 1, 4096, 512, 64) / cost.fa_flops(1, 128, 1, 4096, 128, 64)
    assert round(ratio, 1) == g["flops_ratio_vs_fa"]


def test_mla_asymptote_and_constant():
    # the t -> infinity limit of the absorbed-MLA intensity is h (2k + p) / (k + p)
    h, k, p = 128, 512, 64
    big_t = cost.mla_flops(1, h, 1, 10**9, k, p) / cost.mla_bytes(1, h, 1, 10**9, k, p)
    assert round(big_t) == GOLD["mla_ai_asymptote"]["ai"]
    const = big_t / h
    g = GOLD["summary_table"]
    assert g["mla_constant_lo"] < const < g["mla_constant_hi"]


def test_grouped_head_ai_summary_rows():
    # MHA -> 1, GQA -> Hq/Hkv, MQA -> Hq for long contexts; independent of d and t
    for d in (64, 128, 256):
        for t in (1 << 16, 1 << 20):
            for hq, hkv in ((64, 64), (64, 8), (24, 4), (24, 1)):
                ai = cost.gqa_flops(1, hq, 1, t, d) / cost.gqa_bytes(1, hq, hkv, 1, t, d)
                assert ai == pytest.approx(hq / hkv, rel=hq / t * 2)


def test_gqa_is_fa_with_p0_for_mha():
    # with Hkv = Hq and p = 0 the grouped-head count equals the FlashAttention count
    assert cost.gqa_flops(3, 16, 2, 100, 64) == cost.fa_flops(3, 16, 2, 100, 64, 0)
    assert cost.gqa_bytes(3, 16, 16, 2, 100, 64) == cost.fa_bytes(3, 16, 2, 100, 64, 0)


def test_split_latent_interpolates():
    # n = 0: latent-only; o = 0: decompressed-only ("MLAvar6+ Design" interpolation)
    b, h, s, d, p, k, t = 2, 128, 4, 128, 64, 512, 4096
    f_lat = cost.split_latent_flops(b, h, s, t, 0, d, p, k)
    assert f_lat == cost.mla_flops(b, h, s, t, k, p)
    f_dec = cost.split_latent_flops(b, h, s, 0, t, d, p, k)
    assert f_dec == cost.fa_flops(b, h, s, t, d, p)


def test_kv_accounting_70b():
    g = GOLD["kv_example_70b"]
    mha = cost.kv_bytes_per_token(g["layers"], g["hq"], g["d"])
    gqa = cost.kv_bytes_per_token(g["layers"], 8, g["d"])
    assert mha == g["mha_bytes_per_token"]
    assert gqa == g["gqa8_bytes_per_token"]
    assert cost.kv_cache_bytes(g["tokens"], g["layers"], g["hq"], g["d"]) == g["mha_cache_gib"] * GIB
    assert cost.kv_cache_bytes(g["tokens"], g["layers"], 8, g["d"]) == g["gqa8_cache_gib"] * GIB


def test_kv_accounting_qwen():
    g = GOLD["kv_example_qwen"]
    assert cost.kv_bytes_per_token_layer(g["hq"], g["d"]) == g["mha_kib_per_token_layer"] * KIB
    assert cost.kv_bytes_per_token_layer(g["hkv"], g["d"]) == g["gqa_kib_per_token_layer"] * KIB
    assert cost.kv_bytes_per_token_layer(1, g["d"]) == g["mqa_kib_per_token_layer"] * KIB
    assert cost.kv_bytes_per_token(g["layers"], g["hkv"], g["d"]) == g["gqa_kib_per_token"] * KIB
    assert cost.kv_bytes_per_token(g["layers"], g["hq"], g["d"]) == g["mha_kib_per_token"] * KIB
    assert cost.kv_bytes_per_token(g["layers"], 1, g["d"]) == g["mqa_kib_per_token"] * KIB
    assert cost.kv_cache_bytes(g["tokens"], g["layers"], g["hkv"], g["d"]) == g["gqa_gib_per_seq"] * GIB
    assert cost.kv_cache_bytes(g["tokens"], g["layers"], g["hq"], g["d"]) == g["mha_gib_per_seq"] * GIB
    assert cost.kv_cache_bytes(g["tokens"], g["layers"], 1, g["d"]) == g["mqa_gib_per_seq"] * GIB


def test_rtx5090_ratios():
    g = GOLD["rtx5090_timings_us"]
    assert round(g["s1"]["fa"] / g["s1"]["flashmla"]) == g["claimed_decode_speedup"]
    assert round(100 * (1 - g["s16"]["mlavar6_v3"] / g["s16"]["flashmla"])) == g["claimed_v3_gain_pct"]


def test_exact_counts_reduce_to_formula():
    # s = 1 and equal lengths: the executed count equals the pages' formula
    assert cost.mla_flops_exact(128, 512, 64, [4096] * 3, 1) == cost.mla_flops(3, 128, 1, 4096, 512, 64)
    assert cost.mla_bytes_exact(128, 512, 64, [4096] * 3, 1) == cost.mla_bytes(3, 128, 1, 4096, 512, 64)
    assert cost.gqa_flops_exact(64, 128, [4096] * 2, 1) == cost.gqa_flops(2, 64, 1, 4096, 128)
    assert cost.gqa_bytes_exact(64, 8, 128, [4096] * 2, 1) == cost.gqa_bytes(2, 64, 8, 1, 4096, 128)
    # causal window: token i of s sees L - s + i + 1 keys
    assert cost.causal_keys(10, 3) == 8 + 9 + 10


def test_mtp_crosses_ridge_between_s1_and_s2():
    # with a ridge near 277 FLOP/B, absorbed MLA at t = 4096 sits below it at
    # s = 1 and above it at s = 2 (the MTP tipping point of the pages)
    r = 277.0
    ai1 = cost.mla_flops(1, 128, 1, 4096, 512, 64) / cost.mla_bytes(1, 128, 1, 4096, 512, 64)
    ai2 = cost.mla_flops(1, 128, 2, 4096, 512, 64) / cost.mla_bytes(1, 128, 2, 4096, 512, 64)
    assert ai1 < r < ai2


# ---------------------------------------------------------------------------
# counts pinned against the tensors they describe: bytes are the nbytes of
# arrays of a 2-byte type shaped as the method reads and writes them, FLOPs
# are numpy's own count of the contraction (einsum_path) or a loop count.

W2 = "float16"  # any 2-byte element type stands in for bf16


def _nbytes(*shapes):
    import numpy as np

    return sum(np.zeros(sh, dtype=W2).nbytes for sh in shapes)


def _einsum_flops(spec, *shapes):
    """numpy's naive FLOP count of the contraction. The report prints four
    significant digits, so the shapes are kept small enough to be exact."""
    import numpy as np

    ops = [np.zeros(sh) for sh in shapes]
    report = np.einsum_path(spec, *ops, optimize="optimal")[1]
    for line in report.splitlines():
        if "Naive FLOP count" in line:
            n = float(line.split(":")[1])
            assert n < 1e4, "count too large to be printed exactly"
            return int(round(n))
    raise AssertionError(report)


@pytest.mark.parametrize("b,h,s,din,dout", [(2, 3, 5, 4, 7), (32, 128, 1, 128, 512), (1, 1, 3, 512, 128)])
def test_proj_flops_and_bytes_from_tensors(b, h, s, din, dout):
    # absorb-style GEMM: activations [b,h,s,din] x weights [h,din,dout] -> [b,h,s,dout]
    if 2 * b * h * s * din * dout < 10**4:
        assert cost.proj_flops(b, h, s, din, dout) == _einsum_flops("bhsd,hdk->bhsk", (b, h, s, din), (h, din, dout))
    n_madd = 0
    for _ in range(b * h * s):          # one output row per (sequence, head, token)
        for _ in range(dout):           # each output column
            n_madd += din               # one multiply-add per reduction element
    assert cost.proj_flops(b, h, s, din, dout) == 2 * n_madd
    assert cost.proj_bytes(b, h, s, din, dout) == _nbytes((b, h, s, din), (h, din, dout), (b, h, s, dout))


def test_split_latent_bytes_term_by_term():
    # "Mla Analysis", Cost Models, MLAvar6+: the nine byte terms are, in order, the
    # tensors the split method moves: q_pe [b,h,s,p], q_nope [b,h,s,d], Qz [b,h,s,k],
    # old latents Z [b,o,k], RoPE keys of all t tokens [b,t,p], decompressed K and V
    # of the n new tokens [b,h,n,d] each, the output [b,h,s,d] and the latent output
    # [b,h,s,k]. Distinct primes make every term identifiable.
    b, h, s, o, n, d, p, k = 2, 3, 5, 7, 11, 13, 17, 19
    t = o + n
    shapes = [(b, h, s, p), (b, h, s, d), (b, h, s, k), (b, o, k), (b, t, p), (b, h, n, d), (b, h, n, d),
              (b, h, s, d), (b, h, s, k)]
    assert cost.split_latent_bytes(b, h, s, o, n, d, p, k) == _nbytes(*shapes)
    b, h, s, o, n, d, p, k = 1, 2, 3, 2, 3, 5, 7, 11  # small enough for exact FLOP reports
    t = o + n
    # FLOPs: RoPE scores over all t keys, scores + values over the n decompressed keys
    # (d each), scores + values over the o latent keys (k each)
    f = (_einsum_flops("bhsp,btp->bhst", (b, h, s, p), (b, t, p))
         + 2 * _einsum_flops("bhsd,bhnd->bhsn", (b, h, s, d), (b, h, n, d))
         + 2 * _einsum_flops("bhsk,bok->bhso", (b, h, s, k), (b, o, k)))
    assert cost.split_latent_flops(b, h, s, o, n, d, p, k) == f


def test_mla_and_fa_counts_from_tensors():
    # FlashMLA bytes: Qz, q_pe in, O_lat out per row; Z and K_pe per cached token
    b, h, s, t, k, p, d = 2, 3, 5, 7, 11, 13, 17
    assert cost.mla_bytes(b, h, s, t, k, p) == _nbytes((b, h, s, k), (b, h, s, p), (b, h, s, k), (b, t, k), (b, t, p))
    b, h, s, t, k, p = 1, 2, 3, 5, 7, 11
    f = (_einsum_flops("bhsk,btk->bhst", (b, h, s, k), (b, t, k)) + _einsum_flops("bhsp,btp->bhst", (b, h, s, p), (b, t, p))
         + _einsum_flops("bhst,btk->bhsk", (b, h, s, t), (b, t, k)))
    assert cost.mla_flops(b, h, s, t, k, p) == f
    b, h, s, t, k, p, d = 1, 2, 3, 5, 7, 11, 13
    # FlashAttention over expanded keys [d + p] and values [d], per head
    assert cost.fa_bytes(b, h, s, t, d, p) == _nbytes((b, h, s, d + p), (b, h, s, d), (b, h, t, d + p), (b, h, t, d))
    d, p = 3, 2
    f = (_einsum_flops("bhsc,bhtc->bhst", (b, h, s, d + p), (b, h, t, d + p))
         + _einsum_flops("bhst,bhtd->bhsd", (b, h, s, t), (b, h, t, d)))
    assert cost.fa_flops(b, h, s, t, d, p) == f


def test_expanded_exact_counts_from_tensors():
    # executed counts of the expanded form, ragged lengths and a causal window: the
    # bytes of the tensors it reads and writes, the FLOPs of its two contractions
    # token by token (each new token i of sequence b sees L_b - s + i + 1 keys)
    h, d, p, s = 3, 5, 2, 2
    seqlens = [4, 7, 0]
    b = len(seqlens)
    nb = _nbytes((b, h, s, d + p), (b, h, s, d)) + sum(_nbytes((L, h, d + p), (L, h, d)) for L in seqlens)
    assert cost.fa_bytes_exact(h, d, p, seqlens, s) == nb
    f = 0
    for L in seqlens:
        for i in range(s):
            n = L - s + i + 1 if L else 0
            if n > 0:
                f += (_einsum_flops("hc,hnc->hn", (h, d + p), (h, n, d + p))
                      + _einsum_flops("hn,hnd->hd", (h, n), (h, n, d)))
    assert cost.fa_flops_exact(h, d, p, seqlens, s) == f
    # equal lengths and s = 1: the pages' formulas
    assert cost.fa_flops_exact(h, d, p, [7] * 4, 1) == cost.fa_flops(4, h, 1, 7, d, p)
    assert cost.fa_bytes_exact(h, d, p, [7] * 4, 1) == cost.fa_bytes(4, h, 1, 7, d, p)


def test_gqa_fp8_bytes_from_tensors():
    import numpy as np

    hq, hkv, d, s = 6, 2, 8, 3
    seqlens = [5, 0, 9]
    b = len(seqlens)
    q = np.zeros((b, hq, s, d), np.float16)  # bf16-sized query and output rows
    kv = sum(np.zeros((L, hkv, d), np.uint8).nbytes for L in seqlens) * 2
    assert cost.gqa_fp8_bytes_exact(hq, hkv, d, seqlens, s) == 2 * q.nbytes + kv
    # with a two-byte cache it is the bf16 count
    assert cost.gqa_fp8_bytes_exact(hq, hkv, d, seqlens, s, w_cache=2) == cost.gqa_bytes_exact(hq, hkv, d, seqlens, s)


def test_decompress_counts_from_tensors():
    rows, h, d, k, p = 5, 3, 4, 6, 2
    f = (_einsum_flops("mk,hdk->mhd", (rows, k), (h, d, k)) + _einsum_flops("mk,hkd->mhd", (rows, k), (h, k, d)))
    assert cost.decompress_flops(rows, h, d, k) == f
    assert cost.decompress_bytes(rows, h, d, k, p) == _nbytes((rows, k), (rows, p), (h, d, k), (h, k, d),
                                                              (rows, h, d + p), (rows, h, d))


def test_gqa_counts_from_tensors():
    b, hq, hkv, s, t, d = 2, 6, 3, 5, 7, 8
    assert cost.gqa_bytes(b, hq, hkv, s, t, d) == _nbytes((b, hq, s, d), (b, hq, s, d), (b, t, hkv, d), (b, t, hkv, d))
    f = (_einsum_flops("bhsd,bhtd->bhst", (b, hq, s, d), (b, hq, t, d))
         + _einsum_flops("bhst,bhtd->bhsd", (b, hq, s, t), (b, hq, t, d)))
    assert cost.gqa_flops(b, hq, s, t, d) == f


def test_mla_cache_bytes_per_token_layer():
    # "MQA, GQA & MLA" lesson: the MLA cache holds one latent vector plus the decoupled
    # RoPE key per token and layer; DeepSeek-V3 shapes (k = 512, p = 64) -> 1152 bytes
    assert cost.mla_cache_bytes_per_token_layer(512, 64) == _nbytes((512,), (64,)) == 1152
    assert cost.mla_cache_bytes_per_token_layer(64, 16) == _nbytes((1, 64), (1, 16))
    # a grouped-head cache of the same token: K and V of every KV head
    assert cost.kv_bytes_per_token_layer(8, 128) == _nbytes((8, 128), (8, 128))


def test_roofline_time_and_attainable_by_hand():
    # compute-bound: 2e12 FLOP at 1e15 FLOP/s = 2 ms beats 1e9 B at 1e12 B/s = 1 ms
    assert cost.roofline_time(2e12, 1e9, 1e15, 1e12) == pytest.approx(2e-3)
    # memory-bound: 1e12 FLOP (1 ms) vs 3e9 B (3 ms)
    assert cost.roofline_time(1e12, 3e9, 1e15, 1e12) == pytest.approx(3e-3)
    # attainable throughput, H100 row of the ridge table (989.5 TFLOP/s, 3.35 TB/s):
    # AI 1 (FlashAttention decode) -> 3.35 TFLOP/s; AI 819 (s = 1024) -> the 989.5 peak
    assert cost.attainable_flops(1.0, 989.5e12, 3.35e12) == pytest.approx(3.35e12)
    assert cost.attainable_flops(819.0, 989.5e12, 3.35e12) == pytest.approx(989.5e12)
    # at the ridge both limits meet
    r = cost.ridge_point(989.5e12, 3.35e12)
    assert cost.attainable_flops(r, 989.5e12, 3.35e12) == pytest.approx(989.5e12)
    # time and throughput agree: flops / roofline_time == attainable(flops / bytes)
    for fl, by in ((2e12, 1e9), (1e12, 3e9), (5e11, 5e8)):
        assert fl / cost.roofline_time(fl, by, 989.5e12, 3.35e12) == pytest.approx(
            cost.attainable_flops(fl / by, 989.5e12, 3.35e12))
