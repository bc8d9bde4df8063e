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
