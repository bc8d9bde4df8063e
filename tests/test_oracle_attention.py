"""Pins of the fp64 attention oracle against things other than itself:
a library routine (torch scaled_dot_product_attention in float64), brute force
with pure-Python loops on tiny inputs, closed-form special cases, and the
algebraic identities the pages state (absorbed MLA == expanded MLA)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A

RNG = np.random.default_rng(1234)


def rand(*shape, std=1.0):
    return RNG.standard_normal(shape) * std


# ---------------------------------------------------------------------------
# library cross-check


def sdpa_gqa(q, k_seqs, v_seqs, seqlens, scale):
    """torch SDPA in float64 with K/V repeated per group and an explicit
    bottom-right causal mask built here; returns (out, lse)."""
    b, hq, s, d = q.shape
    out = np.zeros(q.shape[:3] + (v_seqs[0].shape[-1],))
    lse = np.full((b, hq, s), -np.inf)
    for bi in range(b):
        L = seqlens[bi]
        if L == 0:
            continue
        K = torch.from_numpy(np.ascontiguousarray(k_seqs[bi][:L]))  # [L, hkv, d]
        V = torch.from_numpy(np.ascontiguousarray(v_seqs[bi][:L]))
        G = hq // K.shape[1]
        Kr = K.permute(1, 0, 2).repeat_interleave(G, dim=0)  # [hq, L, d]
        Vr = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        mask = torch.zeros(s, L, dtype=torch.bool)
        for i in range(s):
            mask[i, : L - s + i + 1] = True
        Q = torch.from_numpy(np.ascontiguousarray(q[bi]))
        o = F.scaled_dot_product_attention(Q, Kr, Vr, attn_mask=mask, scale=scale)
        out[bi] = o.numpy()
        logits = torch.einsum("hsd,hld->hsl", Q, Kr) * scale
        logits = logits.masked_fill(~mask, -math.inf)
        lse[bi] = torch.logsumexp(logits, dim=-1).numpy()
    return out, lse


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (6, 1), (12, 3)])
@pytest.mark.parametrize("s", [1, 3])
def test_gqa_vs_sdpa(hq, hkv, s):
    b, d = 3, 16
    seqlens = [5, 17, 33]
    q = rand(b, hq, s, d)
    ks = [rand(L, hkv, d) for L in seqlens]
    vs = [rand(L, hkv, d) for L in seqlens]
    scale = 1 / math.sqrt(d)
    o, l = A.gqa_ref(q, ks, vs, seqlens, scale)
    o2, l2 = sdpa_gqa(q, ks, vs, seqlens, scale)
    np.testing.assert_allclose(o, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l, l2, atol=1e-12, rtol=0)


def test_gqa_brute_force_loops():
    # pure-Python loops, math.exp / math.fsum, on a tiny case
    b, hq, hkv, s, d = 2, 4, 2, 2, 3
    seqlens = [3, 4]
    q = rand(b, hq, s, d)
    ks = [rand(L, hkv, d) for L in seqlens]
    vs = [rand(L, hkv, d) for L in seqlens]
    scale = 0.7
    o, l = A.gqa_ref(q, ks, vs, seqlens, scale)
    for bi in range(b):
        L = seqlens[bi]
        for j in range(hq):
            g = j // (hq // hkv)
            for i in range(s):
                n = L - s + i + 1
                x = [scale * math.fsum(q[bi, j, i, c] * ks[bi][m, g, c] for c in range(d)) for m in range(n)]
                mx = max(x)
                den = math.fsum(math.exp(v - mx) for v in x)
                assert l[bi, j, i] == pytest.approx(mx + math.log(den), abs=1e-13)
                for c in range(d):
                    num = math.fsum(math.exp(x[m] - mx) * vs[bi][m, g, c] for m in range(n))
                    assert o[bi, j, i, c] == pytest.approx(num / den, abs=1e-13)


# ---------------------------------------------------------------------------
# closed-form special cases


def test_single_key_returns_that_value():
    q = rand(1, 4, 1, 8)
    k = [rand(1, 2, 8)]
    v = [rand(1, 2, 8)]
    o, l = A.gqa_ref(q, k, v, [1], 0.5)
    for j in range(4):
        g = j // 2
        np.testing.assert_array_equal(o[0, j, 0], v[0][0, g])
        assert l[0, j, 0] == pytest.approx(0.5 * q[0, j, 0] @ k[0][0, g], abs=1e-14)


def test_identical_keys_give_mean_value():
    L, d = 37, 8
    q = rand(1, 2, 1, d)
    key = rand(d)
    k = [np.tile(key, (L, 1, 1)).reshape(L, 1, d)]
    v = [rand(L, 1, d)]
    o, l = A.gqa_ref(q, k, v, [L], 0.3)
    for j in range(2):
        np.testing.assert_allclose(o[0, j, 0], v[0][:, 0].mean(axis=0), atol=1e-13)
        assert l[0, j, 0] == pytest.approx(0.3 * q[0, j, 0] @ key + math.log(L), abs=1e-12)


def test_contiguous_grouping():
    # value rows of KV head g hold the constant g: query head j must read j // G
    hq, hkv, L, d = 12, 4, 9, 4
    q = rand(1, hq, 1, d)
    k = [rand(L, hkv, d)]
    v = [np.stack([np.full((L, d), float(g)) for g in range(hkv)], axis=1)]
    o, _ = A.gqa_ref(q, k, v, [L], 1.0)
    for j in range(hq):
        np.testing.assert_allclose(o[0, j, 0], np.full(d, float(j // (hq // hkv))), atol=1e-13)


def test_empty_and_invalid_sequences():
    q = rand(2, 2, 2, 4)
    k = [rand(0, 1, 4), rand(5, 1, 4)]
    v = [rand(0, 1, 4), rand(5, 1, 4)]
    o, l = A.gqa_ref(q, k, v, [0, 5], 1.0)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    assert np.all(np.isfinite(l[1]))
    with pytest.raises(ValueError):
        A.gqa_ref(q, [rand(1, 1, 4)], [rand(1, 1, 4)], [1], 1.0)


def test_causal_rows_reduce_to_single_token():
    # token i of s equals a one-token decode over the first L - s + i + 1 keys
    b, hq, hkv, s, d, L = 1, 4, 2, 4, 8, 11
    q = rand(b, hq, s, d)
    k = [rand(L, hkv, d)]
    v = [rand(L, hkv, d)]
    o, l = A.gqa_ref(q, k, v, [L], 0.4)
    for i in range(s):
        n = L - s + i + 1
        o1, l1 = A.gqa_ref(q[:, :, i:i + 1], [k[0][:n]], [v[0][:n]], [n], 0.4)
        np.testing.assert_allclose(o[:, :, i], o1[:, :, 0], atol=1e-14)
        np.testing.assert_allclose(l[:, :, i], l1[:, :, 0], atol=1e-14)


# ---------------------------------------------------------------------------
# split merge and paging


def test_merge_partials_any_partition():
    R, L, d = 5, 40, 6
    q = rand(R, d)
    keys = rand(L, d)
    vals = rand(L, d)
    full_o, full_l = A.attend_rows(q, keys, vals, np.full(R, L), 0.9)
    for cuts in ([0, 40], [0, 13, 40], [0, 1, 2, 39, 40], [0, 7, 7, 30, 40]):
        outs, lses = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, l = A.attend_rows(q, keys[a:b], vals[a:b], np.full(R, b - a), 0.9)
            outs.append(o)
            lses.append(l)
        mo, ml = A.merge_partials_ref(outs, lses)
        np.testing.assert_allclose(mo, full_o, atol=1e-13)
        np.testing.assert_allclose(ml, full_l, atol=1e-13)
    # all empty
    mo, ml = A.merge_partials_ref([np.zeros((R, d))] * 2, [np.full(R, -np.inf)] * 2)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_paged_gather_matches_contiguous():
    L, ps, hkv, d = 150, 64, 2, 4
    contig = rand(L, hkv, d)
    n = 3
    perm = np.array([5, 0, 3])
    pool = rand(6, ps, hkv, d)
    for i in range(n):
        chunk = contig[i * ps:(i + 1) * ps]
        pool[perm[i], :chunk.shape[0]] = chunk
    got = A.gather_paged(pool, perm, L, ps)
    np.testing.assert_array_equal(got, contig)


# ---------------------------------------------------------------------------
# MLA: absorbed == expanded (the absorption identity), expanded == SDPA


def mla_case(b, h, d, k, p, s, seqlens, wstd=None):
    wstd = wstd or 1 / math.sqrt(k)
    q_nope = rand(b, h, s, d)
    q_pe = rand(b, h, s, p)
    zs = [rand(L, k) for L in seqlens]
    kpes = [rand(L, p) for L in seqlens]
    w_uk = rand(h, d, k, std=wstd)
    w_uv = rand(h, k, d, std=wstd)
    return q_nope, q_pe, zs, kpes, w_uk, w_uv


@pytest.mark.parametrize("b,h,d,k,p,s,seqlens", [
    (2, 16, 32, 64, 16, 1, [256, 256]),      # the tiny MLA workload's shapes
    (2, 4, 8, 24, 4, 3, [7, 20]),
    (3, 2, 16, 8, 6, 2, [2, 0, 9]),           # k < d and an empty sequence
])
def test_mla_absorbed_equals_expanded(b, h, d, k, p, s, seqlens):
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(b, h, d, k, p, s, seqlens)
    scale = 1 / math.sqrt(d + p)
    o1, l1, _, _ = A.mla_absorbed_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale)
    o2, l2 = A.mla_expanded_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale)
    np.testing.assert_allclose(o1, o2, atol=1e-10, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-10, rtol=0)


def test_mla_expanded_vs_sdpa():
    b, h, d, k, p, s = 2, 3, 8, 12, 4, 2
    seqlens = [6, 11]
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(b, h, d, k, p, s, seqlens)
    scale = 0.37
    o, l = A.mla_expanded_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale)
    for bi in range(b):
        L = seqlens[bi]
        Z = torch.from_numpy(zs[bi])
        KPE = torch.from_numpy(kpes[bi])
        Wk = torch.from_numpy(w_uk)
        Wv = torch.from_numpy(w_uv)
        K = torch.cat([torch.einsum("lk,hdk->hld", Z, Wk), KPE.expand(h, L, p)], dim=-1)
        V = torch.einsum("lk,hkd->hld", Z, Wv)
        Q = torch.cat([torch.from_numpy(q_nope[bi]), torch.from_numpy(q_pe[bi])], dim=-1)
        mask = torch.zeros(s, L, dtype=torch.bool)
        for i in range(s):
            mask[i, : L - s + i + 1] = True
        ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(o[bi], ref.numpy(), atol=1e-12)
        logits = (Q @ K.transpose(-1, -2) * scale).masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(l[bi], torch.logsumexp(logits, -1).numpy(), atol=1e-12)


def test_mla_decompress_brute_force():
    # every element of the decompressed cache by explicit loops over the latent dims
    rows, h, d, k, p = 3, 2, 3, 4, 2
    z = rand(rows, k)
    kpe = rand(rows, p)
    w_uk = rand(h, d, k)
    w_uv = rand(h, k, d)
    K, V = A.mla_decompress_ref(z, kpe, w_uk, w_uv)
    assert K.shape == (rows, h, d + p) and V.shape == (rows, h, d)
    for m in range(rows):
        for j in range(h):
            for c in range(d):
                kn = sum(z[m, x] * w_uk[j, c, x] for x in range(k))
                vv = sum(z[m, x] * w_uv[j, x, c] for x in range(k))
                assert abs(K[m, j, c] - kn) < 1e-12 and abs(V[m, j, c] - vv) < 1e-12
            for c in range(p):
                assert K[m, j, d + c] == kpe[m, c]
    # any leading row shape: [b, capacity] rows give the same rows
    K2, V2 = A.mla_decompress_ref(z.reshape(1, rows, k), kpe.reshape(1, rows, p), w_uk, w_uv)
    np.testing.assert_array_equal(K2[0], K)
    np.testing.assert_array_equal(V2[0], V)


def test_mla_expanded_is_mha_over_the_decompressed_cache():
    # the expanded form is grouped-head attention with Hkv = Hq = h, keys d + p wide
    # and values d wide, over the decompressed cache: the grouped-head definition
    # (pinned against SDPA above) gives the same result
    b, h, d, k, p, s = 2, 3, 8, 12, 4, 2
    seqlens = [6, 13]
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(b, h, d, k, p, s, seqlens)
    scale = 1 / math.sqrt(d + p)
    o1, l1 = A.mla_expanded_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale)
    ks, vs = zip(*(A.mla_decompress_ref(zs[i], kpes[i], w_uk, w_uv) for i in range(b)))
    q = np.concatenate([q_nope, q_pe], axis=-1)
    o2, l2 = A.gqa_ref(q, ks, vs, seqlens, scale)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("s,seqlens,n_recent", [
    (1, [40, 9], [1, 9]),          # one recent key; all keys recent (no latent part)
    (3, [30, 12], [3, 7]),         # recent part exactly the new tokens; a mixed split
    (2, [25, 25], [13, 24]),
])
def test_mla_split_latent_equals_absorbed(s, seqlens, n_recent):
    # "MLAvar6+ Design": splitting the keys into a latent and a decompressed part and
    # merging the two softmaxes changes nothing but rounding
    b, h, d, k, p = len(seqlens), 3, 8, 12, 4
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(b, h, d, k, p, s, seqlens)
    scale = 1 / math.sqrt(d + p)
    o1, l1, _, _ = A.mla_absorbed_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale)
    o2, l2 = A.mla_split_latent_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, scale, n_recent)
    np.testing.assert_allclose(o2, o1, atol=1e-10, rtol=0)
    np.testing.assert_allclose(l2, l1, atol=1e-10, rtol=0)


def test_mla_split_latent_uses_both_parts():
    # a wrong split (older keys dropped, or the recent part not causal) is caught:
    # perturbing one older key's latent changes the result, and so does the last key
    s, seqlens, n_recent = 2, [20], [5]
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(1, 2, 6, 10, 4, s, seqlens)
    base, _ = A.mla_split_latent_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, 0.4, n_recent)
    for m in (3, 19):
        z2 = [zs[0].copy()]
        z2[0][m] += 1.0
        o, _ = A.mla_split_latent_ref(q_nope, q_pe, z2, kpes, w_uk, w_uv, seqlens, 0.4, n_recent)
        assert np.abs(o - base).max() > 1e-4
    # the last key is seen only by the last new token (causal among the new tokens)
    z3 = [zs[0].copy()]
    z3[0][19] += 1.0
    o, _ = A.mla_split_latent_ref(q_nope, q_pe, z3, kpes, w_uk, w_uv, seqlens, 0.4, n_recent)
    np.testing.assert_array_equal(o[:, :, 0], base[:, :, 0])
    with pytest.raises(ValueError):
        A.mla_split_latent_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, 0.4, [1])  # n < s


def test_mla_rope_part_matters():
    # dropping the q_pe K_pe^T term would change the result: the expanded path
    # carries it in its keys, so the identity above fails without it
    b, h, d, k, p, s = 1, 2, 4, 8, 4, 1
    seqlens = [10]
    q_nope, q_pe, zs, kpes, w_uk, w_uv = mla_case(b, h, d, k, p, s, seqlens)
    o1, _, _, _ = A.mla_absorbed_ref(q_nope, q_pe, zs, kpes, w_uk, w_uv, seqlens, 0.5)
    o2, _, _, _ = A.mla_absorbed_ref(q_nope, np.zeros_like(q_pe), zs, kpes, w_uk, w_uv, seqlens, 0.5)
    assert np.max(np.abs(o1 - o2)) > 1e-3


def test_projection_gemms_brute_force():
    b, h, s, d, k = 2, 3, 2, 4, 5
    q = rand(b, h, s, d)
    w = rand(h, d, k)
    qz = A.mla_absorb_ref(q, w, 0.5)
    o_lat = rand(b, h, s, k)
    wv = rand(h, k, d)
    out = A.mla_out_proj_ref(o_lat, wv, 2.0)
    for bi in range(b):
        for j in range(h):
            for i in range(s):
                for c in range(k):
                    assert qz[bi, j, i, c] == pytest.approx(
                        0.5 * math.fsum(q[bi, j, i, e] * w[j, e, c] for e in range(d)), abs=1e-13)
                for c in range(d):
                    assert out[bi, j, i, c] == pytest.approx(
                        2.0 * math.fsum(o_lat[bi, j, i, e] * wv[j, e, c] for e in range(k)), abs=1e-13)


# ---------------------------------------------------------------------------
# FP8 (E4M3) cache


def test_e4m3_decoding_matches_library_and_hand_values():
    codes = np.arange(256, dtype=np.uint8)
    got = A.e4m3_to_float(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(lib)) and np.isnan(got).sum() == 2
    np.testing.assert_array_equal(got[~np.isnan(got)], lib[~np.isnan(lib)])
    # by hand: 1.0 = 0.0111.000, 448 = 0.1111.110, -1.75 = 1.0111.110, smallest subnormal 2^-9,
    # largest subnormal 7/8 * 2^-6, smallest normal 2^-6
    for code, val in ((0x38, 1.0), (0x7E, 448.0), (0xBE, -1.75), (0x01, 2.0 ** -9), (0x07, 7 / 8 * 2.0 ** -6),
                      (0x08, 2.0 ** -6), (0x00, 0.0)):
        assert A.e4m3_to_float(np.array([code], np.uint8))[0] == val


def test_gqa_fp8_ref_is_gqa_over_the_scaled_values():
    # values exactly representable in E4M3 (encoded by the library), times per-tensor
    # scales: the FP8 reference equals the grouped-head definition on k_scale*K, v_scale*V
    rng = np.random.default_rng(5)
    b, hq, hkv, d, s = 2, 4, 2, 8, 2
    seqlens = [9, 5]
    grid = A.e4m3_to_float(np.arange(0, 0x7F, dtype=np.uint8))  # every finite non-negative value
    def cache(L):
        x = rng.choice(grid, size=(L + 3, hkv, d)) * rng.choice([-1.0, 1.0], size=(L + 3, hkv, d))
        codes = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        codes[L:] = 0x7F  # NaN past the end: never decoded into the result
        return x, codes
    kc = [cache(L) for L in seqlens]
    vc = [cache(L) for L in seqlens]
    q = rand(b, hq, s, d)
    ks_, vs_ = 0.03, 0.7
    o1, l1 = A.gqa_fp8_ref(q, [c for _, c in kc], [c for _, c in vc], seqlens, 0.3, ks_, vs_)
    o2, l2 = A.gqa_ref(q, [ks_ * x[:L] for (x, _), L in zip(kc, seqlens)], [vs_ * x[:L] for (x, _), L in zip(vc, seqlens)],
                       seqlens, 0.3)
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-12, rtol=0)
    # the two scales act on different tensors
    o3, _ = A.gqa_fp8_ref(q, [c for _, c in kc], [c for _, c in vc], seqlens, 0.3, vs_, ks_)
    assert np.abs(o3 - o1).max() > 1e-3

