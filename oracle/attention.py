"""Plain float64 definitions of decode attention (test infrastructure; see the
package docstring).

Citations name the page and its section:
  [FIGHT]  "Why MLA and MTP Fight Each Other: Attention Through Arithmetic
           Intensity" (blog post), summary table of the four attention forms.
  [SKILL]  "Mla Analysis" skill page: "Absorption Trick (FlashMLA)",
           "Tensor Shapes (DeepSeek-V3 defaults)".
  [QA]     "MHA vs GQA: same inference speed?" Q&A, section 1 "What changes
           between MHA and GQA?".
  [LESSON] "MQA, GQA & MLA" lesson, "01 Concept".

Readings taken where the pages leave a step open:
  * query head j reads KV head j // G with G = Hq / Hkv: contiguous groups,
    as in [LESSON] "24 query heads in 4 groups of 6";
  * seqlens[b] counts every key of sequence b including the s new tokens;
    token i (0-based) of the s new ones sees keys 0 .. L - s + i (a causal
    window aligned to the bottom-right); for s = 1 that is all L keys;
  * the softmax scale multiplies the whole score (both the latent and the
    RoPE part for MLA); LSE is the natural-log log-sum-exp of the scaled
    scores;
  * an empty sequence (L = 0) yields output 0 and LSE = -inf; 0 < L < s is
    invalid;
  * W_uk is stored [h, d, k] and W_uv [h, k, d]: Qz = q_nope W_uk[j] and
    O = O_lat W_uv[j]; the expanded keys are K_j = Z W_uk[j]^T.
Nothing is rounded: inputs are the exact bf16 values widened to float64.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# one row of softmax attention


def attend_rows(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray,
                n_keys: np.ndarray, scale: float):
    """Softmax attention of R query rows over a prefix of L keys each.

    q_rows [R, Dk], keys [L, Dk], values [L, Dv]; row r attends to keys
    0 .. n_keys[r]-1. Returns (out [R, Dv], lse [R]).
    x_m = scale * <q, k_m>;  lse = log sum_m exp(x_m);  out = sum_m exp(x_m - lse) v_m
    (the plain definition of softmax(Q K^T) V, [FIGHT] summary table rows).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    R = q_rows.shape[0]
    out = np.zeros((R, values.shape[1]), dtype=np.float64)
    lse = np.full((R,), -np.inf, dtype=np.float64)
    if keys.shape[0] == 0 or R == 0:
        return out, lse
    logits = scale * (q_rows @ keys.T)  # [R, L]
    for r in range(R):
        n = int(n_keys[r])
        if n <= 0:
            continue
        x = logits[r, :n]
        m = x.max()
        e = np.exp(x - m)
        l = e.sum()
        lse[r] = m + np.log(l)
        out[r] = (e / l) @ values[:n]
    return out, lse


def causal_key_counts(L: int, s: int) -> np.ndarray:
    """Keys seen by each of the s new tokens: L - s + i + 1 for token i."""
    if L == 0:
        return np.zeros(s, dtype=np.int64)
    if L < s:
        raise ValueError(f"sequence holds {L} keys but {s} new tokens")
    return np.array([L - s + i + 1 for i in range(s)], dtype=np.int64)


# ---------------------------------------------------------------------------
# paged cache


def gather_paged(pool: np.ndarray, block_table: np.ndarray, L: int, page_size: int):
    """Token j of the sequence lives in page block_table[j // page_size], row
    j % page_size of the pool [num_pages, page_size, ...]. Returns the first L
    tokens in logical order, so the attention below never sees page order."""
    n_pages = (L + page_size - 1) // page_size
    if n_pages == 0:
        return pool[:0, 0]
    rows = [pool[int(block_table[i])] for i in range(n_pages)]
    return np.concatenate(rows, axis=0)[:L]


# ---------------------------------------------------------------------------
# grouped-head decode: MHA (Hkv = Hq), GQA, MQA (Hkv = 1)


def gqa_ref(q: np.ndarray, k_seqs, v_seqs, seqlens, scale: float):
    """Grouped-head decode attention ([QA] section 1; [FIGHT] table rows MHA,
    GQA, MQA; [LESSON] grouping).

    q [b, Hq, s, d]; k_seqs[b], v_seqs[b]: [L_b, Hkv, d] (cache of sequence b,
    first L_b tokens); seqlens[b] = L_b. Query head j uses KV head j // G.
    Returns out [b, Hq, s, d] and lse [b, Hq, s].
    """
    b, hq, s, d = q.shape
    out = np.zeros((b, hq, s, v_seqs[0].shape[-1] if b else d), dtype=np.float64)
    lse = np.full((b, hq, s), -np.inf, dtype=np.float64)
    for bi in range(b):
        L = int(seqlens[bi])
        counts = causal_key_counts(L, s)
        if L == 0:
            continue
        K = np.asarray(k_seqs[bi][:L], dtype=np.float64)
        V = np.asarray(v_seqs[bi][:L], dtype=np.float64)
        hkv = K.shape[1]
        if hq % hkv:
            raise ValueError("Hq must be a multiple of Hkv")
        G = hq // hkv
        for j in range(hq):
            g = j // G
            o, l = attend_rows(q[bi, j], K[:, g, :], V[:, g, :], counts, scale)
            out[bi, j] = o
            lse[bi, j] = l
    return out, lse


def e4m3_to_float(codes) -> np.ndarray:
    """Values of FP8 E4M3 bytes (the OCP 8-bit floating-point format: bit 7 sign,
    bits 6-3 exponent E with bias 7, bits 2-0 mantissa M; E = 0 is subnormal,
    M/8 * 2^-6; E = 15 with M = 7 is NaN; no infinities; largest value 448)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def gqa_fp8_ref(q, k8_seqs, v8_seqs, seqlens, scale: float, k_scale: float, v_scale: float):
    """Grouped-head decode over an FP8 cache ([LESSON] deployment paragraph: a
    quantised cache): the cached bytes stand for k_scale * K and v_scale * V; the
    attention is gqa_ref on those values (only the first L_b rows are decoded)."""
    ks = [k_scale * e4m3_to_float(np.asarray(k)[:int(L)]) for k, L in zip(k8_seqs, seqlens)]
    vs = [v_scale * e4m3_to_float(np.asarray(v)[:int(L)]) for v, L in zip(v8_seqs, seqlens)]
    return gqa_ref(q, ks, vs, seqlens, scale)


# ---------------------------------------------------------------------------
# absorbed latent MLA ([SKILL] "Absorption Trick (FlashMLA)": scores
# Q K^T = (Q Wk^T) Z^T = Qz Z^T, values softmax(A) V = (softmax(A) Z) Wv; the
# decompression of O_latent is a separate step; the decoupled RoPE key K_pe
# [B, T, P] is shared by all heads, q_pe is [B, H, S, P] ([SKILL] "Tensor
# Shapes"; [LESSON] MLA paragraph).


def mla_absorb_ref(q_nope: np.ndarray, w_uk: np.ndarray, scale_out: float = 1.0):
    """Qz[b, j, i, :] = scale_out * q_nope[b, j, i, :] @ W_uk[j]  (W_uk [h, d, k])."""
    return scale_out * np.einsum("bhsd,hdk->bhsk", np.asarray(q_nope, np.float64),
                                 np.asarray(w_uk, np.float64))


def mla_latent_ref(qz: np.ndarray, q_pe: np.ndarray, z_seqs, kpe_seqs, seqlens, scale: float):
    """Latent attention: x_m = scale (<Qz, Z_m> + <q_pe, K_pe,m>), softmax over
    the causal window, O_lat = sum_m P_m Z_m. qz [b,h,s,k], q_pe [b,h,s,p],
    z_seqs[b] [L_b, k], kpe_seqs[b] [L_b, p]. Returns (O_lat [b,h,s,k], lse [b,h,s])."""
    b, h, s, k = qz.shape
    out = np.zeros((b, h, s, k), dtype=np.float64)
    lse = np.full((b, h, s), -np.inf, dtype=np.float64)
    for bi in range(b):
        L = int(seqlens[bi])
        counts = causal_key_counts(L, s)
        if L == 0:
            continue
        Z = np.asarray(z_seqs[bi][:L], dtype=np.float64)
        KPE = np.asarray(kpe_seqs[bi][:L], dtype=np.float64)
        keys = np.concatenate([Z, KPE], axis=1)  # [L, k + p]
        for j in range(h):
            qrow = np.concatenate([qz[bi, j], q_pe[bi, j]], axis=1)  # [s, k + p]
            o, l = attend_rows(qrow, keys, Z, counts, scale)
            out[bi, j] = o
            lse[bi, j] = l
    return out, lse


def mla_out_proj_ref(o_lat: np.ndarray, w_uv: np.ndarray, scale_out: float = 1.0):
    """O[b, j, i, :] = scale_out * O_lat[b, j, i, :] @ W_uv[j]  (W_uv [h, k, d])."""
    return scale_out * np.einsum("bhsk,hkd->bhsd", np.asarray(o_lat, np.float64),
                                 np.asarray(w_uv, np.float64))


def mla_absorbed_ref(q_nope, q_pe, z_seqs, kpe_seqs, w_uk, w_uv, seqlens, scale):
    """The absorbed pipeline: absorb, latent attention, output projection.
    Returns (out [b,h,s,d], lse [b,h,s], qz, o_lat)."""
    qz = mla_absorb_ref(q_nope, w_uk)
    o_lat, lse = mla_latent_ref(qz, q_pe, z_seqs, kpe_seqs, seqlens, scale)
    return mla_out_proj_ref(o_lat, w_uv), lse, qz, o_lat


def mla_decompress_ref(z, k_pe, w_uk, w_uv):
    """The per-head keys and values a latent cache stands for ([SKILL]
    "Absorption Trick": K = Z Wk, V = Z Wv with the up-projections; "Cost
    Models - FlashAttention": keys of d + p values, values of d).

    z [..., k] and k_pe [..., p] (any leading row shape), W_uk [h, d, k],
    W_uv [h, k, d]. Returns K [..., h, d + p] with K[..., j, :d] = z W_uk[j]^T
    and K[..., j, d:] = k_pe (the RoPE part every head shares), and
    V [..., h, d] with V[..., j, :] = z W_uv[j]."""
    z = np.asarray(z, np.float64)
    kpe = np.asarray(k_pe, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    h = w_uk.shape[0]
    nope = np.einsum("...k,hdk->...hd", z, w_uk)
    rope = np.broadcast_to(kpe[..., None, :], kpe.shape[:-1] + (h, kpe.shape[-1]))
    K = np.concatenate([nope, rope], axis=-1)
    V = np.einsum("...k,hkd->...hd", z, w_uv)
    return K, V


def mla_expanded_ref(q_nope, q_pe, z_seqs, kpe_seqs, w_uk, w_uv, seqlens, scale):
    """Brute force with decompressed per-head keys and values (mla_decompress_ref):
    K_j = [Z W_uk[j]^T | K_pe] (L x (d + p)), V_j = Z W_uv[j] (L x d), query
    [q_nope | q_pe], then plain per-head attention. The expanded form of the
    pages' regime comparison, and the check of the absorbed form."""
    b, h, s, d = q_nope.shape
    out = np.zeros((b, h, s, w_uv.shape[2]), dtype=np.float64)
    lse = np.full((b, h, s), -np.inf, dtype=np.float64)
    for bi in range(b):
        L = int(seqlens[bi])
        counts = causal_key_counts(L, s)
        if L == 0:
            continue
        K, V = mla_decompress_ref(z_seqs[bi][:L], kpe_seqs[bi][:L], w_uk, w_uv)
        for j in range(h):
            qrow = np.concatenate([np.asarray(q_nope[bi, j], np.float64),
                                   np.asarray(q_pe[bi, j], np.float64)], axis=1)
            o, l = attend_rows(qrow, K[:, j, :], V[:, j, :], counts, scale)
            out[bi, j] = o
            lse[bi, j] = l
    return out, lse


def mla_split_latent_ref(q_nope, q_pe, z_seqs, kpe_seqs, w_uk, w_uv, seqlens, scale, n_recent):
    """The hybrid form ([SKILL] "MLAvar6+ Design"): of the L_b keys of sequence b
    the o_b = L_b - n_b older ones are attended in latent form (scores Qz Z^T +
    q_pe K_pe^T, values O_lat, projected by W_uv) and the n_b most recent ones in
    expanded form (decompressed keys and values); the two softmaxes over disjoint
    key sets are joined by merge_partials_ref. n_recent[b] >= s (the new tokens
    are the last keys and see each other causally); every new token sees all o_b
    older keys. Exactly the full attention up to rounding.
    Returns (out [b, h, s, d], lse [b, h, s])."""
    b, h, s, d = q_nope.shape
    out = np.zeros((b, h, s, w_uv.shape[2]), dtype=np.float64)
    lse = np.full((b, h, s), -np.inf, dtype=np.float64)
    qz = mla_absorb_ref(q_nope, w_uk)
    for bi in range(b):
        L, n = int(seqlens[bi]), int(n_recent[bi])
        if L == 0:
            continue
        if not s <= n <= L:
            raise ValueError(f"recent keys {n} must cover the {s} new tokens and fit in {L}")
        o = L - n
        # latent part: every one of the h*s rows sees all o older keys (one token per row)
        qz_rows = qz[bi:bi + 1].reshape(1, h * s, 1, -1)
        qpe_rows = np.asarray(q_pe[bi:bi + 1], np.float64).reshape(1, h * s, 1, -1)
        lat, l_a = mla_latent_ref(qz_rows, qpe_rows, [z_seqs[bi][:o]], [kpe_seqs[bi][:o]], [o], scale)
        o_a = mla_out_proj_ref(lat.reshape(1, h, s, -1), w_uv)[0]
        # expanded part: the n recent keys, causal among the s new tokens at their end
        o_b, l_b = mla_expanded_ref(q_nope[bi:bi + 1], q_pe[bi:bi + 1], [z_seqs[bi][o:L]], [kpe_seqs[bi][o:L]],
                                    w_uk, w_uv, [n], scale)
        m_o, m_l = merge_partials_ref([o_a, o_b[0]], [l_a.reshape(h, s), l_b[0]])
        out[bi] = m_o
        lse[bi] = m_l
    return out, lse


# ---------------------------------------------------------------------------
# merging split partials (log-sum-exp merge; exact up to rounding)


def merge_partials_ref(outs, lses):
    """Given partial results (o_c, lse_c) of disjoint key subsets of the same
    rows, return the result over their union:
    lse = log sum_c exp(lse_c);  o = sum_c exp(lse_c - lse) o_c.
    Subsets with lse_c = -inf contribute nothing; all empty -> (0, -inf)."""
    outs = [np.asarray(o, np.float64) for o in outs]
    lses = np.stack([np.asarray(l, np.float64) for l in lses], axis=0)
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lses - m_safe)  # exp(-inf) = 0
    total = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), -np.inf)
    o = np.zeros_like(outs[0])
    for c, oc in enumerate(outs):
        coef = np.where(finite, w[c] / np.where(finite, total, 1.0), 0.0)
        o = o + coef[..., None] * oc
    return o, lse
