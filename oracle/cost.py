"""Analytic cost counter: FLOPs, HBM bytes, arithmetic intensity, ridge points
and KV-cache accounting (test infrastructure; see the package docstring).

Notation follows the "Mla Analysis" skill page, section "Cost Models
(DeepSeek-V3-like: h=128, d=128, k=512, p=64)": b batch, h query heads,
s new (query) tokens per sequence, t context length, d head dim, p decoupled
RoPE dim, k latent dim, w bytes per element (2 for BF16, the precision the
"Why MLA and MTP Fight Each Other" post assumes for the KV cache).

Only the attention core is counted (scores and value contraction); the
softmax and the WO projection are left out, as the "Why MLA and MTP Fight
Each Other" post, section 1 ("What arithmetic intensity is"), does. The
absorption and output-projection GEMMs of the absorbed MLA pipeline are
counted separately by ``proj_flops`` / ``proj_bytes``.
"""
from __future__ import annotations

BF16_BYTES = 2


# --- arithmetic intensity and the roofline ("Why MLA and MTP Fight Each Other",
# section 1 "What arithmetic intensity is": AI = FLOPs / bytes moved from HBM;
# the hardware balance point is peak FLOP/s divided by HBM bandwidth; below it a
# kernel is memory-bound, above it compute-bound).

def arithmetic_intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes


def ridge_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """Balance point in FLOP/byte (same table of that section)."""
    return peak_flops / bandwidth_bytes


def roofline_time(flops: float, nbytes: float, peak_flops: float, bandwidth_bytes: float) -> float:
    """Ideal time of the idealised roofline: the slower of compute and traffic."""
    return max(flops / peak_flops, nbytes / bandwidth_bytes)


def attainable_flops(ai: float, peak_flops: float, bandwidth_bytes: float) -> float:
    """min(peak, AI x bandwidth)."""
    return min(peak_flops, ai * bandwidth_bytes)


# --- FlashAttention over expanded K/V ("Mla Analysis", Cost Models, FlashAttention).

def fa_flops(b, h, s, t, d, p):
    """2 b h s t (2d + p): QK^T over d+p plus PV over d."""
    return 2 * b * h * s * t * (2 * d + p)


def fa_bytes(b, h, s, t, d, p, w=BF16_BYTES):
    """w b h (s + t)(2d + p): s query rows (q of d+p, output of d) and t cached
    rows (K of d+p, V of d) per head."""
    return w * b * h * (s + t) * (2 * d + p)


# --- absorbed latent MLA ("Mla Analysis", Cost Models, FlashMLA).

def mla_flops(b, h, s, t, k, p):
    """2 b h s t (2k + p): Qz Z^T over k, q_pe K_pe^T over p, P Z over k."""
    return 2 * b * h * s * t * (2 * k + p)


def mla_bytes(b, h, s, t, k, p, w=BF16_BYTES):
    """w (b h s (2k + p) + b t (k + p)): per query row Qz (k) + q_pe (p) in and
    O_lat (k) out; per cached token one latent (k) plus one RoPE key (p),
    shared by all heads."""
    return w * (b * h * s * (2 * k + p) + b * t * (k + p))


# --- split latent + decompressed ("Mla Analysis", Cost Models, MLAvar6+).

def split_latent_flops(b, h, s, o, n, d, p, k):
    """2bhstp + 4bhsnd + 4bhsok with t = o + n."""
    t = o + n
    return 2 * b * h * s * t * p + 4 * b * h * s * n * d + 4 * b * h * s * o * k


def split_latent_bytes(b, h, s, o, n, d, p, k, w=BF16_BYTES):
    """w (bhsp + bhsd + bhsk + bok + btp + bhnd + bhnd + bhsd + bhsk), t = o + n,
    term by term as the page lists it."""
    t = o + n
    terms = (b * h * s * p, b * h * s * d, b * h * s * k, b * o * k, b * t * p,
             b * h * n * d, b * h * n * d, b * h * s * d, b * h * s * k)
    return w * sum(terms)


# --- grouped-head decode (MHA / GQA / MQA). The "Why MLA and MTP Fight Each
# Other" post says the first three rows of its summary table are one formula
# with different KV-head counts; it is the FlashAttention count with p = 0
# and the t cached rows read once per KV head instead of once per query head.

def gqa_flops(b, hq, s, t, d):
    """2 b Hq s t (2d): QK^T and PV, each 2 b Hq s t d."""
    return 2 * b * hq * s * t * 2 * d


def gqa_bytes(b, hq, hkv, s, t, d, w=BF16_BYTES):
    """w (b Hq s 2d + b Hkv t 2d): query and output rows per query head, K and V
    rows per KV head."""
    return w * (b * hq * s * 2 * d + b * hkv * t * 2 * d)


# --- exact executed counts with a bottom-right causal window among the s new
# tokens (token i of s sees keys 0 .. L - s + i, L = keys including the new s).

def causal_keys(L: int, s: int) -> int:
    """Number of (query token, key) pairs one head evaluates for one sequence."""
    return sum(L - s + i + 1 for i in range(s))


def gqa_flops_exact(hq, d, seqlens, s):
    return sum(2 * hq * causal_keys(L, s) * 2 * d for L in seqlens if L > 0)


def gqa_bytes_exact(hq, hkv, d, seqlens, s, w=BF16_BYTES):
    rows = sum(1 for L in seqlens) * hq * s * 2 * d
    kv = sum(L for L in seqlens) * hkv * 2 * d
    return w * (rows + kv)


def gqa_fp8_bytes_exact(hq, hkv, d, seqlens, s, w=BF16_BYTES, w_cache=1):
    """Grouped-head decode over an FP8 cache: query and output rows in bf16 (w), K
    and V in one byte per value (w_cache)."""
    rows = len(seqlens) * hq * s * 2 * d
    kv = sum(seqlens) * hkv * 2 * d
    return w * rows + w_cache * kv


def mla_flops_exact(h, k, p, seqlens, s):
    return sum(2 * h * causal_keys(L, s) * (2 * k + p) for L in seqlens if L > 0)


def mla_bytes_exact(h, k, p, seqlens, s, w=BF16_BYTES):
    rows = len(seqlens) * h * s * (2 * k + p)
    cache = sum(seqlens) * (k + p)
    return w * (rows + cache)


def fa_flops_exact(h, d, p, seqlens, s):
    """Expanded form (FlashAttention over decompressed keys of d + p and values of d,
    one KV head per query head): 2 (2d + p) per (query token, key) pair and head."""
    return sum(2 * h * causal_keys(L, s) * (2 * d + p) for L in seqlens if L > 0)


def fa_bytes_exact(h, d, p, seqlens, s, w=BF16_BYTES):
    """Query rows (d + p) in and output rows (d) out per head and new token; K (d + p)
    and V (d) of every head per cached key."""
    rows = len(seqlens) * h * s * (2 * d + p)
    cache = sum(seqlens) * h * (2 * d + p)
    return w * (rows + cache)


# --- decompression of the latent cache into the expanded form: per cache row and
# head, K_nope = z W_uk^T (d outputs over k) and V = z W_uv (d outputs over k)

def decompress_flops(rows, h, d, k):
    return 2 * rows * h * d * k * 2


def decompress_bytes(rows, h, d, k, p, w=BF16_BYTES):
    """Read the latent rows (k + p) and both weights (h d k each); write K (d + p) and
    V (d) of every head per row."""
    return w * (rows * (k + p) + 2 * h * d * k + rows * h * (2 * d + p))


# --- absorption and output-projection GEMMs (per-head, weights [h, d, k] and
# [h, k, d]); both are weight-times-activation products outside the attention
# core, like the projections the "Why MLA and MTP Fight Each Other" post leaves
# out of its count.

def proj_flops(b, h, s, d, k):
    return 2 * b * h * s * d * k


def proj_bytes(b, h, s, d, k, w=BF16_BYTES):
    """Read activations [b,h,s,d_in] and weights [h,d,k], write [b,h,s,d_out]."""
    return w * (b * h * s * d + h * d * k + b * h * s * k)


# --- KV-cache size accounting.

def kv_bytes_per_token_layer(hkv, d, w=BF16_BYTES):
    """Grouped-head cache: K and V, Hkv heads of d elements ("MQA, GQA & MLA"
    lesson, Concept: proportional to Hkv x head dim x 2 x bytes)."""
    return 2 * hkv * d * w


def kv_bytes_per_token(n_layers, hkv, d, w=BF16_BYTES):
    """Across caching layers ("MHA vs GQA" Q&A, numerical example)."""
    return n_layers * kv_bytes_per_token_layer(hkv, d, w)


def kv_cache_bytes(n_tokens, n_layers, hkv, d, w=BF16_BYTES):
    return n_tokens * kv_bytes_per_token(n_layers, hkv, d, w)


def mla_cache_bytes_per_token_layer(k, p, w=BF16_BYTES):
    """One latent of k plus one decoupled RoPE key of p per token ("MQA, GQA &
    MLA" lesson: the cache holds a latent vector plus the RoPE part)."""
    return (k + p) * w
