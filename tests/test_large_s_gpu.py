"""Parity at large numbers of new tokens per sequence (the prefill-sized end of
"Mla Analysis", Regime Selection; s = 64 .. 1024, causal among the new tokens),
for the three paths, through the C ABI against the fp64 oracle:
  * absorbed MLA (absorb -> latent attention -> W_uv): many 128-row tiles per
    sequence, each holding consecutive tokens of one head;
  * expanded MLA (decompression -> grouped-head decode, 192 / 128 wide);
  * grouped-head decode with many query rows per KV head (G * s rows).
The checks follow the decode-sized tests: stage-wise on the GPU's own bf16
intermediates and end to end from the bf16 inputs."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import (assert_lse_close, assert_out_close, cache_rows, f64, gqa_rows, key_rounding_lse_bound,
                           mla_rows, qz_rounding_lse_bound)

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


def make_mla(b, h, d, k, p, s, seqlens, paged=False, seed=0):
    from decode_attention_18_b300 import workloads as W

    return W.make_mla(b, h, d, k, p, s, seqlens, paged=paged, seed=seed, device=DEV)


@pytest.mark.parametrize("h,s,seqlens,paged", [
    (2, 128, [300, 128], False),   # 2 row tiles per sequence; the second sequence's first token sees 1 key
    (3, 64, [200, 97], True),      # 192 rows: a tile spans two heads; paged cache
    (1, 1024, [1100], False),      # prefill-sized: 8 tiles of one head
])
def test_absorbed_mla_large_s(h, s, seqlens, paged):
    import decode_attention_18_b300 as da

    d, k, p = 128, 512, 64
    inp = make_mla(len(seqlens), h, d, k, p, s, seqlens, paged=paged, seed=s)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse, qz, o_lat = da.mla_forward(inp.q_nope, inp.q_pe, inp.z, inp.k_pe, inp.w_uk, inp.w_uv, sl,
                                         scale=inp.scale, max_seqlen=max(seqlens),
                                         block_table=inp.block_table if paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    b = len(seqlens)
    zs = [mla_rows(inp, i, "z") for i in range(b)]
    kp = [mla_rows(inp, i, "kpe") for i in range(b)]
    what = f"h{h} s{s}"
    assert_out_close(f64(qz), A.mla_absorb_ref(f64(inp.q_nope), f64(inp.w_uk)), what + " absorb")
    ro_lat, rl = A.mla_latent_ref(f64(qz), f64(inp.q_pe), zs, kp, seqlens, inp.scale)
    assert_out_close(f64(o_lat), ro_lat, what + " latent")
    assert_lse_close(f64(lse), rl, what + " latent lse")
    assert_out_close(f64(out), A.mla_out_proj_ref(f64(o_lat), f64(inp.w_uv)), what + " out_proj")
    eo, el, eqz, eolat = A.mla_absorbed_ref(f64(inp.q_nope), f64(inp.q_pe), zs, kp, f64(inp.w_uk), f64(inp.w_uv),
                                            seqlens, inp.scale)
    assert_out_close(f64(out), eo, what + " end to end")
    assert_lse_close(f64(lse), el, what + " end to end lse", tol=qz_rounding_lse_bound(eqz, eolat, inp.scale))


@pytest.mark.parametrize("h,s,seqlens", [(2, 128, [300, 128]), (1, 512, [700])])
def test_expanded_mla_large_s(h, s, seqlens):
    import decode_attention_18_b300 as da

    d, k, p = 128, 512, 64
    inp = make_mla(len(seqlens), h, d, k, p, s, seqlens, seed=40 + s)
    kf, vf = da.mla_decompress_kv(inp.z, inp.k_pe, inp.w_uk, inp.w_uv)
    q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).contiguous()  # the expanded query [q_nope || q_pe]
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode_dv(q, kf, vf, sl, scale=inp.scale, max_seqlen=max(seqlens))
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    b = len(seqlens)
    what = f"expanded h{h} s{s}"
    ks = [cache_rows(kf, i, seqlens[i]) for i in range(b)]
    vs = [cache_rows(vf, i, seqlens[i]) for i in range(b)]
    o_s, l_s = A.gqa_ref(f64(q), ks, vs, seqlens, inp.scale)
    assert_out_close(f64(out), o_s, what + " stage-wise")
    assert_lse_close(f64(lse), l_s, what + " stage-wise lse")
    zs = [mla_rows(inp, i, "z") for i in range(b)]
    kp = [mla_rows(inp, i, "kpe") for i in range(b)]
    o_e, l_e = A.mla_expanded_ref(f64(inp.q_nope), f64(inp.q_pe), zs, kp, f64(inp.w_uk), f64(inp.w_uv), seqlens,
                                  inp.scale)
    assert_out_close(f64(out), o_e, what + " end to end")
    bound = np.zeros(l_e.shape)
    for bi, L in enumerate(seqlens):
        K, _ = A.mla_decompress_ref(zs[bi], kp[bi], f64(inp.w_uk), f64(inp.w_uv))
        counts = A.causal_key_counts(L, s)
        for j in range(h):
            qrow = np.concatenate([f64(inp.q_nope[bi, j]), f64(inp.q_pe[bi, j])], axis=1)
            bound[bi, j] = key_rounding_lse_bound(qrow, K[:, j], slice(0, d), l_e[bi, j], counts, inp.scale)
    assert_lse_close(f64(lse), l_e, what + " end to end lse", tol=bound)


@pytest.mark.parametrize("b,hq,hkv,d,s,seqlens,paged", [
    (2, 8, 2, 128, 64, [200, 74], False),    # G * s = 256 rows per KV head: 8 row blocks
    (1, 4, 4, 64, 1024, [1500], False),      # MHA, prefill-sized
    (2, 6, 1, 256, 96, [400, 96], True),     # MQA, 576 rows per KV head, paged
])
def test_grouped_head_large_s(b, hq, hkv, d, s, seqlens, paged):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, seed=s, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens),
                             block_table=cache.block_table if paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    ks = [gqa_rows(cache, i, "k") for i in range(b)]
    vs = [gqa_rows(cache, i, "v") for i in range(b)]
    ro, rl = A.gqa_ref(f64(q), ks, vs, seqlens, 1 / math.sqrt(d))
    assert_out_close(f64(out), ro, f"gqa s{s}")
    assert_lse_close(f64(lse), rl, f"gqa s{s} lse")


def test_s_limit():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W
    from decode_attention_18_b300._native import DecAttnError

    q, cache = W.make_gqa(1, 1, 1, 64, 1025, [1100], seed=1, device=DEV)
    sl = torch.tensor([1100], dtype=torch.int32, device=DEV)
    with pytest.raises(DecAttnError) as e:
        da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=1100)
    assert e.value.status == 1
