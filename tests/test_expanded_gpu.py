"""Parity of the expanded MLA form against the fp64 oracle, through the C ABI:
the tcgen05 decompression GEMM (mla_decompress_kv: K = [Z W_uk^T || K_pe],
V = Z W_uv) and grouped-head decode with key width d + p = 192 and value width
d = 128 over the decompressed cache (gqa_decode_dv, Hkv = Hq = h).

Stage-wise: the decompression against oracle.mla_decompress_ref on the same bf16
latent rows, the attention against oracle.gqa_ref on the GPU's own bf16 K / V.
End to end: oracle.mla_expanded_ref from the bf16 inputs, nothing rounded; there
the LSE is held to the first-order bound of storing the decompressed keys in bf16
(tests.helpers.key_rounding_lse_bound), the outputs to the usual bounds."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import assert_lse_close, assert_out_close, cache_rows, f64, key_rounding_lse_bound, mla_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
D, P, KL = 128, 64, 512


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da

    da.set_forced_splits(0)
    yield
    da.set_forced_splits(0)


def make(b, h, s, seqlens, paged=False, capacity=None, seed=0, k=KL):
    from decode_attention_18_b300 import workloads as W

    return W.make_mla(b, h, D, k, P, s, seqlens, paged=paged, capacity=capacity, seed=seed, device=DEV)


def decompress(inp):
    import decode_attention_18_b300 as da

    kf, vf = da.mla_decompress_kv(inp.z, inp.k_pe, inp.w_uk, inp.w_uv)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    return kf, vf


def assert_decompressed_close(got_k, got_v, ref_k, ref_v, what=""):
    """bf16 outputs of fp32 sums: each element within 2^-8 of its magnitude (round to
    nearest even gives 2^-9) plus 1e-5 for the fp32 accumulation; the RoPE part is a
    copy and must be exact."""
    nope, rope = got_k[..., :D], got_k[..., D:]
    for g, r, n in ((nope, ref_k[..., :D], "K nope"), (got_v, ref_v, "V")):
        err = np.abs(g - r)
        bound = 2.0 ** -8 * np.abs(r) + 1e-5
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), f"{what} {n}: err {err[worst]:.3e} at {worst} > {bound[worst]:.3e}"
    np.testing.assert_array_equal(rope, ref_k[..., D:], err_msg=f"{what} K rope")


@pytest.mark.parametrize("b,h,cap,k", [(2, 8, 200, 512), (1, 10, 131, 256), (3, 3, 64, 64)])
def test_decompress_matches_oracle(b, h, cap, k):
    # cache rows not a multiple of the 128-row tile, head counts not a multiple of the
    # 8-head group, latent widths 512 / 256 / 64
    inp = make(b, h, 1, [cap] * b, capacity=cap, seed=3, k=k)
    kf, vf = decompress(inp)
    assert kf.shape == (b, cap, h, D + P) and vf.shape == (b, cap, h, D)
    rk, rv = A.mla_decompress_ref(f64(inp.z), f64(inp.k_pe), f64(inp.w_uk), f64(inp.w_uv))
    assert_decompressed_close(f64(kf), f64(vf), rk, rv, f"b{b} h{h} cap{cap} k{k}")


def test_decompress_paged_pool_keeps_row_order():
    inp = make(3, 4, 1, [100, 64, 257], paged=True, seed=5)
    kf, vf = decompress(inp)
    assert kf.shape[:2] == inp.z.shape[:2]
    rk, rv = A.mla_decompress_ref(f64(inp.z), f64(inp.k_pe), f64(inp.w_uk), f64(inp.w_uv))
    assert_decompressed_close(f64(kf), f64(vf), rk, rv, "paged pool")


def test_decompress_argument_errors():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300._native import DecAttnError

    inp = make(1, 2, 1, [64], capacity=64)
    with pytest.raises(DecAttnError) as e:  # d = 64: no compiled instance
        da.mla_decompress_kv(inp.z, inp.k_pe, inp.w_uk[:, :64].contiguous(), inp.w_uv[:, :, :64].contiguous())
    assert e.value.status == 2
    with pytest.raises(DecAttnError) as e:  # k not a multiple of 64
        da.mla_decompress_kv(inp.z[..., :96].contiguous(), inp.k_pe, inp.w_uk[..., :96].contiguous(),
                             inp.w_uv[:, :96].contiguous())
    assert e.value.status == 2


def run_expanded(inp, seqlens):
    import decode_attention_18_b300 as da

    kf, vf = decompress(inp)
    q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).contiguous()  # the expanded query [q_nope || q_pe]
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = da.gqa_decode_dv(q, kf, vf, sl, scale=inp.scale, max_seqlen=max(max(seqlens), 1),
                                block_table=inp.block_table if inp.paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    return q, kf, vf, out, lse


def check_expanded(inp, seqlens, what):
    q, kf, vf, out, lse = run_expanded(inp, seqlens)
    b = len(seqlens)
    bt = inp.block_table if inp.paged else None
    # stage-wise: the attention over the GPU's own decompressed cache
    ks = [cache_rows(kf, i, seqlens[i], bt) for i in range(b)]
    vs = [cache_rows(vf, i, seqlens[i], bt) for i in range(b)]
    o_s, l_s = A.gqa_ref(f64(q), ks, vs, seqlens, inp.scale)
    assert_out_close(f64(out), o_s, f"{what} stage-wise")
    assert_lse_close(f64(lse), l_s, f"{what} stage-wise lse")
    # end to end from the bf16 inputs
    zs = [mla_rows(inp, i, "z") for i in range(b)]
    kp = [mla_rows(inp, i, "kpe") for i in range(b)]
    o_e, l_e = A.mla_expanded_ref(f64(inp.q_nope), f64(inp.q_pe), zs, kp, f64(inp.w_uk), f64(inp.w_uv), seqlens,
                                  inp.scale)
    assert_out_close(f64(out), o_e, f"{what} end to end")
    # the cache holds the decompressed keys in bf16 while the oracle keeps them exact:
    # the end-to-end LSE is held to the first-order bound of that rounding
    bound = np.full(l_e.shape, 1e-3)
    qn, qp = f64(inp.q_nope), f64(inp.q_pe)
    w_uk, w_uv = f64(inp.w_uk), f64(inp.w_uv)
    h = qn.shape[1]
    for bi, L in enumerate(seqlens):
        if L == 0:
            continue
        K, _ = A.mla_decompress_ref(zs[bi], kp[bi], w_uk, w_uv)
        counts = A.causal_key_counts(L, inp.q_nope.shape[2])
        for j in range(h):
            qrow = np.concatenate([qn[bi, j], qp[bi, j]], axis=1)
            bound[bi, j] = key_rounding_lse_bound(qrow, K[:, j], slice(0, D), l_e[bi, j], counts, inp.scale)
    assert_lse_close(f64(lse), l_e, f"{what} end to end lse", tol=bound)
    return out, lse


@pytest.mark.parametrize("s,seqlens", [(1, [517, 1, 300]), (1, [0, 70]), (4, [400, 129, 64]), (2, [2, 191])])
def test_expanded_attention_vs_oracle(s, seqlens):
    inp = make(len(seqlens), 8, s, seqlens, seed=11 + s)
    check_expanded(inp, seqlens, f"s{s} {seqlens}")


def test_expanded_paged_equals_contiguous_bitwise():
    import decode_attention_18_b300 as da

    seqlens = [300, 77, 129]
    inp = make(3, 4, 1, seqlens, paged=True, seed=21)
    out_p, lse_p = check_expanded(inp, seqlens, "paged")
    # the same rows laid out contiguously
    cap = max(seqlens)
    z = torch.zeros((3, cap, KL), dtype=torch.bfloat16, device=DEV)
    kpe = torch.zeros((3, cap, P), dtype=torch.bfloat16, device=DEV)
    for i, L in enumerate(seqlens):
        z[i, :L] = torch.from_numpy(mla_rows(inp, i, "z")).to(DEV, torch.bfloat16)
        kpe[i, :L] = torch.from_numpy(mla_rows(inp, i, "kpe")).to(DEV, torch.bfloat16)
    kf, vf = da.mla_decompress_kv(z, kpe, inp.w_uk, inp.w_uv)
    q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).contiguous()
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out_c, lse_c = da.gqa_decode_dv(q, kf, vf, sl, scale=inp.scale, max_seqlen=cap)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_c)
    assert torch.equal(lse_p, lse_c)


@pytest.mark.parametrize("nsplit", [1, 3])
def test_expanded_forced_splits(nsplit):
    import decode_attention_18_b300 as da

    seqlens = [700, 333]
    inp = make(2, 4, 1, seqlens, seed=31)
    da.set_forced_splits(nsplit)
    try:
        check_expanded(inp, seqlens, f"splits {nsplit}")
        assert da.last_num_splits() == nsplit
    finally:
        da.set_forced_splits(0)


def test_full_size_dsv3_sampled():
    # b = 32 sequences of 4096 keys, h = 128 heads: the decompressed cache is 10.7 GB.
    # Sampled checks: decompressed rows, and whole (sequence, head) outputs.
    seqlens = [4096] * 32
    inp = make(32, 128, 1, seqlens, seed=0)
    q, kf, vf, out, lse = run_expanded(inp, seqlens)
    rng = np.random.default_rng(7)
    w_uk, w_uv = f64(inp.w_uk), f64(inp.w_uv)
    for bi, m in zip(rng.integers(0, 32, 3), rng.integers(0, 4096, 3)):
        rk, rv = A.mla_decompress_ref(f64(inp.z[bi, m:m + 1]), f64(inp.k_pe[bi, m:m + 1]), w_uk, w_uv)
        assert_decompressed_close(f64(kf[bi, m:m + 1]), f64(vf[bi, m:m + 1]), rk, rv, f"row ({bi},{m})")
    for bi, j in zip(rng.integers(0, 32, 4), rng.integers(0, 128, 4)):
        Z = f64(inp.z[bi])
        KPE = f64(inp.k_pe[bi])
        o_e, l_e = A.mla_expanded_ref(f64(inp.q_nope[bi:bi + 1, j:j + 1]), f64(inp.q_pe[bi:bi + 1, j:j + 1]), [Z],
                                      [KPE], w_uk[j:j + 1], w_uv[j:j + 1], [4096], inp.scale)
        assert_out_close(f64(out[bi:bi + 1, j:j + 1]), o_e, f"({bi},{j})")
        K, _ = A.mla_decompress_ref(Z, KPE, w_uk[j:j + 1], w_uv[j:j + 1])
        qrow = np.concatenate([f64(inp.q_nope[bi, j]), f64(inp.q_pe[bi, j])], axis=1)
        bound = key_rounding_lse_bound(qrow, K[:, 0], slice(0, D), l_e[0, 0], [4096], inp.scale)
        assert_lse_close(f64(lse[bi:bi + 1, j:j + 1]), l_e, f"({bi},{j}) lse", tol=bound[None, None])
    del kf, vf
    torch.cuda.empty_cache()
