"""Parity of the hybrid MLA form ("Mla Analysis", MLAvar6+ Design) against the
fp64 oracle, through the C ABI: the older keys of each sequence attended in
latent form (absorb -> latent kernel -> W_uv), the most recent ones in
decompressed form (gqa_decode_dv over mla_decompress_kv's output), the two
joined by attn_merge_lse.

Stage-wise, every step is fed the GPU's own bf16 intermediates; end to end the
result is held against the plain full attention (the split changes nothing but
rounding), with the LSE bound of the two roundings the pipeline makes (Qz of
the latent part, the stored keys of the recent part)."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import (assert_lse_close, assert_out_close, cache_rows, f64, key_rounding_lse_bound, mla_rows,
                           qz_rounding_lse_bound)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
D, K, P = 128, 512, 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da

    da.set_forced_splits(0)
    yield
    da.set_forced_splits(0)


def recent_cache(inp, seqlens, n_recent):
    """The decompressed cache of each sequence's n most recent keys (rows o .. L-1 of
    the latent cache, gathered with the oracle's paged gather when paged), written
    by mla_decompress_kv: [b, max n, h, d + p] and [b, max n, h, d]."""
    import decode_attention_18_b300 as da

    b = len(seqlens)
    cap = max(n_recent)
    z = torch.zeros((b, cap, K), dtype=torch.bfloat16, device=DEV)
    kpe = torch.zeros((b, cap, P), dtype=torch.bfloat16, device=DEV)
    for i, (L, n) in enumerate(zip(seqlens, n_recent)):
        z[i, :n] = torch.from_numpy(mla_rows(inp, i, "z")[L - n:L]).to(DEV, torch.bfloat16)
        kpe[i, :n] = torch.from_numpy(mla_rows(inp, i, "kpe")[L - n:L]).to(DEV, torch.bfloat16)
    return da.mla_decompress_kv(z, kpe, inp.w_uk, inp.w_uv)


@pytest.mark.parametrize("s,seqlens,n_recent,paged", [
    (1, [600, 200], [64, 200], False),    # the second sequence is all recent: empty latent part
    (4, [500, 130], [4, 100], False),     # recent part = the new tokens only; a mixed split
    (1, [333, 97, 64], [128, 1, 64], True),
    (8, [700, 300], [256, 40], True),
])
def test_split_latent_vs_oracle(s, seqlens, n_recent, paged):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    b, h = len(seqlens), 8
    inp = W.make_mla(b, h, D, K, P, s, seqlens, paged=paged, seed=50 + s, device=DEV)
    kr, vr = recent_cache(inp, seqlens, n_recent)
    old = [L - n for L, n in zip(seqlens, n_recent)]
    sl_old = torch.tensor(old, dtype=torch.int32, device=DEV)
    sl_rec = torch.tensor(n_recent, dtype=torch.int32, device=DEV)
    q_full = torch.cat([inp.q_nope, inp.q_pe], dim=-1).contiguous()
    bt = inp.block_table if paged else None
    # the steps one by one
    qz = da.mla_absorb_q(inp.q_nope, inp.w_uk)
    o_lat, lse_a = da.mla_decode(qz.view(b, h * s, 1, K), inp.q_pe.view(b, h * s, 1, P), inp.z, inp.k_pe, sl_old,
                                 scale=inp.scale, max_seqlen=max(max(old), 1), block_table=bt)
    out_a = da.mla_out_proj(o_lat.view(b, h, s, K), inp.w_uv)
    out_b, lse_b = da.gqa_decode_dv(q_full, kr, vr, sl_rec, scale=inp.scale, max_seqlen=max(n_recent))
    out, lse = da.attn_merge_lse(out_a, lse_a.view(b, h, s), out_b, lse_b)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    what = f"s{s} {seqlens} recent {n_recent}"

    # stage-wise
    zs = [mla_rows(inp, i, "z") for i in range(b)]
    kp = [mla_rows(inp, i, "kpe") for i in range(b)]
    ro_lat, rl_a = A.mla_latent_ref(f64(qz).reshape(b, h * s, 1, K), f64(inp.q_pe).reshape(b, h * s, 1, P),
                                    [zs[i][:old[i]] for i in range(b)], [kp[i][:old[i]] for i in range(b)], old,
                                    inp.scale)
    assert_out_close(f64(o_lat), ro_lat, what + " latent part")
    assert_lse_close(f64(lse_a), rl_a, what + " latent part lse")
    assert_out_close(f64(out_a), A.mla_out_proj_ref(f64(o_lat).reshape(b, h, s, K), f64(inp.w_uv)), what + " W_uv")
    ks = [cache_rows(kr, i, n_recent[i]) for i in range(b)]
    vs = [cache_rows(vr, i, n_recent[i]) for i in range(b)]
    ro_b, rl_b = A.gqa_ref(f64(q_full), ks, vs, n_recent, inp.scale)
    assert_out_close(f64(out_b), ro_b, what + " recent part")
    assert_lse_close(f64(lse_b), rl_b, what + " recent part lse")
    rm, rlm = A.merge_partials_ref([f64(out_a), f64(out_b)], [f64(lse_a).reshape(b, h, s), f64(lse_b)])
    assert_out_close(f64(out), rm, what + " merge")
    assert_lse_close(f64(lse), rlm, what + " merge lse", tol=1e-5)

    # the composite call runs the same kernels on the same inputs: bitwise equal
    out_c, lse_c = da.mla_split_forward(inp.q_nope, inp.q_pe, q_full, inp.z, inp.k_pe, kr, vr, inp.w_uk, inp.w_uv,
                                        sl_old, sl_rec, scale=inp.scale, max_old=max(max(old), 1),
                                        max_recent=max(n_recent), block_table=bt)
    torch.cuda.synchronize()
    assert torch.equal(out_c, out) and torch.equal(lse_c, lse)

    # end to end: the plain full attention from the bf16 inputs
    eo, el, _, _ = A.mla_absorbed_ref(f64(inp.q_nope), f64(inp.q_pe), zs, kp, f64(inp.w_uk), f64(inp.w_uv), seqlens,
                                      inp.scale)
    assert_out_close(f64(out), eo, what + " end to end")
    # LSE bound: the merged LSE is a convex combination of the two parts' LSEs, so its
    # error is at most the larger part error; the sum of both parts' bounds covers it
    eqz = A.mla_absorb_ref(f64(inp.q_nope), f64(inp.w_uk)).reshape(b, h * s, 1, K)
    e_lat, _ = A.mla_latent_ref(eqz, f64(inp.q_pe).reshape(b, h * s, 1, P), [zs[i][:old[i]] for i in range(b)],
                                [kp[i][:old[i]] for i in range(b)], old, inp.scale)
    bound = qz_rounding_lse_bound(eqz, e_lat, inp.scale).reshape(b, h, s)
    for i, (L, n) in enumerate(zip(seqlens, n_recent)):
        Kx, _ = A.mla_decompress_ref(zs[i][L - n:L], kp[i][L - n:L], f64(inp.w_uk), f64(inp.w_uv))
        counts = A.causal_key_counts(n, s)
        _, l_rec = A.mla_expanded_ref(f64(inp.q_nope[i:i + 1]), f64(inp.q_pe[i:i + 1]), [zs[i][L - n:L]],
                                      [kp[i][L - n:L]], f64(inp.w_uk), f64(inp.w_uv), [n], inp.scale)
        for j in range(h):
            qrow = np.concatenate([f64(inp.q_nope[i, j]), f64(inp.q_pe[i, j])], axis=1)
            bound[i, j] += key_rounding_lse_bound(qrow, Kx[:, j], slice(0, D), l_rec[0, j], counts, inp.scale)
    assert_lse_close(f64(lse), el, what + " end to end lse", tol=bound)


def test_merge_edge_cases():
    # one side empty (-inf), both empty, and NaN in an empty side's rows: never used
    import decode_attention_18_b300 as da

    rows, d = 5, 64
    g = torch.Generator(device="cpu").manual_seed(3)
    oa = torch.randn(rows, d, generator=g).to(DEV, torch.bfloat16)
    ob = torch.randn(rows, d, generator=g).to(DEV, torch.bfloat16)
    la = torch.tensor([0.5, -np.inf, 2.0, -np.inf, 30.0], dtype=torch.float32, device=DEV)
    lb = torch.tensor([1.5, 0.25, -np.inf, -np.inf, -30.0], dtype=torch.float32, device=DEV)
    oa[1] = float("nan")
    ob[2] = float("nan")
    ob[3] = float("nan")
    out, lse = da.attn_merge_lse(oa, la, ob, lb)
    torch.cuda.synchronize()
    fa, fb = f64(oa), f64(ob)
    fa[1] = 0.0
    fb[2] = 0.0
    fb[3] = 0.0
    rm, rl = A.merge_partials_ref([fa, fb], [f64(la), f64(lb)])
    assert np.all(np.isfinite(f64(out)))
    assert_out_close(f64(out), rm, "merge edges")
    assert_lse_close(f64(lse), rl, "merge edges lse", tol=1e-5)
    assert np.all(f64(out)[3] == 0.0)
