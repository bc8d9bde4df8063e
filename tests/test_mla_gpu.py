"""Parity of the absorbed-MLA kernels (absorb GEMM, tcgen05 latent attention +
combine, W_uv projection) against the fp64 oracle, through the C ABI.

Two comparisons per case: stage-wise (the oracle step is fed the very bf16
tensor the GPU step received, e.g. the GPU's Qz) and end to end (the oracle
runs the whole pipeline from the bf16 inputs without rounding anything)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from tests.helpers import mla_rows, as_device_bf16, assert_lse_close, assert_out_close, f64, qz_rounding_lse_bound

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


def make(b, h, d, k, p, s, seqlens, paged=False, capacity=None, seed=0, q_std=1.0):
    from decode_attention_18_b300 import workloads as W

    return W.make_mla(b, h, d, k, p, s, seqlens, paged=paged, capacity=capacity, seed=seed, device=DEV,
                      q_std=q_std)


def forward(inp):
    import decode_attention_18_b300 as da

    sl = torch.tensor(inp.seqlens, dtype=torch.int32, device=DEV)
    out, lse, qz, o_lat = da.mla_forward(inp.q_nope, inp.q_pe, inp.z, inp.k_pe, inp.w_uk, inp.w_uv, sl,
                                         scale=inp.scale, max_seqlen=max(inp.seqlens),
                                         block_table=inp.block_table if inp.paged else None)
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    return out, lse, qz, o_lat


def seq_inputs(inp, seqs):
    zs = [mla_rows(inp, i, "z") for i in seqs]
    kp = [mla_rows(inp, i, "kpe") for i in seqs]
    return zs, kp


def check(inp, res, seqs=None, what="", e2e_max_abs=None, e2e_mean_abs=None):
    out, lse, qz, o_lat = res
    seqs = list(range(len(inp.seqlens))) if seqs is None else seqs
    sl = [inp.seqlens[i] for i in seqs]
    zs, kp = seq_inputs(inp, seqs)
    # stage 1: absorb against the oracle on the same bf16 inputs (rows of
    # empty sequences are zero by the entry point's contract)
    rq = A.mla_absorb_ref(f64(inp.q_nope[seqs]), f64(inp.w_uk))
    for n, L in enumerate(sl):
        if L == 0:
            rq[n] = 0.0
    assert_out_close(f64(qz[seqs]), rq, what + " absorb")
    # stage 2: latent attention fed the GPU's bf16 Qz
    ro_lat, rl = A.mla_latent_ref(f64(qz[seqs]), f64(inp.q_pe[seqs]), zs, kp, sl, inp.scale)
    assert_out_close(f64(o_lat[seqs]), ro_lat, what + " latent")
    assert_lse_close(f64(lse[seqs]), rl, what + " lse")
    # stage 3: projection fed the GPU's bf16 O_lat
    ro = A.mla_out_proj_ref(f64(o_lat[seqs]), f64(inp.w_uv))
    assert_out_close(f64(out[seqs]), ro, what + " out_proj")
    # end to end from the bf16 inputs, nothing rounded in between
    eo, el, eqz, eolat = A.mla_absorbed_ref(f64(inp.q_nope[seqs]), f64(inp.q_pe[seqs]), zs, kp, f64(inp.w_uk),
                                            f64(inp.w_uv), sl, inp.scale)
    kw = {}
    if e2e_max_abs is not None:
        kw["max_abs"] = e2e_max_abs
    if e2e_mean_abs is not None:
        kw["mean_abs"] = e2e_mean_abs
    assert_out_close(f64(out[seqs]), eo, what + " end-to-end", **kw)
    assert_lse_close(f64(lse[seqs]), el, what + " end-to-end lse", tol=qz_rounding_lse_bound(eqz, eolat, inp.scale))


def test_tiny_workload():
    # b=2, h=16, d=32, k=64, p=16, t=256, s=1, scale 1/sqrt(48), seed 0
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS["mla_tiny"]
    inp = make(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed)
    check(inp, forward(inp), what="tiny")


@pytest.mark.parametrize("b,h,s,seqlens", [
    (2, 128, 1, [333, 100]),     # one full 128-row tile, ragged tails
    (3, 16, 1, [64, 65, 31]),    # fewer rows than a tile
    (2, 128, 2, [300, 40]),      # MTP s=2: two row tiles, causal
    (1, 64, 4, [97]),            # s=4
    (2, 8, 32, [64, 200]),       # s=32
    (2, 16, 16, [300, 40]),      # s=16: two row tiles
    (1, 128, 16, [200]),         # s=16 at h=128: 2048 rows, 16 row tiles, short context
])
def test_dsv3_shapes_small(b, h, s, seqlens):
    inp = make(b, h, 128, 512, 64, s, seqlens, capacity=max(seqlens) + 5, seed=1)
    check(inp, forward(inp), what=f"b{b} h{h} s{s}")


def test_edge_lengths():
    seqlens = [0, 1, 31, 32, 33, 64, 65]
    inp = make(7, 16, 128, 512, 64, 1, seqlens, seed=2)
    res = forward(inp)
    check(inp, res, what="edges")
    out, lse, _, o_lat = res
    assert torch.all(o_lat[0] == 0) and torch.all(out[0] == 0)
    assert torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("b,h,s,seqlens", [
    (2, 64, 2, [190, 66]),        # two row tiles per sequence; a last tile of 2 keys (one page)
    (3, 16, 8, [129, 64, 300]),   # s=8: a page-sized sequence and a 1-key last tile
])
def test_paged_mtp(b, h, s, seqlens):
    """Paged latent cache with s > 1 new tokens (causal among them): the producer's
    per-page boxes, the RoPE chunk's own ring item and the causal limits together."""
    inp = make(b, h, 128, 512, 64, s, seqlens, paged=True, seed=21)
    check(inp, forward(inp), what=f"paged b{b} h{h} s{s}")


def test_paged_vs_oracle_and_bitwise_contiguous():
    import decode_attention_18_b300 as da

    seqlens = [700, 64, 129]
    inp = make(3, 128, 128, 512, 64, 1, seqlens, paged=True, seed=3)
    res = forward(inp)
    check(inp, res, what="paged")
    cap = max(seqlens)
    z = torch.zeros((3, cap, 512), dtype=torch.bfloat16, device=DEV)
    kpe = torch.zeros((3, cap, 64), dtype=torch.bfloat16, device=DEV)
    for i, L in enumerate(seqlens):
        z[i, :L] = as_device_bf16(mla_rows(inp, i, "z"), z)
        kpe[i, :L] = as_device_bf16(mla_rows(inp, i, "kpe"), kpe)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    o2, l2 = da.mla_decode(res[2], inp.q_pe, z, kpe, sl, scale=inp.scale, max_seqlen=cap)
    torch.cuda.synchronize()
    assert torch.equal(o2, res[3])
    assert torch.equal(l2, res[1])


def test_sharp_queries():
    # queries x 8: logits of a few units, a peaked softmax. Every stage keeps
    # the 2e-2 / 2e-3 bounds against the oracle fed the same bf16 tensor. End
    # to end, the bf16 rounding of the Qz intermediate (round-to-nearest,
    # relative error uniform in +-2^-9, RMS 2^-9/sqrt(3), on |Qz| ~ 8*sqrt(d/k)
    # = 4) moves a logit by scale * dQz . Z, RMS ~ 2^-9/sqrt(3) * 4 *
    # sqrt(512) / sqrt(192) ~ 7.4e-3. With a few keys dominating, an output
    # moves by about that times |v| (unit scale): mean ~ 0.8 * 7.4e-3 * 0.8
    # ~ 5e-3 at worst, max a few times the RMS. So the end-to-end bounds here
    # are max-abs 5e-2 and mean-abs 5e-3 (rel-RMS bound unchanged).
    inp = make(2, 128, 128, 512, 64, 1, [400, 900], seed=4, q_std=8.0)
    check(inp, forward(inp), what="sharp", e2e_max_abs=5e-2, e2e_mean_abs=5e-3)


@pytest.mark.parametrize("nsplit", [1, 2, 5])
def test_split_invariance(nsplit):
    import decode_attention_18_b300 as da

    inp = make(2, 128, 128, 512, 64, 1, [1500, 700], seed=5)
    base = forward(inp)
    da.set_forced_splits(nsplit)
    try:
        sl = torch.tensor(inp.seqlens, dtype=torch.int32, device=DEV)
        o2, l2 = da.mla_decode(base[2], inp.q_pe, inp.z, inp.k_pe, sl, scale=inp.scale, max_seqlen=1500)
        torch.cuda.synchronize()
        chunk = -(-(-(-1500 // nsplit)) // 128) * 128  # chunks are whole 128-key latent tiles
        assert da.last_num_splits() == -(-1500 // chunk)
    finally:
        da.set_forced_splits(0)
    a, b2 = f64(base[3]), f64(o2)
    assert np.sqrt(np.mean((a - b2) ** 2)) / np.sqrt(np.mean(a ** 2)) <= 1e-2
    assert np.abs(f64(base[1]) - f64(l2)).max() <= 1e-4


def test_projection_gemms_alone():
    import decode_attention_18_b300 as da

    g = torch.Generator(device=DEV).manual_seed(9)
    o_lat = torch.randn((5, 16, 3, 512), generator=g, device=DEV).bfloat16()
    w = (torch.randn((16, 512, 128), generator=g, device=DEV) / math.sqrt(512)).bfloat16()
    sl = torch.tensor([3, 0, 9, 4, 5], dtype=torch.int32, device=DEV)
    out = da.mla_out_proj(o_lat, w, sl, scale=0.5)
    q = torch.randn((5, 16, 3, 128), generator=g, device=DEV).bfloat16()
    wk = (torch.randn((16, 128, 512), generator=g, device=DEV) / math.sqrt(512)).bfloat16()
    qz = da.mla_absorb_q(q, wk, None, scale=2.0)
    torch.cuda.synchronize()
    ro = A.mla_out_proj_ref(f64(o_lat), f64(w), 0.5)
    ro[1] = 0.0  # empty sequence -> zero rows
    assert_out_close(f64(out), ro, "out_proj")
    assert_out_close(f64(qz), A.mla_absorb_ref(f64(q), f64(wk), 2.0), "absorb", max_abs=4e-2, mean_abs=4e-3)


def test_tail_split_last_wave():
    # more (sequence, row tile) units than cluster slots, with a short last wave: the
    # units of that wave are cut into chunks (merged by their own combine), the others run
    # whole; an empty sequence and several lengths fall in the cut units
    import decode_attention_18_b300 as da

    seqlens = [1500 - 37 * i for i in range(19)] + [0]
    inp = make(20, 128, 128, 512, 64, 4, seqlens, seed=13)
    res = forward(inp)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    units = 20 * 4  # 512 rows per sequence: 4 row tiles
    if units > pairs and units % pairs and pairs // (units % pairs) >= 2:
        assert da.last_num_splits() == pairs // (units % pairs)
    check(inp, res, seqs=[0, 17, 18, 19], what="tail split")


def test_full_size_dsv3_sampled():
    # b=32, h=128, d=128, k=512, p=64, t=4096, s=1: the headline workload
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS["mla_dsv3"]
    inp = make(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed)
    check(inp, forward(inp), seqs=[0, 19, 31], what="dsv3")


def test_full_size_mtp_s8_sampled():
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS["mla_mtp_s8"]
    inp = make(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed)
    check(inp, forward(inp), seqs=[0, 31], what="mtp s8")


@pytest.mark.parametrize("s", [16, 32])
def test_full_size_mtp_sampled(s):
    # b=32, h=128, t=4096 prior + s new tokens: 2048 / 4096 query rows per sequence
    # (16 / 32 row tiles), the s-sweep's largest shapes
    from decode_attention_18_b300 import workloads as W

    wl = W.WORKLOADS[f"mla_mtp_s{s}"]
    inp = make(wl.b, wl.heads, wl.d, wl.k, wl.p, wl.s, wl.seqlens(), seed=wl.seed)
    check(inp, forward(inp), seqs=[0, 31], what=f"mtp s{s}")


def test_multi_wave_split_grid_then_combine():
    # 64 sequences x 2 column halves x 3 chunks = 384 latent CTAs (more than two waves of
    # one CTA per SM), each launched as a programmatic dependent, then the combine: the
    # combine may only start once every latent CTA has started, and must see all partials
    import decode_attention_18_b300 as da

    seqlens = [1500 - 7 * i for i in range(64)]
    inp = make(64, 128, 128, 512, 64, 1, seqlens, seed=11)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    qz = da.mla_absorb_q(inp.q_nope, inp.w_uk, sl)
    da.set_forced_splits(3)
    try:
        o, lse = da.mla_decode(qz, inp.q_pe, inp.z, inp.k_pe, sl, scale=inp.scale, max_seqlen=max(seqlens))
        torch.cuda.synchronize()
        assert da.last_num_splits() == 3
    finally:
        da.set_forced_splits(0)
    assert da.check_errors() == 0
    seqs = [0, 21, 42, 63]
    zs, kp = seq_inputs(inp, seqs)
    ro, rl = A.mla_latent_ref(f64(qz[seqs]), f64(inp.q_pe[seqs]), zs, kp, [seqlens[i] for i in seqs], inp.scale)
    assert_out_close(f64(o[seqs]), ro, "multi-wave latent")
    assert_lse_close(f64(lse[seqs]), rl, "multi-wave lse")


@pytest.mark.parametrize("paged", [False, True])
def test_nan_past_the_end_is_never_read(paged):
    seqlens = [300, 45, 129]
    inp = make(3, 128, 128, 512, 64, 1, seqlens, paged=paged, capacity=None if paged else 400, seed=14)
    for t in (inp.z, inp.k_pe):
        for i, L in enumerate(seqlens):
            if not paged:
                t[i, L:] = float("nan")
            elif L % 64:
                t[int(inp.block_table[i, (L - 1) // 64])][L % 64:] = float("nan")
    res = forward(inp)
    assert torch.isfinite(res[3].float()).all() and torch.isfinite(res[0].float()).all()
    check(inp, res, what=f"nan past end paged={paged}")
