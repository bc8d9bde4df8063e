"""Over-write detection: every buffer a call writes (outputs, LSE, the split
workspace) is placed between guard regions filled with a canary byte pattern,
and the guards are checked byte for byte after the call, on ragged, paged and
split shapes of each entry point. (Over-reads are covered by the NaN-poisoning
tests: cache rows past each sequence's end are never read.)"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 8192  # bytes before and after each buffer (a multiple of every alignment in use)
CANARY = 0xA7


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    import decode_attention_18_b300 as da

    da.set_forced_splits(0)
    yield
    da.set_forced_splits(0)


class Guarded:
    """A tensor of `shape` / `dtype` inside a byte buffer with canary guards."""

    def __init__(self, shape, dtype, nbytes=None):
        elem = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * elem if nbytes is None else int(nbytes)
        n = max(n, 16)
        self.n = n
        self.buf = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        inner = self.buf[GUARD:GUARD + n]
        self.t = inner if nbytes is not None else inner.view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.n:]
        for part, where in ((head, "before"), (tail, "after")):
            bad = torch.nonzero(part != CANARY)
            assert bad.numel() == 0, f"{what}: {bad.numel()} guard bytes changed {where} the buffer " \
                                     f"(first at offset {int(bad[0])})"


@pytest.mark.parametrize("case", ["balanced_paged", "forced_split3", "many_rows", "unsplit"])
def test_grouped_head_writes_stay_inside(case):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    b, hq, hkv, d, s, seqlens, paged, forced = {
        "balanced_paged": (3, 8, 2, 128, 1, [700, 65, 1], True, 0),
        "forced_split3": (2, 8, 8, 64, 1, [500, 130], False, 3),
        "many_rows": (2, 24, 1, 256, 4, [333, 97], True, 0),
        "unsplit": (64, 8, 8, 128, 1, [128] * 64, False, 1),
    }[case]
    q, cache = W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, seed=2, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    da.set_forced_splits(forced)
    try:
        wsb = da.ops.load().gqa_decode_workspace_size(b, s, hq, hkv, d, max(seqlens))
        out = Guarded((b, hq, s, d), torch.bfloat16)
        lse = Guarded((b, hq, s), torch.float32)
        ws = Guarded(None, torch.uint8, nbytes=wsb)
        da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens),
                      block_table=cache.block_table if paged else None, out=out.t, lse=lse.t,
                      workspace=ws.t if wsb else None)
        assert da.check_errors() == 0
    finally:
        da.set_forced_splits(0)
    out.check(case + " out")
    lse.check(case + " lse")
    ws.check(case + " workspace")
    assert not torch.all(out.t.view(torch.uint8) == CANARY)  # the call did write its output


@pytest.mark.parametrize("paged,forced,s", [(True, 2, 1), (False, 0, 4), (False, 1, 1), (True, 0, 16)])
def test_mla_pipeline_writes_stay_inside(paged, forced, s):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [300, 70, 129] if s == 1 else [300, 70, 129][:2]
    b, h, d, k, p = len(seqlens), 16, 128, 512, 64
    inp = W.make_mla(b, h, d, k, p, s, seqlens, paged=paged, seed=4, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    bt = inp.block_table if paged else None
    qz = Guarded((b, h, s, k), torch.bfloat16)
    o_lat = Guarded((b, h, s, k), torch.bfloat16)
    lse = Guarded((b, h, s), torch.float32)
    out = Guarded((b, h, s, d), torch.bfloat16)
    da.set_forced_splits(forced)
    try:
        wsb = da.ops.load().mla_decode_workspace_size(b, s, h, k, max(seqlens))
        ws = Guarded(None, torch.uint8, nbytes=wsb)
        da.mla_absorb_q(inp.q_nope, inp.w_uk, sl, out=qz.t)
        da.mla_decode(qz.t, inp.q_pe, inp.z, inp.k_pe, sl, scale=inp.scale, max_seqlen=max(seqlens), block_table=bt,
                      out=o_lat.t, lse=lse.t, workspace=ws.t if wsb else None)
        da.mla_out_proj(o_lat.t, inp.w_uv, sl, out=out.t)
        assert da.check_errors() == 0
    finally:
        da.set_forced_splits(0)
    for g, n in ((qz, "qz"), (o_lat, "o_lat"), (lse, "lse"), (out, "out"), (ws, "workspace")):
        g.check(f"mla paged={paged} splits={forced} s={s} {n}")


def test_expanded_writes_stay_inside():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    seqlens = [200, 77]
    b, h, d, k, p = 2, 10, 128, 512, 64  # 400 cache rows (a ragged 128-row tile), 10 heads (a ragged group)
    inp = W.make_mla(b, h, d, k, p, 1, seqlens, seed=6, device=DEV)
    cap = inp.z.shape[1]
    kf = Guarded((b, cap, h, d + p), torch.bfloat16)
    vf = Guarded((b, cap, h, d), torch.bfloat16)
    da.mla_decompress_kv(inp.z, inp.k_pe, inp.w_uk, inp.w_uv, k_out=kf.t, v_out=vf.t)
    kf.check("decompressed K")
    vf.check("decompressed V")
    q = torch.cat([inp.q_nope, inp.q_pe], dim=-1).contiguous()
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    wsb = da.ops.load().gqa_decode_dv_workspace_size(b, 1, h, h, d + p, d, max(seqlens))
    out = Guarded((b, h, 1, d), torch.bfloat16)
    lse = Guarded((b, h, 1), torch.float32)
    ws = Guarded(None, torch.uint8, nbytes=wsb)
    da.gqa_decode_dv(q, kf.t, vf.t, sl, scale=inp.scale, max_seqlen=max(seqlens), out=out.t, lse=lse.t,
                     workspace=ws.t if wsb else None)
    assert da.check_errors() == 0
    for g, n in ((out, "out"), (lse, "lse"), (ws, "workspace")):
        g.check("expanded " + n)
