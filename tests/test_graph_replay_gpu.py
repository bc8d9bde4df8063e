"""The kernels launched as programmatic dependents (each may start while the kernel
before it on the stream finishes, and waits for it before reading) give the same
results when the calls are captured in a CUDA graph and replayed back to back with
new inputs copied into the captured buffers: every replay must equal, bit for bit,
eager calls on the same inputs, and one replay is checked against the oracle."""
import math

import pytest
import torch

from oracle import attention as A
from tests.helpers import gqa_rows, mla_rows, assert_lse_close, assert_out_close, f64

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


def _capture(fn, stream):
    with torch.cuda.stream(stream):
        fn()  # first-call set-up (kernel attributes) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def test_mla_pipeline_graph_replays():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    stream = torch.cuda.Stream()
    seqlens = [1500, 700, 0, 129]  # split context (the combine runs), an empty sequence
    b, h, d, k, p, s = 4, 128, 128, 512, 64, 1
    sets = [W.make_mla(b, h, d, k, p, s, seqlens, seed=40 + r, device=DEV) for r in range(3)]
    buf = W.make_mla(b, h, d, k, p, s, seqlens, seed=39, device=DEV)  # the captured input buffers
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    qz = torch.empty((b, h, s, k), dtype=torch.bfloat16, device=DEV)
    o_lat = torch.empty_like(qz)
    lse = torch.empty((b, h, s), dtype=torch.float32, device=DEV)
    out = torch.empty((b, h, s, d), dtype=torch.bfloat16, device=DEV)

    def step():
        da.mla_absorb_q(buf.q_nope, buf.w_uk, sl, out=qz, stream=stream)
        da.mla_decode(qz, buf.q_pe, buf.z, buf.k_pe, sl, scale=buf.scale, max_seqlen=max(seqlens), out=o_lat,
                      lse=lse, workspace=ws, stream=stream)
        da.mla_out_proj(o_lat, buf.w_uv, sl, out=out, stream=stream)

    g = _capture(step, stream)
    assert da.last_num_splits() > 1
    results = []
    with torch.cuda.stream(stream):
        for x in sets:  # back-to-back replays, inputs replaced in between on the same stream
            for name in ("q_nope", "q_pe", "z", "k_pe", "w_uk", "w_uv"):
                getattr(buf, name).copy_(getattr(x, name))
            g.replay()
            results.append(tuple(t.clone() for t in (qz, o_lat, lse, out)))
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    for x, (gqz, go, gl, gout) in zip(sets, results):
        eout, else_, eqz, eo = da.mla_forward(x.q_nope, x.q_pe, x.z, x.k_pe, x.w_uk, x.w_uv, sl, scale=x.scale,
                                              max_seqlen=max(seqlens))
        torch.cuda.synchronize()
        assert torch.equal(gqz, eqz) and torch.equal(go, eo) and torch.equal(gl, else_) and torch.equal(gout, eout)
    # the last replay against the oracle (latent stage fed the replay's own Qz)
    x = sets[-1]
    gqz, go, gl, _ = results[-1]
    zs = [mla_rows(x, i, "z") for i in range(b)]
    kp = [mla_rows(x, i, "kpe") for i in range(b)]
    ro, rl = A.mla_latent_ref(f64(gqz), f64(x.q_pe), zs, kp, seqlens, x.scale)
    assert_out_close(f64(go), ro, "graph replay latent")
    assert_lse_close(f64(gl), rl, "graph replay lse")


@pytest.mark.parametrize("hkv,d,paged", [(4, 128, True), (8, 128, False), (1, 256, True)])
def test_gqa_graph_replays(hkv, d, paged):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    stream = torch.cuda.Stream()
    seqlens = [3000, 0, 65, 1800, 7]
    b, hq, s = 5, 32, 1
    sets = [W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, seed=50 + r, device=DEV) for r in range(3)]
    q0, c0 = W.make_gqa(b, hq, hkv, d, s, seqlens, paged=paged, seed=49, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(q0)
    lse = torch.empty((b, hq, s), dtype=torch.float32, device=DEV)
    bt = c0.block_table if paged else None

    def step():
        da.gqa_decode(q0, c0.k, c0.v, sl, max_seqlen=max(seqlens), block_table=bt, out=out, lse=lse, workspace=ws,
                      stream=stream)

    g = _capture(step, stream)
    # the context was cut: fixed chunks (> 1), or the tensor-core kernel's balanced pieces (0)
    assert da.last_num_splits() != 1
    results = []
    with torch.cuda.stream(stream):
        for q, c in sets:
            q0.copy_(q)
            c0.k.copy_(c.k)
            c0.v.copy_(c.v)
            if paged:
                bt.copy_(c.block_table)
            g.replay()
            results.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert da.check_errors() == 0
    for (q, c), (go, gl) in zip(sets, results):
        eo, el = da.gqa_decode(q, c.k, c.v, sl, max_seqlen=max(seqlens), block_table=c.block_table if paged else None)
        torch.cuda.synchronize()
        assert torch.equal(go, eo) and torch.equal(gl, el)
    q, c = sets[-1]
    ks = [gqa_rows(c, i, "k") for i in range(b)]
    vs = [gqa_rows(c, i, "v") for i in range(b)]
    ro, rl = A.gqa_ref(f64(q), ks, vs, seqlens, 1 / math.sqrt(d))
    assert_out_close(f64(results[-1][0]), ro, "graph replay gqa")
    assert_lse_close(f64(results[-1][1]), rl, "graph replay gqa lse")
