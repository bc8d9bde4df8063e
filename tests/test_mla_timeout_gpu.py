"""The timeout path of the latent kernel, exercised without hanging the GPU:
a test-only switch makes one wait of each CTA poll a barrier that nothing
signals, with a 1 ms limit. The kernels must record the time-out, wind down
(wait for their own copies, free Tensor Memory) and return; the host reads
DECATTN_ERR_TIMEOUT, and the context stays usable."""
import math

import pytest
import torch

from oracle import attention as A
from tests.helpers import mla_rows, assert_lse_close, assert_out_close, f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(inp):
    import decode_attention_18_b300 as da

    sl = torch.tensor(inp.seqlens, dtype=torch.int32, device=DEV)
    qz = da.mla_absorb_q(inp.q_nope, inp.w_uk, sl)
    o, lse = da.mla_decode(qz, inp.q_pe, inp.z, inp.k_pe, sl, scale=inp.scale, max_seqlen=max(inp.seqlens))
    return qz, o, lse


def test_forced_timeout_reports_status_and_context_survives():
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import build, workloads as W

    build.build()
    inp = W.make_mla(2, 128, 128, 512, 64, 1, [300, 200], seed=21, device=DEV)
    assert da.check_errors() == 0
    da.test_force_timeout(True)
    try:
        _run(inp)
        rc = da.check_errors()
    finally:
        da.test_force_timeout(False)
    assert rc == 5  # DECATTN_ERR_TIMEOUT
    # the same call afterwards runs normally and is correct
    qz, o, lse = _run(inp)
    assert da.check_errors() == 0
    zs = [mla_rows(inp, i, "z") for i in range(2)]
    kp = [mla_rows(inp, i, "kpe") for i in range(2)]
    ro, rl = A.mla_latent_ref(f64(qz), f64(inp.q_pe), zs, kp, inp.seqlens, inp.scale)
    assert_out_close(f64(o), ro, "after timeout")
    assert_lse_close(f64(lse), rl, "after timeout")
