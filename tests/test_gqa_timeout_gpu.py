"""The timeout path of the grouped-head kernels, exercised without hanging the
GPU: a test-only switch makes the first tile wait of every CTA also poll a
barrier that nothing signals, with a 1 ms limit. Each CTA must record the
time-out, let the copies it already requested land, stop (the balanced
schedule still writes the meta entries the combine reads) and return; the host
reads DECATTN_ERR_TIMEOUT, and the next call on the same context is correct."""
import math

import pytest
import torch

from oracle import attention as A
from tests.helpers import assert_lse_close, assert_out_close, f64, gqa_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_attention_18_b300 import build

    build.build()
    yield


@pytest.mark.parametrize("b,hq,hkv,d,seqlens,forced,paged", [
    (2, 8, 2, 128, [300, 200], 1, False),        # one chunk: final rows written by the kernel
    (2, 8, 2, 128, [300, 200], 3, True),         # fixed chunks + combine, paged
    (3, 8, 2, 128, [5000, 1000, 64], 0, False),  # planner's split: balanced schedule + its combine
    (2, 24, 1, 256, [700, 129], 0, True),        # two m-tiles per CTA (24-row MQA, d = 256)
])
def test_forced_timeout_reports_status_and_context_survives(b, hq, hkv, d, seqlens, forced, paged):
    import decode_attention_18_b300 as da
    from decode_attention_18_b300 import workloads as W

    q, cache = W.make_gqa(b, hq, hkv, d, 1, seqlens, paged=paged, seed=31, device=DEV)
    sl = torch.tensor(seqlens, dtype=torch.int32, device=DEV)

    def call():
        return da.gqa_decode(q, cache.k, cache.v, sl, max_seqlen=max(seqlens),
                             block_table=cache.block_table if paged else None)

    assert da.check_errors() == 0
    da.set_forced_splits(forced)
    try:
        da.test_force_timeout(True)
        try:
            call()
            rc = da.check_errors()
        finally:
            da.test_force_timeout(False)
        assert rc == 5  # DECATTN_ERR_TIMEOUT
        out, lse = call()
        assert da.check_errors() == 0
    finally:
        da.set_forced_splits(0)
    ks = [gqa_rows(cache, i, "k") for i in range(b)]
    vs = [gqa_rows(cache, i, "v") for i in range(b)]
    ro, rl = A.gqa_ref(f64(q), ks, vs, seqlens, 1 / math.sqrt(d))
    assert_out_close(f64(out), ro, "after timeout")
    assert_lse_close(f64(lse), rl, "after timeout")
