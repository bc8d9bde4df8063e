"""Shared test utilities: tolerance checks and oracle calls on torch inputs.

Tolerances (float outputs, bf16 out / fp32 accumulate):
  max |gpu - oracle| <= 2e-2, mean |gpu - oracle| <= 2e-3,
  relative RMS ||gpu - oracle|| / ||oracle|| <= 1e-2 (bf16 output rounding
  alone is about 2^-9 = 2e-3 relative), LSE within 1e-3 absolute.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
REL_RMS = 1e-2
LSE_ABS = 1e-3


def f64(t):
    return t.detach().float().double().cpu().numpy()


def assert_out_close(got, ref, what="", max_abs=MAX_ABS, mean_abs=MEAN_ABS, rel_rms=REL_RMS):
    """The absolute bounds are stated for unit-scale outputs: outputs whose
    RMS exceeds 1 (e.g. sharp-softmax cases, absorbed queries of large
    inputs) are first divided by that RMS."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    unit = max(1.0, float(np.sqrt(np.mean(ref ** 2)))) if ref.size else 1.0
    got, ref = got / unit, ref / unit
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max|err| {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean|err| {err.mean():.3e} > {mean_abs}"
    den = np.sqrt(np.mean(ref ** 2))
    if den > 0:
        rr = np.sqrt(np.mean(err ** 2)) / den
        assert rr <= rel_rms, f"{what}: rel-RMS {rr:.3e} > {rel_rms}"


def assert_lse_close(got, ref, what="", tol=LSE_ABS):
    """tol may be a scalar or an array of per-row bounds."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), f"{what}: -inf pattern differs"
    if fin.any():
        tol = np.broadcast_to(np.asarray(tol, np.float64), ref.shape)
        e = np.abs(got[fin] - ref[fin])
        worst = int(np.argmax(e - tol[fin]))
        assert np.all(e <= tol[fin]), f"{what}: LSE err {e[worst]:.3e} > bound {tol[fin][worst]:.3e}"
    assert np.all(got[~fin] == -np.inf)


def qz_rounding_lse_bound(qz_exact, o_lat_exact, scale):
    """Per-row bound on the LSE change caused by rounding Qz to bf16 between
    the absorb and latent kernels (the pipeline's stage boundary):
    to first order dLSE = scale * dQz . O_lat with |dQz_i| <= 2^-9 |Qz_i|
    (bf16 round-to-nearest), so |dLSE| <= scale * 2^-9 * sum_i |Qz_i| |O_lat_i|.
    Returned with the 1e-3 allowance added."""
    return LSE_ABS + scale * 2.0 ** -9 * np.sum(np.abs(qz_exact) * np.abs(o_lat_exact), axis=-1)


def key_rounding_lse_bound(q_rows, keys_exact, rounded_cols, lse_exact, counts, scale):
    """Per-row bound on the LSE change caused by storing keys in bf16 (the expanded
    form's decompressed cache; the oracle keeps them exact): to first order
    dLSE = sum_m P_m dx_m with dx_m = scale * sum_i q_i dK_mi and |dK_mi| <= 2^-9 |K_mi|
    on the rounded columns, so |dLSE| <= scale * 2^-9 * sum_m P_m sum_i |q_i| |K_mi|.
    q_rows [R, dk], keys_exact [L, dk], counts[r] keys seen by row r, P from the exact
    logits and LSE. Returned with the 1e-3 allowance added."""
    q_rows = np.asarray(q_rows, np.float64)
    keys_exact = np.asarray(keys_exact, np.float64)
    x = scale * (q_rows @ keys_exact.T)
    mag = np.abs(keys_exact[:, rounded_cols]) @ np.abs(q_rows[:, rounded_cols]).T  # [L, R]
    out = np.full(q_rows.shape[0], LSE_ABS)
    for r in range(q_rows.shape[0]):
        n = int(counts[r])
        if n > 0 and np.isfinite(lse_exact[r]):
            P = np.exp(x[r, :n] - lse_exact[r])
            out[r] += scale * 2.0 ** -9 * float(P @ mag[:n, r])
    return out


# ---------------------------------------------------------------------------
# the checker's view of a cache: sequence rows in logical order, gathered from a
# paged pool by the oracle's own gather_paged (the package's helpers are not used
# on the checker side)


class _LazyPool:
    """Indexable like a [num_pages, 64, ...] array: pool[page] is that page in
    float64, fetched from the device on demand (optionally one KV head only)."""

    def __init__(self, t, kv_head=None):
        self.t, self.kv_head = t, kv_head

    def _page(self, x):
        if self.kv_head is not None:
            x = x[:, self.kv_head:self.kv_head + 1]
        return f64(x)

    def __getitem__(self, idx):
        if isinstance(idx, tuple):  # pool[:0, 0]: the empty case
            return np.zeros((0,) + self._page(self.t[0]).shape[1:])
        return self._page(self.t[int(idx)])


def cache_rows(t, i, L, block_table=None, kv_head=None, page_size=64):
    """Rows [L, ...] of sequence i in logical order as float64: a contiguous
    cache [b, capacity, ...] is sliced, a paged pool [num_pages, 64, ...] is
    gathered with oracle.attention.gather_paged through block_table [b, max_pages]."""
    from oracle import attention as A

    if block_table is None:
        x = t[i, :L]
        if kv_head is not None:
            x = x[:, kv_head:kv_head + 1]
        return f64(x)
    return A.gather_paged(_LazyPool(t, kv_head), block_table[i].cpu().numpy(), L, page_size)


def gqa_rows(cache, i, which, kv_head=None):
    """K or V rows of sequence i of a workloads.KVCache (checker side)."""
    t = cache.k if which == "k" else cache.v
    return cache_rows(t, i, cache.seqlens[i], cache.block_table if cache.paged else None, kv_head)


def mla_rows(inp, i, which):
    """Z or K_pe rows of sequence i of workloads.MLAInputs (checker side)."""
    t = inp.z if which == "z" else inp.k_pe
    return cache_rows(t, i, inp.seqlens[i], inp.block_table if inp.paged else None)


def as_device_bf16(rows, like):
    """fp64 rows (exact bf16 values) back to a bf16 tensor on `like`'s device."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(rows)).to(device=like.device, dtype=torch.bfloat16)
