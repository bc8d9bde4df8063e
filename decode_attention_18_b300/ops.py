"""Python binding of the C ABI: argument marshalling only.

Every function takes CUDA torch tensors (bf16 unless stated), derives the
sizes from their shapes, allocates outputs and the split workspace with torch
when the caller passes none, and calls the same-named C entry point on the
current torch stream. All computation happens in the native kernels; a
non-zero status raises DecAttnError.
"""
from __future__ import annotations

import ctypes
import math

import torch

from ._native import KV, check, load

_BF16 = torch.bfloat16


def _need(t, name, dtype=_BF16):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _kv_desc(cache, block_table, page_size=64):
    if block_table is None:
        return KV(0, int(cache.shape[1]), None, 0, 0, 0)
    _need(block_table, "block_table", torch.int32)
    return KV(1, 0, block_table.data_ptr(), int(block_table.shape[1]), int(page_size), int(cache.shape[0]))


def _max_seqlen(seqlens, max_seqlen):
    return int(seqlens.max().item()) if max_seqlen is None else int(max_seqlen)


def _workspace(nbytes, workspace, device):
    if nbytes == 0:
        return None, 0
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace, workspace.numel() * workspace.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def gqa_decode(q, k, v, seqlens, *, max_seqlen=None, scale=None, block_table=None, out=None, lse=None,
               return_lse=True, workspace=None, stream=None):
    """Grouped-head decode attention (MHA / GQA / MQA).

    q [b, Hq, s, d]; k, v contiguous [b, capacity, Hkv, d] or, with
    block_table [b, max_pages] int32, paged [num_pages, 64, Hkv, d];
    seqlens int32 [b] on the device (keys including the s new tokens).
    Returns (out [b, Hq, s, d] bf16, lse [b, Hq, s] fp32 or None)."""
    lib = load()
    _need(q, "q"), _need(k, "k"), _need(v, "v"), _need(seqlens, "seqlens", torch.int32)
    b, hq, s, d = (int(x) for x in q.shape)
    hkv = int(k.shape[2])
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    L = _max_seqlen(seqlens, max_seqlen)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((b, hq, s), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(lib.gqa_decode_workspace_size(b, s, hq, hkv, d, L), workspace, q.device)
    check(lib.gqa_decode(_p(q), _p(k), _p(v), _kv_desc(k, block_table), _p(seqlens), L, b, s, hq, hkv, d, scale,
                         _p(out), _p(lse), _p(ws), wsb, _stream(stream)), "gqa_decode")
    return out, lse


def gqa_decode_dv(q, k, v, seqlens, *, scale, max_seqlen=None, block_table=None, out=None, lse=None,
                  return_lse=True, workspace=None, stream=None):
    """Grouped-head decode with value rows of their own width: q [b, Hq, s, dk],
    k [b, capacity, Hkv, dk], v [b, capacity, Hkv, dv] (or paged pools with
    block_table). Returns (out [b, Hq, s, dv] bf16, lse [b, Hq, s] or None)."""
    lib = load()
    _need(q, "q"), _need(k, "k"), _need(v, "v"), _need(seqlens, "seqlens", torch.int32)
    b, hq, s, dk = (int(x) for x in q.shape)
    hkv, dv = int(k.shape[2]), int(v.shape[3])
    L = _max_seqlen(seqlens, max_seqlen)
    if out is None:
        out = torch.empty((b, hq, s, dv), dtype=_BF16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((b, hq, s), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(lib.gqa_decode_dv_workspace_size(b, s, hq, hkv, dk, dv, L), workspace, q.device)
    check(lib.gqa_decode_dv(_p(q), _p(k), _p(v), _kv_desc(k, block_table), _p(seqlens), L, b, s, hq, hkv, dk, dv,
                            float(scale), _p(out), _p(lse), _p(ws), wsb, _stream(stream)), "gqa_decode_dv")
    return out, lse


def gqa_decode_fp8(q, k8, v8, seqlens, *, k_scale, v_scale, max_seqlen=None, scale=None, block_table=None, out=None,
                   lse=None, return_lse=True, workspace=None, stream=None):
    """Grouped-head decode over an FP8 (E4M3) cache: k8, v8 uint8 tensors in the
    layouts of gqa_decode (one byte per value) standing for k_scale * K and
    v_scale * V. q [b, Hq, s, d] bf16. Returns (out [b, Hq, s, d] bf16, lse)."""
    lib = load()
    _need(q, "q"), _need(k8, "k8", torch.uint8), _need(v8, "v8", torch.uint8)
    _need(seqlens, "seqlens", torch.int32)
    b, hq, s, d = (int(x) for x in q.shape)
    hkv = int(k8.shape[2])
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    L = _max_seqlen(seqlens, max_seqlen)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((b, hq, s), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(lib.gqa_decode_fp8_workspace_size(b, s, hq, hkv, d, L), workspace, q.device)
    check(lib.gqa_decode_fp8(_p(q), _p(k8), _p(v8), _kv_desc(k8, block_table), _p(seqlens), L, b, s, hq, hkv, d, scale,
                             float(k_scale), float(v_scale), _p(out), _p(lse), _p(ws), wsb, _stream(stream)),
          "gqa_decode_fp8")
    return out, lse


def mla_decompress_kv(z, k_pe, w_uk, w_uv, *, k_out=None, v_out=None, stream=None):
    """Expanded-form cache: K = [Z W_uk^T || K_pe], V = Z W_uv for every cache row.
    z [..., k] and k_pe [..., p] with the same leading (row) shape, w_uk [h, d, k],
    w_uv [h, k, d]. Returns (k_out [..., h, d + p], v_out [..., h, d])."""
    lib = load()
    for t, n in ((z, "z"), (k_pe, "k_pe"), (w_uk, "w_uk"), (w_uv, "w_uv")):
        _need(t, n)
    lead = tuple(int(x) for x in z.shape[:-1])
    rows = int(math.prod(lead))
    k, p = int(z.shape[-1]), int(k_pe.shape[-1])
    h, d = int(w_uk.shape[0]), int(w_uk.shape[1])
    if k_out is None:
        k_out = torch.empty(lead + (h, d + p), dtype=_BF16, device=z.device)
    if v_out is None:
        v_out = torch.empty(lead + (h, d), dtype=_BF16, device=z.device)
    check(lib.mla_decompress_kv(_p(z), _p(k_pe), _p(w_uk), _p(w_uv), rows, h, d, k, p, _p(k_out), _p(v_out),
                                _stream(stream)), "mla_decompress_kv")
    return k_out, v_out


def mla_absorb_q(q_nope, w_uk, seqlens=None, *, scale=1.0, out=None, stream=None):
    """Qz = scale * q_nope @ W_uk per head. q_nope [b, h, s, d], w_uk [h, d, k]."""
    lib = load()
    _need(q_nope, "q_nope"), _need(w_uk, "w_uk")
    b, h, s, d = (int(x) for x in q_nope.shape)
    k = int(w_uk.shape[2])
    if out is None:
        out = torch.empty((b, h, s, k), dtype=_BF16, device=q_nope.device)
    if seqlens is not None:
        _need(seqlens, "seqlens", torch.int32)
    check(lib.mla_absorb_q(_p(q_nope), _p(w_uk), _p(out), _p(seqlens), b, s, h, d, k, float(scale),
                           _stream(stream)), "mla_absorb_q")
    return out


def mla_decode(qz, q_pe, z, k_pe, seqlens, *, scale, max_seqlen=None, block_table=None, out=None, lse=None,
               return_lse=True, workspace=None, stream=None):
    """Latent attention. qz [b, h, s, k], q_pe [b, h, s, p]; z [b, cap, k] and
    k_pe [b, cap, p] (or paged [num_pages, 64, k] / [num_pages, 64, p] with
    block_table). Returns (o_lat [b, h, s, k] bf16, lse [b, h, s] or None)."""
    lib = load()
    for t, n in ((qz, "qz"), (q_pe, "q_pe"), (z, "z"), (k_pe, "k_pe")):
        _need(t, n)
    _need(seqlens, "seqlens", torch.int32)
    b, h, s, k = (int(x) for x in qz.shape)
    p = int(q_pe.shape[3])
    L = _max_seqlen(seqlens, max_seqlen)
    if out is None:
        out = torch.empty_like(qz)
    if lse is None and return_lse:
        lse = torch.empty((b, h, s), dtype=torch.float32, device=qz.device)
    ws, wsb = _workspace(lib.mla_decode_workspace_size(b, s, h, k, L), workspace, qz.device)
    check(lib.mla_decode(_p(qz), _p(q_pe), _p(z), _p(k_pe), _kv_desc(z, block_table), _p(seqlens), L, b, s, h, k, p,
                         float(scale), _p(out), _p(lse), _p(ws), wsb, _stream(stream)), "mla_decode")
    return out, lse


def mla_out_proj(o_lat, w_uv, seqlens=None, *, scale=1.0, out=None, stream=None):
    """O = scale * o_lat @ W_uv per head. o_lat [b, h, s, k], w_uv [h, k, d]."""
    lib = load()
    _need(o_lat, "o_lat"), _need(w_uv, "w_uv")
    b, h, s, k = (int(x) for x in o_lat.shape)
    d = int(w_uv.shape[2])
    if out is None:
        out = torch.empty((b, h, s, d), dtype=_BF16, device=o_lat.device)
    if seqlens is not None:
        _need(seqlens, "seqlens", torch.int32)
    check(lib.mla_out_proj(_p(o_lat), _p(w_uv), _p(out), _p(seqlens), b, s, h, k, d, float(scale),
                           _stream(stream)), "mla_out_proj")
    return out


def mla_forward(q_nope, q_pe, z, k_pe, w_uk, w_uv, seqlens, *, scale, max_seqlen=None, block_table=None,
                workspace=None, stream=None):
    """The absorbed pipeline: absorb -> latent attention (+ combine) -> W_uv.
    Returns (out [b, h, s, d], lse, qz, o_lat)."""
    qz = mla_absorb_q(q_nope, w_uk, seqlens, stream=stream)
    o_lat, lse = mla_decode(qz, q_pe, z, k_pe, seqlens, scale=scale, max_seqlen=max_seqlen,
                            block_table=block_table, workspace=workspace, stream=stream)
    out = mla_out_proj(o_lat, w_uv, seqlens, stream=stream)
    return out, lse, qz, o_lat


def attn_merge_lse(out_a, lse_a, out_b, lse_b, *, out=None, lse=None, stream=None):
    """LSE merge of two results over disjoint key sets of the same rows:
    out_a, out_b [..., d] bf16 and lse_a, lse_b [...] fp32. Returns (out, lse)."""
    lib = load()
    _need(out_a, "out_a"), _need(out_b, "out_b")
    _need(lse_a, "lse_a", torch.float32), _need(lse_b, "lse_b", torch.float32)
    d = int(out_a.shape[-1])
    rows = int(out_a.numel()) // d
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    check(lib.attn_merge_lse(_p(out_a), _p(lse_a), _p(out_b), _p(lse_b), rows, d, _p(out), _p(lse),
                             _stream(stream)), "attn_merge_lse")
    return out, lse


def mla_split_forward(q_nope, q_pe, q_full, z, k_pe, k_recent, v_recent, w_uk, w_uv, seqlens_old, seqlens_recent, *,
                      scale, max_old, max_recent, block_table=None, recent_block_table=None, workspace=None,
                      stream=None):
    """The hybrid form ("Mla Analysis", MLAvar6+ Design): the o_i older keys of
    sequence i attended in latent form, its n_i most recent keys in decompressed
    form, the two merged by log-sum-exp.

    z [b, cap, k] / k_pe [b, cap, p] (or paged with block_table): the latent cache,
    of which keys 0 .. o_i - 1 are read (seqlens_old = o_i). k_recent
    [b, cap_r, h, d + p] / v_recent [b, cap_r, h, d] (or paged with
    recent_block_table): the decompressed recent keys, o_i .. o_i + n_i - 1, as
    mla_decompress_kv writes them (seqlens_recent = n_i >= s: the s new tokens are
    the last of them, causal among themselves). q_full = [q_nope || q_pe] per head.
    Every new token sees all o_i older keys. Returns (out [b, h, s, d], lse)."""
    b, h, s, k = int(q_nope.shape[0]), int(q_nope.shape[1]), int(q_nope.shape[2]), int(w_uk.shape[2])
    p = int(q_pe.shape[3])
    qz = mla_absorb_q(q_nope, w_uk, stream=stream)
    # the older keys precede every new token: the h*s query rows of a sequence attend
    # to all o_i of them, which is the latent call with one token per row ([b, h*s, 1, .])
    o_lat, lse_a = mla_decode(qz.view(b, h * s, 1, k), q_pe.view(b, h * s, 1, p), z, k_pe, seqlens_old, scale=scale,
                              max_seqlen=max_old, block_table=block_table, workspace=workspace, stream=stream)
    out_a = mla_out_proj(o_lat.view(b, h, s, k), w_uv, stream=stream)
    out_b, lse_b = gqa_decode_dv(q_full, k_recent, v_recent, seqlens_recent, scale=scale, max_seqlen=max_recent,
                                 block_table=recent_block_table, stream=stream)
    return attn_merge_lse(out_a, lse_a.view(b, h, s), out_b, lse_b, out=out_a, stream=stream)


def check_errors(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().decattn_check_errors(_stream(stream)))


def set_forced_splits(n: int):
    load().decattn_set_forced_splits(int(n))


def last_num_splits() -> int:
    return int(load().decattn_last_num_splits())


def set_wait_limit_ns(ns: int):
    load().decattn_set_wait_limit_ns(int(ns))


def set_grouped_kernel(mode: int):
    """0 automatic, 1 split-KV kernels, 2 tensor-core kernel (diagnostics and tests)."""
    load().decattn_set_grouped_kernel(int(mode))


def test_force_timeout(on: bool):
    load().decattn_test_force_timeout(1 if on else 0)
