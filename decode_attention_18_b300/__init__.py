"""B300-native (sm_103a) decode attention: grouped-head (MHA / GQA / MQA)
split-KV decode, absorbed latent MLA and the expanded (decompressed) MLA form,
behind the C ABI of include/decattn.h. The native library is loaded on first
use."""
from ._native import DecAttnError, LIB_PATH, SYMBOLS  # noqa: F401
from .ops import (  # noqa: F401
    attn_merge_lse,
    check_errors,
    gqa_decode,
    gqa_decode_dv,
    gqa_decode_fp8,
    last_num_splits,
    mla_absorb_q,
    mla_decode,
    mla_decompress_kv,
    mla_forward,
    mla_out_proj,
    mla_split_forward,
    set_forced_splits,
    set_grouped_kernel,
    set_wait_limit_ns,
    test_force_timeout,
)

__all__ = [
    "gqa_decode", "gqa_decode_dv", "gqa_decode_fp8", "mla_decompress_kv", "mla_absorb_q", "mla_decode", "mla_out_proj", "mla_forward",
    "attn_merge_lse", "mla_split_forward",
    "check_errors", "set_forced_splits", "set_grouped_kernel", "last_num_splits", "set_wait_limit_ns", "test_force_timeout", "DecAttnError",
]
