"""Paged-KV attention for mixed decode / extend / prefill batches on NVIDIA GB300 (sm_103a).

The computation lives in libpkv.so (hand-written CUDA behind the C ABI of include/pkv.h);
this package only builds, loads and calls it.
"""
from .binding import (  # noqa: F401
    CLASS_DECODE, CLASS_EXTEND, CLASS_PREFILL, LayerHandoff, PkvError, Reqs, batch_classify_reorder,
    device_errors, extend_attn, extend_fp8_workspace_size, kv_block_pack, kv_block_unpack, kv_cache_write, launch_count, make_cache,
    mla_decode_attn, mla_decode_workspace_size, paged_decode_attn, paged_decode_attn_noalloc,
    paged_decode_workspace_size, selftest_bounded_wait, varlen_prefill_attn)
from ._lib import lib_path, load  # noqa: F401
