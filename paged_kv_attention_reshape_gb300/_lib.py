"""ctypes declarations of libpkv.so (include/pkv.h). Loading fails loudly when the library is
missing: there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

P = ctypes.c_void_p
i32, i64, f32, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

PKV_OK = 0
NOALLOC_SCRATCH_BYTES = 32 << 20  # PKV_NOALLOC_SCRATCH_BYTES
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace", 4: "CUDA error",
          5: "device-side index error"}
DEVERR = {0x1: "slot", 0x2: "block", 0x4: "reqs", 0x8: "len", 0x10: "timeout"}
CLASS_DECODE, CLASS_EXTEND, CLASS_PREFILL = 0, 1, 2


KV_BF16, KV_FP8_E4M3 = 0, 1


class PkvCache(ctypes.Structure):
    _fields_ = [("k", P), ("v", P), ("num_blocks", i64), ("block_size", i32),
                ("num_kv_heads", i32), ("head_dim", i32), ("stride_block", i64),
                ("kv_dtype", i32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class PkvReqs(ctypes.Structure):
    _fields_ = [("order", P), ("bounds", P), ("cls", i32), ("max_reqs", i32), ("batch_reqs", i32)]


# (name, restype, argtypes) of every exported entry point; the tests check this list against
# include/pkv.h and the library's symbol table.
SIGNATURES = [
    ("pkv_status_string", ctypes.c_char_p, [i32]),
    ("pkv_kv_cache_write", i32, [P, P, P, i64, PkvCache, P]),
    ("pkv_batch_classify_reorder", i32, [P, P, i32, i32, P, P, P, P, i64, P]),
    ("pkv_paged_decode_workspace_size", sz, [i32, i32, i32, i32, i32]),
    ("pkv_paged_decode_attn", i32, [P, PkvCache, P, i32, P, P, PkvReqs, i32, i32, f32, P, P, P, sz, P]),
    ("pkv_paged_decode_attn_noalloc", i32, [P, PkvCache, P, i32, P, P, PkvReqs, i32, i32, f32, P, P, P]),
    ("pkv_mla_decode_workspace_size", sz, [i32, i32, i32]),
    ("pkv_extend_fp8_workspace_size", sz, [i32, i32, i32, i32, i32, i32]),
    ("pkv_mla_decode_attn", i32, [P, PkvCache, P, i32, P, P, PkvReqs, i32, i32, f32, i32, P, P, P, sz, P]),
    ("pkv_extend_workspace_size", sz, [i32, i32, i32, i32, i32]),
    ("pkv_extend_attn", i32, [P, P, P, i64, P, P, PkvCache, P, i32, PkvReqs, i32, i32, i32, i32, f32,
                              P, P, P, sz, P]),
    ("pkv_varlen_prefill_attn", i32, [P, P, P, i64, P, PkvReqs, i32, i32, i32, i32, f32, P, P, P]),
    ("pkv_kv_block_pack", i32, [PkvCache, P, i32, P, P]),
    ("pkv_kv_block_unpack", i32, [P, P, i32, PkvCache, P]),
    ("pkv_handoff_create", i32, [i32, P, P]),
    ("pkv_handoff_stage", i32, [P, i32, PkvCache, P, i32, P, P]),
    ("pkv_handoff_ready", i32, [P, i32, P]),
    ("pkv_handoff_release", i32, [P, i32, P]),
    ("pkv_handoff_destroy", i32, [P]),
    ("pkv_selftest_bounded_wait", i32, [ctypes.c_uint64, P]),
    ("pkv_device_errors", i32, [P, i32, P]),
    ("pkv_launch_count", i64, [i32]),
]

_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libpkv.so (building it first when it is missing and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path) or not _build.up_to_date():
            if not build_if_missing:
                raise RuntimeError(f"libpkv.so not built at {path}; run __graft_entry__.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
