"""ctypes front end of the fp64 CPU oracle (``pkv_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg
use this module; the CUDA library never imports or links it, and it imports nothing from
the library. See ``pkv_oracle.cpp`` for the definitions and the passages they follow.

All array arguments are numpy arrays on the host. bf16 data is passed as its raw bits
(``np.uint16``); results come back as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler; returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_kv_bytes_per_token.argtypes = [i32, i32, i32, i32]
            lib.oracle_kv_bytes_per_token.restype = i64
            lib.oracle_kv_cache_write.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P]
            lib.oracle_kv_cache_write.restype = i64
            lib.oracle_kv_block_pack.argtypes = [P, P, i64, i64, P, i32, P]
            lib.oracle_kv_block_pack.restype = i32
            lib.oracle_kv_block_unpack.argtypes = [P, P, i32, P, P, i64, i64]
            lib.oracle_kv_block_unpack.restype = i32
            lib.oracle_batch_classify_reorder.argtypes = [P, P, i32, i32, P, P, P, P]
            lib.oracle_batch_classify_reorder.restype = None
            lib.oracle_lse_merge.argtypes = [P, P, P, P, i64, i32, P, P]
            lib.oracle_lse_merge.restype = None
            lib.oracle_paged_decode.argtypes = [P, P, P, i64, i32, i32, i32, P, i32, P, P, P,
                                                i32, i32, f64, P, P, i32]
            lib.oracle_paged_decode.restype = None
            f32 = ctypes.c_float
            lib.oracle_e4m3_decode.argtypes = [P, i64, P]
            lib.oracle_e4m3_decode.restype = None
            lib.oracle_e4m3_encode.argtypes = [P, i64, P]
            lib.oracle_e4m3_encode.restype = None
            lib.oracle_kv_cache_write_fp8.argtypes = [P, P, P, i64, i32, i32, i32, i64, f32, f32, P, P]
            lib.oracle_kv_cache_write_fp8.restype = i64
            lib.oracle_paged_decode_fp8.argtypes = [P, P, P, i64, i32, i32, i32, P, i32, P, P, P,
                                                    i32, i32, f64, f64, f64, P, P, i32]
            lib.oracle_paged_decode_fp8.restype = None
            lib.oracle_mla_decode.argtypes = [P, P, i64, i32, i32, i32, P, i32, P, P, P, i32, i32, f64, P, P, i32]
            lib.oracle_mla_decode.restype = None
            lib.oracle_extend.argtypes = [P, P, P, P, P, P, P, i64, i32, P, i32, P, i32, i32,
                                          i32, i32, f64, P, P, P, i32]
            lib.oracle_extend.restype = None
            lib.oracle_extend_fp8.argtypes = [P, P, P, P, P, P, P, i64, i32, P, i32, P, i32, i32, i32, i32,
                                              f64, f64, f64, P, P, P, i32]
            lib.oracle_extend_fp8.restype = None
            lib.oracle_extend_chunked.argtypes = [P, P, P, P, P, P, P, i64, i32, P, i32, i32,
                                                  i32, i32, i32, f64, i64, P, P]
            lib.oracle_extend_chunked.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of the given dtype (no copy when it already is one)."""
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, elem_bytes=2) -> int:
    return int(_load().oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim, elem_bytes))


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache):
    """In-place write of key/value [T, Hkv, D] (uint16 bits) into caches
    [num_blocks, bs, Hkv, D]. Returns the count of out-of-range slots."""
    lib = _load()
    key, value = _c(key, np.uint16), _c(value, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    nb, bs, hkv, d = k_cache.shape
    return int(lib.oracle_kv_cache_write(_ptr(key), _ptr(value), _ptr(slot_mapping),
                                         slot_mapping.shape[0], hkv, d, bs, nb,
                                         _ptr(k_cache), _ptr(v_cache)))


def kv_block_pack(k_cache, v_cache, block_ids, dst=None):
    """Gather whole blocks: returns dst [2, n, bs, Hkv, D] (uint16 bits)."""
    lib = _load()
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_ids = _c(block_ids, np.int32)
    nb = k_cache.shape[0]
    block_elems = int(np.prod(k_cache.shape[1:]))
    n = block_ids.shape[0]
    if dst is None:
        dst = np.zeros((2, n) + tuple(k_cache.shape[1:]), dtype=np.uint16)
    bad = lib.oracle_kv_block_pack(_ptr(k_cache), _ptr(v_cache), nb, block_elems,
                                   _ptr(block_ids), n, _ptr(dst))
    return dst, int(bad)


def kv_block_unpack(src, block_ids, k_cache, v_cache):
    """Scatter packed blocks src [2, n, bs, Hkv, D] into the caches in place (uint16 bits);
    returns the count of ids outside the pool."""
    lib = _load()
    src = _c(src, np.uint16)
    block_ids = _c(block_ids, np.int32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    nb = k_cache.shape[0]
    block_elems = int(np.prod(k_cache.shape[1:]))
    n = block_ids.shape[0]
    assert src.shape[0] == 2 and src.shape[1] == n and int(np.prod(src.shape[2:])) == block_elems
    return int(lib.oracle_kv_block_unpack(_ptr(src), _ptr(block_ids), n, _ptr(k_cache), _ptr(v_cache),
                                          nb, block_elems))


def e4m3_decode(codes):
    """float64 values of E4M3 codes (uint8)."""
    lib = _load()
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    lib.oracle_e4m3_decode(_ptr(codes), codes.size, _ptr(out))
    return out


def e4m3_encode(x):
    """E4M3 codes (round to nearest even, saturating at +-448) of float32 values."""
    lib = _load()
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib.oracle_e4m3_encode(_ptr(x), x.size, _ptr(out))
    return out


def kv_cache_write_fp8(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """Quantise bf16 rows (bits) into E4M3 caches (uint8, in place); returns bad-slot count."""
    lib = _load()
    key, value = _c(key, np.uint16), _c(value, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, hkv, D = key.shape
    nb, bs = k_cache.shape[:2]
    return int(lib.oracle_kv_cache_write_fp8(_ptr(key), _ptr(value), _ptr(slot_mapping), T, hkv, D, bs, nb,
                                             float(k_scale), float(v_scale), _ptr(k_cache), _ptr(v_cache)))


def paged_decode_fp8(q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale, v_scale, cu_q=None,
                     req_ids=None, n_req=None, nthreads=None, out=None, lse=None):
    """paged_decode over E4M3 caches (uint8 codes [nb, bs, Hkv, D]) with per-tensor scales."""
    lib = _load()
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint8), _c(v_cache, np.uint8)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    cu_q, req_ids = _c(cu_q, np.int32), _c(req_ids, np.int32)
    T, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == D and Hq % hkv == 0
    if n_req is None:
        n_req = req_ids.shape[0] if req_ids is not None else seq_lens.shape[0]
    if out is None:
        out = np.full((T, Hq, D), np.nan)
    if lse is None:
        lse = np.full((T, Hq), np.nan)
    lib.oracle_paged_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, D, _ptr(block_tables),
                                block_tables.shape[1], _ptr(seq_lens), _ptr(cu_q), _ptr(req_ids), n_req, Hq,
                                float(scale), float(k_scale), float(v_scale), _ptr(out), _ptr(lse),
                                nthreads or default_threads())
    return out, lse


def mla_decode(q, cache, block_tables, seq_lens, scale, v_dim, cu_q=None, req_ids=None, n_req=None,
               nthreads=None, out=None, lse=None):
    """Absorbed MLA decode: q [T, Hq, Dk] bits, latent cache [nb, bs, 1, Dk] bits (keys = all
    Dk dims, values = the first v_dim). Returns (out [T, Hq, v_dim], lse [T, Hq]) float64."""
    lib = _load()
    q = _c(q, np.uint16)
    cache = _c(cache, np.uint16)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    cu_q, req_ids = _c(cu_q, np.int32), _c(req_ids, np.int32)
    T, Hq, Dk = q.shape
    nb, bs = cache.shape[:2]
    assert int(np.prod(cache.shape[2:])) == Dk
    if n_req is None:
        n_req = req_ids.shape[0] if req_ids is not None else seq_lens.shape[0]
    if out is None:
        out = np.full((T, Hq, v_dim), np.nan)
    if lse is None:
        lse = np.full((T, Hq), np.nan)
    lib.oracle_mla_decode(_ptr(q), _ptr(cache), nb, bs, Dk, int(v_dim), _ptr(block_tables), block_tables.shape[1],
                          _ptr(seq_lens), _ptr(cu_q), _ptr(req_ids), n_req, Hq, float(scale), _ptr(out), _ptr(lse),
                          nthreads or default_threads())
    return out, lse


def batch_classify_reorder(cu_q, seq_lens, threshold=1):
    """Returns (perm, bounds[4], cu_q_reordered[R+1], token_map[T])."""
    lib = _load()
    cu_q, seq_lens = _c(cu_q, np.int32), _c(seq_lens, np.int32)
    R = seq_lens.shape[0]
    T = int(cu_q[R]) if R > 0 else 0
    perm = np.zeros(R, np.int32)
    bounds = np.zeros(4, np.int32)
    cu_r = np.zeros(R + 1, np.int32)
    tmap = np.zeros(T, np.int32)
    lib.oracle_batch_classify_reorder(_ptr(cu_q), _ptr(seq_lens), R, threshold, _ptr(perm),
                                      _ptr(bounds), _ptr(cu_r), _ptr(tmap))
    return perm, bounds, cu_r, tmap


def lse_merge(o_a, lse_a, o_b, lse_b):
    lib = _load()
    o_a, o_b = _c(o_a, np.float64), _c(o_b, np.float64)
    lse_a, lse_b = _c(lse_a, np.float64), _c(lse_b, np.float64)
    rows, D = o_a.reshape(-1, o_a.shape[-1]).shape
    o = np.empty_like(o_a)
    lse = np.empty_like(lse_a)
    lib.oracle_lse_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, D, _ptr(o), _ptr(lse))
    return o, lse


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, cu_q=None, req_ids=None,
                 n_req=None, nthreads=None, out=None, lse=None):
    """q [T, Hq, D] bits; caches [nb, bs, Hkv, D] bits. Returns (out, lse) float64 with
    NaN in rows that were not computed."""
    lib = _load()
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    cu_q, req_ids = _c(cu_q, np.int32), _c(req_ids, np.int32)
    T, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == D and Hq % hkv == 0
    if n_req is None:
        n_req = req_ids.shape[0] if req_ids is not None else seq_lens.shape[0]
    if out is None:
        out = np.full((T, Hq, D), np.nan)
    if lse is None:
        lse = np.full((T, Hq), np.nan)
    lib.oracle_paged_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, D,
                            _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                            _ptr(cu_q), _ptr(req_ids), n_req, Hq, float(scale), _ptr(out),
                            _ptr(lse), nthreads or default_threads())
    return out, lse


def extend(q, k_new, v_new, cu_q, scale, seq_lens=None, k_cache=None, v_cache=None,
           block_tables=None, req_ids=None, n_req=None, row_mask=None, nthreads=None,
           out=None, lse=None):
    """Extend (seq_lens given) or prefill (seq_lens None). Returns (out, lse) float64."""
    lib = _load()
    q, k_new, v_new = _c(q, np.uint16), _c(k_new, np.uint16), _c(v_new, np.uint16)
    cu_q = _c(cu_q, np.int32)
    seq_lens, req_ids = _c(seq_lens, np.int32), _c(req_ids, np.int32)
    T, Hq, D = q.shape
    hkv = k_new.shape[1]
    if k_cache is not None:
        k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        block_tables = _c(block_tables, np.int32)
        nb, bs = k_cache.shape[0], k_cache.shape[1]
        max_blocks = block_tables.shape[1]
    else:
        assert seq_lens is None
        nb, bs, max_blocks = 0, 16, 0
    if n_req is None:
        n_req = req_ids.shape[0] if req_ids is not None else cu_q.shape[0] - 1
    if row_mask is not None:
        row_mask = _c(row_mask, np.uint8)
    if out is None:
        out = np.full((T, Hq, D), np.nan)
    if lse is None:
        lse = np.full((T, Hq), np.nan)
    lib.oracle_extend(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens),
                      _ptr(k_cache), _ptr(v_cache), nb, bs, _ptr(block_tables), max_blocks,
                      _ptr(req_ids), n_req, Hq, hkv, D, float(scale), _ptr(row_mask),
                      _ptr(out), _ptr(lse), nthreads or default_threads())
    return out, lse


def prefill(q, k, v, cu_seqlens, scale, req_ids=None, n_req=None, row_mask=None, nthreads=None):
    return extend(q, k, v, cu_seqlens, scale, req_ids=req_ids, n_req=n_req, row_mask=row_mask,
                  nthreads=nthreads)


def extend_fp8(q, k_new, v_new, cu_q, seq_lens, k_cache, v_cache, block_tables, scale, k_scale, v_scale,
               req_ids=None, n_req=None, row_mask=None, nthreads=None, out=None, lse=None):
    """Extend over an FP8 cache: k_cache / v_cache uint8 E4M3 codes [nb, bs, Hkv, D] standing for
    e4m3(code) * k_scale / v_scale; new tokens bf16 bits. Returns (out, lse) float64."""
    lib = _load()
    q, k_new, v_new = _c(q, np.uint16), _c(k_new, np.uint16), _c(v_new, np.uint16)
    cu_q, seq_lens, req_ids = _c(cu_q, np.int32), _c(seq_lens, np.int32), _c(req_ids, np.int32)
    k_cache, v_cache = _c(k_cache, np.uint8), _c(v_cache, np.uint8)
    block_tables = _c(block_tables, np.int32)
    T, Hq, D = q.shape
    hkv = k_new.shape[1]
    if n_req is None:
        n_req = req_ids.shape[0] if req_ids is not None else cu_q.shape[0] - 1
    if row_mask is not None:
        row_mask = _c(row_mask, np.uint8)
    if out is None:
        out = np.full((T, Hq, D), np.nan)
    if lse is None:
        lse = np.full((T, Hq), np.nan)
    lib.oracle_extend_fp8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens), _ptr(k_cache),
                          _ptr(v_cache), k_cache.shape[0], k_cache.shape[1], _ptr(block_tables),
                          block_tables.shape[1], _ptr(req_ids), n_req, Hq, hkv, D, float(scale), float(k_scale),
                          float(v_scale), _ptr(row_mask), _ptr(out), _ptr(lse), nthreads or default_threads())
    return out, lse


def extend_chunked(q, k_new, v_new, cu_q, seq_lens, k_cache, v_cache, block_tables, scale,
                   chunk_tokens):
    lib = _load()
    q, k_new, v_new = _c(q, np.uint16), _c(k_new, np.uint16), _c(v_new, np.uint16)
    cu_q, seq_lens = _c(cu_q, np.int32), _c(seq_lens, np.int32)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    T, Hq, D = q.shape
    hkv = k_new.shape[1]
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    lib.oracle_extend_chunked(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens),
                              _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], k_cache.shape[1],
                              _ptr(block_tables), block_tables.shape[1], seq_lens.shape[0], Hq,
                              hkv, D, float(scale), int(chunk_tokens), _ptr(out), _ptr(lse))
    return out, lse
