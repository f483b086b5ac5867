"""Python binding of the C ABI: torch tensors in, data pointers and sizes out.

Argument marshalling only: every step of the computation runs in libpkv.so's CUDA kernels.
Tensors must be CUDA tensors on the current device; outputs that are not passed in are
allocated here with torch (the library itself never allocates). Calls are asynchronous on the
current torch stream unless ``stream`` is given.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

CLASS_DECODE, CLASS_EXTEND, CLASS_PREFILL = _lib.CLASS_DECODE, _lib.CLASS_EXTEND, _lib.CLASS_PREFILL


class PkvError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != _lib.PKV_OK:
        raise PkvError(f"{what}: {_lib.STATUS.get(status, status)}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, dtype, name: str, contiguous: bool = True):
    if not t.is_cuda:
        raise PkvError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise PkvError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise PkvError(f"{name} must be contiguous")


def make_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: float = 1.0,
               v_scale: float = 1.0) -> "_lib.PkvCache":
    """Describe one layer's paged cache: k_cache / v_cache [num_blocks, block_size, Hkv, D]
    with contiguous blocks (any stride between blocks). bf16 tensors are a bf16 cache; uint8
    or float8_e4m3fn tensors are an FP8 (E4M3) cache whose codes stand for e4m3(code) * scale."""
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    want = k_cache.dtype if fp8 else torch.bfloat16
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, want, n, contiguous=False)
        nb, bs, hkv, d = t.shape
        if t.stride()[1:] != (hkv * d, d, 1):
            raise PkvError(f"{n}: each block must be contiguous [block_size, Hkv, D]")
    if k_cache.shape != v_cache.shape or k_cache.stride(0) != v_cache.stride(0):
        raise PkvError("k_cache and v_cache must have the same shape and block stride")
    nb, bs, hkv, d = k_cache.shape
    return _lib.PkvCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, k_cache.stride(0),
                         _lib.KV_FP8_E4M3 if fp8 else _lib.KV_BF16, float(k_scale), float(v_scale))


@dataclass
class Reqs:
    """A request set (pkv_reqs): order[bounds[cls]:bounds[cls+1]] when bounds is given, else
    order[:max_reqs] (or 0..max_reqs-1 without order). batch_reqs = R of the batch arrays."""
    max_reqs: int
    batch_reqs: int
    order: Optional[torch.Tensor] = None
    bounds: Optional[torch.Tensor] = None
    cls: int = 0

    def c(self) -> "_lib.PkvReqs":
        return _lib.PkvReqs(self.order.data_ptr() if self.order is not None else None,
                            self.bounds.data_ptr() if self.bounds is not None else None,
                            self.cls, self.max_reqs, self.batch_reqs)


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache, stream=None, k_scale=1.0, v_scale=1.0):
    """Scatter key/value [T, Hkv, D] into the cache slots given by slot_mapping (int64 [T]);
    into an FP8 cache, quantised with the per-tensor scales."""
    lib = _lib.load()
    _need(key, torch.bfloat16, "key")
    _need(value, torch.bfloat16, "value")
    _need(slot_mapping, torch.int64, "slot_mapping")
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    _check(lib.pkv_kv_cache_write(_ptr(key), _ptr(value), _ptr(slot_mapping), slot_mapping.numel(),
                                  cache, _stream(stream)), "kv_cache_write")


def kv_block_pack(k_cache, v_cache, block_ids, dst=None, stream=None):
    """dst [2, n, block_size, Hkv, D] = (k_cache[block_ids], v_cache[block_ids])."""
    lib = _lib.load()
    _need(block_ids, torch.int32, "block_ids")
    cache = make_cache(k_cache, v_cache)
    n = block_ids.numel()
    if dst is None:
        dst = torch.empty((2, n) + tuple(k_cache.shape[1:]), dtype=k_cache.dtype, device=k_cache.device)
    _need(dst, k_cache.dtype, "dst")
    _check(lib.pkv_kv_block_pack(cache, _ptr(block_ids), n, _ptr(dst), _stream(stream)), "kv_block_pack")
    return dst


def kv_block_unpack(src, block_ids, k_cache, v_cache, stream=None):
    """k_cache[block_ids[i]] = src[0][i], v_cache[block_ids[i]] = src[1][i] (in place)."""
    lib = _lib.load()
    _need(src, k_cache.dtype, "src")
    _need(block_ids, torch.int32, "block_ids")
    cache = make_cache(k_cache, v_cache)
    n = block_ids.numel()
    if tuple(src.shape) != (2, n) + tuple(k_cache.shape[1:]):
        raise ValueError(f"src shape {tuple(src.shape)} does not match 2 x {n} blocks of {tuple(k_cache.shape[1:])}")
    _check(lib.pkv_kv_block_unpack(_ptr(src), _ptr(block_ids), n, cache, _stream(stream)), "kv_block_unpack")


class LayerHandoff:
    """Per-layer handoff staging on a copy stream of its own (pkv_handoff_*): stage(slot, ...)
    packs one layer's blocks into dst after the work already on the compute stream, without
    holding up the compute stream; ready(slot, stream) orders a consumer after that pack;
    release(slot, stream) orders the slot's next stage after the consumer."""

    def __init__(self, num_slots: int, copy_stream: Optional[torch.cuda.Stream] = None):
        lib = _lib.load()
        self.copy_stream = copy_stream if copy_stream is not None else torch.cuda.Stream()
        self.num_slots = int(num_slots)
        h = ctypes.c_void_p()
        _check(lib.pkv_handoff_create(self.num_slots, _stream(self.copy_stream), ctypes.byref(h)), "handoff_create")
        self._h = h

    def stage(self, slot, k_cache, v_cache, block_ids, dst=None, compute_stream=None):
        lib = _lib.load()
        _need(block_ids, torch.int32, "block_ids")
        cache = make_cache(k_cache, v_cache)
        n = block_ids.numel()
        if dst is None:
            # allocated on the copy stream's behalf: the caching allocator must not hand it to
            # other work before the pack that writes it is done
            with torch.cuda.stream(self.copy_stream):
                dst = torch.empty((2, n) + tuple(k_cache.shape[1:]), dtype=k_cache.dtype, device=k_cache.device)
        _need(dst, k_cache.dtype, "dst")
        _check(lib.pkv_handoff_stage(self._h, int(slot), cache, _ptr(block_ids), n, _ptr(dst), _stream(compute_stream)),
               "handoff_stage")
        return dst

    def ready(self, slot, stream=None):
        _check(_lib.load().pkv_handoff_ready(self._h, int(slot), _stream(stream)), "handoff_ready")

    def release(self, slot, stream=None):
        _check(_lib.load().pkv_handoff_release(self._h, int(slot), _stream(stream)), "handoff_release")

    def close(self):
        if self._h is not None and self._h.value:
            _check(_lib.load().pkv_handoff_destroy(self._h), "handoff_destroy")
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def selftest_bounded_wait(limit_ns=10_000_000, stream=None):
    """Run a kernel whose barrier wait must run out after limit_ns (sets the TIMEOUT bit of the
    device error word; the context stays usable)."""
    _check(_lib.load().pkv_selftest_bounded_wait(int(limit_ns), _stream(stream)), "selftest_bounded_wait")


def batch_classify_reorder(cu_q, seq_lens, decode_threshold=1, perm=None, bounds=None,
                           cu_q_reordered=None, token_map=None, with_token_map=False,
                           num_tokens=None, stream=None):
    """Returns (perm, bounds[4], cu_q_reordered, token_map or None)."""
    lib = _lib.load()
    _need(cu_q, torch.int32, "cu_q")
    _need(seq_lens, torch.int32, "seq_lens")
    R = seq_lens.numel()
    dev = seq_lens.device
    perm = perm if perm is not None else torch.empty(R, dtype=torch.int32, device=dev)
    bounds = bounds if bounds is not None else torch.empty(4, dtype=torch.int32, device=dev)
    cu_q_reordered = cu_q_reordered if cu_q_reordered is not None else torch.empty(R + 1, dtype=torch.int32, device=dev)
    if with_token_map and token_map is None:
        if num_tokens is None:
            raise PkvError("num_tokens (host) is needed for the token map")
        token_map = torch.empty(num_tokens, dtype=torch.int32, device=dev)
    T = token_map.numel() if token_map is not None else (num_tokens or 0)
    _check(lib.pkv_batch_classify_reorder(_ptr(cu_q), _ptr(seq_lens), R, decode_threshold, _ptr(perm),
                                          _ptr(bounds), _ptr(cu_q_reordered), _ptr(token_map), T,
                                          _stream(stream)), "batch_classify_reorder")
    return perm, bounds, cu_q_reordered, token_map


def _scale(scale, D):
    return float(scale) if scale is not None else 1.0 / math.sqrt(D)


def paged_decode_workspace_size(max_reqs, Hq, Hkv, D, max_seq_len) -> int:
    return int(_lib.load().pkv_paged_decode_workspace_size(max_reqs, Hq, Hkv, D, max_seq_len))


def paged_decode_attn(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, cu_q=None,
                      reqs: Optional[Reqs] = None, scale=None, out=None, lse=None, workspace=None,
                      stream=None, k_scale=1.0, v_scale=1.0):
    """One query token per request against its paged context. q [T, Hq, D]. An FP8 cache is
    dequantised with the per-tensor scales as it is read."""
    lib = _lib.load()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    T, Hq, D = q.shape
    R = seq_lens.numel()
    reqs = reqs or Reqs(max_reqs=R, batch_reqs=R)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    need = lib.pkv_paged_decode_workspace_size(reqs.max_reqs, Hq, cache.num_kv_heads, D, max_seq_len)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.pkv_paged_decode_attn(_ptr(q), cache, _ptr(block_tables), block_tables.shape[1],
                                     _ptr(seq_lens), _ptr(cu_q), reqs.c(), Hq, max_seq_len,
                                     _scale(scale, D), _ptr(out), _ptr(lse), _ptr(workspace),
                                     need, _stream(stream)), "paged_decode_attn")
    return out, lse


def paged_decode_attn_noalloc(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, out, lse,
                              cu_q=None, reqs: Optional[Reqs] = None, scale=None, stream=None,
                              k_scale=1.0, v_scale=1.0):
    """paged_decode_attn for callers that cannot allocate: the library uses its own fixed
    device scratch (NOALLOC_SCRATCH_BYTES per GPU) and the caller passes out and lse."""
    lib = _lib.load()
    _need(q, torch.bfloat16, "q")
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    T, Hq, D = q.shape
    R = seq_lens.numel()
    reqs = reqs or Reqs(max_reqs=R, batch_reqs=R)
    _check(lib.pkv_paged_decode_attn_noalloc(_ptr(q), cache, _ptr(block_tables), block_tables.shape[1],
                                             _ptr(seq_lens), _ptr(cu_q), reqs.c(), Hq, max_seq_len,
                                             _scale(scale, D), _ptr(out), _ptr(lse), _stream(stream)),
           "paged_decode_attn_noalloc")
    return out, lse


def mla_decode_attn(q, latent_cache, block_tables, seq_lens, max_seq_len, scale, v_dim=512, cu_q=None,
                    reqs: Optional[Reqs] = None, out=None, lse=None, workspace=None, stream=None):
    """Absorbed MLA decode. q [T, Hq, 576]; latent_cache [num_blocks, 16, 1, 576] bf16 (keys =
    all 576 dims of a token's latent row, values = its first v_dim). Returns out [T, Hq, v_dim]
    and lse [T, Hq]. The softmax scale is the model's (no default)."""
    lib = _lib.load()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    cache = make_cache(latent_cache, latent_cache)
    T, Hq, Dk = q.shape
    R = seq_lens.numel()
    reqs = reqs or Reqs(max_reqs=R, batch_reqs=R)
    if out is None:
        out = torch.empty((T, Hq, v_dim), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    need = lib.pkv_mla_decode_workspace_size(reqs.max_reqs, Hq, max_seq_len)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.pkv_mla_decode_attn(_ptr(q), cache, _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                   _ptr(cu_q), reqs.c(), Hq, max_seq_len, float(scale), int(v_dim), _ptr(out),
                                   _ptr(lse), _ptr(workspace), need, _stream(stream)), "mla_decode_attn")
    return out, lse


def mla_decode_workspace_size(max_reqs, num_q_heads, max_seq_len) -> int:
    return int(_lib.load().pkv_mla_decode_workspace_size(max_reqs, num_q_heads, max_seq_len))


def extend_attn(q, k_new, v_new, cu_q, seq_lens, k_cache, v_cache, block_tables, max_q_len,
                max_seq_len, reqs: Optional[Reqs] = None, chunk_budget_tokens=32768, scale=None,
                out=None, lse=None, stream=None, k_scale=1.0, v_scale=1.0, workspace=None):
    """New tokens attend to their cached context (paged) and causally to themselves. An FP8
    cache (uint8 / float8 codes with per-tensor scales) is read as codes and converted in the
    kernel at head_dim 128; at head_dim 64 it is gathered into a bf16 workspace of the set's
    context first (allocated here when not given)."""
    lib = _lib.load()
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n)
    _need(cu_q, torch.int32, "cu_q")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(block_tables, torch.int32, "block_tables")
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    T, Hq, D = q.shape
    R = seq_lens.numel()
    reqs = reqs or Reqs(max_reqs=R, batch_reqs=R)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    need = 0
    if cache.kv_dtype == _lib.KV_FP8_E4M3:
        need = extend_fp8_workspace_size(reqs.max_reqs, reqs.batch_reqs, max_seq_len, block_tables.shape[1],
                                         cache.num_kv_heads, cache.head_dim)
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.pkv_extend_attn(_ptr(q), _ptr(k_new), _ptr(v_new), T, _ptr(cu_q), _ptr(seq_lens), cache,
                               _ptr(block_tables), block_tables.shape[1], reqs.c(), Hq, max_q_len,
                               max_seq_len, chunk_budget_tokens, _scale(scale, D), _ptr(out),
                               _ptr(lse), _ptr(workspace) if need else None, need, _stream(stream)), "extend_attn")
    return out, lse


def extend_fp8_workspace_size(max_reqs, batch_reqs, max_seq_len, max_blocks, num_kv_heads, head_dim) -> int:
    return int(_lib.load().pkv_extend_fp8_workspace_size(max_reqs, batch_reqs, max_seq_len, max_blocks,
                                                         num_kv_heads, head_dim))


def varlen_prefill_attn(q, k, v, cu_seqlens, max_seqlen, reqs: Optional[Reqs] = None, scale=None,
                        out=None, lse=None, stream=None):
    """Causal attention over packed variable-length prompts."""
    lib = _lib.load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    R = cu_seqlens.numel() - 1
    reqs = reqs or Reqs(max_reqs=R, batch_reqs=R)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    _check(lib.pkv_varlen_prefill_attn(_ptr(q), _ptr(k), _ptr(v), T, _ptr(cu_seqlens), reqs.c(), Hq,
                                       Hkv, D, max_seqlen, _scale(scale, D), _ptr(out), _ptr(lse),
                                       _stream(stream)), "varlen_prefill_attn")
    return out, lse


def device_errors(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return (then clear) the device error word."""
    lib = _lib.load()
    flags = ctypes.c_uint32(0)
    st = lib.pkv_device_errors(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    if st not in (0, 5):
        _check(st, "device_errors")
    return int(flags.value)


def launch_count(reset: bool = False) -> int:
    return int(_lib.load().pkv_launch_count(1 if reset else 0))
