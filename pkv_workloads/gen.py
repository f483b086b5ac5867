"""Seeded synthetic workloads: request lengths, block tables, slot mappings and bf16 values.

Recipe (shared by the tests and the benchmark):
  * values: fp32 N(0, 1) drawn by ``torch.randn`` and rounded to bf16 (round to nearest even),
    optionally multiplied by ``q_scale`` before rounding (the "peaked" variant);
  * metadata (lengths, request order, block permutation) always comes from a CPU
    ``torch.Generator`` seeded with ``seed``, so it is identical on every machine; bulk values
    come from a generator on the target device seeded with ``seed + 1``, so a batch built on
    the GPU differs in its values (not its shapes) from one built on the CPU;
  * physical blocks: a pool of ``num_blocks`` blocks, shuffled by ``randperm``; each request
    takes the next ceil(seq_len / block_size) blocks of the shuffled pool, in order, as its
    block table; unused table entries are 0;
  * the new tokens of a request sit at positions seq_len - q_len .. seq_len - 1; token i's
    slot is table[pos // block_size] * block_size + pos % block_size;
  * every pool block, referenced or not, holds random values.

Nothing here computes attention, classifies requests or moves KV data.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

DECODE, EXTEND, PREFILL = "decode", "extend", "prefill"


def randn_bf16(shape, gen: torch.Generator, device, scale: float = 1.0,
               chunk: int = 1 << 26) -> torch.Tensor:
    """bf16 tensor of N(0, scale^2) values, drawn in fp32 chunks to bound temporary memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e].copy_(x)
    return out


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    return g


def uniform_ints(lo: int, hi: int, n: int, gen: torch.Generator) -> List[int]:
    """n integers uniform in [lo, hi] (both ends included)."""
    if n == 0:
        return []
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


@dataclass
class Batch:
    """One mixed batch in arrival order, plus one layer's paged KV cache."""
    kinds: List[str]             # recipe label of each request (what the generator built)
    q_lens: List[int]
    seq_lens_list: List[int]
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    max_blocks: int
    cu_q: torch.Tensor           # int32 [R+1]
    seq_lens: torch.Tensor       # int32 [R]
    block_tables: torch.Tensor   # int32 [R, max_blocks]
    slot_mapping: torch.Tensor   # int64 [T]
    q: torch.Tensor              # bf16 [T, Hq, D]
    k_new: torch.Tensor          # bf16 [T, Hkv, D]
    v_new: torch.Tensor          # bf16 [T, Hkv, D]
    k_cache: torch.Tensor        # bf16 [num_blocks, block_size, Hkv, D]
    v_cache: torch.Tensor
    extra: Dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return len(self.q_lens)

    @property
    def T(self) -> int:
        return int(sum(self.q_lens))

    def to(self, device) -> "Batch":
        kw = dict(self.__dict__)
        for k, v in list(kw.items()):
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return Batch(**kw)


def make_batch(kinds: List[str], q_lens: List[int], seq_lens: List[int], *, Hq: int, Hkv: int,
               D: int, block_size: int = 16, num_blocks: Optional[int] = None,
               pool_factor: float = 1.2, seed: int = 0, device="cpu", q_scale: float = 1.0,
               max_blocks: Optional[int] = None, gen: Optional[torch.Generator] = None) -> Batch:
    """Lay out a batch whose request lengths are already chosen."""
    assert len(kinds) == len(q_lens) == len(seq_lens)
    g = gen if gen is not None else _cpu_gen(seed)
    R = len(q_lens)
    need = [math.ceil(s / block_size) for s in seq_lens]
    total_need = sum(need)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * total_need))
    assert num_blocks >= total_need, "pool too small"
    if max_blocks is None:
        max_blocks = max([1] + need)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    tables = torch.zeros((R, max_blocks), dtype=torch.int32)
    cur = 0
    for r in range(R):
        tables[r, :need[r]] = perm[cur:cur + need[r]]
        cur += need[r]
    cu_q = torch.zeros(R + 1, dtype=torch.int32)
    if R:
        cu_q[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu_q[-1])
    slots = torch.empty(T, dtype=torch.int64)
    tab64 = tables.to(torch.int64)
    for r in range(R):
        n, s = q_lens[r], seq_lens[r]
        if n == 0:
            continue
        pos = torch.arange(s - n, s, dtype=torch.int64)
        slots[int(cu_q[r]):int(cu_q[r + 1])] = tab64[r, pos // block_size] * block_size + pos % block_size
    dg = _dev_gen(seed, device)
    q = randn_bf16((T, Hq, D), dg, device, q_scale)
    k_new = randn_bf16((T, Hkv, D), dg, device)
    v_new = randn_bf16((T, Hkv, D), dg, device)
    k_cache = randn_bf16((num_blocks, block_size, Hkv, D), dg, device)
    v_cache = randn_bf16((num_blocks, block_size, Hkv, D), dg, device)
    dev = torch.device(device)
    return Batch(kinds=list(kinds), q_lens=list(q_lens), seq_lens_list=list(seq_lens), Hq=Hq,
                 Hkv=Hkv, D=D, block_size=block_size, num_blocks=num_blocks,
                 max_blocks=max_blocks, cu_q=cu_q.to(dev),
                 seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=dev),
                 block_tables=tables.to(dev), slot_mapping=slots.to(dev), q=q, k_new=k_new,
                 v_new=v_new, k_cache=k_cache, v_cache=v_cache)


def decode_batch(B: int, ctx_lo: int, ctx_hi: int, *, Hq: int, Hkv: int, D: int,
                 block_size: int = 16, num_blocks: Optional[int] = None, pool_factor=1.2,
                 seed: int = 0, device="cpu", q_scale: float = 1.0) -> Batch:
    """B decode requests (one new token each); context length (the new token included)
    uniform in [ctx_lo, ctx_hi]."""
    g = _cpu_gen(seed)
    seq = uniform_ints(ctx_lo, ctx_hi, B, g)
    return make_batch([DECODE] * B, [1] * B, seq, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                      num_blocks=num_blocks, pool_factor=pool_factor, seed=seed, device=device,
                      q_scale=q_scale, gen=g)


def mixed_batch(n_decode: int, decode_ctx, n_extend: int, extend_new: int, extend_ctx,
                n_prefill: int, prefill_len, *, Hq: int, Hkv: int, D: int, block_size: int = 16,
                pool_factor=1.2, seed: int = 0, device="cpu", q_scale: float = 1.0,
                shuffle: bool = True) -> Batch:
    """Decode requests (context in decode_ctx, new token included), extend requests
    (extend_new new tokens over a cached context in extend_ctx) and prefill prompts (length in
    prefill_len), in a seeded random arrival order when shuffle is set."""
    g = _cpu_gen(seed)
    dec = uniform_ints(decode_ctx[0], decode_ctx[1], n_decode, g)
    ext = uniform_ints(extend_ctx[0], extend_ctx[1], n_extend, g)
    pre = uniform_ints(prefill_len[0], prefill_len[1], n_prefill, g)
    reqs = ([(DECODE, 1, s) for s in dec] + [(EXTEND, extend_new, c + extend_new) for c in ext]
            + [(PREFILL, L, L) for L in pre])
    if shuffle and reqs:
        order = torch.randperm(len(reqs), generator=g).tolist()
        reqs = [reqs[i] for i in order]
    kinds = [r[0] for r in reqs]
    return make_batch(kinds, [r[1] for r in reqs], [r[2] for r in reqs], Hq=Hq, Hkv=Hkv, D=D,
                      block_size=block_size, pool_factor=pool_factor, seed=seed, device=device,
                      q_scale=q_scale, gen=g)


def prefill_batch(lengths: List[int], *, Hq: int, Hkv: int, D: int, seed: int = 0, device="cpu",
                  q_scale: float = 1.0) -> Batch:
    """Prefill prompts of the given lengths (cache sized for the prompts)."""
    return make_batch([PREFILL] * len(lengths), list(lengths), list(lengths), Hq=Hq, Hkv=Hkv,
                      D=D, seed=seed, device=device, q_scale=q_scale)


def extend_batch(new_lens: List[int], ctx_lens: List[int], *, Hq: int, Hkv: int, D: int,
                 seed: int = 0, device="cpu", q_scale: float = 1.0, pool_factor=1.2) -> Batch:
    """Extend requests: new_lens[i] new tokens over ctx_lens[i] cached tokens."""
    return make_batch([EXTEND] * len(new_lens), list(new_lens),
                      [c + n for c, n in zip(ctx_lens, new_lens)], Hq=Hq, Hkv=Hkv, D=D,
                      seed=seed, device=device, q_scale=q_scale, pool_factor=pool_factor)


@dataclass
class WritePackLayer:
    key: torch.Tensor            # bf16 [T, Hkv, D]
    value: torch.Tensor
    slot_mapping: torch.Tensor   # int64 [T]
    block_ids: torch.Tensor      # int32 [n]: the prompt's blocks in request order
    k_cache: torch.Tensor        # bf16 [num_blocks, bs, Hkv, D]
    v_cache: torch.Tensor


def write_pack_layers(num_layers: int, T: int, *, Hkv: int, D: int, block_size: int = 16,
                      num_blocks: Optional[int] = None, seed: int = 0, device="cpu",
                      shuffled_pack: bool = False) -> List[WritePackLayer]:
    """Per layer: one prompt of T tokens, its ceil(T / bs) blocks drawn at random distinct ids
    from the layer's pool, the matching slot mapping, and fresh random K/V rows. With
    shuffled_pack the pack order of the blocks is a random permutation of the table."""
    g = _cpu_gen(seed)
    dg = _dev_gen(seed, device)
    nblk = math.ceil(T / block_size)
    if num_blocks is None:
        num_blocks = math.ceil(1.2 * nblk)
    layers = []
    pos = torch.arange(T, dtype=torch.int64)
    for _ in range(num_layers):
        table = torch.randperm(num_blocks, generator=g)[:nblk].to(torch.int64)
        slots = table[pos // block_size] * block_size + pos % block_size
        ids = table.to(torch.int32)
        if shuffled_pack:
            ids = ids[torch.randperm(nblk, generator=g)]
        layers.append(WritePackLayer(
            key=randn_bf16((T, Hkv, D), dg, device), value=randn_bf16((T, Hkv, D), dg, device),
            slot_mapping=slots.to(device), block_ids=ids.to(device),
            k_cache=randn_bf16((num_blocks, block_size, Hkv, D), dg, device),
            v_cache=randn_bf16((num_blocks, block_size, Hkv, D), dg, device)))
    return layers


@dataclass
class MlaBatch:
    """Decode requests over a latent cache: q [B, Hq, Dk]; latent [num_blocks, block_size, 1, Dk]
    (one latent row per token); block_tables [B, max_blocks]; seq_lens [B]."""
    q: torch.Tensor
    latent: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    seq_lens_list: List[int]
    Hq: int
    Dk: int
    block_size: int
    num_blocks: int

    @property
    def R(self) -> int:
        return len(self.seq_lens_list)


def mla_batch(B: int, ctx_lo: int, ctx_hi: int, *, Hq: int, Dk: int = 576, block_size: int = 16,
              pool_factor: float = 1.2, seed: int = 0, device="cpu", q_scale: float = 1.0,
              seq_lens: Optional[List[int]] = None) -> MlaBatch:
    """B decode requests against a latent cache (the recipe above, with one latent head of Dk
    dims per token in place of separate K and V); context lengths uniform in [ctx_lo, ctx_hi]
    unless given."""
    g = _cpu_gen(seed)
    seq = list(seq_lens) if seq_lens is not None else uniform_ints(ctx_lo, ctx_hi, B, g)
    need = [math.ceil(s / block_size) for s in seq]
    num_blocks = max(1, math.ceil(pool_factor * sum(need)))
    max_blocks = max([1] + need)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    tables = torch.zeros((len(seq), max_blocks), dtype=torch.int32)
    cur = 0
    for r, n in enumerate(need):
        tables[r, :n] = perm[cur:cur + n]
        cur += n
    dg = _dev_gen(seed, device)
    q = randn_bf16((len(seq), Hq, Dk), dg, device, q_scale)
    latent = randn_bf16((num_blocks, block_size, 1, Dk), dg, device)
    dev = torch.device(device)
    return MlaBatch(q=q, latent=latent, block_tables=tables.to(dev),
                    seq_lens=torch.tensor(seq, dtype=torch.int32, device=dev), seq_lens_list=seq, Hq=Hq,
                    Dk=Dk, block_size=block_size, num_blocks=num_blocks)


def fp8_codes(t: torch.Tensor, scale: float) -> torch.Tensor:
    """E4M3 codes (uint8, same shape and device) standing for t / scale: an FP8 cache's content
    synthesised from values, with torch's float8_e4m3fn conversion (round to nearest even) after
    clamping to the finite range. Input synthesis only: the library's quantiser is not used."""
    x = (t.float() / scale).clamp_(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_scale(amax: float) -> float:
    """Per-tensor scale mapping |x| <= amax onto the E4M3 range."""
    return float(amax) / 448.0


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a bf16 tensor as a host uint16 array (the oracle's input format)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ---- the workloads the benchmark and the full-size tests use -------------------------------

TINY_DECODE = dict(B=4, ctx_lo=16, ctx_hi=200, Hq=8, Hkv=2, D=64, num_blocks=64, seed=0)
DECODE_QWEN3 = dict(B=256, ctx_lo=2000, ctx_hi=3000, Hq=64, Hkv=4, D=128, seed=1)
MIXED_LLAMA70B = dict(n_decode=192, decode_ctx=(1000, 8000), n_extend=8, extend_new=512,
                      extend_ctx=(4000, 32000), n_prefill=4, prefill_len=(2000, 8000), Hq=64,
                      Hkv=8, D=128, seed=2)
LONG_EXTEND = dict(new_lens=[2048, 2048], ctx_lens=[100000, 100000], Hq=64, Hkv=8, D=128,
                   seed=3)
WRITE_PACK_LLAMA70B = dict(num_layers=80, T=10000, Hkv=8, D=128, seed=4)
# DeepSeek-R1-like MLA layer under tensor parallelism 8: 16 query heads per GPU over one
# 576-wide latent (512 value dims + 64 rotary dims); 128 concurrent requests of a 10K-token
# prompt part-way through 1K generated tokens. Softmax scale 1/sqrt(128 + 64), the model's
# query-key head width.
MLA_DEEPSEEK_TP8 = dict(B=128, ctx_lo=10000, ctx_hi=11000, Hq=16, Dk=576, seed=5)
MLA_DV = 512
MLA_SCALE = 1.0 / math.sqrt(192.0)
