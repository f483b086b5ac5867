"""GPU parity at the benchmark's full sizes, in the launch configuration bench.py times.
Attention outputs are checked on sampled rows the oracle computes one by one (every head of the
sampled rows); write, pack and reorder are compared bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
from pkv_workloads import gen

from helpers import bits, compare_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_attention_reshape_gb300 as m
    m.load()
    return m


def _host(t):
    return bits(t)


def test_decode_qwen3_full(pkv):
    """256 sequences, context U[2000, 3000], 64 Q / 4 KV heads, D 128 (the headline workload):
    reorder + write + decode as the benchmark step runs them; 24 sampled sequences checked."""
    b = gen.decode_batch(**gen.DECODE_QWEN3, device="cuda")
    kc0, vc0 = _host(b.k_cache).copy(), _host(b.v_cache).copy()
    R = b.R
    perm, bounds, _, _ = pkv.batch_classify_reorder(b.cu_q, b.seq_lens)
    pkv.kv_cache_write(b.k_new, b.v_new, b.slot_mapping, b.k_cache, b.v_cache)
    out, lse = pkv.paged_decode_attn(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                     max(b.seq_lens_list), cu_q=b.cu_q,
                                     reqs=pkv.Reqs(R, R, perm, bounds, pkv.CLASS_DECODE),
                                     scale=1 / math.sqrt(b.D))
    assert pkv.device_errors() == 0
    oracle.kv_cache_write(_host(b.k_new), _host(b.v_new), b.slot_mapping.cpu().numpy(), kc0, vc0)
    assert np.array_equal(_host(b.k_cache), kc0) and np.array_equal(_host(b.v_cache), vc0)
    assert perm.tolist() == list(range(R)) and bounds.tolist() == [0, R, R, R]
    sample = np.sort(np.random.default_rng(0).choice(R, 24, replace=False)).astype(np.int32)
    ref, ref_lse = oracle.paged_decode(_host(b.q), kc0, vc0, b.block_tables.cpu().numpy(),
                                       b.seq_lens.cpu().numpy(), 1 / math.sqrt(b.D),
                                       cu_q=b.cu_q.cpu().numpy(), req_ids=sample)
    rows = np.zeros(b.T, bool)
    rows[sample] = True
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="decode qwen3 full"))


def test_decode_qwen3_fp8_full(pkv):
    """The headline workload over an FP8 (E4M3) cache: the caches hold codes, the new tokens
    are quantised by kv_cache_write, decode dequantises as it reads; the written caches bit for
    bit, 24 sampled sequences against the oracle."""
    b = gen.decode_batch(**gen.DECODE_QWEN3, device="cuda")
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    del b.k_cache, b.v_cache
    kc0, vc0 = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    R = b.R
    perm, bounds, _, _ = pkv.batch_classify_reorder(b.cu_q, b.seq_lens)
    pkv.kv_cache_write(b.k_new, b.v_new, b.slot_mapping, kc, vc, k_scale=ks, v_scale=vs)
    out, lse = pkv.paged_decode_attn(b.q, kc, vc, b.block_tables, b.seq_lens, max(b.seq_lens_list), cu_q=b.cu_q,
                                     reqs=pkv.Reqs(R, R, perm, bounds, pkv.CLASS_DECODE),
                                     scale=1 / math.sqrt(b.D), k_scale=ks, v_scale=vs)
    assert pkv.device_errors() == 0
    assert oracle.kv_cache_write_fp8(_host(b.k_new), _host(b.v_new), b.slot_mapping.cpu().numpy(), kc0, vc0,
                                     ks, vs) == 0
    assert np.array_equal(kc.cpu().numpy(), kc0) and np.array_equal(vc.cpu().numpy(), vc0)
    sample = np.sort(np.random.default_rng(0).choice(R, 24, replace=False)).astype(np.int32)
    ref, ref_lse = oracle.paged_decode_fp8(_host(b.q), kc0, vc0, b.block_tables.cpu().numpy(),
                                           b.seq_lens.cpu().numpy(), 1 / math.sqrt(b.D), ks, vs,
                                           cu_q=b.cu_q.cpu().numpy(), req_ids=sample)
    rows = np.zeros(b.T, bool)
    rows[sample] = True
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="decode qwen3 fp8 full"))


def test_mla_deepseek_tp8_full(pkv):
    """The MLA decode workload at full size (128 requests over 10K-11K tokens of a 576-wide
    latent, 16 query heads): 16 sampled requests against the oracle, every head."""
    b = gen.mla_batch(**gen.MLA_DEEPSEEK_TP8, device="cuda")
    out, lse = pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, max(b.seq_lens_list),
                                   gen.MLA_SCALE)
    torch.cuda.synchronize()
    assert pkv.device_errors() == 0
    sample = np.sort(np.random.default_rng(1).choice(b.R, 16, replace=False)).astype(np.int32)
    ref, ref_lse = oracle.mla_decode(_host(b.q), _host(b.latent), b.block_tables.cpu().numpy(),
                                     b.seq_lens.cpu().numpy(), gen.MLA_SCALE, gen.MLA_DV, req_ids=sample)
    rows = np.zeros(b.R, bool)
    rows[sample] = True
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="mla deepseek tp8 full"))


def test_mla_deepseek_128_heads_full(pkv):
    """The same latent batch with all 128 query heads of the layer (no tensor parallelism), the
    tensor-core kernel on clusters of two CTAs: 8 sampled requests against the oracle, every
    head; the bench times this call as its 128-head line."""
    b = gen.mla_batch(**{**gen.MLA_DEEPSEEK_TP8, "Hq": 128}, device="cuda")
    out, lse = pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, max(b.seq_lens_list),
                                   gen.MLA_SCALE)
    torch.cuda.synchronize()
    assert pkv.device_errors() == 0
    sample = np.sort(np.random.default_rng(2).choice(b.R, 8, replace=False)).astype(np.int32)
    ref, ref_lse = oracle.mla_decode(_host(b.q), _host(b.latent), b.block_tables.cpu().numpy(),
                                     b.seq_lens.cpu().numpy(), gen.MLA_SCALE, gen.MLA_DV, req_ids=sample)
    rows = np.zeros(b.R, bool)
    rows[sample] = True
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="mla deepseek 128 heads full"))


def test_mixed_llama70b_full(pkv):
    """192 decode + 8 extend (512 over 4k-32k) + 4 prefill (2k-8k), shuffled: the full step;
    sampled rows of every class checked."""
    b = gen.mixed_batch(**gen.MIXED_LLAMA70B, device="cuda")
    kc0, vc0 = _host(b.k_cache).copy(), _host(b.v_cache).copy()
    R, T = b.R, b.T
    kinds = b.kinds
    n_dec = sum(k == gen.DECODE for k in kinds)
    n_ext = sum(k == gen.EXTEND for k in kinds)
    n_pre = sum(k == gen.PREFILL for k in kinds)
    perm, bounds, cu_r, tmap = pkv.batch_classify_reorder(b.cu_q, b.seq_lens, with_token_map=True, num_tokens=T)
    pkv.kv_cache_write(b.k_new, b.v_new, b.slot_mapping, b.k_cache, b.v_cache)
    out = torch.full_like(b.q, float("nan"))
    lse = torch.full((T, b.Hq), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1 / math.sqrt(b.D)
    maxs = max(b.seq_lens_list)
    pkv.paged_decode_attn(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                          max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.DECODE), cu_q=b.cu_q,
                          reqs=pkv.Reqs(n_dec, R, perm, bounds, pkv.CLASS_DECODE), scale=scale, out=out, lse=lse)
    pkv.extend_attn(b.q, b.k_new, b.v_new, b.cu_q, b.seq_lens, b.k_cache, b.v_cache, b.block_tables,
                    max(q for k, q in zip(kinds, b.q_lens) if k == gen.EXTEND), maxs,
                    reqs=pkv.Reqs(n_ext, R, perm, bounds, pkv.CLASS_EXTEND), chunk_budget_tokens=32768,
                    scale=scale, out=out, lse=lse)
    pkv.varlen_prefill_attn(b.q, b.k_new, b.v_new, b.cu_q, max(q for k, q in zip(kinds, b.q_lens) if k == gen.PREFILL),
                            reqs=pkv.Reqs(n_pre, R, perm, bounds, pkv.CLASS_PREFILL), scale=scale, out=out, lse=lse)
    assert pkv.device_errors() == 0
    # indexing calls, bit for bit
    e_perm, e_bounds, e_cu, e_map = oracle.batch_classify_reorder(b.cu_q.cpu().numpy(), b.seq_lens.cpu().numpy())
    assert np.array_equal(perm.cpu().numpy(), e_perm) and np.array_equal(bounds.cpu().numpy(), e_bounds)
    assert np.array_equal(cu_r.cpu().numpy(), e_cu) and np.array_equal(tmap.cpu().numpy(), e_map)
    assert e_bounds.tolist() == [0, n_dec, n_dec + n_ext, R]
    oracle.kv_cache_write(_host(b.k_new), _host(b.v_new), b.slot_mapping.cpu().numpy(), kc0, vc0)
    assert np.array_equal(_host(b.k_cache), kc0) and np.array_equal(_host(b.v_cache), vc0)
    # attention on sampled rows: 16 decode requests, and in every extend / prefill request its
    # first row, last row and 6 random rows
    rng = np.random.default_rng(1)
    cu = b.cu_q.cpu().numpy()
    d_ids = e_perm[:n_dec]
    d_sample = np.sort(rng.choice(d_ids, 16, replace=False)).astype(np.int32)
    rows = np.zeros(T, bool)
    for r in d_sample:
        rows[cu[r]] = True
    for r in e_perm[n_dec:]:
        n = cu[r + 1] - cu[r]
        pick = {0, n - 1, *rng.choice(n, 6, replace=False).tolist()}
        for i in pick:
            rows[cu[r] + i] = True
    ref = np.full((T, b.Hq, b.D), np.nan)
    ref_lse = np.full((T, b.Hq), np.nan)
    qb, kb, vb = _host(b.q), _host(b.k_new), _host(b.v_new)
    bt, sl = b.block_tables.cpu().numpy(), b.seq_lens.cpu().numpy()
    oracle.paged_decode(qb, kc0, vc0, bt, sl, scale, cu_q=cu, req_ids=d_sample, out=ref, lse=ref_lse)
    oracle.extend(qb, kb, vb, cu, scale, seq_lens=sl, k_cache=kc0, v_cache=vc0, block_tables=bt,
                  req_ids=e_perm[n_dec:n_dec + n_ext], row_mask=rows, out=ref, lse=ref_lse)
    oracle.extend(qb, kb, vb, cu, scale, req_ids=e_perm[n_dec + n_ext:], row_mask=rows, out=ref, lse=ref_lse)
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="mixed llama70b full"))


def test_mixed_llama70b_fp8_full(pkv):
    """The mixed step over an FP8 (E4M3) cache: quantising write, decode dequantising as it
    reads, extend through the gather of its context into bf16; the written caches bit for bit,
    sampled decode and extend rows against the FP8 oracles."""
    b = gen.mixed_batch(**gen.MIXED_LLAMA70B, device="cuda")
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    del b.k_cache, b.v_cache
    kc0, vc0 = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    R, T = b.R, b.T
    kinds = b.kinds
    n_dec = sum(k == gen.DECODE for k in kinds)
    n_ext = sum(k == gen.EXTEND for k in kinds)
    perm, bounds, _, _ = pkv.batch_classify_reorder(b.cu_q, b.seq_lens)
    pkv.kv_cache_write(b.k_new, b.v_new, b.slot_mapping, kc, vc, k_scale=ks, v_scale=vs)
    out = torch.full_like(b.q, float("nan"))
    lse = torch.full((T, b.Hq), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1 / math.sqrt(b.D)
    pkv.paged_decode_attn(b.q, kc, vc, b.block_tables, b.seq_lens,
                          max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.DECODE), cu_q=b.cu_q,
                          reqs=pkv.Reqs(n_dec, R, perm, bounds, pkv.CLASS_DECODE), scale=scale, out=out, lse=lse,
                          k_scale=ks, v_scale=vs)
    pkv.extend_attn(b.q, b.k_new, b.v_new, b.cu_q, b.seq_lens, kc, vc, b.block_tables,
                    max(q for k, q in zip(kinds, b.q_lens) if k == gen.EXTEND),
                    max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.EXTEND),
                    reqs=pkv.Reqs(n_ext, R, perm, bounds, pkv.CLASS_EXTEND), scale=scale, out=out, lse=lse,
                    k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkv.device_errors() == 0
    assert oracle.kv_cache_write_fp8(_host(b.k_new), _host(b.v_new), b.slot_mapping.cpu().numpy(), kc0, vc0,
                                     ks, vs) == 0
    assert np.array_equal(kc.cpu().numpy(), kc0) and np.array_equal(vc.cpu().numpy(), vc0)
    e_perm, e_bounds, _, _ = oracle.batch_classify_reorder(b.cu_q.cpu().numpy(), b.seq_lens.cpu().numpy())
    rng = np.random.default_rng(2)
    cu = b.cu_q.cpu().numpy()
    d_sample = np.sort(rng.choice(e_perm[:n_dec], 16, replace=False)).astype(np.int32)
    rows = np.zeros(T, bool)
    for r in d_sample:
        rows[cu[r]] = True
    for r in e_perm[n_dec:n_dec + n_ext]:
        n = cu[r + 1] - cu[r]
        for i in {0, n - 1, *rng.choice(n, 4, replace=False).tolist()}:
            rows[cu[r] + i] = True
    ref = np.full((T, b.Hq, b.D), np.nan)
    ref_lse = np.full((T, b.Hq), np.nan)
    qb, kb, vb = _host(b.q), _host(b.k_new), _host(b.v_new)
    bt, sl = b.block_tables.cpu().numpy(), b.seq_lens.cpu().numpy()
    oracle.paged_decode_fp8(qb, kc0, vc0, bt, sl, scale, ks, vs, cu_q=cu, req_ids=d_sample, out=ref, lse=ref_lse)
    oracle.extend_fp8(qb, kb, vb, cu, sl, kc0, vc0, bt, scale, ks, vs, req_ids=e_perm[n_dec:n_dec + n_ext],
                      row_mask=rows, out=ref, lse=ref_lse)
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="mixed llama70b fp8 full"))


def test_long_extend_full(pkv):
    """2 x (100000 cached + 2048 new), budget 32768: 24 sampled rows (first/last of each request)."""
    b = gen.extend_batch(**gen.LONG_EXTEND, device="cuda")
    out, lse = pkv.extend_attn(b.q, b.k_new, b.v_new, b.cu_q, b.seq_lens, b.k_cache, b.v_cache,
                               b.block_tables, max(b.q_lens), max(b.seq_lens_list),
                               chunk_budget_tokens=32768, scale=1 / math.sqrt(b.D))
    assert pkv.device_errors() == 0
    rng = np.random.default_rng(2)
    cu = b.cu_q.cpu().numpy()
    rows = np.zeros(b.T, bool)
    for r in range(b.R):
        n = cu[r + 1] - cu[r]
        for i in {0, 127, 128, n - 1, *rng.choice(n, 8, replace=False).tolist()}:
            rows[cu[r] + i] = True
    ref, ref_lse = oracle.extend(_host(b.q), _host(b.k_new), _host(b.v_new), cu, 1 / math.sqrt(b.D),
                                 seq_lens=b.seq_lens.cpu().numpy(), k_cache=_host(b.k_cache),
                                 v_cache=_host(b.v_cache), block_tables=b.block_tables.cpu().numpy(),
                                 row_mask=rows)
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="long extend full"))


def test_prefill_4x8k_full(pkv):
    b = gen.prefill_batch([8192] * 4, Hq=64, Hkv=8, D=128, seed=5, device="cuda")
    out, lse = pkv.varlen_prefill_attn(b.q, b.k_new, b.v_new, b.cu_q, 8192, scale=1 / math.sqrt(b.D))
    rng = np.random.default_rng(3)
    cu = b.cu_q.cpu().numpy()
    rows = np.zeros(b.T, bool)
    for r in range(b.R):
        for i in {0, 1, 127, 128, 8191, *rng.choice(8192, 6, replace=False).tolist()}:
            rows[cu[r] + i] = True
    ref, ref_lse = oracle.prefill(_host(b.q), _host(b.k_new), _host(b.v_new), cu, 1 / math.sqrt(b.D),
                                  row_mask=rows)
    print(compare_attention(out, lse, ref, ref_lse, rows=rows, what="prefill 4x8k full"))


def test_write_pack_llama70b_full(pkv):
    """80 layers x 10000 tokens, Hkv 8, D 128 (320 KiB/token): all 80 layers written and packed as
    in the benchmark; 8 sampled layers compared bit for bit (caches and packed buffers), a
    shuffled-order pack of one layer, and its unpack into another pool."""
    layers = gen.write_pack_layers(**gen.WRITE_PACK_LLAMA70B, device="cuda")
    sample = set(np.random.default_rng(4).choice(len(layers), 8, replace=False).tolist())
    before = {i: (_host(L.k_cache).copy(), _host(L.v_cache).copy()) for i, L in enumerate(layers) if i in sample}
    packed = {}
    for i, L in enumerate(layers):
        pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache)
        dst = pkv.kv_block_pack(L.k_cache, L.v_cache, L.block_ids)
        if i in sample:
            packed[i] = _host(dst)
    assert pkv.device_errors() == 0
    for i in sample:
        L = layers[i]
        kc, vc = before[i]
        assert oracle.kv_cache_write(_host(L.key), _host(L.value), L.slot_mapping.cpu().numpy(), kc, vc) == 0
        assert np.array_equal(_host(L.k_cache), kc) and np.array_equal(_host(L.v_cache), vc)
        exp, bad = oracle.kv_block_pack(kc, vc, L.block_ids.cpu().numpy())
        assert bad == 0 and np.array_equal(packed[i], exp)
        # 10000 tokens = 625 whole blocks: the packed K rows are the prompt's K rows
        assert np.array_equal(packed[i][0].reshape(-1, 8, 128)[:10000], _host(L.key))
    L = layers[0]
    shuf = L.block_ids[torch.randperm(L.block_ids.numel(), generator=torch.Generator().manual_seed(9))
                       .to(L.block_ids.device)].contiguous()
    dst = pkv.kv_block_pack(L.k_cache, L.v_cache, shuf)
    exp, _ = oracle.kv_block_pack(_host(L.k_cache), _host(L.v_cache), shuf.cpu().numpy())
    assert np.array_equal(_host(dst), exp)
    # the receiving side: land the packed layer in another pool's blocks (as the benchmark's
    # handoff does), bit for bit the oracle's
    g = torch.Generator().manual_seed(10)
    recv_k = gen.randn_bf16(tuple(L.k_cache.shape), g, "cpu")
    recv_v = gen.randn_bf16(tuple(L.v_cache.shape), g, "cpu")
    recv_ids = torch.randperm(L.k_cache.shape[0], generator=g)[:shuf.numel()].to(torch.int32)
    rk, rv = recv_k.to(L.k_cache.device), recv_v.to(L.k_cache.device)
    pkv.kv_block_unpack(dst, recv_ids.to(L.k_cache.device), rk, rv)
    assert pkv.device_errors() == 0
    ek, ev = _host(recv_k).copy(), _host(recv_v).copy()
    assert oracle.kv_block_unpack(exp, recv_ids.numpy(), ek, ev) == 0
    assert np.array_equal(_host(rk), ek) and np.array_equal(_host(rv), ev)
