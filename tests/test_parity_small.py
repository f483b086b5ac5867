"""GPU parity of every call against the oracle at sizes the oracle finishes in seconds, covering
several tiles, ragged tails and the degenerate cases. Indexing calls bit-exact; attention within
the stated tolerances (tests/helpers.py)."""
import math

import numpy as np
import pytest
import torch

import oracle
from pkv_workloads import gen

from helpers import bits, compare_attention, default_scale, oracle_decode, oracle_extend, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_attention_reshape_gb300 as m
    m.load()
    assert torch.cuda.is_available()
    return m


DEV = "cuda"


def _errors(pkv):
    return pkv.device_errors(clear=True)


# ---- kv_cache_write --------------------------------------------------------------------------

@pytest.mark.parametrize("Hkv,D", [(2, 64), (8, 128), (1, 8)])
def test_kv_cache_write_bit_exact(pkv, Hkv, D):
    b = gen.mixed_batch(5, (3, 70), 3, 20, (1, 50), 2, (1, 45), Hq=Hkv, Hkv=Hkv, D=D, seed=D + Hkv)
    slots = b.slot_mapping.clone()
    slots[::7] = -1
    g = b.to(DEV)
    pkv.kv_cache_write(g.k_new, g.v_new, slots.to(DEV), g.k_cache, g.v_cache)
    kc, vc = bits(b.k_cache).copy(), bits(b.v_cache).copy()
    assert oracle.kv_cache_write(bits(b.k_new), bits(b.v_new), slots.numpy(), kc, vc) == 0
    assert np.array_equal(bits(g.k_cache), kc) and np.array_equal(bits(g.v_cache), vc)
    assert _errors(pkv) == 0


def test_kv_cache_write_strided_cache_and_bad_slots(pkv):
    """K and V in one allocation [nb, 2, bs, H, D]; out-of-range slots are skipped and flagged."""
    nb, bs, H, D = 12, 16, 2, 64
    both = gen.randn_bf16((nb, 2, bs, H, D), torch.Generator().manual_seed(3), "cpu")
    key = gen.randn_bf16((9, H, D), torch.Generator().manual_seed(4), "cpu")
    val = gen.randn_bf16((9, H, D), torch.Generator().manual_seed(5), "cpu")
    slots = torch.tensor([0, 5, 17, 191, -1, 40, nb * bs, 1000, 33], dtype=torch.int64)
    g = both.to(DEV)
    pkv.kv_cache_write(key.to(DEV), val.to(DEV), slots.to(DEV), g[:, 0], g[:, 1])
    kc, vc = bits(both[:, 0]).copy(), bits(both[:, 1]).copy()
    assert oracle.kv_cache_write(bits(key), bits(val), slots.numpy(), kc, vc) == 2
    gb = bits(g)
    assert np.array_equal(gb[:, 0], kc) and np.array_equal(gb[:, 1], vc)
    assert _errors(pkv) & 0x1


@pytest.mark.parametrize("bs", [1, 8, 32, 64])
def test_write_pack_unpack_other_block_sizes(pkv, bs):
    """kv_cache_write, kv_block_pack and kv_block_unpack take any block size: bit for bit the
    oracle's at 1, 8, 32 and 64 tokens per block (the attention calls take 16)."""
    L = gen.write_pack_layers(1, 150, Hkv=2, D=64, block_size=bs, seed=70 + bs)[0]
    gk, gv = L.k_cache.to(DEV), L.v_cache.to(DEV)
    pkv.kv_cache_write(L.key.to(DEV), L.value.to(DEV), L.slot_mapping.to(DEV), gk, gv)
    kc, vc = bits(L.k_cache).copy(), bits(L.v_cache).copy()
    assert oracle.kv_cache_write(bits(L.key), bits(L.value), L.slot_mapping.numpy(), kc, vc) == 0
    assert np.array_equal(bits(gk), kc) and np.array_equal(bits(gv), vc)
    packed = pkv.kv_block_pack(gk, gv, L.block_ids.to(DEV))
    exp, bad = oracle.kv_block_pack(kc, vc, L.block_ids.numpy())
    assert bad == 0 and np.array_equal(bits(packed), exp)
    # the prompt's rows come back in order from the blocks in table order
    assert np.array_equal(exp[0].reshape(-1, 2, 64)[:150], bits(L.key))
    rk, rv = torch.zeros_like(gk), torch.zeros_like(gv)
    ids = torch.flip(L.block_ids, [0]).contiguous()
    pkv.kv_block_unpack(packed, ids.to(DEV), rk, rv)
    ek, ev = np.zeros_like(kc), np.zeros_like(vc)
    assert oracle.kv_block_unpack(exp, ids.numpy(), ek, ev) == 0
    assert np.array_equal(bits(rk), ek) and np.array_equal(bits(rv), ev)
    assert _errors(pkv) == 0


def test_kv_cache_write_empty(pkv):
    c = torch.zeros((2, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device=DEV)
    pkv.kv_cache_write(e, e, torch.empty(0, dtype=torch.int64, device=DEV), c, c)
    assert _errors(pkv) == 0 and c.abs().sum().item() == 0


# ---- kv_block_pack ---------------------------------------------------------------------------

@pytest.mark.parametrize("shuffled", [False, True])
def test_kv_block_pack_bit_exact(pkv, shuffled):
    L = gen.write_pack_layers(1, 300, Hkv=8, D=128, seed=8, shuffled_pack=shuffled)[0]
    gk, gv = L.k_cache.to(DEV), L.v_cache.to(DEV)
    pkv.kv_cache_write(L.key.to(DEV), L.value.to(DEV), L.slot_mapping.to(DEV), gk, gv)
    dst = pkv.kv_block_pack(gk, gv, L.block_ids.to(DEV))
    kc, vc = bits(L.k_cache).copy(), bits(L.v_cache).copy()
    oracle.kv_cache_write(bits(L.key), bits(L.value), L.slot_mapping.numpy(), kc, vc)
    exp, bad = oracle.kv_block_pack(kc, vc, L.block_ids.numpy())
    assert bad == 0 and np.array_equal(bits(dst), exp)
    assert _errors(pkv) == 0


def test_kv_block_pack_duplicates_and_bad_ids(pkv):
    kc = gen.randn_bf16((6, 16, 2, 64), torch.Generator().manual_seed(1), "cpu")
    vc = gen.randn_bf16((6, 16, 2, 64), torch.Generator().manual_seed(2), "cpu")
    ids = torch.tensor([5, 5, 0, 6, -3, 2], dtype=torch.int32)
    dst0 = torch.zeros((2, 6, 16, 2, 64), dtype=torch.bfloat16)
    dst = pkv.kv_block_pack(kc.to(DEV), vc.to(DEV), ids.to(DEV), dst=dst0.to(DEV))
    exp = np.zeros((2, 6, 16, 2, 64), np.uint16)
    exp, bad = oracle.kv_block_pack(bits(kc), bits(vc), ids.numpy(), dst=exp)
    assert bad == 2 and np.array_equal(bits(dst), exp)
    assert _errors(pkv) & 0x2


# ---- kv_block_unpack -------------------------------------------------------------------------

@pytest.mark.parametrize("Hkv,D", [(8, 128), (2, 64), (1, 8)])
def test_kv_block_unpack_bit_exact(pkv, Hkv, D):
    """Pack from one pool, unpack into another at different ids: bit for bit the oracle's."""
    g = torch.Generator().manual_seed(21 + Hkv)
    nb, n = 300, 97
    src_k, src_v = gen.randn_bf16((nb, 16, Hkv, D), g, "cpu"), gen.randn_bf16((nb, 16, Hkv, D), g, "cpu")
    dst_k, dst_v = gen.randn_bf16((nb, 16, Hkv, D), g, "cpu"), gen.randn_bf16((nb, 16, Hkv, D), g, "cpu")
    src_ids = torch.randperm(nb, generator=g)[:n].to(torch.int32)
    dst_ids = torch.randperm(nb, generator=g)[:n].to(torch.int32)
    gk, gv = dst_k.to(DEV), dst_v.to(DEV)
    packed = pkv.kv_block_pack(src_k.to(DEV), src_v.to(DEV), src_ids.to(DEV))
    pkv.kv_block_unpack(packed, dst_ids.to(DEV), gk, gv)
    exp_packed, _ = oracle.kv_block_pack(bits(src_k), bits(src_v), src_ids.numpy())
    ek, ev = bits(dst_k).copy(), bits(dst_v).copy()
    assert oracle.kv_block_unpack(exp_packed, dst_ids.numpy(), ek, ev) == 0
    assert np.array_equal(bits(gk), ek) and np.array_equal(bits(gv), ev)
    assert _errors(pkv) == 0


def test_kv_block_unpack_strided_cache_and_bad_ids(pkv):
    """Caches that are slices of a wider pool (block stride > block), and ids outside the
    pool: skipped, flagged, the rest landed."""
    g = torch.Generator().manual_seed(5)
    pool = gen.randn_bf16((10, 2, 16, 2, 64), g, "cpu")       # [blocks][K|V][16][Hkv][D]
    src = gen.randn_bf16((2, 4, 16, 2, 64), g, "cpu")
    ids = torch.tensor([3, 11, -1, 7], dtype=torch.int32)
    gpool = pool.to(DEV)
    gk, gv = gpool[:, 0], gpool[:, 1]
    pkv.kv_block_unpack(src.to(DEV), ids.to(DEV), gk, gv)
    ek, ev = bits(pool[:, 0]).copy(), bits(pool[:, 1]).copy()
    assert oracle.kv_block_unpack(bits(src), ids.numpy(), ek, ev) == 2
    assert np.array_equal(bits(gk.contiguous()), ek) and np.array_equal(bits(gv.contiguous()), ev)
    assert _errors(pkv) & 0x2


# ---- FP8 (E4M3) cache -----------------------------------------------------------------------------

def _codes(t):
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


@pytest.mark.parametrize("Hkv,D", [(8, 128), (4, 128), (2, 64), (1, 16)])
def test_kv_cache_write_fp8_bit_exact(pkv, Hkv, D):
    """Quantising write: code = E4M3(float(x) * (1/scale)), round to nearest even, saturating;
    bit for bit the oracle's (which is pinned to torch's float8 conversion)."""
    L = gen.write_pack_layers(1, 300, Hkv=Hkv, D=D, seed=40 + Hkv)[0]
    nb = L.k_cache.shape[0]
    g = torch.Generator().manual_seed(41)
    kc0 = torch.randint(0, 0x7F, (nb, 16, Hkv, D), generator=g, dtype=torch.uint8)
    vc0 = torch.randint(0x80, 0xFF, (nb, 16, Hkv, D), generator=g, dtype=torch.uint8)
    ks, vs = 0.0213, 0.00071   # the V scale saturates the larger values at +-448
    gk, gv = kc0.to(DEV), vc0.to(DEV)
    pkv.kv_cache_write(L.key.to(DEV), L.value.to(DEV), L.slot_mapping.to(DEV), gk, gv, k_scale=ks, v_scale=vs)
    ek, ev = kc0.numpy().copy(), vc0.numpy().copy()
    assert oracle.kv_cache_write_fp8(bits(L.key), bits(L.value), L.slot_mapping.numpy(), ek, ev, ks, vs) == 0
    assert np.array_equal(_codes(gk), ek) and np.array_equal(_codes(gv), ev)
    assert (ev == 0x7E).any() or (ev == 0xFE).any()   # saturation exercised
    assert _errors(pkv) == 0


def test_kv_block_pack_unpack_fp8_bit_exact(pkv):
    g = torch.Generator().manual_seed(42)
    nb, n = 200, 61
    kc = torch.randint(0, 256, (nb, 16, 4, 128), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 256, (nb, 16, 4, 128), generator=g, dtype=torch.uint8)
    ids = torch.randperm(nb, generator=g)[:n].to(torch.int32)
    dst_ids = torch.randperm(nb, generator=g)[:n].to(torch.int32)
    packed = pkv.kv_block_pack(kc.to(DEV), vc.to(DEV), ids.to(DEV))
    assert packed.dtype == torch.uint8
    assert np.array_equal(_codes(packed[0]), kc.numpy()[ids.numpy()])
    assert np.array_equal(_codes(packed[1]), vc.numpy()[ids.numpy()])
    rk, rv = torch.zeros_like(kc).to(DEV), torch.zeros_like(vc).to(DEV)
    pkv.kv_block_unpack(packed, dst_ids.to(DEV), rk, rv)
    ek, ev = np.zeros_like(kc.numpy()), np.zeros_like(vc.numpy())
    ek[dst_ids.numpy()] = kc.numpy()[ids.numpy()]
    ev[dst_ids.numpy()] = vc.numpy()[ids.numpy()]
    assert np.array_equal(_codes(rk), ek) and np.array_equal(_codes(rv), ev)


def _fp8_decode_case(B, lo, hi, Hq, Hkv, seed, q_scale=1.0):
    b = gen.decode_batch(B, lo, hi, Hq=Hq, Hkv=Hkv, D=128, seed=seed, q_scale=q_scale)
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    return b, gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs), ks, vs


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_decode_fp8_group_sizes(pkv, G):
    b, kc, vc, ks, vs = _fp8_decode_case(5, 1, 300, Hq=2 * G, Hkv=2, seed=50 + G)
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), kc.to(DEV), vc.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(b.seq_lens_list), scale=1 / math.sqrt(128),
                                     k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                           b.seq_lens.numpy(), 1 / math.sqrt(128), ks, vs)
    compare_attention(out, lse, ref, ref_lse, what=f"decode fp8 G={G}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hkv", [1, 3, 6, 8, 16])
def test_decode_fp8_kv_head_counts(pkv, Hkv):
    """The FP8 kernel's CTA layouts (12 warps a CTA: 12 one-warp shares at Hkv 1 and 3, 6 x 2 at
    6, 3 x 4 at 8 and 16)."""
    b, kc, vc, ks, vs = _fp8_decode_case(7, 1, 900, Hq=2 * Hkv, Hkv=Hkv, seed=400 + Hkv)
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), kc.to(DEV), vc.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(b.seq_lens_list), scale=1 / math.sqrt(128),
                                     k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                           b.seq_lens.numpy(), 1 / math.sqrt(128), ks, vs)
    compare_attention(out, lse, ref, ref_lse, what=f"decode fp8 Hkv={Hkv}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("ctxs", [[1, 16, 17, 31, 32, 33], [4096, 1, 7000, 15]])
def test_decode_fp8_edge_lengths_and_nan_codes_past_the_end(pkv, ctxs):
    """Ragged and cut sequences; codes past each sequence's end are NaN codes (0x7F), which
    must not reach the result."""
    b = gen.make_batch([gen.DECODE] * len(ctxs), [1] * len(ctxs), ctxs, Hq=32, Hkv=4, D=128, seed=60)
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.0)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    for r, n in enumerate(ctxs):
        last = int(b.block_tables[r, (n - 1) // 16])
        kc[last, (n - 1) % 16 + 1:] = 0x7F
        vc[last, (n - 1) % 16 + 1:] = 0x7F
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), kc.to(DEV), vc.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(ctxs), scale=1 / math.sqrt(128), k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                           b.seq_lens.numpy(), 1 / math.sqrt(128), ks, vs)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, what="decode fp8 edges")


def test_decode_fp8_peaked_softmax(pkv):
    b, kc, vc, ks, vs = _fp8_decode_case(8, 100, 2000, Hq=64, Hkv=4, seed=61, q_scale=4.0)
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), kc.to(DEV), vc.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(b.seq_lens_list), scale=1 / math.sqrt(128),
                                     k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                           b.seq_lens.numpy(), 1 / math.sqrt(128), ks, vs)
    compare_attention(out, lse, ref, ref_lse, what="decode fp8 peaked")


def _fp8_extend_ref(b, kc, vc, ks, vs, scale, **kw):
    return oracle.extend_fp8(bits(b.q), bits(b.k_new), bits(b.v_new), b.cu_q.cpu().numpy(), b.seq_lens.cpu().numpy(),
                             kc, vc, b.block_tables.cpu().numpy(), scale, ks, vs, **kw)


@pytest.mark.parametrize("G,D", [(1, 64), (4, 128), (8, 128), (16, 64)])
def test_extend_fp8_ragged(pkv, G, D):
    """Extend over an E4M3 cache: the set's context gathered into a bf16 pool of the E4M3
    values, the scales applied in the attention; ragged new and cached lengths."""
    Hkv = 2
    new = [1, 63, 64, 65, 130, 7]
    ctx = [0, 1, 15, 16, 100, 300]
    b = gen.extend_batch(new, ctx, Hq=G * Hkv, Hkv=Hkv, D=D, seed=G * 11 + D)
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kc.to(DEV), vc.to(DEV), g.block_tables,
                               max(new), max(b.seq_lens_list), scale=scale, k_scale=ks, v_scale=vs)
    ref, ref_lse = _fp8_extend_ref(b, kc.numpy(), vc.numpy(), ks, vs, scale)
    compare_attention(out, lse, ref, ref_lse, what=f"extend fp8 G={G} D={D}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_shared_prefix_blocks(pkv, fp8):
    """Prefix reuse: the block tables of several requests point at the same physical blocks
    for a common prefix (60 whole blocks, 960 tokens), as a prefix cache hands them out. Decode
    and extend read the shared blocks in place (the FP8 extend gathers them once per request);
    the results equal the oracle's over the same tables."""
    kinds = [gen.DECODE] * 4 + [gen.EXTEND] * 3
    q_lens = [1, 1, 1, 1, 40, 200, 129]
    seq_lens = [2000, 1500, 3100, 2049, 1840, 2700, 1329]
    b = gen.make_batch(kinds, q_lens, seq_lens, Hq=32, Hkv=4, D=128, seed=123)
    bt = b.block_tables.clone()
    bt[1:, :60] = bt[0, :60]
    b.block_tables = bt
    g = b.to(DEV)
    scale = default_scale(b.D)
    kw, kc, vc = {}, g.k_cache, g.v_cache
    if fp8:
        ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
        kc8, vc8 = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
        kw, kc, vc = dict(k_scale=ks, v_scale=vs), kc8.to(DEV), vc8.to(DEV)
    dec = pkv.Reqs(max_reqs=4, batch_reqs=b.R)  # requests 0..3
    ext = pkv.Reqs(max_reqs=3, batch_reqs=b.R, order=torch.tensor([4, 5, 6], dtype=torch.int32, device=DEV))
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((b.T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_attn(g.q, kc, vc, g.block_tables, g.seq_lens, max(seq_lens), cu_q=g.cu_q, reqs=dec,
                          scale=scale, out=out, lse=lse, **kw)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kc, vc, g.block_tables, max(q_lens), max(seq_lens),
                    reqs=ext, scale=scale, out=out, lse=lse, **kw)
    assert _errors(pkv) == 0
    ref = np.full((b.T, b.Hq, b.D), np.nan)
    ref_lse = np.full((b.T, b.Hq), np.nan)
    if fp8:
        oracle.paged_decode_fp8(bits(b.q), _codes(kc8), _codes(vc8), bt.numpy(), b.seq_lens.numpy(), scale, ks, vs,
                                cu_q=b.cu_q.numpy(), req_ids=[0, 1, 2, 3], out=ref, lse=ref_lse)
        _fp8_extend_ref(b, _codes(kc8), _codes(vc8), ks, vs, scale, req_ids=[4, 5, 6], out=ref, lse=ref_lse)
    else:
        oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale, req_ids=[0, 1, 2, 3], out=ref, lse=ref_lse)
        oracle_extend(b, bits(b.k_cache), bits(b.v_cache), scale, req_ids=[4, 5, 6], out=ref, lse=ref_lse)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, what=f"shared prefix fp8={fp8}")


def test_extend_fp8_request_set_and_peaked(pkv):
    """A request set from the reorder's outputs over a shuffled batch, peaked queries, and
    NaN codes past the end of each context (never gathered into a sum)."""
    b = gen.mixed_batch(4, (20, 90), 5, 70, (10, 400), 3, (5, 80), Hq=16, Hkv=2, D=128, seed=63, q_scale=3.0)
    ks, vs = gen.fp8_scale(6.0), gen.fp8_scale(5.0)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    bt = b.block_tables.numpy()
    for r in range(b.R):
        C = b.seq_lens_list[r] - b.q_lens[r]
        if C % 16:
            kc[bt[r, C // 16], C % 16:] = 0x7F
            vc[bt[r, C // 16], C % 16:] = 0xFF
    g = b.to(DEV)
    R = b.R
    perm, bounds, _, _ = pkv.batch_classify_reorder(g.cu_q, g.seq_lens)
    reqs = pkv.Reqs(max_reqs=R, batch_reqs=R, order=perm, bounds=bounds, cls=pkv.CLASS_EXTEND)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((b.T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    scale = default_scale(128)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kc.to(DEV), vc.to(DEV), g.block_tables,
                    max(b.q_lens), max(b.seq_lens_list), reqs=reqs, scale=scale, k_scale=ks, v_scale=vs,
                    out=out, lse=lse)
    o_perm, o_bounds, _, _ = oracle.batch_classify_reorder(b.cu_q.numpy(), b.seq_lens.numpy())
    ids = o_perm[o_bounds[1]:o_bounds[2]]
    ref, ref_lse = _fp8_extend_ref(b, kc.numpy(), vc.numpy(), ks, vs, scale, req_ids=ids)
    compare_attention(out, lse, ref, ref_lse, what="extend fp8 set")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("G", [2, 8, 16])
def test_extend_fp8_codes_converted_in_the_kernel(pkv, G):
    """head_dim 128 over an E4M3 cache: the kernel loads the context's codes and converts them
    in shared memory (no workspace). Contexts of many tiles with ragged ends, new tokens over
    several tiles, a small value scale (new values stored divided by it), peaked queries."""
    Hkv = 2
    new = [300, 129, 1, 128]
    ctx = [5000, 2047, 700, 0]
    b = gen.extend_batch(new, ctx, Hq=G * Hkv, Hkv=Hkv, D=128, seed=700 + G, q_scale=2.0)
    ks, vs = gen.fp8_scale(0.5), gen.fp8_scale(0.2)
    kc, vc = gen.fp8_codes(b.k_cache * 0.1, ks), gen.fp8_codes(b.v_cache * 0.05, vs)
    assert pkv.extend_fp8_workspace_size(b.R, b.R, max(b.seq_lens_list), b.block_tables.shape[1], Hkv, 128) == 0
    g = b.to(DEV)
    scale = default_scale(128)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((b.T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kc.to(DEV), vc.to(DEV), g.block_tables,
                    max(new), max(b.seq_lens_list), scale=scale, k_scale=ks, v_scale=vs, out=out, lse=lse)
    ref, ref_lse = _fp8_extend_ref(b, kc.numpy(), vc.numpy(), ks, vs, scale)
    compare_attention(out, lse, ref, ref_lse, what=f"extend fp8 in-kernel G={G}")
    assert _errors(pkv) == 0


# ---- randomized shapes -------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_random_mixed_batches(pkv, seed):
    """Random mixes of decode, extend and prefill requests (lengths from 1 token to several
    tiles, random head counts and head dims, shuffled arrival order) through the whole step:
    reorder, write, then the three attention calls on the reorder's sets; every row checked."""
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    n_dec, n_ext, n_pre = (int(x) for x in rng.integers(0, 6, size=3))
    if n_dec + n_ext + n_pre == 0:
        n_dec = 1
    b = gen.mixed_batch(n_dec, (1, int(rng.integers(2, 900))), n_ext, int(rng.integers(1, 300)),
                        (1, int(rng.integers(2, 700))), n_pre, (1, int(rng.integers(2, 400))),
                        Hq=G * Hkv, Hkv=Hkv, D=D, seed=2000 + seed)
    g = b.to(DEV)
    R, T = b.R, b.T
    perm, bounds, _, _ = pkv.batch_classify_reorder(g.cu_q, g.seq_lens)
    pkv.kv_cache_write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    scale = default_scale(D)
    maxs, maxq = max(b.seq_lens_list), max(b.q_lens)
    mk = lambda c: pkv.Reqs(max_reqs=R, batch_reqs=R, order=perm, bounds=bounds, cls=c)
    pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, maxs, cu_q=g.cu_q,
                          reqs=mk(pkv.CLASS_DECODE), scale=scale, out=out, lse=lse)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, g.k_cache, g.v_cache, g.block_tables, maxq, maxs,
                    reqs=mk(pkv.CLASS_EXTEND), scale=scale, out=out, lse=lse)
    pkv.varlen_prefill_attn(g.q, g.k_new, g.v_new, g.cu_q, maxq, reqs=mk(pkv.CLASS_PREFILL), scale=scale,
                            out=out, lse=lse)
    assert _errors(pkv) == 0
    kc, vc = bits(b.k_cache).copy(), bits(b.v_cache).copy()
    assert oracle.kv_cache_write(bits(b.k_new), bits(b.v_new), b.slot_mapping.numpy(), kc, vc) == 0
    o_perm, o_bounds, _, _ = oracle.batch_classify_reorder(b.cu_q.numpy(), b.seq_lens.numpy())
    assert np.array_equal(perm.cpu().numpy(), o_perm) and np.array_equal(bounds.cpu().numpy(), o_bounds)
    ref = np.full((T, b.Hq, D), np.nan)
    ref_lse = np.full((T, b.Hq), np.nan)
    qb = bits(b.q)
    oracle.paged_decode(qb, kc, vc, b.block_tables.numpy(), b.seq_lens.numpy(), scale, cu_q=b.cu_q.numpy(),
                        req_ids=o_perm[o_bounds[0]:o_bounds[1]], out=ref, lse=ref_lse)
    oracle_extend(b, kc, vc, scale, req_ids=o_perm[o_bounds[1]:o_bounds[2]], out=ref, lse=ref_lse)
    oracle_prefill(b, scale, req_ids=o_perm[o_bounds[2]:o_bounds[3]], out=ref, lse=ref_lse)
    compare_attention(out, lse, ref, ref_lse, what=f"random mix {seed}: D={D} Hkv={Hkv} G={G}")


@pytest.mark.parametrize("seed", range(6))
def test_random_mla_batches(pkv, seed):
    rng = np.random.default_rng(3000 + seed)
    Hq = int(rng.choice([16, 32, 64, 128]))
    R = int(rng.integers(1, 40))
    lens = [int(x) for x in rng.integers(0, int(rng.choice([50, 2000, 20000])), size=R)]
    b = gen.mla_batch(R, 0, 0, Hq=Hq, seq_lens=lens, seed=4000 + seed)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what=f"random mla {seed}: Hq={Hq} R={R}")
    assert _errors(pkv) == 0


# ---- failure detection -----------------------------------------------------------------------

def test_bounded_wait_runs_out_and_the_context_stays_usable(pkv):
    """A barrier nothing completes: the library's bounded wait gives up after the limit, the
    TIMEOUT bit shows in the device error word, and the next calls run normally."""
    pkv.device_errors(clear=True)
    pkv.selftest_bounded_wait(limit_ns=20_000_000)
    assert pkv.device_errors(clear=True) & 0x10
    b = gen.decode_batch(**gen.TINY_DECODE)
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), b.k_cache.to(DEV), b.v_cache.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(b.seq_lens_list), scale=1 / math.sqrt(b.D))
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), 1 / math.sqrt(b.D))
    compare_attention(out, lse, ref, ref_lse, what="decode after a timed-out wait")
    assert pkv.device_errors() == 0


# ---- batch_classify_reorder ------------------------------------------------------------------

def _reorder_case(R, seed, thr=1):
    rng = np.random.default_rng(seed)
    kind = rng.integers(0, 3, R)
    q = np.where(kind == 0, rng.integers(0, 2, R), rng.integers(1, 300, R))
    cached = np.where(kind == 1, rng.integers(1, 1000, R), 0)
    cached = np.where(kind == 0, rng.integers(0, 5000, R), cached)
    seq = q + cached
    cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    return cu, seq.astype(np.int32), thr


@pytest.mark.parametrize("R,seed,thr", [(0, 0, 1), (1, 1, 1), (204, 2, 1), (1024, 3, 1),
                                        (1025, 4, 1), (3001, 5, 1), (500, 6, 4), (64, 7, 0)])
def test_reorder_bit_exact(pkv, R, seed, thr):
    cu, seq, thr = _reorder_case(R, seed, thr)
    T = int(cu[-1])
    perm, bounds, cu_r, tmap = pkv.batch_classify_reorder(
        torch.from_numpy(cu).to(DEV), torch.from_numpy(seq).to(DEV), decode_threshold=thr,
        with_token_map=True, num_tokens=T)
    e_perm, e_bounds, e_cu, e_map = oracle.batch_classify_reorder(cu, seq, thr)
    assert np.array_equal(perm.cpu().numpy(), e_perm)
    assert np.array_equal(bounds.cpu().numpy(), e_bounds)
    assert np.array_equal(cu_r.cpu().numpy(), e_cu)
    assert np.array_equal(tmap.cpu().numpy(), e_map)


def test_reorder_single_class(pkv):
    cu = np.arange(0, 11, dtype=np.int32)          # ten decode requests
    seq = np.full(10, 50, np.int32)
    perm, bounds, _, _ = pkv.batch_classify_reorder(torch.from_numpy(cu).to(DEV), torch.from_numpy(seq).to(DEV))
    assert perm.tolist() == list(range(10)) and bounds.tolist() == [0, 10, 10, 10]


# ---- paged_decode_attn -----------------------------------------------------------------------

@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_group_sizes(pkv, G, D):
    Hkv = 2
    b = gen.decode_batch(6, 1, 300, Hq=G * Hkv, Hkv=Hkv, D=D, seed=10 * G + D)
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                     max(b.seq_lens_list), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what=f"decode G={G} D={D}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hkv", [1, 3, 5, 6, 12, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_kv_head_counts(pkv, Hkv, D):
    """KV head counts that lay the CTAs out differently: a CTA runs several shares side by side,
    each with a divisor of Hkv as its warps (Hkv 3 and 5: one warp per share and one head group
    per head; 6: two; 12 and 16: several head groups). Lengths cut sequences at share edges."""
    b = gen.decode_batch(7, 1, 900, Hq=2 * Hkv, Hkv=Hkv, D=D, seed=300 + 7 * Hkv + D)
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                     max(b.seq_lens_list), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what=f"decode Hkv={Hkv} D={D}")
    assert _errors(pkv) == 0


def test_decode_tiny_config(pkv):
    """4 sequences, context U[16,200], 8 Q / 2 KV heads, head_dim 64, pool of 64 blocks, seed 0."""
    b = gen.decode_batch(**gen.TINY_DECODE)
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                     max(b.seq_lens_list), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what="decode tiny")


@pytest.mark.parametrize("ctxs", [[1, 16, 17, 31, 32, 33], [0, 5, 0], [4096, 1, 7000, 15]])
def test_decode_edge_lengths_and_splits(pkv, ctxs):
    b = gen.make_batch([gen.DECODE] * len(ctxs), [1] * len(ctxs), ctxs, Hq=16, Hkv=1, D=128, seed=len(ctxs))
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                     max(ctxs), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what=f"decode {ctxs}")
    empty = np.array(ctxs) == 0
    if empty.any():
        o = out.float().cpu().numpy()[empty]
        assert np.all(o == 0) and np.all(np.isneginf(lse.cpu().numpy()[empty]))


@pytest.mark.parametrize("ctxs", [[256], [640], [2048], [2176], [8320], [80000], [192000], [50000, 7, 30000]])
def test_decode_long_sequences_merge_tree(pkv, ctxs):
    """A few long sequences spread over all the CTAs: each is cut into up to one piece per
    share, and the pieces are merged along the fan-in-4 tree (depths 1 to 6 here, including
    partly filled groups)."""
    b = gen.make_batch([gen.DECODE] * len(ctxs), [1] * len(ctxs), ctxs, Hq=16, Hkv=1, D=128, seed=sum(ctxs) % 101)
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, max(ctxs),
                                     cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what=f"decode long {ctxs}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hq,Hkv,D,fp8,longs,seed", [
    (64, 4, 128, True, [83746], 3),           # FP8, 3 shares of 4 warps a CTA (the headline shape)
    (64, 4, 128, True, [150633, 60000], 7),
    (64, 4, 128, False, [120000], 11),        # bf16, 2 shares of 4 warps a CTA
    (24, 6, 64, False, [153387], 10),         # bf16 D 64 at Hkv 6
    (16, 4, 128, False, [192000], 5),
])
def test_decode_long_sequences_several_shares_per_cta(pkv, Hq, Hkv, D, fp8, longs, seed):
    """Long sequences (cut into hundreds of pieces) among short ones, at head counts where one
    CTA runs several shares side by side, so the launch holds more shares than CTAs: the merge
    counters of different tree levels must be distinct (levels a whole launch's shares apart).
    Counters shared by two nodes only go wrong when their arrivals interleave, so every call is
    repeated."""
    rnd = np.random.default_rng(seed)
    ctxs = list(longs) + [int(x) for x in rnd.integers(0, 3000, size=int(rnd.integers(8, 30)))]
    rnd.shuffle(ctxs)
    b = gen.make_batch([gen.DECODE] * len(ctxs), [1] * len(ctxs), ctxs, Hq=Hq, Hkv=Hkv, D=D, seed=seed)
    g = b.to(DEV)
    scale = default_scale(b.D)
    kw, kc, vc = {}, g.k_cache, g.v_cache
    if fp8:
        ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
        kc8, vc8 = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
        kw, kc, vc = dict(k_scale=ks, v_scale=vs), kc8.to(DEV), vc8.to(DEV)
        ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc8), _codes(vc8), b.block_tables.numpy(),
                                               b.seq_lens.numpy(), scale, ks, vs)
    else:
        ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    for rep in range(6):
        out, lse = pkv.paged_decode_attn(g.q, kc, vc, g.block_tables, g.seq_lens, max(ctxs), cu_q=g.cu_q,
                                         scale=scale, **kw)
        compare_attention(out, lse, ref, ref_lse, what=f"decode long Hq {Hq} Hkv {Hkv} D {D} fp8={fp8} call {rep}")
    assert _errors(pkv) == 0


def test_decode_peaked_softmax(pkv):
    b = gen.decode_batch(8, 100, 900, Hq=32, Hkv=4, D=128, seed=77, q_scale=4.0)
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                     max(b.seq_lens_list), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what="decode peaked")


def test_decode_nonfinite_past_the_end_is_ignored(pkv):
    """Cache rows after the last valid token of a block may hold anything (NaN here)."""
    b = gen.decode_batch(3, 5, 40, Hq=8, Hkv=2, D=64, seed=5)
    kc = b.k_cache.clone()
    vc = b.v_cache.clone()
    bt = b.block_tables.numpy()
    for r, n in enumerate(b.seq_lens_list):
        last = bt[r, (n - 1) // 16]
        kc[last, n % 16 or 16:] = float("nan")
        vc[last, n % 16 or 16:] = float("nan")
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.paged_decode_attn(g.q, kc.to(DEV), vc.to(DEV), g.block_tables, g.seq_lens,
                                     max(b.seq_lens_list), cu_q=g.cu_q, scale=scale)
    ref, ref_lse = oracle_decode(b, bits(kc), bits(vc), scale)
    compare_attention(out, lse, ref, ref_lse, what="decode nan tail")


# ---- MLA absorbed decode ---------------------------------------------------------------------

def _mla(pkv, b, scale, **kw):
    return pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, max(b.seq_lens_list), scale, **kw)


def _mla_ref(b, scale, latent=None, **kw):
    lat = bits(b.latent if latent is None else latent)
    return oracle.mla_decode(bits(b.q), lat, b.block_tables.cpu().numpy(), b.seq_lens.cpu().numpy(), scale,
                             gen.MLA_DV, **kw)


@pytest.mark.parametrize("Hq", [16, 32, 128])
def test_mla_decode_head_groups(pkv, Hq):
    """16 query heads per CTA group: one, two and eight groups over the same latent rows."""
    b = gen.mla_batch(5, 1, 700, Hq=Hq, seed=90 + Hq)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    assert out.shape == (5, Hq, gen.MLA_DV)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what=f"mla Hq={Hq}")
    assert _errors(pkv) == 0


def _to_dev(b):
    return gen.MlaBatch(**{**b.__dict__, "q": b.q.to(DEV), "latent": b.latent.to(DEV),
                           "block_tables": b.block_tables.to(DEV), "seq_lens": b.seq_lens.to(DEV)})


@pytest.mark.parametrize("Hq", [16, 128])
@pytest.mark.parametrize("ctxs", [[1, 16, 17, 31, 32, 33], [0, 5, 0], [4096, 1, 7000, 15], [30000, 20000]])
def test_mla_decode_edge_lengths_and_cuts(pkv, ctxs, Hq):
    """Partial last blocks, empty contexts (out 0, lse -inf), and a few long sequences that the
    shares cut into many pieces (merged in several passes). At 128 heads the tensor-core kernel
    runs: tiles of 112 keys, partial tiles at piece ends, the merge of cut sequences."""
    b = gen.mla_batch(len(ctxs), 0, 0, Hq=Hq, seq_lens=ctxs, seed=len(ctxs) + sum(ctxs) % 97)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what=f"mla {ctxs} Hq={Hq}")
    empty = np.array(ctxs) == 0
    if empty.any():
        assert np.all(out.float().cpu().numpy()[empty] == 0)
        assert np.all(np.isneginf(lse.cpu().numpy()[empty]))
    assert _errors(pkv) == 0


@pytest.mark.parametrize("ctxs,Hq", [([640], 16), ([8320], 16), ([80000], 16), ([3, 41000, 9000], 16),
                                     ([640], 128), ([8320], 128), ([3, 41000, 9000], 128)])
def test_mla_decode_long_sequences_merge_tree(pkv, ctxs, Hq):
    b = gen.mla_batch(len(ctxs), 0, 0, Hq=Hq, seq_lens=ctxs, seed=sum(ctxs) % 89)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what=f"mla long {ctxs} Hq={Hq}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hq", [16, 128])
def test_mla_decode_peaked_softmax(pkv, Hq):
    b = gen.mla_batch(6, 100, 2000, Hq=Hq, seed=93, q_scale=3.0)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what=f"mla peaked Hq={Hq}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hq", [16, 128])
def test_mla_decode_running_max_grows_late(pkv, Hq):
    """Each sequence's first 200 latent rows are scaled down 20x, so the scores of its first key
    tiles are small and the running max grows by far more than the lazy-rescale threshold
    (8 in log2 units) later on: the kernels must rescale the accumulated output (at 128 heads,
    CTA 1 of the pair rescales O in tensor memory when CTA 0 reports it)."""
    b = gen.mla_batch(5, 600, 3000, Hq=Hq, seed=97, q_scale=3.0)
    lat = b.latent.clone()
    bt = b.block_tables.numpy()
    for r, n in enumerate(b.seq_lens_list):
        for j in range(min(n, 200)):
            blk, off = bt[r, j // 16], j % 16
            lat[blk, off] = (lat[blk, off].float() * 0.05).to(torch.bfloat16)
    out, lse = pkv.mla_decode_attn(b.q.to(DEV), lat.to(DEV), b.block_tables.to(DEV), b.seq_lens.to(DEV),
                                   max(b.seq_lens_list), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE, latent=lat)
    compare_attention(out, lse, ref, ref_lse, what=f"mla late max Hq={Hq}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hq", [16, 128])
def test_mla_decode_nonfinite_past_the_end_is_ignored(pkv, Hq):
    b = gen.mla_batch(4, 5, 90, Hq=Hq, seed=94)
    lat = b.latent.clone()
    bt = b.block_tables.numpy()
    for r, n in enumerate(b.seq_lens_list):
        lat[bt[r, (n - 1) // 16], n % 16 or 16:] = float("nan")
    out, lse = pkv.mla_decode_attn(b.q.to(DEV), lat.to(DEV), b.block_tables.to(DEV), b.seq_lens.to(DEV),
                                   max(b.seq_lens_list), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE, latent=lat)
    compare_attention(out, lse, ref, ref_lse, what=f"mla nan tail Hq={Hq}")


@pytest.mark.parametrize("Hq", [16, 128])
def test_mla_decode_request_set_and_query_rows(pkv, Hq):
    """A request set given by order/bounds (the decode class of a reordered batch) with query
    rows taken through cu_q: only the set's rows are written."""
    R = 9
    b = gen.mla_batch(R, 1, 900, Hq=Hq, seed=95)
    order = torch.tensor([7, 2, 5, 0, 8, 1, 3, 4, 6], dtype=torch.int32)
    bounds = torch.tensor([2, 7, 9, 9], dtype=torch.int32)  # the set: order[2:7]
    cu_q = torch.tensor([3 * r for r in range(R + 1)], dtype=torch.int32)  # query row of r = 3r
    q = gen.randn_bf16((3 * R, Hq, 576), torch.Generator().manual_seed(6), "cpu")
    out = torch.full((3 * R, Hq, gen.MLA_DV), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((3 * R, Hq), float("nan"), dtype=torch.float32, device=DEV)
    pkv.mla_decode_attn(q.to(DEV), b.latent.to(DEV), b.block_tables.to(DEV), b.seq_lens.to(DEV),
                        max(b.seq_lens_list), gen.MLA_SCALE, cu_q=cu_q.to(DEV),
                        reqs=pkv.Reqs(5, R, order.to(DEV), bounds.to(DEV), 0), out=out, lse=lse)
    members = order[2:7].numpy()
    ref, ref_lse = oracle.mla_decode(bits(q), bits(b.latent), b.block_tables.numpy(), b.seq_lens.numpy(),
                                     gen.MLA_SCALE, gen.MLA_DV, cu_q=cu_q.numpy(), req_ids=members)
    rows = np.zeros(3 * R, bool)
    rows[3 * members] = True
    compare_attention(out, lse, ref, ref_lse, rows=rows, what="mla set")
    assert torch.isnan(out.float().cpu()[~torch.from_numpy(rows)]).all()
    assert _errors(pkv) == 0


@pytest.mark.parametrize("Hq,v_dim,dk", [(8, 512, 576), (16, 256, 576), (16, 512, 512), (144, 512, 576)])
def test_mla_decode_rejects_other_shapes(pkv, Hq, v_dim, dk):
    b = gen.mla_batch(2, 1, 40, Hq=Hq, Dk=dk, seed=96)
    with pytest.raises(pkv.PkvError):
        pkv.mla_decode_attn(b.q.to(DEV), b.latent.to(DEV), b.block_tables.to(DEV), b.seq_lens.to(DEV), 40,
                            gen.MLA_SCALE, v_dim=v_dim)


# ---- extend / prefill ------------------------------------------------------------------------

@pytest.mark.parametrize("G,D", [(1, 64), (4, 128), (8, 128), (16, 64), (2, 128)])
def test_extend_ragged(pkv, G, D):
    Hkv = 2
    new = [1, 63, 64, 65, 130, 7]
    ctx = [0, 1, 15, 16, 100, 300]
    b = gen.extend_batch(new, ctx, Hq=G * Hkv, Hkv=Hkv, D=D, seed=G * 7 + D)
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, g.k_cache, g.v_cache,
                               g.block_tables, max(new), max(b.seq_lens_list), scale=scale)
    ref, ref_lse = oracle_extend(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what=f"extend G={G} D={D}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_extend_nonfinite_past_the_context_end_is_ignored(pkv, D):
    """Cache rows after a context's last token (in its last block) may hold anything: NaN and
    +inf keys and inf values here, with peaked queries. The context's last key tile masks those
    columns before any arithmetic, and their value rows are zeroed."""
    Hkv = 2
    new = [1, 40, 130, 7, 64]
    ctx = [5, 100, 300, 17, 129]
    b = gen.extend_batch(new, ctx, Hq=4 * Hkv, Hkv=Hkv, D=D, seed=70 + D, q_scale=3.0)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    bt = b.block_tables.numpy()
    for r, C in enumerate(ctx):
        if C % 16:
            last = bt[r, C // 16]
            kc[last, C % 16:] = float("nan")
            kc[last, C % 16::3] = float("inf")
            vc[last, C % 16:] = float("inf")
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kc.to(DEV), vc.to(DEV), g.block_tables,
                               max(new), max(b.seq_lens_list), scale=scale)
    ref, ref_lse = oracle_extend(b, bits(kc), bits(vc), scale)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, what=f"extend nonfinite tail D={D}")
    assert _errors(pkv) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_ragged(pkv, D):
    lens = [1, 17, 64, 65, 200, 128, 3]
    b = gen.prefill_batch(lens, Hq=16, Hkv=4, D=D, seed=D)
    g = b.to(DEV)
    scale = default_scale(D)
    out, lse = pkv.varlen_prefill_attn(g.q, g.k_new, g.v_new, g.cu_q, max(lens), scale=scale)
    ref, ref_lse = oracle_prefill(b, scale)
    compare_attention(out, lse, ref, ref_lse, what=f"prefill D={D}")
    assert _errors(pkv) == 0


def test_prefill_peaked(pkv):
    b = gen.prefill_batch([300, 77], Hq=8, Hkv=1, D=128, seed=9, q_scale=4.0)
    g = b.to(DEV)
    scale = default_scale(b.D)
    out, lse = pkv.varlen_prefill_attn(g.q, g.k_new, g.v_new, g.cu_q, 300, scale=scale)
    ref, ref_lse = oracle_prefill(b, scale)
    compare_attention(out, lse, ref, ref_lse, what="prefill peaked")


# ---- the mixed batch through the reorder -----------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
def test_mixed_batch_pipeline(pkv, D):
    b = gen.mixed_batch(20, (10, 400), 3, 70, (30, 300), 3, (10, 150), Hq=16, Hkv=2, D=D, seed=31 + D)
    g = b.to(DEV)
    scale = default_scale(D)
    R, T = b.R, b.T
    perm, bounds, _, _ = pkv.batch_classify_reorder(g.cu_q, g.seq_lens)
    pkv.kv_cache_write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    maxs, maxq = max(b.seq_lens_list), max(b.q_lens)
    mk = lambda c: pkv.Reqs(max_reqs=R, batch_reqs=R, order=perm, bounds=bounds, cls=c)
    pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, maxs, cu_q=g.cu_q,
                          reqs=mk(pkv.CLASS_DECODE), scale=scale, out=out, lse=lse)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, g.k_cache, g.v_cache, g.block_tables,
                    maxq, maxs, reqs=mk(pkv.CLASS_EXTEND), scale=scale, out=out, lse=lse)
    pkv.varlen_prefill_attn(g.q, g.k_new, g.v_new, g.cu_q, maxq, reqs=mk(pkv.CLASS_PREFILL),
                            scale=scale, out=out, lse=lse)
    assert _errors(pkv) == 0
    kc, vc = bits(b.k_cache).copy(), bits(b.v_cache).copy()
    oracle.kv_cache_write(bits(b.k_new), bits(b.v_new), b.slot_mapping.numpy(), kc, vc)
    assert np.array_equal(bits(g.k_cache), kc)
    e_perm, e_b, _, _ = oracle.batch_classify_reorder(b.cu_q.numpy(), b.seq_lens.numpy())
    ref = np.full((T, b.Hq, D), np.nan)
    ref_lse = np.full((T, b.Hq), np.nan)
    oracle_decode(b, kc, vc, scale, req_ids=e_perm[e_b[0]:e_b[1]], out=ref, lse=ref_lse)
    oracle_extend(b, kc, vc, scale, req_ids=e_perm[e_b[1]:e_b[2]], out=ref, lse=ref_lse)
    oracle_prefill(b, scale, req_ids=e_perm[e_b[2]:e_b[3]], out=ref, lse=ref_lse)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, rows=np.ones(T, bool), what=f"mixed D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_mixed_batch_unified_single_call(pkv, D):
    """The unified variant (vLLM blog "rocm-attention-backend", "Unified attention backends":
    one kernel for every token type): the whole batch in arrival order through one extend_attn
    call — decode requests are extend requests with one new token, prefill requests extend
    requests with no cached tokens. Same results as the three routed calls, against the oracle."""
    b = gen.mixed_batch(20, (10, 400), 3, 70, (30, 300), 3, (10, 150), Hq=16, Hkv=2, D=D, seed=33 + D)
    g = b.to(DEV)
    scale = default_scale(D)
    R, T = b.R, b.T
    pkv.kv_cache_write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    out, lse = pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, g.k_cache, g.v_cache, g.block_tables,
                               max(b.q_lens), max(b.seq_lens_list), scale=scale)
    assert _errors(pkv) == 0
    kc, vc = bits(b.k_cache).copy(), bits(b.v_cache).copy()
    oracle.kv_cache_write(bits(b.k_new), bits(b.v_new), b.slot_mapping.numpy(), kc, vc)
    e_perm, e_b, _, _ = oracle.batch_classify_reorder(b.cu_q.numpy(), b.seq_lens.numpy())
    ref = np.full((T, b.Hq, D), np.nan)
    ref_lse = np.full((T, b.Hq), np.nan)
    oracle_decode(b, kc, vc, scale, req_ids=e_perm[e_b[0]:e_b[1]], out=ref, lse=ref_lse)
    oracle_extend(b, kc, vc, scale, req_ids=e_perm[e_b[1]:e_b[2]], out=ref, lse=ref_lse)
    oracle_prefill(b, scale, req_ids=e_perm[e_b[2]:e_b[3]], out=ref, lse=ref_lse)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, rows=np.ones(T, bool), what=f"unified D={D}")


@pytest.mark.parametrize("G,Hkv,D,fp8", [(2, 4, 128, False), (4, 2, 64, False), (8, 2, 128, False),
                                          (16, 1, 64, False), (8, 3, 128, True), (1, 4, 128, False)])
def test_extend_one_token_requests_pack_heads(pkv, G, Hkv, D, fp8):
    """One-token requests inside extend_attn (decodes sent through the extend call): their G query
    heads share one tile (one item per KV head), beside ordinary extend requests in the same
    launch. Ragged and empty contexts, non-finite values past each context's end."""
    ctx = [0, 1, 15, 16, 17, 300, 1000, 4095]
    new = [1] * len(ctx) + [70, 129]
    ctx = ctx + [50, 200]
    b = gen.extend_batch(new, ctx, Hq=G * Hkv, Hkv=Hkv, D=D, seed=900 + G * 10 + D + fp8)
    bt = b.block_tables.numpy()
    g = b.to(DEV)
    scale = default_scale(D)
    kw = {}
    if fp8:
        ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
        kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
        for r, C in enumerate(ctx):
            if C % 16:
                kc[bt[r, C // 16], C % 16:] = 0x7F
                vc[bt[r, C // 16], C % 16:] = 0xFF
        kw = dict(k_scale=ks, v_scale=vs)
        kcd, vcd = kc.to(DEV), vc.to(DEV)
    else:
        kc, vc = b.k_cache.clone(), b.v_cache.clone()
        for r, C in enumerate(ctx):
            if C % 16:
                kc[bt[r, C // 16], C % 16:] = float("nan")
                vc[bt[r, C // 16], C % 16:] = float("inf")
        kcd, vcd = kc.to(DEV), vc.to(DEV)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((b.T, b.Hq), float("nan"), dtype=torch.float32, device=DEV)
    pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, kcd, vcd, g.block_tables, max(new),
                    max(b.seq_lens_list), scale=scale, out=out, lse=lse, **kw)
    if fp8:
        ref, ref_lse = _fp8_extend_ref(b, kc.numpy(), vc.numpy(), ks, vs, scale)
    else:
        ref, ref_lse = oracle_extend(b, bits(kc), bits(vc), scale)
    assert not np.isnan(ref).any()
    compare_attention(out, lse, ref, ref_lse, rows=np.ones(b.T, bool), what=f"extend one-token G={G} D={D} fp8={fp8}")
    assert _errors(pkv) == 0


def test_request_set_cut_to_max_reqs_is_flagged(pkv):
    b = gen.decode_batch(6, 10, 60, Hq=4, Hkv=1, D=64, seed=2)
    g = b.to(DEV)
    bounds = torch.tensor([0, 6, 6, 6], dtype=torch.int32, device=DEV)
    order = torch.arange(6, dtype=torch.int32, device=DEV)
    reqs = pkv.Reqs(max_reqs=4, batch_reqs=6, order=order, bounds=bounds, cls=0)
    out = torch.zeros_like(g.q)
    pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, 60, cu_q=g.cu_q,
                          reqs=reqs, out=out)
    assert _errors(pkv) & 0x4
    assert out[4:].abs().sum().item() == 0  # requests past the bound are not computed


# ---- request sets larger than one launch holds (1024 requests) -------------------------------

def test_decode_request_sets_larger_than_one_launch(pkv):
    """1500 short decode sequences: more than the 1024 requests one launch holds, so two launches
    serve them. Every row against the oracle; once as the plain set, once as the decode class of
    a reordered batch whose size the host only bounds (max_reqs 2048), in a shuffled order."""
    R = 1500
    b = gen.decode_batch(R, 1, 300, Hq=16, Hkv=2, D=128, seed=1500)
    g = b.to(DEV)
    scale = default_scale(128)
    ref, ref_lse = oracle_decode(b, bits(b.k_cache), bits(b.v_cache), scale)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((g.T, g.Hq), float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, max(b.seq_lens_list),
                          cu_q=g.cu_q, scale=scale, out=out, lse=lse)
    compare_attention(out, lse, ref, ref_lse, what="decode 1500 requests")
    assert _errors(pkv) == 0
    order = torch.randperm(R, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    bounds = torch.tensor([0, R, R, R], dtype=torch.int32)
    reqs = pkv.Reqs(max_reqs=2048, batch_reqs=R, order=order.to(DEV), bounds=bounds.to(DEV), cls=0)
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    pkv.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens, max(b.seq_lens_list),
                          cu_q=g.cu_q, reqs=reqs, scale=scale, out=out, lse=lse)
    compare_attention(out, lse, ref, ref_lse, what="decode 1500 requests, reordered set")
    assert _errors(pkv) == 0


def test_decode_fp8_request_set_larger_than_one_launch(pkv):
    b, kc, vc, ks, vs = _fp8_decode_case(1100, 1, 200, Hq=32, Hkv=4, seed=1100)
    out, lse = pkv.paged_decode_attn(b.q.to(DEV), kc.to(DEV), vc.to(DEV), b.block_tables.to(DEV),
                                     b.seq_lens.to(DEV), max(b.seq_lens_list), scale=1 / math.sqrt(128),
                                     k_scale=ks, v_scale=vs)
    ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                           b.seq_lens.numpy(), 1 / math.sqrt(128), ks, vs)
    compare_attention(out, lse, ref, ref_lse, what="decode fp8 1100 requests")
    assert _errors(pkv) == 0


def test_mla_decode_request_set_larger_than_one_launch(pkv):
    b = gen.mla_batch(1100, 1, 120, Hq=16, seed=1101)
    out, lse = _mla(pkv, _to_dev(b), gen.MLA_SCALE)
    ref, ref_lse = _mla_ref(b, gen.MLA_SCALE)
    compare_attention(out, lse, ref, ref_lse, what="mla 1100 requests")
    assert _errors(pkv) == 0


def test_prefill_and_extend_request_sets_larger_than_one_launch(pkv):
    """1100 short prompts (prefill), and 1030 short extends: each needs two launches."""
    lens = gen.uniform_ints(1, 40, 1100, torch.Generator().manual_seed(1102))
    b = gen.prefill_batch(lens, Hq=8, Hkv=2, D=64, seed=1102)
    g = b.to(DEV)
    scale = default_scale(64)
    out, lse = pkv.varlen_prefill_attn(g.q, g.k_new, g.v_new, g.cu_q, max(lens), scale=scale)
    ref, ref_lse = oracle_prefill(b, scale)
    compare_attention(out, lse, ref, ref_lse, what="prefill 1100 requests")
    assert _errors(pkv) == 0
    gr = torch.Generator().manual_seed(1103)
    new = gen.uniform_ints(1, 20, 1030, gr)
    ctx = gen.uniform_ints(1, 60, 1030, gr)
    b = gen.extend_batch(new, ctx, Hq=8, Hkv=2, D=128, seed=1103)
    g = b.to(DEV)
    scale = default_scale(128)
    out, lse = pkv.extend_attn(g.q, g.k_new, g.v_new, g.cu_q, g.seq_lens, g.k_cache, g.v_cache,
                               g.block_tables, max(new), max(b.seq_lens_list), scale=scale)
    ref, ref_lse = oracle_extend(b, bits(b.k_cache), bits(b.v_cache), scale)
    compare_attention(out, lse, ref, ref_lse, what="extend 1030 requests")
    assert _errors(pkv) == 0
