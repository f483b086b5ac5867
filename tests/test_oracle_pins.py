"""Pins of the fp64 oracle to facts that do not come from the oracle itself: library
routines (torch's scaled_dot_product_attention in float64, numpy indexing, Python's stable
sort, scipy's logsumexp), closed forms, invariants the pages state, and the printed numbers
of the pages (tests/golden). CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from pkv_workloads import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    """bf16 bits -> float64, through torch's own bf16 conversion."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def dense_kv(batch, r, upto):
    """The logical key/value sequence of request r (positions 0..upto-1), gathered with numpy
    fancy indexing from the paged cache."""
    bs = batch.block_size
    pos = np.arange(upto)
    blk = batch.block_tables.numpy()[r, pos // bs]
    kc, vc = gen.bf16_bits(batch.k_cache), gen.bf16_bits(batch.v_cache)
    return f64(kc[blk, pos % bs]), f64(vc[blk, pos % bs])   # [n, Hkv, D]


def sdpa(q, k, v, scale, causal_offset=None):
    """torch SDPA in float64. q [n_q, Hq, D], k/v [n_k, Hkv, D]; GQA by repeat_interleave
    (query head h reads KV head h // G). causal_offset c: query i sees keys 0..c+i."""
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1).transpose(0, 1)
    vv = v.repeat_interleave(G, dim=1).transpose(0, 1)
    qq = q.transpose(0, 1)
    mask = None
    if causal_offset is not None:
        nq, nk = q.shape[0], k.shape[0]
        mask = torch.arange(nk)[None, :] <= (causal_offset + torch.arange(nq))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    return o.transpose(0, 1).numpy()


def lse_ref(q, k, scale, causal_offset=None):
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1)
    s = torch.einsum("qhd,khd->qhk", q, kk).numpy() * scale
    if causal_offset is not None:
        nq, nk = q.shape[0], k.shape[0]
        allowed = np.arange(nk)[None, :] <= (causal_offset + np.arange(nq))[:, None]
        s = np.where(allowed[:, None, :], s, -np.inf)
    return logsumexp(s, axis=-1)


# ---- sizes -------------------------------------------------------------------------------------

def test_kv_bytes_per_token_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "kv_size_llama70b.json")))
    b = oracle.kv_bytes_per_token(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert b == g["bytes_per_token"] == 320 * 1024
    total = b * g["prompt_tokens"]
    assert abs(total - g["prompt_bytes_approx"]) / g["prompt_bytes_approx"] < 0.1


# ---- write / pack ------------------------------------------------------------------------------

def test_write_matches_numpy_scatter_and_skips_negative():
    b = gen.mixed_batch(3, (5, 40), 2, 7, (10, 50), 2, (3, 30), Hq=4, Hkv=2, D=8, seed=11)
    slots = b.slot_mapping.numpy().copy()
    slots[::5] = -1                      # padding tokens
    kc, vc = gen.bf16_bits(b.k_cache).copy(), gen.bf16_bits(b.v_cache).copy()
    ek, ev = kc.copy(), vc.copy()
    key, val = gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new)
    bad = oracle.kv_cache_write(key, val, slots, kc, vc)
    assert bad == 0
    keep = slots >= 0
    rows_k = ek.reshape(-1, *ek.shape[2:])
    rows_v = ev.reshape(-1, *ev.shape[2:])
    rows_k[slots[keep]] = key[keep]
    rows_v[slots[keep]] = val[keep]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_write_counts_out_of_range_slots():
    kc = np.zeros((4, 16, 1, 8), np.uint16)
    vc = np.zeros_like(kc)
    key = np.ones((3, 1, 8), np.uint16)
    bad = oracle.kv_cache_write(key, key, np.array([0, 64, 1000], np.int64), kc, vc)
    assert bad == 2
    assert kc[0, 0].sum() == 8 and kc.sum() == 8


def test_pack_matches_numpy_take_and_roundtrips_write():
    layers = gen.write_pack_layers(2, 100, Hkv=2, D=16, block_size=16, seed=5)
    for shuffled in (False, True):
        for L in gen.write_pack_layers(1, 100, Hkv=2, D=16, seed=6, shuffled_pack=shuffled) + layers:
            kc, vc = gen.bf16_bits(L.k_cache).copy(), gen.bf16_bits(L.v_cache).copy()
            key, val = gen.bf16_bits(L.key), gen.bf16_bits(L.value)
            oracle.kv_cache_write(key, val, L.slot_mapping.numpy(), kc, vc)
            ids = L.block_ids.numpy()
            dst, bad = oracle.kv_block_pack(kc, vc, ids)
            assert bad == 0
            assert np.array_equal(dst[0], np.take(kc, ids, axis=0))
            assert np.array_equal(dst[1], np.take(vc, ids, axis=0))
            if not shuffled:
                # blocks in request order, flattened, give back the prompt's rows
                T = key.shape[0]
                assert np.array_equal(dst[0].reshape(-1, *key.shape[1:])[:T], key)
                assert np.array_equal(dst[1].reshape(-1, *key.shape[1:])[:T], val)


def test_pack_flags_bad_ids():
    kc = np.arange(4 * 16 * 8, dtype=np.uint16).reshape(4, 16, 1, 8)
    dst, bad = oracle.kv_block_pack(kc, kc, np.array([3, 4, -1, 0], np.int32))
    assert bad == 2
    assert np.array_equal(dst[0, 0], kc[3]) and np.array_equal(dst[0, 3], kc[0])


def test_unpack_matches_numpy_assignment_and_inverts_pack():
    """MORI-IO "Read mode vs write mode": the receiving instance lands each layer's blocks in
    the ids it allocated. unpack == numpy fancy-index assignment; pack then unpack into a
    second pool moves exactly the listed blocks and nothing else."""
    rng = np.random.default_rng(11)
    nb, n = 40, 13
    kc = rng.integers(0, 1 << 16, size=(nb, 16, 2, 8), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(nb, 16, 2, 8), dtype=np.uint16)
    src_ids = rng.permutation(nb)[:n].astype(np.int32)
    dst_ids = rng.permutation(nb)[:n].astype(np.int32)
    packed, bad = oracle.kv_block_pack(kc, vc, src_ids)
    assert bad == 0
    k2 = rng.integers(0, 1 << 16, size=kc.shape, dtype=np.uint16)
    v2 = rng.integers(0, 1 << 16, size=vc.shape, dtype=np.uint16)
    ek, ev = k2.copy(), v2.copy()
    ek[dst_ids] = kc[src_ids]
    ev[dst_ids] = vc[src_ids]
    assert oracle.kv_block_unpack(packed, dst_ids, k2, v2) == 0
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    # the round trip onto the same ids restores the listed blocks of the source pool
    k3, v3 = np.zeros_like(kc), np.zeros_like(vc)
    oracle.kv_block_unpack(packed, src_ids, k3, v3)
    assert np.array_equal(k3[src_ids], kc[src_ids]) and np.array_equal(v3[src_ids], vc[src_ids])
    others = np.setdiff1d(np.arange(nb), src_ids)
    assert not k3[others].any() and not v3[others].any()


def test_unpack_skips_and_counts_bad_ids():
    src = np.arange(2 * 3 * 16 * 8, dtype=np.uint16).reshape(2, 3, 16, 1, 8)
    kc = np.zeros((4, 16, 1, 8), np.uint16)
    vc = np.zeros_like(kc)
    assert oracle.kv_block_unpack(src, np.array([2, 7, -3], np.int32), kc, vc) == 2
    assert np.array_equal(kc[2], src[0, 0]) and np.array_equal(vc[2], src[1, 0])
    assert kc.sum() == src[0, 0].sum()


# ---- reorder -----------------------------------------------------------------------------------

def _classify_brute(q_lens, seq_lens, thr):
    return [0 if q <= thr else (1 if s > q else 2) for q, s in zip(q_lens, seq_lens)]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("thr", [0, 1, 4])
def test_reorder_matches_stable_sort(seed, thr):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(0, 40))
    q_lens = rng.integers(0, 6, R) * rng.integers(0, 2, R) + rng.integers(1, 3, R) * (rng.random(R) < 0.5)
    cached = rng.integers(0, 3, R) * rng.integers(0, 20, R)
    seq = q_lens + cached
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    perm, bounds, cu_r, tmap = oracle.batch_classify_reorder(cu, seq, thr)
    cls = _classify_brute(q_lens, seq, thr)
    exp_perm = sorted(range(R), key=lambda i: cls[i])          # Python's sort is stable
    assert perm.tolist() == exp_perm
    counts = np.bincount(np.array(cls, dtype=np.int64), minlength=3) if R else np.zeros(3, int)
    assert bounds.tolist() == [0, counts[0], counts[0] + counts[1], R]
    assert cu_r.tolist() == [0] + np.cumsum([q_lens[i] for i in exp_perm]).tolist()
    exp_map = [t for i in exp_perm for t in range(cu[i], cu[i + 1])]
    assert tmap.tolist() == exp_map


def test_reorder_walkthrough_from_page():
    g = json.load(open(os.path.join(GOLDEN, "reorder_walkthrough.json")))
    for it in g["iterations"]:
        reqs = it["reqs"]
        q = [r["q_len"] for r in reqs]
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        perm, bounds, _, _ = oracle.batch_classify_reorder(cu, [r["seq_len"] for r in reqs], g["threshold"])
        assert [reqs[i]["name"] for i in perm] == it["order"], it["it"]
        assert bounds.tolist() == it["bounds"], it["it"]
        for j, i in enumerate(perm):
            cls = 0 if j < bounds[1] else (1 if j < bounds[2] else 2)
            assert cls == reqs[i]["cls"]


# ---- attention ---------------------------------------------------------------------------------

TOL = 1e-12


@pytest.mark.parametrize("G,D", [(1, 16), (4, 64), (8, 32), (16, 16)])
def test_decode_matches_torch_sdpa(G, D):
    Hkv = 2
    b = gen.decode_batch(5, 1, 70, Hq=G * Hkv, Hkv=Hkv, D=D, seed=G + D)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.paged_decode(gen.bf16_bits(b.q), gen.bf16_bits(b.k_cache),
                                   gen.bf16_bits(b.v_cache), b.block_tables.numpy(),
                                   b.seq_lens.numpy(), scale, cu_q=b.cu_q.numpy())
    qf = f64(gen.bf16_bits(b.q))
    for r in range(b.R):
        n = b.seq_lens_list[r]
        k, v = dense_kv(b, r, n)
        exp = sdpa(qf[r:r + 1], k, v, scale)
        assert np.abs(out[r] - exp[0]).max() < TOL
        assert np.abs(lse[r] - lse_ref(qf[r:r + 1], k, scale)[0]).max() < TOL


@pytest.mark.parametrize("G,D", [(1, 8), (2, 16), (4, 32)])
def test_prefill_matches_torch_sdpa_causal(G, D):
    Hkv = 2
    b = gen.prefill_batch([1, 17, 40], Hq=G * Hkv, Hkv=Hkv, D=D, seed=3)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.prefill(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                              b.cu_q.numpy(), scale)
    qf, kf, vf = (f64(gen.bf16_bits(t)) for t in (b.q, b.k_new, b.v_new))
    cu = b.cu_q.numpy()
    for r in range(b.R):
        s, e = cu[r], cu[r + 1]
        exp = sdpa(qf[s:e], kf[s:e], vf[s:e], scale, causal_offset=0)
        assert np.abs(out[s:e] - exp).max() < TOL
        assert np.abs(lse[s:e] - lse_ref(qf[s:e], kf[s:e], scale, 0)).max() < TOL


def _extend_case(seed=7, G=4, D=32, q_scale=1.0):
    return gen.extend_batch([1, 5, 23], [0, 37, 50], Hq=2 * G, Hkv=2, D=D, seed=seed, q_scale=q_scale)


def test_extend_matches_torch_sdpa_masked():
    b = _extend_case()
    scale = 1 / math.sqrt(b.D)
    out, lse = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                             b.cu_q.numpy(), scale, seq_lens=b.seq_lens.numpy(),
                             k_cache=gen.bf16_bits(b.k_cache), v_cache=gen.bf16_bits(b.v_cache),
                             block_tables=b.block_tables.numpy())
    qf, kf, vf = (f64(gen.bf16_bits(t)) for t in (b.q, b.k_new, b.v_new))
    cu = b.cu_q.numpy()
    for r in range(b.R):
        s, e = cu[r], cu[r + 1]
        C = b.seq_lens_list[r] - b.q_lens[r]
        kc, vc = dense_kv(b, r, C)
        k = torch.cat([kc, kf[s:e]])
        v = torch.cat([vc, vf[s:e]])
        exp = sdpa(qf[s:e], k, v, scale, causal_offset=C)
        assert np.abs(out[s:e] - exp).max() < TOL
        assert np.abs(lse[s:e] - lse_ref(qf[s:e], k, scale, C)).max() < TOL


def test_results_invariant_to_physical_block_relabeling():
    b = _extend_case(seed=9)
    scale = 1 / math.sqrt(b.D)
    args = dict(seq_lens=b.seq_lens.numpy())
    kc, vc = gen.bf16_bits(b.k_cache), gen.bf16_bits(b.v_cache)
    out1, lse1 = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                               b.cu_q.numpy(), scale, k_cache=kc, v_cache=vc,
                               block_tables=b.block_tables.numpy(), **args)
    sigma = np.random.default_rng(0).permutation(b.num_blocks)   # old id -> new id
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[sigma], vc2[sigma] = kc, vc
    bt2 = sigma[b.block_tables.numpy()].astype(np.int32)
    out2, lse2 = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                               b.cu_q.numpy(), scale, k_cache=kc2, v_cache=vc2, block_tables=bt2,
                               **args)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    # and a relabeling that breaks the table (no longer consistent) must change the result
    out3, _ = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                            b.cu_q.numpy(), scale, k_cache=kc2, v_cache=vc2,
                            block_tables=b.block_tables.numpy(), **args)
    assert not np.allclose(out1[~np.isnan(out1)], out3[~np.isnan(out3)])


@pytest.mark.parametrize("chunk", [1, 16, 17, 40, 32768, 10 ** 9])
def test_chunked_extend_with_lse_merge_equals_single_pass(chunk):
    b = _extend_case(seed=12, q_scale=4.0)
    scale = 1 / math.sqrt(b.D)
    common = (gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new), b.cu_q.numpy())
    out, lse = oracle.extend(*common, scale, seq_lens=b.seq_lens.numpy(),
                             k_cache=gen.bf16_bits(b.k_cache), v_cache=gen.bf16_bits(b.v_cache),
                             block_tables=b.block_tables.numpy())
    out_c, lse_c = oracle.extend_chunked(*common, b.seq_lens.numpy(), gen.bf16_bits(b.k_cache),
                                         gen.bf16_bits(b.v_cache), b.block_tables.numpy(), scale,
                                         chunk)
    assert np.abs(out - out_c).max() < 1e-12
    assert np.abs(lse - lse_c).max() < 1e-12


def test_lse_merge_special_cases():
    o_a = np.array([[1.0, 2.0]]); o_b = np.array([[3.0, -1.0]])
    # an empty partial has weight zero, whichever side it is on
    o, l = oracle.lse_merge(o_a, np.array([0.5]), o_b, np.array([-np.inf]))
    assert np.array_equal(o, o_a) and l[0] == 0.5
    o, l = oracle.lse_merge(o_a, np.array([-np.inf]), o_b, np.array([2.0]))
    assert np.array_equal(o, o_b) and l[0] == 2.0
    o, l = oracle.lse_merge(o_a, np.array([-np.inf]), o_b, np.array([-np.inf]))
    assert np.array_equal(o, np.zeros_like(o)) and l[0] == -np.inf
    # equal lse: plain average, lse + ln 2
    o, l = oracle.lse_merge(o_a, np.array([1.0]), o_b, np.array([1.0]))
    assert np.allclose(o, (o_a + o_b) / 2, rtol=0, atol=1e-15) and abs(l[0] - (1 + math.log(2))) < 1e-15
    # weights e^la : e^lb
    o, l = oracle.lse_merge(o_a, np.array([0.0]), o_b, np.array([math.log(3.0)]))
    assert np.allclose(o, (o_a + 3 * o_b) / 4, atol=1e-15) and abs(l[0] - math.log(4.0)) < 1e-15


def _decode_single(q_bits, k_rows, v_rows, scale, bs=16):
    """One sequence of len(k_rows) tokens laid into a shuffled small pool, decoded by the oracle."""
    n, Hkv, D = k_rows.shape
    nblk = (n + bs - 1) // bs
    nb = nblk + 3
    tab = np.random.default_rng(n).permutation(nb)[:nblk].astype(np.int32)
    kc = np.zeros((nb, bs, Hkv, D), np.uint16); vc = np.zeros_like(kc)
    pos = np.arange(n)
    kc[tab[pos // bs], pos % bs] = k_rows
    vc[tab[pos // bs], pos % bs] = v_rows
    out, lse = oracle.paged_decode(q_bits[None], kc, vc, tab[None], np.array([n], np.int32), scale)
    return out[0], lse[0]


def _bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_closed_forms():
    rng = np.random.default_rng(1)
    D, scale = 16, 0.25
    q = _bits(rng.standard_normal((2, D)))
    k = _bits(rng.standard_normal((33, 1, D)))
    v = _bits(rng.standard_normal((33, 1, D)))
    qd, kd, vd = f64(q).numpy(), f64(k).numpy(), f64(v).numpy()
    # one key: o = v_0, lse = s_0
    o, l = _decode_single(q, k[:1], v[:1], scale)
    assert np.abs(o - vd[0, 0][None]).max() < TOL
    assert np.abs(l - scale * qd @ kd[0, 0]).max() < TOL
    # q = 0: uniform weights, o = mean(V), lse = ln n
    o, l = _decode_single(np.zeros_like(q), k, v, scale)
    assert np.abs(o - vd[:, 0].mean(0)[None]).max() < 1e-12
    assert np.abs(l - math.log(33)).max() < 1e-12
    # identical keys: uniform weights, lse = s + ln n
    kk = np.repeat(k[:1], 33, axis=0)
    o, l = _decode_single(q, kk, v, scale)
    assert np.abs(o - vd[:, 0].mean(0)[None]).max() < 1e-12
    assert np.abs(l - (scale * qd @ kd[0, 0] + math.log(33))).max() < 1e-12
    # all-ones values: softmax weights sum to one
    ones = _bits(np.ones((33, 1, D)))
    o, _ = _decode_single(q, k, ones, scale)
    assert np.abs(o - 1.0).max() < 1e-13


def test_cross_path_consistency():
    """decode over n tokens == last row of prefill over the same n tokens == extend of 1 new
    token over n-1 cached ones."""
    rng = np.random.default_rng(2)
    n, Hq, Hkv, D = 45, 8, 2, 32
    scale = 1 / math.sqrt(D)
    q = _bits(rng.standard_normal((n, Hq, D)))
    k = _bits(rng.standard_normal((n, Hkv, D)))
    v = _bits(rng.standard_normal((n, Hkv, D)))
    o_p, l_p = oracle.prefill(q, k, v, np.array([0, n], np.int32), scale)
    # lay the n tokens into a paged pool
    bs, nblk = 16, (n + 15) // 16
    tab = np.array([[5, 0, 3]], np.int32)
    kc = np.zeros((6, bs, Hkv, D), np.uint16); vc = np.zeros_like(kc)
    pos = np.arange(n)
    kc[tab[0, pos // bs], pos % bs] = k
    vc[tab[0, pos // bs], pos % bs] = v
    o_d, l_d = oracle.paged_decode(q[n - 1:], kc, vc, tab, np.array([n], np.int32), scale)
    o_e, l_e = oracle.extend(q[n - 1:], k[n - 1:], v[n - 1:], np.array([0, 1], np.int32), scale,
                             seq_lens=np.array([n], np.int32), k_cache=kc, v_cache=vc,
                             block_tables=tab)
    assert np.abs(o_d[0] - o_p[n - 1]).max() < TOL and np.abs(l_d[0] - l_p[n - 1]).max() < TOL
    assert np.abs(o_e[0] - o_p[n - 1]).max() < TOL and np.abs(l_e[0] - l_p[n - 1]).max() < TOL


def test_numpy_brute_force_tiny():
    """An independent pure-numpy loop over a tiny extend batch."""
    b = gen.extend_batch([3, 2], [5, 0], Hq=4, Hkv=2, D=8, seed=21)
    scale = 1 / math.sqrt(8)
    out, lse = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                             b.cu_q.numpy(), scale, seq_lens=b.seq_lens.numpy(),
                             k_cache=gen.bf16_bits(b.k_cache), v_cache=gen.bf16_bits(b.v_cache),
                             block_tables=b.block_tables.numpy(), nthreads=1)
    qf = f64(gen.bf16_bits(b.q)).numpy(); kn = f64(gen.bf16_bits(b.k_new)).numpy()
    vn = f64(gen.bf16_bits(b.v_new)).numpy()
    kc = f64(gen.bf16_bits(b.k_cache)).numpy(); vc = f64(gen.bf16_bits(b.v_cache)).numpy()
    bt = b.block_tables.numpy(); cu = b.cu_q.numpy()
    for r in range(2):
        C = b.seq_lens_list[r] - b.q_lens[r]
        for i in range(b.q_lens[r]):
            t = cu[r] + i
            for h in range(4):
                kh = h // 2
                keys, vals = [], []
                for j in range(C):
                    keys.append(kc[bt[r, j // 16], j % 16, kh]); vals.append(vc[bt[r, j // 16], j % 16, kh])
                for j in range(i + 1):
                    keys.append(kn[cu[r] + j, kh]); vals.append(vn[cu[r] + j, kh])
                s = [scale * sum(qf[t, h, d] * kk[d] for d in range(8)) for kk in keys]
                m = max(s)
                p = [math.exp(x - m) for x in s]
                z = sum(p)
                o = [sum(p[j] * vals[j][d] for j in range(len(p))) / z for d in range(8)]
                assert max(abs(o[d] - out[t, h, d]) for d in range(8)) < 1e-12
                assert abs(m + math.log(z) - lse[t, h]) < 1e-12


def test_empty_key_set_gives_zero_and_minus_inf():
    q = np.zeros((1, 2, 8), np.uint16)
    kc = np.zeros((2, 16, 1, 8), np.uint16)
    out, lse = oracle.paged_decode(q, kc, kc, np.zeros((1, 1), np.int32), np.array([0], np.int32), 1.0)
    assert np.array_equal(out[0], np.zeros((2, 8))) and np.all(lse[0] == -np.inf)


def test_planted_mistake_is_caught():
    """A transposed-GQA oracle (h % Hkv instead of h // G), planted here on the CPU, must fail
    the SDPA pin: the pins are sharp enough to see index mistakes."""
    b = gen.decode_batch(2, 5, 40, Hq=8, Hkv=2, D=16, seed=4)
    scale = 0.25
    out, _ = oracle.paged_decode(gen.bf16_bits(b.q), gen.bf16_bits(b.k_cache),
                                 gen.bf16_bits(b.v_cache), b.block_tables.numpy(),
                                 b.seq_lens.numpy(), scale)
    qf = f64(gen.bf16_bits(b.q))
    wrong = gen.bf16_bits(b.q).copy()
    G = 4
    for h in range(8):   # feed query head h where the oracle expects h' with the other mapping
        wrong[:, h] = gen.bf16_bits(b.q)[:, (h % 2) * G + h // 2]
    out_w, _ = oracle.paged_decode(wrong, gen.bf16_bits(b.k_cache), gen.bf16_bits(b.v_cache),
                                   b.block_tables.numpy(), b.seq_lens.numpy(), scale)
    k, v = dense_kv(b, 0, b.seq_lens_list[0])
    exp = sdpa(qf[0:1], k, v, scale)[0]
    assert np.abs(out[0] - exp).max() < TOL
    assert np.abs(out_w[0] - exp).max() > 1e-3


def test_planted_off_by_one_context_is_caught():
    """An extend oracle that reads one cached key too many (context length off by one), planted
    here on the CPU by passing seq_len + 1, must fail the masked-SDPA pin."""
    b = _extend_case(seed=13)
    scale = 1 / math.sqrt(b.D)
    args = dict(k_cache=gen.bf16_bits(b.k_cache), v_cache=gen.bf16_bits(b.v_cache),
                block_tables=b.block_tables.numpy())
    common = (gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new), b.cu_q.numpy(), scale)
    r = 2   # 23 new tokens over 50 cached: the table has room for the extra key
    out, _ = oracle.extend(*common, seq_lens=b.seq_lens.numpy(), **args)
    out_w, _ = oracle.extend(*common, seq_lens=b.seq_lens.numpy() + 1, **args)
    qf, kf, vf = (f64(gen.bf16_bits(t)) for t in (b.q, b.k_new, b.v_new))
    cu = b.cu_q.numpy()
    s, e = cu[r], cu[r + 1]
    C = b.seq_lens_list[r] - b.q_lens[r]
    kc, vc = dense_kv(b, r, C)
    exp = sdpa(qf[s:e], torch.cat([kc, kf[s:e]]), torch.cat([vc, vf[s:e]]), scale, causal_offset=C)
    assert np.abs(out[s:e] - exp).max() < TOL
    assert np.abs(out_w[s:e] - exp).max() > 1e-3


# ---- FP8 (E4M3) KV cache -------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_float8():
    """All 256 codes against torch's float8_e4m3fn (an independent implementation of the OCP
    E4M3 format): equal values, NaN at the same codes, largest finite 448, smallest subnormal
    2^-9."""
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9


def test_e4m3_encode_rounds_to_nearest_even_and_saturates():
    """Round to nearest, ties to even, against torch's conversion on values below 464 (torch
    turns larger ones into NaN); above that, the saturating definition: +-448."""
    rng = np.random.default_rng(31)
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))          # the 127 finite magnitudes
    mids = (grid[1:] + grid[:-1]) / 2                                   # exact ties
    x = np.concatenate([rng.normal(0, 8, 20000), rng.uniform(-463, 463, 20000), mids, -mids,
                        grid, rng.uniform(0, 2 ** -6, 2000)]).astype(np.float32)
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    big = np.array([464, 470, 1e6, 3.4e38, -500, -1e30], np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E] * 4 + [0xFE] * 2


def test_fp8_write_matches_numpy_quantise_and_scatter():
    """code = E4M3(float(x) * float(1 / scale)) scattered through the slot mapping."""
    layers = gen.write_pack_layers(1, 100, Hkv=2, D=16, seed=33)
    L = layers[0]
    nb = L.k_cache.shape[0]
    kc = np.zeros((nb, 16, 2, 16), np.uint8)
    vc = np.zeros_like(kc)
    ks, vs = 0.037, 0.011
    assert oracle.kv_cache_write_fp8(gen.bf16_bits(L.key), gen.bf16_bits(L.value), L.slot_mapping.numpy(),
                                     kc, vc, ks, vs) == 0
    def quant(t, s):
        inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(s, dtype=torch.float32)
        return (t.float() * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    slots = L.slot_mapping.numpy()
    ek, ev = np.zeros_like(kc), np.zeros_like(vc)
    ek.reshape(-1, 2, 16)[slots] = quant(L.key, ks)
    ev.reshape(-1, 2, 16)[slots] = quant(L.value, vs)
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_fp8_decode_matches_torch_sdpa_on_dequantised_cache():
    """Decode over an E4M3 cache == fp64 SDPA over the dequantised keys/values (codes through
    torch's float8 decoding, times the scales)."""
    b = gen.decode_batch(3, 5, 60, Hq=8, Hkv=2, D=16, seed=34)
    rng = np.random.default_rng(35)
    kc = rng.integers(0, 256, size=tuple(b.k_cache.shape), dtype=np.uint8)
    vc = rng.integers(0, 256, size=tuple(b.v_cache.shape), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x11                                      # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    ks, vs, scale = 0.02, 0.5, 0.25
    out, lse = oracle.paged_decode_fp8(gen.bf16_bits(b.q), kc, vc, b.block_tables.numpy(),
                                       b.seq_lens.numpy(), scale, ks, vs)
    deq = lambda c, s: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64) * s
    kd, vd = deq(kc, ks).numpy(), deq(vc, vs).numpy()
    qf = f64(gen.bf16_bits(b.q))
    for r in range(b.R):
        n = b.seq_lens_list[r]
        pos = np.arange(n)
        blk = b.block_tables.numpy()[r, pos // 16]
        k = torch.from_numpy(kd[blk, pos % 16])
        v = torch.from_numpy(vd[blk, pos % 16])
        exp = sdpa(qf[r:r + 1], k, v, scale)[0]
        assert np.abs(out[r] - exp).max() < TOL
        assert np.abs(lse[r] - lse_ref(qf[r:r + 1], k, scale)[0]).max() < TOL


def test_fp8_extend_matches_torch_sdpa_on_dequantised_context():
    """Extend over an E4M3 cache == fp64 SDPA (causal over the new tokens) with the cached keys
    and values dequantised (codes through torch's float8 decoding, times the scales) and the
    new tokens' bf16 rows as given."""
    b = _extend_case()
    rng = np.random.default_rng(36)
    kc = rng.integers(0, 256, size=tuple(b.k_cache.shape), dtype=np.uint8)
    vc = rng.integers(0, 256, size=tuple(b.v_cache.shape), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x31                                      # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x42
    ks, vs, scale = 0.015, 0.3, 1 / math.sqrt(b.D)
    out, lse = oracle.extend_fp8(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                                 b.cu_q.numpy(), b.seq_lens.numpy(), kc, vc, b.block_tables.numpy(), scale, ks, vs)
    deq = lambda c, s: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64) * s
    kd, vd = deq(kc, ks).numpy(), deq(vc, vs).numpy()
    qf, kf, vf = (f64(gen.bf16_bits(t)) for t in (b.q, b.k_new, b.v_new))
    cu = b.cu_q.numpy()
    for r in range(b.R):
        s, e = cu[r], cu[r + 1]
        C = b.seq_lens_list[r] - b.q_lens[r]
        pos = np.arange(C)
        blk = b.block_tables.numpy()[r, pos // 16]
        k = torch.cat([torch.from_numpy(kd[blk, pos % 16]), kf[s:e]])
        v = torch.cat([torch.from_numpy(vd[blk, pos % 16]), vf[s:e]])
        exp = sdpa(qf[s:e], k, v, scale, causal_offset=C)
        assert np.abs(out[s:e] - exp).max() < TOL
        assert np.abs(lse[s:e] - lse_ref(qf[s:e], k, scale, C)).max() < TOL


def test_fp8_extend_with_power_of_two_scales_is_the_bf16_extend():
    """With scales that are powers of two the dequantised values are exact bf16 numbers: the
    FP8 extend then equals the bf16 extend over a cache holding those numbers."""
    b = _extend_case()
    rng = np.random.default_rng(37)
    kc = rng.integers(0, 256, size=tuple(b.k_cache.shape), dtype=np.uint8)
    vc = rng.integers(0, 256, size=tuple(b.v_cache.shape), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x25
    vc[(vc & 0x7F) == 0x7F] = 0x26
    ks, vs, scale = 2.0 ** -4, 2.0 ** -1, 0.2
    out, lse = oracle.extend_fp8(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new),
                                 b.cu_q.numpy(), b.seq_lens.numpy(), kc, vc, b.block_tables.numpy(), scale, ks, vs)
    to_bf16 = lambda c, s: gen.bf16_bits((torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float32) * s)
                                         .to(torch.bfloat16))
    ref, ref_lse = oracle.extend(gen.bf16_bits(b.q), gen.bf16_bits(b.k_new), gen.bf16_bits(b.v_new), b.cu_q.numpy(),
                                 scale, seq_lens=b.seq_lens.numpy(), k_cache=to_bf16(kc, ks), v_cache=to_bf16(vc, vs),
                                 block_tables=b.block_tables.numpy())
    assert np.abs(out - ref).max() < 1e-12 and np.abs(lse - ref_lse).max() < 1e-12


# ---- MLA absorbed decode ----------------------------------------------------------------------------

def test_mla_decode_matches_torch_sdpa_with_latent_values():
    """Absorbed MLA decode == SDPA in fp64 with keys = the latent rows (all Dk dims) and values =
    their first Dv dims, every query head against the one latent head."""
    Dk, Dv, Hq = 40, 32, 8
    b = gen.decode_batch(3, 5, 70, Hq=Hq, Hkv=1, D=Dk, seed=80)
    scale = 0.11
    out, lse = oracle.mla_decode(gen.bf16_bits(b.q), gen.bf16_bits(b.k_cache), b.block_tables.numpy(),
                                 b.seq_lens.numpy(), scale, Dv)
    qf = f64(gen.bf16_bits(b.q))
    for r in range(b.R):
        k, _ = dense_kv(b, r, b.seq_lens_list[r])          # [n, 1, Dk] latent rows
        v = k[:, :, :Dv].contiguous()
        exp = sdpa(qf[r:r + 1], k, v, scale)[0]
        assert np.abs(out[r] - exp).max() < TOL
        assert np.abs(lse[r] - lse_ref(qf[r:r + 1], k, scale)[0]).max() < TOL


def test_mla_decode_with_full_values_is_the_one_kv_head_decode():
    """With Dv = Dk the latent is both key and value: the generic decode with one KV head
    (whose V cache is the same latent) gives the same result."""
    D = 24
    b = gen.decode_batch(4, 1, 90, Hq=4, Hkv=1, D=D, seed=81)
    lat = gen.bf16_bits(b.k_cache)
    out, lse = oracle.mla_decode(gen.bf16_bits(b.q), lat, b.block_tables.numpy(), b.seq_lens.numpy(), 0.2, D)
    ref, ref_lse = oracle.paged_decode(gen.bf16_bits(b.q), lat, lat, b.block_tables.numpy(), b.seq_lens.numpy(), 0.2)
    assert np.abs(out - ref).max() < 1e-12 and np.abs(lse - ref_lse).max() < 1e-12
