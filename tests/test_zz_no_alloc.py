"""pkv_paged_decode_attn_noalloc: the decode entry point for callers that cannot allocate
device memory (an engine whose memory all belongs to its KV-cache pool, a plug-in whose host
program owns every allocation). It must give the oracle's result, and what pkv_paged_decode_attn
gives with a caller-allocated workspace, call after call, while using only the library's own
fixed scratch, which every call shares and which keeps the last call's contents.

Collected last on purpose (file name), so a run that stops at the first failure has run every
other test before this one; it also passes on its own in a fresh process."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from pkv_workloads import gen

from helpers import LSE_ABS, MAX_ABS, MEAN_ABS, bits, compare_attention

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, pkv, b, kc, vc, out, lse, ks=1.0, vs=1.0, Hq=None):
    """Call the C ABI directly (ctypes), passing only inputs and outputs."""
    cache = pkv.make_cache(kc, vc, ks, vs)
    reqs = pkv.Reqs(max_reqs=b.R, batch_reqs=b.R).c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_decode_attn_noalloc(
        ctypes.c_void_p(b.q.data_ptr()), cache, ctypes.c_void_p(b.block_tables.data_ptr()),
        b.block_tables.shape[1], ctypes.c_void_p(b.seq_lens.data_ptr()),
        ctypes.c_void_p(b.cu_q.data_ptr()), reqs, Hq or b.Hq, max(b.seq_lens_list),
        1.0 / np.sqrt(b.D), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)


def _codes(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype != torch.uint8 else t.cpu().numpy()


# Consecutive calls at different shapes and cache types, so that each call's partials and merge
# counters land on other offsets of the shared scratch than the previous call's (the scratch
# keeps them). Each batch has sequences long enough to be cut across shares, so the scratch is
# really used.
CASES = [
    dict(B=8, lo=1000, hi=4000, Hq=32, Hkv=4, D=128, fp8=False, seed=101),
    dict(B=3, lo=5, hi=9000, Hq=32, Hkv=4, D=128, fp8=False, seed=102),
    dict(B=6, lo=500, hi=6000, Hq=64, Hkv=8, D=64, fp8=False, seed=103),
    dict(B=9, lo=1000, hi=5000, Hq=64, Hkv=4, D=128, fp8=True, seed=104),
    dict(B=5, lo=2000, hi=12000, Hq=16, Hkv=1, D=128, fp8=False, seed=105),
    dict(B=8, lo=1000, hi=4000, Hq=32, Hkv=4, D=128, fp8=False, seed=101),
]


def test_noalloc_decode_matches_oracle_and_workspace_decode_on_consecutive_calls():
    import paged_kv_attention_reshape_gb300 as pkv
    lib = pkv.load()
    for c in CASES:
        b = gen.decode_batch(c["B"], c["lo"], c["hi"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], seed=c["seed"])
        scale = 1.0 / math.sqrt(c["D"])
        if c["fp8"]:
            ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
            kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
            ref, ref_lse = oracle.paged_decode_fp8(bits(b.q), _codes(kc), _codes(vc), b.block_tables.numpy(),
                                                   b.seq_lens.numpy(), scale, ks, vs, cu_q=b.cu_q.numpy())
        else:
            ks = vs = 1.0
            kc, vc = b.k_cache, b.v_cache
            ref, ref_lse = oracle.paged_decode(bits(b.q), bits(kc), bits(vc), b.block_tables.numpy(),
                                               b.seq_lens.numpy(), scale, cu_q=b.cu_q.numpy())
        g = b.to("cuda")
        kc, vc = kc.to("cuda"), vc.to("cuda")
        maxs = max(b.seq_lens_list)
        need = pkv.paged_decode_workspace_size(b.R, b.Hq, b.Hkv, b.D, maxs)
        assert 0 < need <= pkv._lib.NOALLOC_SCRATCH_BYTES   # the split scratch is really used
        ref_out, ref_lse_ws = pkv.paged_decode_attn(g.q, kc, vc, g.block_tables, g.seq_lens, maxs, cu_q=g.cu_q,
                                                    scale=scale, k_scale=ks, v_scale=vs)
        out = torch.full_like(g.q, float("nan"))
        lse = torch.full((g.T, g.Hq), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_call(lib, pkv, g, kc, vc, out, lse, ks, vs) == 0
        torch.cuda.synchronize()
        assert pkv.device_errors() == 0
        what = f"noalloc {c}"
        compare_attention(out, lse, ref, ref_lse, what=what)
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, what
        assert (lse - ref_lse_ws).abs().max().item() <= LSE_ABS, what


def test_noalloc_rejects_a_scratch_need_beyond_its_array_and_enqueues_nothing():
    import paged_kv_attention_reshape_gb300 as pkv
    lib = pkv.load()
    # 64 query heads over 2 KV heads need more split scratch than the array holds (the size
    # check comes before the shape check)
    b = gen.decode_batch(2, 100, 200, Hq=64, Hkv=2, D=128, seed=7).to("cuda")
    need = pkv.paged_decode_workspace_size(b.R, b.Hq, b.Hkv, b.D, max(b.seq_lens_list))
    assert need > pkv._lib.NOALLOC_SCRATCH_BYTES
    out = torch.full_like(b.q, 7.0)
    lse = torch.full((b.T, b.Hq), 7.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    before = lib.pkv_launch_count(0)
    assert _noalloc_call(lib, pkv, b, b.k_cache, b.v_cache, out, lse) == 3  # PKV_ERR_WORKSPACE
    assert lib.pkv_launch_count(0) == before
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
