"""pkv_paged_decode_attn_noalloc: the decode entry point for callers that cannot allocate
device memory (an engine whose memory all belongs to its KV-cache pool, a plug-in whose host
program owns every allocation). It must give what pkv_paged_decode_attn gives with a
caller-allocated workspace, call after call, while using only the library's own fixed scratch.

Collected last on purpose (file name), so a run that stops at the first failure has run every
other test before this one; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from pkv_workloads import gen

from helpers import LSE_ABS, MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, pkv, b, out, lse):
    """Call the C ABI directly (ctypes), passing only inputs and outputs."""
    cache = pkv.make_cache(b.k_cache, b.v_cache)
    reqs = pkv.Reqs(max_reqs=b.R, batch_reqs=b.R).c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_decode_attn_noalloc(
        ctypes.c_void_p(b.q.data_ptr()), cache, ctypes.c_void_p(b.block_tables.data_ptr()),
        b.block_tables.shape[1], ctypes.c_void_p(b.seq_lens.data_ptr()),
        ctypes.c_void_p(b.cu_q.data_ptr()), reqs, b.Hq, max(b.seq_lens_list),
        1.0 / np.sqrt(b.D), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    import paged_kv_attention_reshape_gb300 as pkv
    lib = pkv.load()
    # two different batches back to back: the second call must not see the first one's
    # leftovers in the shared scratch
    cases = [dict(B=8, ctx_lo=1000, ctx_hi=4000, seed=101), dict(B=3, ctx_lo=5, ctx_hi=9000, seed=102)]
    for c in cases:
        b = gen.decode_batch(c["B"], c["ctx_lo"], c["ctx_hi"], Hq=32, Hkv=4, D=128, seed=c["seed"]).to("cuda")
        maxs = max(b.seq_lens_list)
        need = pkv.paged_decode_workspace_size(b.R, b.Hq, b.Hkv, b.D, maxs)
        assert 0 < need <= pkv._lib.NOALLOC_SCRATCH_BYTES   # the split scratch is really used
        ref_out, ref_lse = pkv.paged_decode_attn(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                                 maxs, cu_q=b.cu_q, scale=1.0 / np.sqrt(b.D))
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full((b.T, b.Hq), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc_call(lib, pkv, b, out, lse) == 0
        torch.cuda.synchronize()
        assert pkv.device_errors() == 0
        err = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS
