"""Shared pieces of the parity tests: tolerances, comparisons, and oracle runs over a
pkv_workloads Batch."""
import math

import numpy as np
import torch

import oracle
from pkv_workloads import gen

# Attention tolerances against the fp64 oracle (bf16 inputs, fp32 accumulation, bf16 output).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def compare_attention(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref: np.ndarray,
                      ref_lse: np.ndarray, rows=None, what=""):
    """Element-wise comparison over the rows the oracle computed (rows: bool mask [T] or None
    = every row without NaN in ref)."""
    got = out_gpu.float().cpu().numpy()
    got_lse = lse_gpu.float().cpu().numpy()
    if rows is None:
        rows = ~np.isnan(ref_lse).any(axis=1)
    assert rows.any(), f"{what}: nothing to compare"
    r, g = ref[rows], got[rows]
    assert not np.isnan(r).any(), f"{what}: oracle rows incomplete"
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    rl, gl = ref_lse[rows], got_lse[rows]
    inf = np.isneginf(rl)
    assert np.array_equal(inf, np.isneginf(gl)), f"{what}: -inf lse pattern differs"
    lerr = np.abs(gl[~inf] - rl[~inf]) if (~inf).any() else np.zeros(1)
    # relative error per row, reported for visibility (outputs shrink at long contexts)
    scale = np.maximum(np.abs(r).max(axis=-1, keepdims=True), 1e-6)
    rel = (err / scale).max()
    msg = (f"{what}: max_abs {err.max():.3e} mean_abs {err.mean():.3e} lse {lerr.max():.3e} "
           f"max_rel_row {rel:.3e} rows {int(rows.sum())}")
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS and lerr.max() <= LSE_ABS, msg
    return msg


def bits(t):
    return gen.bf16_bits(t)


def oracle_decode(b: gen.Batch, kc, vc, scale, req_ids=None, out=None, lse=None):
    return oracle.paged_decode(bits(b.q), kc, vc, b.block_tables.cpu().numpy(),
                               b.seq_lens.cpu().numpy(), scale, cu_q=b.cu_q.cpu().numpy(),
                               req_ids=req_ids, out=out, lse=lse)


def oracle_extend(b: gen.Batch, kc, vc, scale, req_ids=None, row_mask=None, out=None, lse=None):
    return oracle.extend(bits(b.q), bits(b.k_new), bits(b.v_new), b.cu_q.cpu().numpy(), scale,
                         seq_lens=b.seq_lens.cpu().numpy(), k_cache=kc, v_cache=vc,
                         block_tables=b.block_tables.cpu().numpy(), req_ids=req_ids,
                         row_mask=row_mask, out=out, lse=lse)


def oracle_prefill(b: gen.Batch, scale, req_ids=None, row_mask=None, out=None, lse=None):
    return oracle.extend(bits(b.q), bits(b.k_new), bits(b.v_new), b.cu_q.cpu().numpy(), scale,
                         req_ids=req_ids, row_mask=row_mask, out=out, lse=lse)


def default_scale(D):
    return 1.0 / math.sqrt(D)
