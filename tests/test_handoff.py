"""Layer handoff staging (pkv_handoff_*, vLLM blog "moriio-kv-connector", "Write mode": each
layer's KV blocks leave as soon as the layer is written, while the next work computes).

On the CPU: the host-side checks. On the GPU: a ring of staging slots over several layers,
each layer packed on the copy stream beside a prefill attention on the compute stream and
landed in a receiving pool by a consumer stream; every received pool must equal, bit for bit,
the oracle's write -> pack -> unpack of the same layer."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from pkv_workloads import gen

from helpers import bits


def test_handoff_host_checks_without_a_gpu():
    import paged_kv_attention_reshape_gb300 as pkv
    from paged_kv_attention_reshape_gb300 import _lib
    lib = pkv.load()
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    h = P()
    assert lib.pkv_handoff_create(0, fake, ctypes.byref(h)) == 1   # no slots
    assert lib.pkv_handoff_create(2, None, ctypes.byref(h)) == 1   # no copy stream
    assert lib.pkv_handoff_create(2, fake, None) == 1              # no output pointer
    cache = _lib.PkvCache(fake, fake, 10, 16, 2, 128, 16 * 2 * 128)
    assert lib.pkv_handoff_stage(None, 0, cache, fake, 1, fake, fake) == 1
    assert lib.pkv_handoff_ready(None, 0, fake) == 1
    assert lib.pkv_handoff_release(None, 0, fake) == 1
    assert lib.pkv_handoff_destroy(None) == 1


def _expected_received(L, recv_ids, nb):
    """The oracle's write of the layer's prompt, pack of its blocks, unpack into a zeroed pool."""
    kc, vc = bits(L.k_cache).copy(), bits(L.v_cache).copy()
    assert oracle.kv_cache_write(bits(L.key), bits(L.value), L.slot_mapping.numpy(), kc, vc) == 0
    packed, bad = oracle.kv_block_pack(kc, vc, L.block_ids.numpy())
    assert bad == 0
    ek, ev = np.zeros_like(kc), np.zeros_like(vc)
    assert oracle.kv_block_unpack(packed, recv_ids.numpy(), ek, ev) == 0
    return ek, ev


@pytest.mark.gpu
@pytest.mark.parametrize("slots", [1, 2, 8])
def test_handoff_ring_over_layers_bit_exact(slots):
    """Six layers through a ring of `slots` staging buffers: a slot is staged again only after
    the consumer released it, so with one slot every layer waits for the previous landing."""
    import paged_kv_attention_reshape_gb300 as pkv
    pkv.load()
    dev = "cuda"
    T, Hkv, D, Hq, nl = 700, 2, 64, 8, 6
    layers = gen.write_pack_layers(nl, T, Hkv=Hkv, D=D, seed=90 + slots, shuffled_pack=True)
    nb = layers[0].k_cache.shape[0]
    nblk = layers[0].block_ids.numel()
    g = torch.Generator().manual_seed(91 + slots)
    recv_ids = [torch.randperm(nb, generator=g)[:nblk].to(torch.int32) for _ in range(nl)]
    q = gen.randn_bf16((T, Hq, D), g, "cpu").to(dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    gl = [(L.key.to(dev), L.value.to(dev), L.slot_mapping.to(dev), L.block_ids.to(dev),
           L.k_cache.to(dev), L.v_cache.to(dev)) for L in layers]
    ids_dev = [r.to(dev) for r in recv_ids]
    recv = [(torch.zeros_like(k), torch.zeros_like(v)) for (_, _, _, _, k, v) in gl]
    bufs = [torch.empty((2, nblk, 16, Hkv, D), dtype=torch.bfloat16, device=dev) for _ in range(slots)]
    outs = [torch.empty_like(q) for _ in range(nl)]
    torch.cuda.synchronize()

    compute, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    ho = pkv.LayerHandoff(slots)
    for l, (key, val, sm, bid, kc, vc) in enumerate(gl):
        s = l % slots
        pkv.kv_cache_write(key, val, sm, kc, vc, stream=compute)
        ho.stage(s, kc, vc, bid, dst=bufs[s], compute_stream=compute)
        pkv.varlen_prefill_attn(q, key, val, cu, T, out=outs[l], stream=compute)  # runs beside the pack
        ho.ready(s, consumer)
        pkv.kv_block_unpack(bufs[s], ids_dev[l], recv[l][0], recv[l][1], stream=consumer)
        ho.release(s, consumer)
    torch.cuda.synchronize()
    ho.close()
    assert pkv.device_errors(clear=True) == 0
    for l, L in enumerate(layers):
        ek, ev = _expected_received(L, recv_ids[l], nb)
        assert np.array_equal(bits(recv[l][0]), ek), f"layer {l} K"
        assert np.array_equal(bits(recv[l][1]), ev), f"layer {l} V"
