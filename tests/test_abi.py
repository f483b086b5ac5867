"""CPU checks of the C ABI: the library loads, exports exactly what include/pkv.h declares, the
binding declares the same calls, and host-side argument checks answer without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import paged_kv_attention_reshape_gb300 as pkv
    return pkv.load()


def test_header_declares_the_six_calls():
    names = header_functions()
    for call in ["kv_cache_write", "batch_classify_reorder", "paged_decode_attn", "extend_attn",
                 "varlen_prefill_attn", "kv_block_pack"]:
        assert f"pkv_{call}" in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_attention_reshape_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (pkv_\w+)", out))
    declared = set(header_functions())
    assert declared <= exported, declared - exported
    assert {n for n, _, _ in _lib.SIGNATURES} == declared
    for name in declared:
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for s in range(6):
        assert lib.pkv_status_string(s)


def test_host_checks_reject_bad_arguments_without_a_gpu(lib):
    from paged_kv_attention_reshape_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its host checks first
    cache = _lib.PkvCache(fake, fake, 10, 16, 2, 128, 16 * 2 * 128)
    # negative token count
    assert lib.pkv_kv_cache_write(fake, fake, fake, -1, cache, None) == 1
    # zero tokens is a no-op
    assert lib.pkv_kv_cache_write(None, None, None, 0, cache, None) == 0
    # misaligned cache pointer
    bad = _lib.PkvCache(P((1 << 20) + 2), fake, 10, 16, 2, 128, 16 * 2 * 128)
    assert lib.pkv_kv_block_pack(bad, fake, 3, fake, None) == 1
    # block stride smaller than a block
    bad = _lib.PkvCache(fake, fake, 10, 16, 2, 128, 100)
    assert lib.pkv_kv_block_pack(bad, fake, 3, fake, None) == 1
    # unsupported head_dim / group size / block size for the attention calls
    reqs = _lib.PkvReqs(None, None, 0, 4, 4)
    c96 = _lib.PkvCache(fake, fake, 10, 16, 2, 96, 16 * 2 * 96)
    assert lib.pkv_paged_decode_attn(fake, c96, fake, 4, fake, None, reqs, 4, 100, 1.0, fake, None,
                                     None, 0, None) == 2
    assert lib.pkv_paged_decode_attn(fake, cache, fake, 4, fake, None, reqs, 6, 100, 1.0, fake, None,
                                     None, 0, None) == 2
    c32 = _lib.PkvCache(fake, fake, 10, 32, 2, 128, 32 * 2 * 128)
    assert lib.pkv_extend_attn(fake, fake, fake, 8, fake, fake, c32, fake, 4, reqs, 4, 8, 100, 0,
                               1.0, fake, None, None, 0, None) == 2
    assert lib.pkv_varlen_prefill_attn(fake, fake, fake, 8, fake, reqs, 64, 2, 128, 8, 1.0, fake,
                                       None, None) == 2
    # unpack: misaligned source, negative count, empty
    assert lib.pkv_kv_block_unpack(P((1 << 20) + 4), fake, 3, cache, None) == 1
    assert lib.pkv_kv_block_unpack(fake, fake, -1, cache, None) == 1
    assert lib.pkv_kv_block_unpack(None, None, 0, cache, None) == 0
    # self-test wait limits outside 1 us .. 2 s
    assert lib.pkv_selftest_bounded_wait(10, None) == 1
    assert lib.pkv_selftest_bounded_wait(3_000_000_000, None) == 1
    # token map without reordered starts
    assert lib.pkv_batch_classify_reorder(fake, fake, 4, 1, fake, fake, None, fake, 10, None) == 1
    # identity set larger than the batch
    big = _lib.PkvReqs(None, None, 0, 5, 4)
    assert lib.pkv_varlen_prefill_attn(fake, fake, fake, 8, fake, big, 4, 2, 128, 8, 1.0, fake,
                                       None, None) == 1
    # empty sets are no-ops
    empty = _lib.PkvReqs(None, None, 0, 0, 4)
    assert lib.pkv_varlen_prefill_attn(fake, fake, fake, 8, fake, empty, 4, 2, 128, 8, 1.0, fake,
                                       None, None) == 0
    # the softmax scale must be positive and finite (checked before the empty-set shortcut)
    for bad_scale in (0.0, -0.125, float("inf"), float("nan")):
        assert lib.pkv_varlen_prefill_attn(fake, fake, fake, 8, fake, empty, 4, 2, 128, 8, bad_scale, fake,
                                           None, None) == 1
        assert lib.pkv_extend_attn(fake, fake, fake, 8, fake, fake, cache, fake, 4, empty, 4, 8, 100, 0,
                                   bad_scale, fake, None, None, 0, None) == 1
        assert lib.pkv_paged_decode_attn(fake, cache, fake, 4, fake, None, empty, 4, 100, bad_scale, fake, None,
                                         None, 0, None) == 1


def test_decode_workspace_query_is_host_only(lib):
    # partials for two cut units per CTA plus the set's block prefix: a few MB, independent of
    # the batch; invalid head counts give 0
    n = lib.pkv_paged_decode_workspace_size(256, 64, 4, 128, 3000)
    assert 0 < n <= 32 << 20
    assert lib.pkv_paged_decode_workspace_size(4, 8, 3, 64, 200) == 0


def test_mla_host_checks_without_a_gpu(lib):
    from paged_kv_attention_reshape_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    reqs = _lib.PkvReqs(None, None, 0, 4, 4)
    lat = _lib.PkvCache(fake, None, 10, 16, 1, 576, 16 * 576)  # v may be NULL: the rows are shared
    n = lib.pkv_mla_decode_workspace_size(128, 16, 11000)
    assert 0 < n <= 64 << 20
    assert lib.pkv_mla_decode_workspace_size(128, 24, 11000) == 0
    assert lib.pkv_mla_decode_workspace_size(128, 144, 11000) == 0
    ws = P(1 << 21)
    args = lambda c, hq, vd: (fake, c, fake, 4, fake, None, reqs, hq, 100, 0.07, vd, fake, None, ws, n, None)
    assert lib.pkv_mla_decode_attn(*args(lat, 8, 512)) == 2             # heads not a multiple of 16
    assert lib.pkv_mla_decode_attn(*args(lat, 16, 256)) == 2            # value width other than 512
    assert lib.pkv_mla_decode_attn(*args(_lib.PkvCache(fake, None, 10, 16, 2, 576, 16 * 2 * 576), 16, 512)) == 2
    assert lib.pkv_mla_decode_attn(*args(_lib.PkvCache(fake, None, 10, 16, 1, 512, 16 * 512), 16, 512)) == 2
    assert lib.pkv_mla_decode_attn(*args(_lib.PkvCache(fake, None, 10, 32, 1, 576, 32 * 576), 16, 512)) == 2
    fp8 = _lib.PkvCache(fake, None, 10, 16, 1, 576, 16 * 576, _lib.KV_FP8_E4M3, 1.0, 1.0)
    assert lib.pkv_mla_decode_attn(*args(fp8, 16, 512)) == 2
    # too small a workspace
    small = (fake, lat, fake, 4, fake, None, reqs, 16, 100, 0.07, 512, fake, None, ws, n - 16, None)
    assert lib.pkv_mla_decode_attn(*small) == 3
    # an empty set is a no-op
    empty = _lib.PkvReqs(None, None, 0, 0, 4)
    assert lib.pkv_mla_decode_attn(fake, lat, fake, 4, fake, None, empty, 16, 100, 0.07, 512, fake, None,
                                   None, 0, None) == 0


def test_product_path_has_no_fallback():
    """The binding only calls libpkv.so: it never imports the oracle or torch compute ops."""
    src = open(os.path.join(ROOT, "paged_kv_attention_reshape_gb300", "binding.py")).read()
    assert "oracle" not in src.replace("no other implementation", "")
    for banned in ["torch.nn.functional", "torch.matmul", "torch.softmax", "scaled_dot_product", "triton"]:
        assert banned not in src
