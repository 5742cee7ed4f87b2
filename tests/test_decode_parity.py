"""Paged KV-cache decode parity: append, split-KV, combine."""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, dev_i32, f64, host

pytestmark = pytest.mark.gpu


def run_small(seed, b, sq, s_new, hq, hkv, d, max_len, page, dtype, num_splits, paged=True, **kw):
    import torch

    from exact_attention_41_gb300 import libattn

    c = syn.decode_case(seed, b, sq, s_new, hq, hkv, d, max_len, page, dtype)
    table = c["block_table"] if paged else None
    kc_bits, vc_bits = c["k_cache"], c["v_cache"]
    if not paged:  # contiguous cache: (b, capacity, hkv, d), one page per entry
        cap = c["block_table"].shape[1] * page
        kc_bits = kc_bits[c["block_table"]].reshape(b, cap, hkv, d)
        vc_bits = vc_bits[c["block_table"]].reshape(b, cap, hkv, d)
    kc, vc = dev(kc_bits, dtype), dev(vc_bits, dtype)
    seqlens = dev_i32(c["cache_seqlens"])
    kn = dev(c["k_new"], dtype) if s_new else None
    vn = dev(c["v_new"], dtype) if s_new else None
    o, lse = libattn.fwd_kvcache(dev(c["q"], dtype), kc, vc, seqlens, k_new=kn, v_new=vn,
                                 block_table=dev_i32(table) if paged else None,
                                 num_splits=num_splits, **kw)
    torch.cuda.synchronize()
    assert (seqlens.cpu().numpy() == c["cache_seqlens"]).all(), "cache_seqlens must not change"
    win = kw.get("window", (-1, -1))
    ro, rl, rk, rv = ref.kvcache_forward(
        f64(c["q"], dtype), f64(kc_bits, dtype), f64(vc_bits, dtype), c["cache_seqlens"],
        1 / math.sqrt(d), f64(c["k_new"], dtype) if s_new else None,
        f64(c["v_new"], dtype) if s_new else None, table if paged else None,
        page if paged else kc_bits.shape[1], kw.get("causal", False), win[0], win[1],
        kw.get("softcap", 0.0))
    assert_close(host(o), ro, dtype, "out")
    assert_lse(host(lse), rl)
    # the cache after the call: appended rows in place, everything else untouched
    np.testing.assert_array_equal(host(kc), rk)
    np.testing.assert_array_equal(host(vc), rv)


@pytest.mark.parametrize("num_splits", [1, 2, 7, 0])
@pytest.mark.parametrize("sq,s_new", [(1, 0), (1, 1), (4, 4), (3, 0)])
def test_small_paged(num_splits, sq, s_new):
    run_small(41, 5, sq, s_new, 8, 2, 128, 700, 128, syn.BF16, num_splits, causal=True)


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
def test_head_dims_and_dtypes(d, dtype):
    run_small(42, 3, 2, 2, 4, 4, d, 600, 256, dtype, 0, causal=True)


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("num_splits", [1, 3])
@pytest.mark.parametrize("sq,s_new", [(1, 1), (4, 4), (8, 0)])
def test_head_dims_gqa_splits(d, num_splits, sq, s_new):
    """d = 64 and 256 on the tensor-core decode: GQA 4:1, so g * sq = 4, 16
    and 32 query rows per KV head (both padded widths), one and several
    splits, ragged caches over 128-token pages."""
    run_small(45, 3, sq, s_new, 8, 2, d, 700, 128, syn.BF16, num_splits, causal=True)


@pytest.mark.parametrize("kw", [dict(causal=True, window=(100, 0)), dict(softcap=30.0),
                                dict(causal=True, softcap=50.0)])
def test_window_softcap(kw):
    run_small(43, 4, 4, 4, 8, 2, 128, 900, 256, syn.BF16, 3, **kw)


@pytest.mark.parametrize("num_splits", [1, 4])
def test_contiguous_cache(num_splits):
    run_small(44, 3, 1, 1, 8, 2, 128, 500, 128, syn.BF16, num_splits, paged=False, causal=True)


@pytest.mark.parametrize("sq", [1, 4])
def test_workload_sampled_entries(sq):
    """b=64, hq=32, hkv=8, d=128, bf16, cache_seqlens U[1, 32768], 256-token
    pages placed by a seeded permutation (8256 pages), s_new = sq, causal,
    auto num_splits: 3 seeded batch entries plus the longest and shortest checked in full, plus the append."""
    import torch

    from exact_attention_41_gb300 import libattn

    b, hq, hkv, d, page = 64, 32, 8, 128, 256
    seqlens, table, npages = syn.decode_layout(8, b, 32768, page, sq)
    kc = syn.device_normal((npages, page, hkv, d), syn.BF16, 80)
    vc = syn.device_normal((npages, page, hkv, d), syn.BF16, 81)
    rng = np.random.default_rng(82)
    q = syn.normal_bits(rng, (b, sq, hq, d), syn.BF16)
    kn = syn.normal_bits(rng, (b, sq, hkv, d), syn.BF16)
    vn = syn.normal_bits(rng, (b, sq, hkv, d), syn.BF16)
    picks = sorted(set(np.random.default_rng(83).choice(b, 3, replace=False).tolist()
                       + [int(np.argmax(seqlens)), int(np.argmin(seqlens))]))
    # the oracle's inputs: the picked entries' pages, copied before the call
    tsel = torch.as_tensor(table[picks].ravel(), device="cuda", dtype=torch.long)
    kpages, vpages = host(kc[tsel]), host(vc[tsel])
    o, lse = libattn.fwd_kvcache(dev(q, syn.BF16), kc, vc, dev_i32(seqlens), k_new=dev(kn, syn.BF16),
                                 v_new=dev(vn, syn.BF16), block_table=dev_i32(table), causal=True)
    npp = table.shape[1]
    local_table = np.arange(len(picks) * npp).reshape(len(picks), npp)
    ro, rl, rk, rv = ref.kvcache_forward(
        f64(q[picks], syn.BF16), kpages, vpages, seqlens[picks], 1 / math.sqrt(d),
        f64(kn[picks], syn.BF16), f64(vn[picks], syn.BF16), local_table, page, causal=True)
    assert_close(host(o)[picks], ro, syn.BF16, "out")
    assert_lse(host(lse)[picks], rl)
    np.testing.assert_array_equal(host(kc[tsel]), rk)
    np.testing.assert_array_equal(host(vc[tsel]), rv)


def test_bad_page_raises_device_error():
    """A block_table entry outside the pool is caught on the device: the
    error word is raised and nothing is read or written out of bounds."""
    import torch

    from exact_attention_41_gb300 import libattn

    libattn.device_error()  # clear
    c = syn.decode_case(45, 2, 1, 1, 4, 4, 128, 300, 128, syn.BF16)
    table = c["block_table"].copy()
    table[1, 0] = 10_000
    kc, vc = dev(c["k_cache"], syn.BF16), dev(c["v_cache"], syn.BF16)
    libattn.fwd_kvcache(dev(c["q"], syn.BF16), kc, vc, dev_i32(c["cache_seqlens"]),
                        k_new=dev(c["k_new"], syn.BF16), v_new=dev(c["v_new"], syn.BF16),
                        block_table=dev_i32(table), causal=True, num_splits=1)
    torch.cuda.synchronize()
    st, word = libattn.device_error()
    assert st == 6 and word & 1
    assert libattn.device_error() == (0, 0)
