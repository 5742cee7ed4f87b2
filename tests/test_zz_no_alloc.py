"""attn_fwd_kvcache_noalloc: the decode entry point for callers that cannot
allocate device memory (for example code running under CUDA graph capture,
or a plugin whose device memory belongs to someone else's pool).  Its split
scratch is a fixed array inside the library; it must give the results of
attn_fwd_kvcache, call after call.  Collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from tests.helpers import TOL, dev, dev_i32, host

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    import torch

    from exact_attention_41_gb300 import libattn

    lib = libattn.lib()
    b, sq, s_new, hq, hkv, d, page = 6, 4, 4, 16, 4, 128, 256
    c = syn.decode_case(91, b, sq, s_new, hq, hkv, d, 3000, page, syn.BF16)
    npages, npp = c["k_cache"].shape[0], c["block_table"].shape[1]
    q = dev(c["q"], syn.BF16)
    kn, vn = dev(c["k_new"], syn.BF16), dev(c["v_new"], syn.BF16)
    seqlens, table = dev_i32(c["cache_seqlens"]), dev_i32(c["block_table"])
    splits = 5
    assert lib.attn_kvcache_workspace_size(b, sq, hq, hkv, d, npp * page, splits) > 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    scale = 1 / math.sqrt(d)

    # the existing entry point, with a caller-provided workspace
    kc, vc = dev(c["k_cache"], syn.BF16), dev(c["v_cache"], syn.BF16)
    ref_out = torch.empty_like(q)
    ref_lse = torch.empty((b, hq, sq), device="cuda", dtype=torch.float32)
    ws = libattn.kvcache_workspace(q, kc, page, npp, splits)
    st = lib.attn_fwd_kvcache(_p(q), _p(kc), _p(vc), _p(kn), _p(vn), _p(seqlens), _p(table),
                              npages, page, npp, _p(ref_out), _p(ref_lse), 1, b, sq, s_new, hq,
                              hkv, d, scale, 1, -1, -1, 0.0, splits, _p(ws), ws.numel(), stream)
    assert st == 0
    torch.cuda.synchronize()
    atol, rtol = TOL[syn.BF16]
    for call in range(2):
        kc2, vc2 = dev(c["k_cache"], syn.BF16), dev(c["v_cache"], syn.BF16)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((b, hq, sq), float("nan"), device="cuda", dtype=torch.float32)
        st = lib.attn_fwd_kvcache_noalloc(_p(q), _p(kc2), _p(vc2), _p(kn), _p(vn), _p(seqlens),
                                          _p(table), npages, page, npp, _p(out), _p(lse), 1, b,
                                          sq, s_new, hq, hkv, d, scale, 1, -1, -1, 0.0, splits,
                                          stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got, want = host(out), host(ref_out)
        assert np.all(np.abs(got - want) <= atol + rtol * np.abs(want)), f"call {call}: out"
        np.testing.assert_allclose(host(lse), host(ref_lse), atol=1e-3, rtol=0)
        assert torch.equal(kc2, kc) and torch.equal(vc2, vc), f"call {call}: cache append"
    assert libattn.device_error() == (0, 0)


def test_noalloc_rejects_oversized_scratch():
    import torch

    from exact_attention_41_gb300 import libattn

    lib = libattn.lib()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check comes first
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # 64 splits x 64 x 4 x 32 x 128 fp32 partials = 128 MiB > the 32 MiB array
    st = lib.attn_fwd_kvcache_noalloc(fake, fake, fake, fake, fake, fake, fake, 8256, 256, 129,
                                      fake, fake, 1, 64, 4, 4, 32, 8, 128, 0.08, 1, -1, -1, 0.0,
                                      64, stream)
    assert st == 3
