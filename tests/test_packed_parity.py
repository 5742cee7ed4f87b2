"""Packed inputs read in place through token strides: qkv (b, s, 3, h, d)
("flash_attn FlashAttention完整说明" §六.1) and kv (b, sk, 2, hkv, d)
(Inference Cookbook FAQ Q7), forward and backward, against the oracle and
bitwise against the same call on contiguous copies (deterministic mode)."""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, f64, host

pytestmark = pytest.mark.gpu


def _check_grads(dq, dk, dv, c, dtype, d, kw):
    win = kw.get("window", (-1, -1))
    rq, rk, rv = ref.backward(f64(c["q"], dtype), f64(c["k"], dtype), f64(c["v"], dtype),
                              f64(c["dout"], dtype), 1 / math.sqrt(d), kw.get("causal", False),
                              win[0], win[1], kw.get("softcap", 0.0), stored_o=dtype)
    assert_close(host(dq), rq, dtype, "dq")
    assert_close(host(dk), rk, dtype, "dk")
    assert_close(host(dv), rv, dtype, "dv")


@pytest.mark.parametrize("d", [128, 64])
def test_qkvpacked_forward_backward(d):
    import torch

    from exact_attention_41_gb300 import libattn

    dtype, b, s, h = syn.BF16, 2, 200, 4
    c = syn.dense_case(61, b, s, s, h, h, d, dtype, with_dout=True)
    q, k, v, do = (dev(c[n], dtype) for n in ("q", "k", "v", "dout"))
    qkv = torch.stack([q, k, v], dim=2).contiguous()          # (b, s, 3, h, d)
    kw = dict(causal=True)
    out, lse = libattn.fwd_qkvpacked(qkv, **kw)
    dqkv = libattn.bwd_qkvpacked(qkv, out, lse, do, deterministic=True, **kw)
    torch.cuda.synchronize()
    ro, rl = ref.forward(f64(c["q"], dtype), f64(c["k"], dtype), f64(c["v"], dtype),
                         1 / math.sqrt(d), True)
    assert_close(host(out), ro, dtype, "out")
    assert_lse(host(lse), rl)
    _check_grads(dqkv[:, :, 0], dqkv[:, :, 1], dqkv[:, :, 2], c, dtype, d, kw)
    # the same call on contiguous tensors gives the same bits
    out2, lse2 = libattn.fwd(q, k, v, **kw)
    g2 = libattn.bwd(q, k, v, out2, lse2, do, deterministic=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    for i in range(3):
        assert torch.equal(dqkv[:, :, i], g2[i]), f"gradient {i} differs from the contiguous call"


@pytest.mark.parametrize("d", [128, 64])
def test_kvpacked_gqa_cross_attention(d):
    import torch

    from exact_attention_41_gb300 import libattn

    dtype, b, sq, sk, hq, hkv = syn.F16, 2, 96, 330, 8, 2
    c = syn.dense_case(62, b, sq, sk, hq, hkv, d, dtype, with_dout=True)
    q, k, v, do = (dev(c[n], dtype) for n in ("q", "k", "v", "dout"))
    kv = torch.stack([k, v], dim=2).contiguous()              # (b, sk, 2, hkv, d)
    kw = dict(window=(100, 20), softcap=4.0)
    out, lse = libattn.fwd_kvpacked(q, kv, **kw)
    dq = torch.empty_like(q)
    dkv = torch.empty_like(kv)
    libattn.bwd(q, kv[:, :, 0], kv[:, :, 1], out, lse, do, dq=dq, dk=dkv[:, :, 0],
                dv=dkv[:, :, 1], **kw)
    torch.cuda.synchronize()
    ro, rl = ref.forward(f64(c["q"], dtype), f64(c["k"], dtype), f64(c["v"], dtype),
                         1 / math.sqrt(d), False, 100, 20, 4.0)
    assert_close(host(out), ro, dtype, "out")
    assert_lse(host(lse), rl)
    _check_grads(dq, dkv[:, :, 0], dkv[:, :, 1], c, dtype, d, kw)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("sq,sk,hq,hkv,kw", [
    (16, 300, 8, 2, dict(causal=True)),                      # short queries: auto packs
    (5, 5, 16, 2, dict(causal=True)),                        # g = 8: 16 positions per tile
    (130, 257, 16, 1, dict(window=(40, 3), softcap=6.0)),    # g = 16, ragged, forced on
    (300, 200, 8, 2, dict(causal=True)),                     # sq > sk: leading rows empty
])
def test_pack_gqa_matches_oracle_and_unpacked(d, sq, sk, hq, hkv, kw):
    """PackGQA (Inference Cookbook FAQ Q15): g query heads share each tile.
    Forced on, off and automatic give the oracle's result, and the packed and
    unpacked kernels agree bitwise (each row's arithmetic is the same)."""
    import torch

    from exact_attention_41_gb300 import libattn

    dtype, b = syn.BF16, 2
    c = syn.dense_case(63, b, sq, sk, hq, hkv, d, dtype)
    q, k, v = (dev(c[n], dtype) for n in ("q", "k", "v"))
    o1, l1 = libattn.fwd(q, k, v, pack_gqa=True, **kw)
    o0, l0 = libattn.fwd(q, k, v, pack_gqa=False, **kw)
    oa, la = libattn.fwd(q, k, v, **kw)
    torch.cuda.synchronize()
    win = kw.get("window", (-1, -1))
    ro, rl = ref.forward(f64(c["q"], dtype), f64(c["k"], dtype), f64(c["v"], dtype),
                         1 / math.sqrt(d), kw.get("causal", False), win[0], win[1],
                         kw.get("softcap", 0.0))
    for o, l, what in ((o1, l1, "packed"), (o0, l0, "unpacked"), (oa, la, "auto")):
        assert_close(host(o), ro, dtype, f"out ({what})")
        assert_lse(host(l), rl, f"lse ({what})")
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_pack_gqa_varlen_short_sequences():
    """Varlen with every sequence <= 128 queries packs automatically."""
    import torch

    from exact_attention_41_gb300 import libattn

    dtype, hq, hkv, d = syn.F16, 8, 2, 128
    lens = np.array([1, 37, 128, 64, 100])
    cu = syn.cu_seqlens(lens)
    c = syn.varlen_case(64, lens, lens, hq, hkv, d, dtype)
    q, k, v = (dev(c[n], dtype) for n in ("q", "k", "v"))
    cu_d = torch.from_numpy(cu).cuda()
    o, lse = libattn.fwd_varlen(q, k, v, cu_d, cu_d, int(lens.max()), int(lens.max()), causal=True)
    torch.cuda.synchronize()
    ro, rl = ref.varlen_forward(f64(c["q"], dtype), f64(c["k"], dtype), f64(c["v"], dtype), cu, cu,
                                1 / math.sqrt(d), True)
    assert_close(host(o), ro, dtype, "varlen out")
    assert_lse(host(lse), rl)
