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
