"""FP8 forward (Inference Cookbook FAQ Q20) against the oracle.

Inputs are E4M3 bytes (seeded N(0,1) draws rounded to E4M3) with per-tensor
descale factors; the oracle evaluates the forward of the dequantized values
in float64.  Tolerance: FAQ Q10's FP8 row, |out - ref| <= 1e-2 + 1e-2*|ref|
(the library's P V runs in bf16, so its error is that of the 16-bit path);
LSE within 1e-3 (S is exact products accumulated in fp32).
"""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_lse, host

pytestmark = pytest.mark.gpu


def _dev8(bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda().view(
        torch.float8_e4m3fn)


@pytest.mark.parametrize("b,sq,sk,hq,hkv,kw", [
    (2, 200, 333, 8, 2, dict(causal=True)),
    (1, 16, 1000, 32, 8, dict(causal=True)),                 # short queries: PackGQA
    (2, 130, 130, 4, 4, dict(window=(50, 7), softcap=8.0)),
    (1, 300, 64, 4, 2, dict(causal=True)),                   # sq > sk: empty leading rows
])
def test_fp8_forward_matches_oracle(b, sq, sk, hq, hkv, kw):
    import torch

    from exact_attention_41_gb300 import libattn

    d = 128
    rng = np.random.default_rng(81)
    q8, k8, v8 = (syn.normal_e4m3(rng, sh) for sh in ((b, sq, hq, d), (b, sk, hkv, d), (b, sk, hkv, d)))
    dq, dk, dv = 0.75, 1.25, 0.5
    out, lse = libattn.fwd_fp8(_dev8(q8), _dev8(k8), _dev8(v8), dq, dk, dv, **kw)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    win = kw.get("window", (-1, -1))
    ro, rl = ref.fp8_forward(syn.e4m3_bits_to_f64(q8), syn.e4m3_bits_to_f64(k8),
                             syn.e4m3_bits_to_f64(v8), dq, dk, dv, 1 / math.sqrt(d),
                             kw.get("causal", False), win[0], win[1], kw.get("softcap", 0.0))
    got = host(out)
    err = np.abs(got - ro)
    bound = 1e-2 + 1e-2 * np.abs(ro)
    assert np.isfinite(got).all()
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}, max err {err.max():.3e}"
    assert_lse(host(lse), rl)


def test_fp8_argument_checks():
    import torch

    from exact_attention_41_gb300 import libattn

    z = torch.zeros((1, 8, 2, 128), device="cuda", dtype=torch.uint8).view(torch.float8_e4m3fn)
    with pytest.raises(libattn.AttnError):
        libattn.fwd_fp8(z, z, z, 0.0, 1.0, 1.0)        # descale must be > 0
    z64 = torch.zeros((1, 8, 2, 64), device="cuda", dtype=torch.uint8).view(torch.float8_e4m3fn)
    with pytest.raises(libattn.AttnError):
        libattn.fwd_fp8(z64, z64, z64)                 # d = 128 only
