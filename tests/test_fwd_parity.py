"""Forward parity: the CUDA path against the float64 oracle on the same seeded bits."""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, f64, host, report

pytestmark = pytest.mark.gpu


def run_dense(seed, b, sq, sk, hq, hkv, d, dtype, scale=None, causal=False, window=(-1, -1),
              softcap=0.0):
    from exact_attention_41_gb300 import libattn

    case = syn.dense_case(seed, b, sq, sk, hq, hkv, d, dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = libattn.fwd(dev(case["q"], dtype), dev(case["k"], dtype), dev(case["v"], dtype),
                         scale=scale, causal=causal, window=window, softcap=softcap)
    ro, rl = ref.forward(f64(case["q"], dtype), f64(case["k"], dtype), f64(case["v"], dtype),
                         scale, causal, window[0], window[1], softcap)
    return host(o), host(lse), ro, rl


def test_tiny_fp16():
    """b=1, s=64, h=4, d=64, scale 1/8, non-causal (Inference Cookbook FAQ Q2 shape)."""
    o, lse, ro, rl = run_dense(0, 1, 64, 64, 4, 4, 64, syn.F16, scale=1 / 8)
    assert o.shape == (1, 64, 4, 64)
    assert_close(o, ro, syn.F16, "out")
    assert_lse(lse, rl)


@pytest.mark.parametrize("seed,h,d", [(1, 32, 64), (2, 16, 128), (3, 8, 256)])
def test_head_dim_sweep_fp16(seed, h, d):
    """b=2, s=1024, non-causal; the three head dims of the sm_86 verification note."""
    o, lse, ro, rl = run_dense(seed, 2, 1024, 1024, h, h, d, syn.F16)
    assert_close(o, ro, syn.F16, "out")
    assert_lse(lse, rl)


@pytest.mark.parametrize("sq,sk", [(128, 1024), (1024, 128)])
@pytest.mark.parametrize("h,d", [(32, 64), (16, 128), (8, 256)])
def test_bottom_right_causal_fp16(sq, sk, h, d):
    o, lse, ro, rl = run_dense(4 if sq < sk else 5, 2, sq, sk, h, h, d, syn.F16, causal=True)
    assert_close(o, ro, syn.F16, "out")
    assert_lse(lse, rl)
    if sq > sk:  # the first sq - sk query rows see no key: O = 0, LSE = -inf
        assert np.all(o[:, : sq - sk] == 0) and np.isneginf(lse[:, :, : sq - sk]).all()


@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
@pytest.mark.parametrize("kw", [
    dict(causal=True),
    dict(window=(37, 0)),
    dict(window=(5, 9)),
    dict(window=(-1, 3)),
    dict(causal=True, softcap=5.0),
    dict(softcap=2.5, window=(64, 64)),
])
@pytest.mark.parametrize("shape", [(2, 197, 197, 8, 2, 128), (1, 300, 77, 4, 4, 64),
                                   (1, 77, 300, 6, 3, 256), (3, 1, 513, 4, 1, 128),
                                   (1, 1100, 1300, 4, 2, 128)])
def test_masks_softcap_gqa_ragged(dtype, kw, shape):
    """d = 128 takes two layouts: one 128-row tile with 64-key steps (two
    CTAs per SM) for windows and sequences of at most 1024 keys, two tiles
    with 128-key steps otherwise; the 1300-key shape keeps the unwindowed
    cases on the second."""
    b, sq, sk, hq, hkv, d = shape
    o, lse, ro, rl = run_dense(11, b, sq, sk, hq, hkv, d, dtype, **kw)
    assert_close(o, ro, dtype, "out")
    assert_lse(lse, rl)


@pytest.mark.parametrize("kw", [dict(causal=True, window=(1100, 0), softcap=20.0),
                                dict(window=(700, 700))])
def test_wide_window_two_tile_layout(kw):
    """Windows wider than 1024 keys at d = 128 run on the two-tile layout:
    its masked tiles at both window edges, with and without softcap."""
    o, lse, ro, rl = run_dense(13, 1, 2000, 2000, 4, 2, 128, syn.BF16, **kw)
    assert_close(o, ro, syn.BF16, "out")
    assert_lse(lse, rl)


def test_empty_keys_give_zero_and_neg_inf():
    o, lse, ro, rl = run_dense(12, 1, 5, 0, 2, 2, 64, syn.BF16)
    assert np.all(o == 0) and np.isneginf(lse).all()


def test_training_shape_sampled_rows():
    """bf16 b=4, s=8192, hq=32, hkv=8, d=128, causal: 256 seeded (b, h, row) slices."""
    from exact_attention_41_gb300 import libattn

    b, s, hq, hkv, d = 4, 8192, 32, 8, 128
    case = syn.dense_case(6, b, s, s, hq, hkv, d, syn.BF16)
    o, lse = libattn.fwd(dev(case["q"], syn.BF16), dev(case["k"], syn.BF16),
                         dev(case["v"], syn.BF16), causal=True)
    rng = np.random.default_rng(600)
    samples = [(int(rng.integers(b)), int(rng.integers(hq)), int(rng.integers(s)))
               for _ in range(256)]
    samples += [(0, 0, 0), (b - 1, hq - 1, s - 1), (1, 5, 127), (2, 9, 128)]
    import torch

    bi, hi, ri = (torch.as_tensor(x, device="cuda") for x in zip(*samples))
    q, k, v = (f64(case[x], syn.BF16) for x in ("q", "k", "v"))
    ro, rl = ref.forward_rows(q, k, v, samples, 1 / math.sqrt(d), causal=True)
    report("training fwd O (260 sampled rows)", host(o[bi, ri, hi]), ro, syn.BF16, "oracle")
    assert_close(host(o[bi, ri, hi]), ro, syn.BF16, "out")
    assert_lse(host(lse[bi, hi, ri]), rl)
