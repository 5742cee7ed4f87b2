"""The debug probability matrix (Inference Cookbook FAQ Q9) and a decode step
captured in a CUDA graph with the on-device length advance (FAQ Q17, Q19).

Probability tolerance: the library forms P_ij = exp(s_ij - LSE_i) from its
own forward's LSE (within 1e-3 of the oracle's, the LSE contract) and an
fp32 dot product of the 16-bit inputs, so
|P_gpu - P_ref| <= P_ref * (|dLSE| + |ds|) + rounding, with |ds| ~ 1e-6 at
these sizes: we allow 1e-5 + 3e-3 * P_ref.  Masked entries and rows that see
no key must be exactly 0.
"""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, dev_i32, f64, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
@pytest.mark.parametrize("sq,sk,kw", [
    (70, 70, dict(causal=True)),
    (40, 130, dict(causal=True)),
    (130, 40, dict(causal=True)),            # rows 0..89 see no key
    (96, 96, dict(window=(8, 3), softcap=5.0)),
    (33, 257, {}),
])
def test_probs_match_oracle(dtype, sq, sk, kw):
    import torch

    from exact_attention_41_gb300 import libattn

    b, hq, hkv, d = 2, 4, 2, 64
    c = syn.dense_case(77, b, sq, sk, hq, hkv, d, dtype)
    q, k, v = (dev(c[n], dtype) for n in ("q", "k", "v"))
    o, lse = libattn.fwd(q, k, v, **kw)
    p = libattn.fwd_probs(q, k, lse, **kw)
    torch.cuda.synchronize()
    win = kw.get("window", (-1, -1))
    want = ref.probs(f64(c["q"], dtype), f64(c["k"], dtype), 1 / math.sqrt(d),
                     kw.get("causal", False), win[0], win[1], kw.get("softcap", 0.0))
    got = host(p)
    assert got.shape == want.shape
    zero = want == 0.0
    assert np.all(got[zero] == 0.0), "masked entries / empty rows must be exactly 0"
    err = np.abs(got - want)
    bound = 1e-5 + 3e-3 * np.abs(want)
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}"


def test_decode_step_captured_in_cuda_graph():
    """FAQ Q19: warm up, capture one decode step (append + attention, then the
    cache_seqlens += s_new advance of FAQ Q17) into a CUDA graph, replay it
    for three steps while only the contents of q / k_new / v_new change, and
    compare every step with the same step run eagerly (bitwise) and the last
    one with the oracle."""
    import torch

    from exact_attention_41_gb300 import libattn

    dtype, b, sq, s_new, hq, hkv, d, page = syn.BF16, 3, 1, 1, 8, 2, 128, 128
    c = syn.decode_case(91, b, sq, s_new, hq, hkv, d, 600, page, dtype)
    steps = 3
    rng = np.random.default_rng(92)
    qs = [syn.normal_bits(rng, (b, sq, hq, d), dtype) for _ in range(steps)]
    kns = [syn.normal_bits(rng, (b, s_new, hkv, d), dtype) for _ in range(steps)]
    vns = [syn.normal_bits(rng, (b, s_new, hkv, d), dtype) for _ in range(steps)]
    table = dev_i32(c["block_table"])
    splits = 2
    max_pages = c["block_table"].shape[1]

    def state():
        return (dev(c["k_cache"], dtype), dev(c["v_cache"], dtype), dev_i32(c["cache_seqlens"]))

    # eager reference run
    kc_e, vc_e, sl_e = state()
    outs_e = []
    for t in range(steps):
        o, _ = libattn.fwd_kvcache(dev(qs[t], dtype), kc_e, vc_e, sl_e, k_new=dev(kns[t], dtype),
                                   v_new=dev(vns[t], dtype), block_table=table, causal=True,
                                   num_splits=splits)
        libattn.kvcache_advance(sl_e, s_new)
        outs_e.append(host(o))
    torch.cuda.synchronize()

    # graph run: fixed buffers, contents refreshed before each replay
    kc, vc, sl = state()
    q_buf = dev(qs[0], dtype)
    kn_buf, vn_buf = dev(kns[0], dtype), dev(vns[0], dtype)
    ws = libattn.kvcache_workspace(q_buf, kc, page, max_pages, splits)
    out = torch.empty_like(q_buf)
    lse = torch.empty((b, hq, sq), device="cuda", dtype=torch.float32)

    def step():
        libattn.fwd_kvcache(q_buf, kc, vc, sl, k_new=kn_buf, v_new=vn_buf, block_table=table,
                            causal=True, num_splits=splits, workspace=ws, out=out, lse=lse)
        libattn.kvcache_advance(sl, s_new)

    # warm up on a scratch copy of the cache state, then restore it
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        saved = (kc.clone(), vc.clone(), sl.clone())
        for _ in range(2):
            step()
        kc.copy_(saved[0]), vc.copy_(saved[1]), sl.copy_(saved[2])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    # capture does not run the work: the state is still the initial one
    assert (sl.cpu().numpy() == c["cache_seqlens"]).all()

    for t in range(steps):
        q_buf.copy_(dev(qs[t], dtype))
        kn_buf.copy_(dev(kns[t], dtype))
        vn_buf.copy_(dev(vns[t], dtype))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out), outs_e[t])
    assert (sl.cpu().numpy() == c["cache_seqlens"] + steps * s_new).all()
    np.testing.assert_array_equal(host(kc), host(kc_e))

    # the last step against the oracle, from the cache state before it
    kc0 = f64(c["k_cache"], dtype)
    vc0 = f64(c["v_cache"], dtype)
    seqlens = c["cache_seqlens"].copy()
    for t in range(steps):
        ro, rl, kc0, vc0 = ref.kvcache_forward(
            f64(qs[t], dtype), kc0, vc0, seqlens, 1 / math.sqrt(d), f64(kns[t], dtype),
            f64(vns[t], dtype), c["block_table"], page, True)
        seqlens = seqlens + s_new
    assert_close(host(out), ro, dtype, "graph step out")
    assert_lse(host(lse), rl)


@pytest.mark.parametrize("d,window", [(128, (-1, -1)), (128, (200, 0)), (64, (-1, -1))])
def test_training_step_captured_in_cuda_graph(d, window):
    """FAQ Q19: a forward + deterministic backward step captured once in a
    CUDA graph and replayed on new inputs (same buffers) gives the eager
    call's bits: the library allocates nothing and never synchronises, and
    its per-device set-up runs on the first, eager, call.  Both forward
    layouts at d = 128 (two 128-row tiles; one tile with two CTAs per SM
    under the window) and the d = 64 one."""
    import torch

    from exact_attention_41_gb300 import libattn

    b, s, hq, hkv = 2, 1536, 8, 2
    kw = dict(causal=True, window=window)
    bufs = {n: dev(syn.dense_case(60 + i, b, s, s, hq, hkv, d, syn.BF16, with_dout=True)[n],
                   syn.BF16) for i, n in enumerate(("q", "k", "v", "dout"))}
    q, k, v, do = (bufs[n] for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty((b, hq, s), device="cuda", dtype=torch.float32)
    ws = libattn.bwd_workspace(q, k, True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        libattn.fwd(q, k, v, out=o, lse=lse, **kw)
        libattn.bwd(q, k, v, o, lse, do, deterministic=True, workspace=ws, dq=dq, dk=dk, dv=dv,
                    **kw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    for t in range(2):
        case = syn.dense_case(70 + t, b, s, s, hq, hkv, d, syn.BF16, with_dout=True)
        for n in ("q", "k", "v", "dout"):
            bufs[n].copy_(dev(case[n], syn.BF16))
        g.replay()
        torch.cuda.synchronize()
        got = [x.clone() for x in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        for x, y in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(x, y)
