"""Varlen (packed cu_seqlens) parity, forward and backward."""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, dev_i32, f64, host, report

pytestmark = pytest.mark.gpu


def run(case, lq, lk, dtype, deterministic=False, with_bwd=True, **kw):
    from exact_attention_41_gb300 import libattn

    q, k, v = (dev(case[x], dtype) for x in ("q", "k", "v"))
    cq, ck = dev_i32(case["cu_seqlens_q"]), dev_i32(case["cu_seqlens_k"])
    o, lse = libattn.fwd_varlen(q, k, v, cq, ck, max(lq), max(lk), **kw)
    grads = None
    if with_bwd:
        do = dev(case["dout"], dtype)
        grads = libattn.bwd_varlen(q, k, v, o, lse, do, cq, ck, max(lq), max(lk),
                                   deterministic=deterministic, **kw)
    return o, lse, grads


@pytest.mark.parametrize("dtype", [syn.F16, syn.BF16])
@pytest.mark.parametrize("kw", [dict(causal=True), dict(causal=True, window=(256, 0), softcap=50.0),
                                dict(), dict(window=(3, 30), softcap=2.0)])
def test_small_packed(dtype, kw):
    lq = [100, 1, 257, 64, 3, 130]
    lk = [100, 9, 129, 64, 1, 300]
    case = syn.varlen_case(31, lq, lk, 8, 2, 128, dtype, with_dout=True)
    o, lse, (dq, dk, dv) = run(case, lq, lk, dtype, **kw)
    win = kw.get("window", (-1, -1))
    args = [f64(case[x], dtype) for x in ("q", "k", "v")]
    a = (case["cu_seqlens_q"], case["cu_seqlens_k"], 1 / math.sqrt(128), kw.get("causal", False),
         win[0], win[1], kw.get("softcap", 0.0))
    ro, rl = ref.varlen_forward(*args, *a)
    assert_close(host(o), ro, dtype, "out")
    assert_lse(host(lse), rl)
    rq, rk, rv = ref.varlen_backward(*args, f64(case["dout"], dtype), *a, stored_o=dtype)
    assert_close(host(dq), rq, dtype, "dq")
    assert_close(host(dk), rk, dtype, "dk")
    assert_close(host(dv), rv, dtype, "dv")


@pytest.mark.parametrize("deterministic", [False, True])
def test_workload_sampled_sequences(deterministic):
    """64 sequences, lengths U[100, 4096] (seed 7), hq=32, hkv=8, d=128, bf16,
    causal + window (256, 0) + softcap 50: 8 seeded sequences checked in full."""
    lens = syn.varlen_lengths(7)
    case = syn.varlen_case(7, lens, lens, 32, 8, 128, syn.BF16, with_dout=True)
    kw = dict(causal=True, window=(256, 0), softcap=50.0)
    o, lse, (dq, dk, dv) = run(case, lens, lens, syn.BF16, deterministic, **kw)
    seqs = sorted(np.random.default_rng(700).choice(64, size=8, replace=False).tolist())
    seqs = sorted(set(seqs + [int(np.argmax(lens)), int(np.argmin(lens))]))
    args = [f64(case[x], syn.BF16) for x in ("q", "k", "v")]
    a = (case["cu_seqlens_q"], case["cu_seqlens_k"], 1 / math.sqrt(128), True, 256, 0, 50.0)
    ro, rl = ref.varlen_forward(*args, *a, seqs=seqs)
    rq, rk, rv = ref.varlen_backward(*args, f64(case["dout"], syn.BF16), *a, seqs=seqs,
                                     stored_o=syn.BF16)
    cu = case["cu_seqlens_q"]
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs])
    mode = "det" if deterministic else "atomic"
    got = {"dq": host(dq)[rows], "dk": host(dk)[rows], "dv": host(dv)[rows]}
    report(f"varlen fwd O ({len(seqs)} sequences)", host(o)[rows], ro[rows], syn.BF16, "oracle")
    for n, r in zip(("dq", "dk", "dv"), (rq, rk, rv)):
        report(f"varlen bwd {n} {mode} ({len(seqs)} sequences)", got[n], r[rows], syn.BF16)
    if not deterministic:
        eq, ek, ev = ref.varlen_backward(*args, f64(case["dout"], syn.BF16), *a, seqs=seqs)
        for n, r in zip(("dq", "dk", "dv"), (eq, ek, ev)):
            report(f"varlen bwd {n} {mode} ({len(seqs)} sequences)", got[n], r[rows], syn.BF16,
                   "oracle, exact gradient")
    assert_close(host(o)[rows], ro[rows], syn.BF16, "out")
    assert_lse(host(lse)[:, rows], rl[:, rows])
    assert_close(host(dq)[rows], rq[rows], syn.BF16, "dq")
    assert_close(host(dk)[rows], rk[rows], syn.BF16, "dk")
    assert_close(host(dv)[rows], rv[rows], syn.BF16, "dv")


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("kw", [dict(causal=True), dict(causal=True, window=(200, 0), softcap=30.0)])
def test_packed_head_dims(deterministic, d, kw):
    """Packed sequences at d = 64 and 256 (the backward's 64-column and
    column-half layouts; ragged lengths, an empty-key sequence, sq != sk).
    The forward is checked against the oracle; the backward is given the
    oracle's O (rounded to bf16) and LSE, so it is checked as a function of
    its inputs."""
    import torch

    from exact_attention_41_gb300 import libattn

    lq = [300, 1, 129, 64, 200]
    lk = [300, 7, 129, 0, 450]
    dtype = syn.BF16
    case = syn.varlen_case(33, lq, lk, 4, 2, d, dtype, with_dout=True)
    o, lse, _ = run(case, lq, lk, dtype, with_bwd=False, **kw)
    win = kw.get("window", (-1, -1))
    args = [f64(case[x], dtype) for x in ("q", "k", "v")]
    a = (case["cu_seqlens_q"], case["cu_seqlens_k"], 1 / math.sqrt(d), True,
         win[0], win[1], kw.get("softcap", 0.0))
    ro, rl = ref.varlen_forward(*args, *a)
    assert_close(host(o), ro, dtype, "out")
    assert_lse(host(lse), rl)
    q, k, v, do = (dev(case[x], dtype) for x in ("q", "k", "v", "dout"))
    cq, ck = dev_i32(case["cu_seqlens_q"]), dev_i32(case["cu_seqlens_k"])
    o_ref = torch.from_numpy(ref.round_to(ro, dtype)).to(torch.bfloat16).cuda()
    lse_ref = torch.from_numpy(rl.astype(np.float32)).cuda()
    dq, dk, dv = libattn.bwd_varlen(q, k, v, o_ref, lse_ref, do, cq, ck, max(lq), max(lk),
                                    deterministic=deterministic, **kw)
    rq, rk, rv = ref.varlen_backward(*args, f64(case["dout"], dtype), *a, stored_o=dtype)
    assert_close(host(dq), rq, dtype, "dq")
    assert_close(host(dk), rk, dtype, "dk")
    assert_close(host(dv), rv, dtype, "dv")
