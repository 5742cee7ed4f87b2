"""Device-side error paths, exercised without faulting the GPU.

* A bounded wait that runs out: with the test hook attn_set_test_stall the
  MMA issuer waits on a barrier that nothing completes, and with a 1 ms
  limit (attn_set_wait_limit_ns) that wait expires; the kernels give up,
  drain their own copies and MMAs, free their TMEM and return; the call
  reports ATTN_ERR_TIMEOUT through attn_get_device_error, and the next call
  with the hook off and the default limit is correct.
* Malformed varlen offsets (a sequence ending past total_q / total_k) are
  skipped and flagged, and nothing is written past the caller's buffers.
* A block-table entry outside the page pool: the split that holds it gives
  the empty result (O = 0, LSE = -inf), the error word says which check
  fired, and the other batch entries are unaffected.
"""
import math

import numpy as np
import pytest

from exact_attention_41_gb300 import synthetic as syn
from oracle import attention as ref
from tests.helpers import assert_close, assert_lse, dev, dev_i32, f64, host

pytestmark = pytest.mark.gpu

ERR_TIMEOUT, ERR_DEVICE = 5, 6
BIT_PAGE, BIT_BAD_SEQLEN, BIT_TIMEOUT = 1, 16, 8


def _clear():
    from exact_attention_41_gb300 import libattn

    libattn.device_error()


def _dense_call(kind, case, dtype, deterministic=False):
    from exact_attention_41_gb300 import libattn

    q, k, v = (dev(case[x], dtype) for x in ("q", "k", "v"))
    o, lse = libattn.fwd(q, k, v, causal=True)
    if kind == "fwd":
        return o, lse
    return libattn.bwd(q, k, v, o, lse, dev(case["dout"], dtype), causal=True,
                       deterministic=deterministic)


@pytest.mark.parametrize("kind,deterministic", [("fwd", False), ("bwd", False), ("bwd", True)])
@pytest.mark.parametrize("s,d", [(384, 128), (1280, 128), (384, 64), (384, 256)])
def test_wait_timeout_is_reported_and_recoverable(kind, deterministic, s, d):
    """Every tensor-core kernel layout: the one-tile two-CTA forward (s = 384)
    and the two-tile one (1280 keys) at d = 128, the d = 64 and d = 256
    forwards, and the backward kernels at each head dim."""
    import torch

    from exact_attention_41_gb300 import libattn

    case = syn.dense_case(51, 2, s, s, 8, 2, d, syn.BF16, with_dout=True)
    _clear()
    prev = libattn.set_wait_limit_ns(1_000_000)
    libattn.set_test_stall(True)
    try:
        _dense_call(kind, case, syn.BF16, deterministic)
        torch.cuda.synchronize()
    finally:
        libattn.set_test_stall(False)
        libattn.set_wait_limit_ns(prev)
    st, word = libattn.device_error()
    assert st == ERR_TIMEOUT and word & BIT_TIMEOUT, (st, word)
    # the same process, default limit: correct again
    out = _dense_call(kind, case, syn.BF16, deterministic)
    torch.cuda.synchronize()
    assert libattn.device_error() == (0, 0)
    q, k, v = (f64(case[x], syn.BF16) for x in ("q", "k", "v"))
    if kind == "fwd":
        ro, rl = ref.forward(q, k, v, 1 / math.sqrt(d), causal=True)
        assert_close(host(out[0]), ro, syn.BF16, "out")
        assert_lse(host(out[1]), rl)
    else:
        rq, rk, rv = ref.backward(q, k, v, f64(case["dout"], syn.BF16), 1 / math.sqrt(d),
                                  causal=True, stored_o=syn.BF16)
        for g, r, n in zip(out, (rq, rk, rv), ("dq", "dk", "dv")):
            assert_close(host(g), r, syn.BF16, n)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_wait_timeout_is_reported_and_recoverable(d):
    import torch

    from exact_attention_41_gb300 import libattn

    c = syn.decode_case(52, 3, 1, 1, 8, 2, d, 900, 128, syn.BF16)
    kc, vc = dev(c["k_cache"], syn.BF16), dev(c["v_cache"], syn.BF16)
    args = (dev(c["q"], syn.BF16), kc, vc, dev_i32(c["cache_seqlens"]))
    kw = dict(k_new=dev(c["k_new"], syn.BF16), v_new=dev(c["v_new"], syn.BF16),
              block_table=dev_i32(c["block_table"]), causal=True, num_splits=2)
    _clear()
    prev = libattn.set_wait_limit_ns(1_000_000)
    libattn.set_test_stall(True)
    try:
        libattn.fwd_kvcache(*args, **kw)
        torch.cuda.synchronize()
    finally:
        libattn.set_test_stall(False)
        libattn.set_wait_limit_ns(prev)
    st, word = libattn.device_error()
    assert st == ERR_TIMEOUT and word & BIT_TIMEOUT, (st, word)
    o, lse = libattn.fwd_kvcache(*args, **kw)
    torch.cuda.synchronize()
    assert libattn.device_error() == (0, 0)
    ro, rl, _, _ = ref.kvcache_forward(
        f64(c["q"], syn.BF16), f64(c["k_cache"], syn.BF16), f64(c["v_cache"], syn.BF16),
        c["cache_seqlens"], 1 / math.sqrt(d), f64(c["k_new"], syn.BF16),
        f64(c["v_new"], syn.BF16), c["block_table"], 128, causal=True)
    assert_close(host(o), ro, syn.BF16, "out")
    assert_lse(host(lse), rl)


def test_wait_limit_setter_round_trip():
    from exact_attention_41_gb300 import libattn

    prev = libattn.set_wait_limit_ns(12345)
    assert libattn.set_wait_limit_ns(0) == 12345
    assert libattn.set_wait_limit_ns(prev) == 2_000_000_000
    assert libattn.set_test_stall(True) is False
    assert libattn.set_test_stall(False) is True


@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_offsets_past_the_tensors_are_rejected(deterministic):
    """cu_seqlens_q / cu_seqlens_k whose last sequence ends one row past
    total_q / total_k: that sequence is skipped (error word: bad length) and
    the guard rows after every output buffer keep their sentinel."""
    import torch

    from exact_attention_41_gb300 import libattn

    lens = [70, 130, 64]
    case = syn.varlen_case(53, lens, lens, 4, 2, 128, syn.BF16, with_dout=True)
    t = sum(lens)
    guard = 16

    def with_guard(bits, fill):
        full = torch.full((t + guard,) + bits.shape[1:], fill, dtype=torch.bfloat16, device="cuda")
        full[:t] = dev(bits, syn.BF16)
        return full

    sentinel = 3.0
    q, k, v, do = (with_guard(case[x], sentinel) for x in ("q", "k", "v", "dout"))
    o_full = torch.full_like(q, sentinel)
    lse_full = torch.full((4 * t + guard,), sentinel, device="cuda")  # LSE is (hq, total_q)
    cu_bad = np.asarray(case["cu_seqlens_q"]).copy()
    cu_bad[-1] += 1
    cq = dev_i32(cu_bad)
    _clear()
    libattn.lib().attn_fwd_varlen(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o_full.data_ptr(), lse_full.data_ptr(),
        cq.data_ptr(), cq.data_ptr(), 3, max(lens) + 1, max(lens) + 1, t, t, 1, 4, 2, 128,
        1 / math.sqrt(128), 1, -1, -1, 0.0, libattn._stream())
    torch.cuda.synchronize()
    st, word = libattn.device_error()
    assert st == ERR_DEVICE and word & BIT_BAD_SEQLEN, (st, word)
    assert torch.all(o_full[t:] == sentinel) and torch.all(lse_full[4 * t:] == sentinel)
    # the backward with the same offsets, gradients with guard rows
    dq_full, dk_full, dv_full = (torch.full_like(x, sentinel) for x in (q, k, v))
    lse = lse_full
    n = libattn.lib().attn_bwd_varlen_workspace_size(3, max(lens) + 1, max(lens) + 1, t, t, 4, 2,
                                                     128, int(deterministic))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    libattn.lib().attn_bwd_varlen(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o_full.data_ptr(), lse.data_ptr(),
        do.data_ptr(), dq_full.data_ptr(), dk_full.data_ptr(), dv_full.data_ptr(), cq.data_ptr(),
        cq.data_ptr(), 3, max(lens) + 1, max(lens) + 1, t, t, 1, 4, 2, 128, 1 / math.sqrt(128),
        1, -1, -1, 0.0, int(deterministic), ws.data_ptr(), n, libattn._stream())
    torch.cuda.synchronize()
    st, word = libattn.device_error()
    assert st == ERR_DEVICE and word & BIT_BAD_SEQLEN, (st, word)
    for x in (dq_full, dk_full, dv_full):
        assert torch.all(x[t:] == sentinel)


@pytest.mark.parametrize("num_splits", [1, 3])
@pytest.mark.parametrize("d,hq", [(128, 8), (64, 4)])
def test_page_outside_pool_gives_empty_row_and_flag(num_splits, d, hq):
    """One batch entry's block table points past the pool at its fourth
    page: the error word says "page out of range" and the other entries match
    the oracle.  The split that holds the bad page gives the empty result
    (O = 0, LSE = -inf), so with one split the entry's output is exactly that,
    and with several it is the merge of the other splits -- the same bits
    whatever the scratch memory held before the call."""
    import torch

    from exact_attention_41_gb300 import libattn

    c = syn.decode_case(54, 3, 1, 0, hq, 2, d, 1000, 128, syn.BF16)
    table = c["block_table"].copy()
    seqlens = c["cache_seqlens"].copy()
    bad = 1
    seqlens[bad] = 600  # pages 0..4 used; page 3 made invalid
    table[bad, 3] = table.max() + 1000
    kc, vc = dev(c["k_cache"], syn.BF16), dev(c["v_cache"], syn.BF16)
    q = dev(c["q"], syn.BF16)
    ws = libattn.kvcache_workspace(q, kc, 128, table.shape[1], num_splits)
    runs = []
    for fill in (0.0, float("nan")):  # scratch contents before the call
        ws.view(torch.uint8).fill_(0)
        if fill != 0.0:
            ws[: ws.numel() // 4 * 4].view(torch.float32).fill_(fill)
        _clear()
        o, lse = libattn.fwd_kvcache(q, kc, vc, dev_i32(seqlens), block_table=dev_i32(table),
                                     causal=True, num_splits=num_splits, workspace=ws)
        torch.cuda.synchronize()
        st, word = libattn.device_error()
        assert st == ERR_DEVICE and word & BIT_PAGE, (st, word)
        runs.append((host(o), host(lse)))
    (o, lse), (o2, lse2) = runs
    np.testing.assert_array_equal(o[bad], o2[bad])
    np.testing.assert_array_equal(lse[bad], lse2[bad])
    assert np.isfinite(o[bad]).all()
    if num_splits == 1:
        assert np.all(o[bad] == 0) and np.isneginf(lse[bad]).all()
    good = [i for i in range(3) if i != bad]
    ro, rl, _, _ = ref.kvcache_forward(
        f64(c["q"], syn.BF16), f64(c["k_cache"], syn.BF16), f64(c["v_cache"], syn.BF16), seqlens,
        1 / math.sqrt(d), None, None, table, 128, causal=True, batches=good)
    assert_close(o[good], ro[good], syn.BF16, "out")
    assert_lse(lse[good], rl[good])
