"""Pins for the float64 oracle: each test checks it against something other
than itself -- a closed form, a fact the pages state, a library routine, an
invariant of the mathematics, or finite differences.  All CPU, all fast."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import attention as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")


def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- softmax rows


def test_probability_rows_sum_to_one_masked_zero():
    rng = np.random.default_rng(1)
    sq, sk, d = 9, 13, 8
    q, k, v = rng.standard_normal((sq, d)), rng.standard_normal((sk, d)), rng.standard_normal((sk, d))
    for causal, wl, wr, cap in [(False, -1, -1, 0.0), (True, -1, -1, 0.0), (False, 2, 1, 0.0),
                                (True, 3, -1, 5.0)]:
        _, lse, p = ref.head_forward(q, k, v, np.arange(sq), sq, sk, 0.3, causal, wl, wr, cap,
                                     return_probs=True)
        mask = ref.visible(np.arange(sq), sq, sk, causal, wl, wr)
        assert (p >= 0).all()
        assert (p[~mask] == 0).all()
        nonempty = mask.any(1)
        np.testing.assert_allclose(p[nonempty].sum(1), 1.0, atol=1e-12)
        assert np.isneginf(lse[~nonempty]).all()


def test_single_key_output_is_v():
    rng = np.random.default_rng(2)
    q, k, v = rng.standard_normal((1, 5, 2, 8)), rng.standard_normal((1, 1, 2, 8)), rng.standard_normal((1, 1, 2, 8))
    o, lse = ref.forward(q, k, v, 0.7)
    for h in range(2):
        np.testing.assert_array_equal(o[0, :, h], np.broadcast_to(v[0, 0, h], (5, 8)))
        np.testing.assert_allclose(lse[0, h], 0.7 * q[0, :, h] @ k[0, 0, h], rtol=1e-14)


def test_window_zero_zero_is_identity():
    q, k, v = rnd(3, 1, 11, 1, 4), rnd(4, 1, 11, 1, 4), rnd(5, 1, 11, 1, 4)
    o, _ = ref.forward(q, k, v, 1.0, win_l=0, win_r=0)
    np.testing.assert_array_equal(o, v)
    o, _ = ref.forward(q, k, v, 1.0, causal=True, win_l=0)
    np.testing.assert_array_equal(o, v)


def test_causal_square_first_row_is_v0():
    q, k, v = rnd(6, 1, 6, 1, 4), rnd(7, 1, 6, 1, 4), rnd(8, 1, 6, 1, 4)
    o, _ = ref.forward(q, k, v, 1.0, causal=True)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0])


@pytest.mark.parametrize("sq,sk", [(6, 6), (3, 7), (7, 3), (1, 9)])
@pytest.mark.parametrize("cap", [0.0, 4.0])
def test_zero_query_gives_mean_of_visible_values(sq, sk, cap):
    """Q = 0 makes all visible scores equal (tanh 0 = 0), so O_i is the mean
    of the visible V rows and LSE_i = ln(#visible).  Visible sets come from
    the bottom-right rule of the Inference Cookbook FAQ Q6: query i sees the
    first i + 1 + (sk - sq) keys (none when that is <= 0)."""
    v = rnd(9, 1, sk, 1, 3)
    q = np.zeros((1, sq, 1, 3))
    k = rnd(10, 1, sk, 1, 3)
    o, lse = ref.forward(q, k, v, 1.0, causal=True, softcap=cap)
    csum = np.cumsum(v[0, :, 0], axis=0)
    for i in range(sq):
        n = i + 1 + (sk - sq)
        if n <= 0:
            assert np.all(o[0, i, 0] == 0) and np.isneginf(lse[0, 0, i])
        else:
            np.testing.assert_allclose(o[0, i, 0], csum[n - 1] / n, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(lse[0, 0, i], math.log(n), rtol=1e-14)
    o, lse = ref.forward(q, k, v, 1.0, causal=False, softcap=cap)
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, :, 0].mean(0), (sq, 3)), atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], math.log(sk), rtol=1e-14)


def test_lse_is_library_logsumexp():
    q, k, v = rnd(11, 1, 7, 2, 5), rnd(12, 1, 9, 2, 5), rnd(13, 1, 9, 2, 5)
    _, lse = ref.forward(q, k, v, 0.4)
    for h in range(2):
        s = 0.4 * np.einsum("id,jd->ij", q[0, :, h], k[0, :, h])
        np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(s, axis=1), rtol=1e-13)


# ---------------------------------------------------------------- masks


def test_golden_window_rows():
    f = facts()["window_example"]
    wl, wr = f["window_size"]
    sq = 1200
    mask = ref.visible(np.arange(sq), sq, sq, False, wl, wr)
    for i, lo, hi in f["rows"]:
        idx = np.flatnonzero(mask[i])
        assert idx[0] == lo and idx[-1] == hi and len(idx) == hi - lo + 1


def test_golden_bottom_right_counts():
    for case in facts()["bottom_right_causal"]["cases"]:
        sq, sk = case["sq"], case["sk"]
        counts = ref.visible(np.arange(sq), sq, sk, True, -1, -1).sum(1)
        assert list(counts) == case["row_visible_counts"]


@pytest.mark.parametrize("sq,sk", [(3, 7), (7, 3), (1, 9), (5, 5)])
def test_bottom_right_causal_is_kv_cache_prefix(sq, sk):
    """Each causal query row equals a single-query, non-causal call on the key
    prefix it may see -- the KV-cache reading of FAQ Q6."""
    q, k, v = rnd(14, 1, sq, 1, 4), rnd(15, 1, sk, 1, 4), rnd(16, 1, sk, 1, 4)
    o, lse = ref.forward(q, k, v, 0.5, causal=True)
    for i in range(sq):
        n = sk - sq + i + 1
        if n <= 0:
            assert np.all(o[0, i] == 0) and np.isneginf(lse[0, 0, i])
            continue
        o1, l1 = ref.forward(q[:, i:i + 1], k[:, :n], v[:, :n], 0.5)
        np.testing.assert_allclose(o[0, i], o1[0, 0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[0, 0, i], l1[0, 0, 0], rtol=1e-13)


@pytest.mark.parametrize("wl,wr", [(2, 1), (0, 3), (4, 0), (-1, 2), (3, -1)])
def test_window_is_key_slice(wl, wr):
    """Window (left, right) row i equals attention over keys
    [max(0, i-left), min(sk-1, i+right)] (FAQ Q21), sq = sk."""
    n = 10
    q, k, v = rnd(17, 1, n, 1, 4), rnd(18, 1, n, 1, 4), rnd(19, 1, n, 1, 4)
    o, _ = ref.forward(q, k, v, 0.5, win_l=wl, win_r=wr)
    for i in range(n):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = n - 1 if wr < 0 else min(n - 1, i + wr)
        o1, _ = ref.forward(q[:, i:i + 1], k[:, lo:hi + 1], v[:, lo:hi + 1], 0.5)
        np.testing.assert_allclose(o[0, i], o1[0, 0], rtol=1e-13, atol=1e-15)


def test_right_zero_window_is_causal():
    q, k, v = rnd(20, 1, 6, 2, 4), rnd(21, 1, 9, 2, 4), rnd(22, 1, 9, 2, 4)
    a = ref.forward(q, k, v, 0.5, causal=True)
    b = ref.forward(q, k, v, 0.5, win_l=-1, win_r=0)
    np.testing.assert_array_equal(a[0], b[0])
    a = ref.forward(q, k, v, 0.5, causal=True, win_l=2)
    b = ref.forward(q, k, v, 0.5, win_l=2, win_r=0)
    np.testing.assert_array_equal(a[0], b[0])


def test_key_permutation_invariance_and_query_equivariance():
    q, k, v = rnd(23, 1, 8, 2, 4), rnd(24, 1, 12, 2, 4), rnd(25, 1, 12, 2, 4)
    o, lse = ref.forward(q, k, v, 0.6, softcap=3.0)
    perm = np.random.default_rng(0).permutation(12)
    o2, lse2 = ref.forward(q, k[:, perm], v[:, perm], 0.6, softcap=3.0)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)
    qp = np.random.default_rng(1).permutation(8)
    o3, lse3 = ref.forward(q[:, qp], k, v, 0.6, softcap=3.0)
    np.testing.assert_allclose(o3, o[:, qp], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse3, lse[:, :, qp], rtol=1e-13)


# ---------------------------------------------------------------- softmax order


def online_softmax_attention(qh, kh, vh, scale, block):
    """Blockwise online softmax (FlashAttention完整说明 section 二.1), written
    independently of the oracle, which is two-pass."""
    m = np.full(qh.shape[0], -np.inf)
    ell = np.zeros(qh.shape[0])
    acc = np.zeros((qh.shape[0], vh.shape[1]))
    for j0 in range(0, kh.shape[0], block):
        s = scale * qh @ kh[j0:j0 + block].T
        m_new = np.maximum(m, s.max(1))
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        ell = alpha * ell + p.sum(1)
        acc = alpha[:, None] * acc + p @ vh[j0:j0 + block]
        m = m_new
    return acc / ell[:, None], m + np.log(ell)


@pytest.mark.parametrize("block", [1, 3, 16])
def test_two_pass_equals_online_rescale(block):
    q, k, v = rnd(26, 7, 8), rnd(27, 37, 8), rnd(28, 37, 8)
    o1, l1 = online_softmax_attention(q, k, v, 0.35, block)
    o2, l2 = ref.head_forward(q, k, v, np.arange(7), 7, 37, 0.35)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)


# ---------------------------------------------------------------- softcap


def test_softcap_large_equals_none_and_bounds():
    q, k, v = rnd(29, 1, 5, 1, 4), rnd(30, 1, 6, 1, 4), rnd(31, 1, 6, 1, 4)
    a = ref.forward(q, k, v, 0.5)
    b = ref.forward(q, k, v, 0.5, softcap=1e7)
    np.testing.assert_allclose(b[0], a[0], rtol=1e-9, atol=1e-12)
    # huge scores: every capped score is within (-c, c), so LSE < c + ln(sk)
    c = 2.0
    _, lse = ref.forward(100 * q, k, v, 1.0, softcap=c)
    assert (lse < c + math.log(6) + 1e-12).all()
    assert (lse > -c + math.log(6) - 1e-12).all()


def test_softcap_two_keys_closed_form():
    """Two keys, one query: P = [1, e^(t2-t1)] / (1 + e^(t2-t1)) with
    t = c * tanh(scale * q.k / c) (FAQ Q22 order: softcap before softmax)."""
    q = np.array([[[[1.0, 2.0]]]])
    k = np.array([[[[3.0, 0.5]], [[-1.0, 1.0]]]])
    v = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    c, scale = 1.5, 0.5
    t1 = c * math.tanh(scale * 4.0 / c)
    t2 = c * math.tanh(scale * 1.0 / c)
    p2 = 1.0 / (1.0 + math.exp(t1 - t2))
    o, lse = ref.forward(q, k, v, scale, softcap=c)
    np.testing.assert_allclose(o[0, 0, 0], [1 - p2, p2], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], math.log(math.exp(t1) + math.exp(t2)), rtol=1e-14)


# ---------------------------------------------------------------- GQA / varlen / cache


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v = rnd(32, 2, 5, 6, 4), rnd(33, 2, 7, 2, 4), rnd(34, 2, 7, 2, 4)
    o, lse = ref.forward(q, k, v, 0.5, causal=True)
    o2, lse2 = ref.forward(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), 0.5, causal=True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    dout = rnd(35, 2, 5, 6, 4)
    g1 = ref.backward(q, k, v, dout, 0.5, causal=True)
    g2 = ref.backward(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), dout, 0.5, causal=True)
    np.testing.assert_allclose(g1[0], g2[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g1[1], g2[1].reshape(2, 7, 2, 3, 4).sum(3), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g1[2], g2[2].reshape(2, 7, 2, 3, 4).sum(3), rtol=1e-12, atol=1e-14)


def test_varlen_equal_lengths_equals_batched_dense():
    b, s, hq, hkv, d = 3, 6, 4, 2, 4
    q, k, v, do = rnd(36, b, s, hq, d), rnd(37, b, s, hkv, d), rnd(38, b, s, hkv, d), rnd(39, b, s, hq, d)
    cu = np.arange(b + 1) * s
    o, lse = ref.forward(q, k, v, 0.5, causal=True, win_l=2, softcap=4.0)
    ov, lv = ref.varlen_forward(q.reshape(b * s, hq, d), k.reshape(b * s, hkv, d),
                                v.reshape(b * s, hkv, d), cu, cu, 0.5, True, 2, -1, 4.0)
    np.testing.assert_array_equal(ov, o.reshape(b * s, hq, d))
    np.testing.assert_array_equal(lv, lse.transpose(1, 0, 2).reshape(hq, b * s))
    g = ref.backward(q, k, v, do, 0.5, causal=True, win_l=2, softcap=4.0)
    gv = ref.varlen_backward(q.reshape(b * s, hq, d), k.reshape(b * s, hkv, d),
                             v.reshape(b * s, hkv, d), do.reshape(b * s, hq, d), cu, cu, 0.5,
                             True, 2, -1, 4.0)
    for a, bb in zip(g, gv):
        np.testing.assert_array_equal(bb, a.reshape(bb.shape))


def test_varlen_sequences_do_not_interact():
    lq, lk = [3, 5, 2], [4, 5, 6]
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, k, v = rnd(40, cq[-1], 2, 4), rnd(41, ck[-1], 1, 4), rnd(42, ck[-1], 1, 4)
    o, _ = ref.varlen_forward(q, k, v, cq, ck, 0.5, causal=True)
    k2 = k.copy()
    k2[ck[0]:ck[1]] += rnd(61, lk[0], 1, 4)  # perturb sequence 0 only
    o2, _ = ref.varlen_forward(q, k2, v, cq, ck, 0.5, causal=True)
    np.testing.assert_array_equal(o[cq[1]:], o2[cq[1]:])
    assert not np.allclose(o[:cq[1]], o2[:cq[1]])


@pytest.mark.parametrize("s_new", [0, 1, 3])
def test_paged_cache_equals_contiguous(s_new):
    rng = np.random.default_rng(43)
    b, hq, hkv, d, page, npp = 3, 4, 2, 4, 4, 5
    sq = max(s_new, 1)
    lens = np.array([0, 7, 13])
    table = rng.permutation(b * npp).reshape(b, npp)
    kc, vc = rng.standard_normal((b * npp, page, hkv, d)), rng.standard_normal((b * npp, page, hkv, d))
    q = rng.standard_normal((b, sq, hq, d))
    kn = rng.standard_normal((b, s_new, hkv, d)) if s_new else None
    vn = rng.standard_normal((b, s_new, hkv, d)) if s_new else None
    o, lse, kc2, vc2 = ref.kvcache_forward(q, kc, vc, lens, 0.5, kn, vn, table, page, causal=True)
    # the same logical cache laid out contiguously: (b, capacity, hkv, d)
    cap = npp * page
    kflat = kc[table].reshape(b, cap, hkv, d)
    vflat = vc[table].reshape(b, cap, hkv, d)
    o2, lse2, kf2, vf2 = ref.kvcache_forward(q, kflat, vflat, lens, 0.5, kn, vn, causal=True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    np.testing.assert_array_equal(kc2[table].reshape(b, cap, hkv, d), kf2)
    for bi in range(b):
        n = lens[bi] + s_new
        if n == 0:
            assert np.isneginf(lse[bi]).all()
            continue
        o3, l3 = ref.forward(q[bi:bi + 1], kf2[bi:bi + 1, :n], vf2[bi:bi + 1, :n], 0.5, causal=True)
        np.testing.assert_array_equal(o[bi], o3[0])
        # appended rows landed at positions lens..lens+s_new, the rest untouched
        if s_new:
            np.testing.assert_array_equal(kf2[bi, lens[bi]:n], kn[bi])
        np.testing.assert_array_equal(kf2[bi, :lens[bi]], kflat[bi, :lens[bi]])
        np.testing.assert_array_equal(kf2[bi, n:], kflat[bi, n:])
    assert list(lens) == [0, 7, 13]  # cache_seqlens is not updated by the call


# ---------------------------------------------------------------- backward


def loss(q, k, v, dout, **kw):
    o, _ = ref.forward(q, k, v, **kw)
    return float((o * dout).sum())


@pytest.mark.parametrize("kw", [
    dict(scale=0.7),
    dict(scale=0.7, causal=True),
    dict(scale=0.7, causal=True, softcap=1.3),
    dict(scale=0.7, win_l=1, win_r=1, softcap=2.0),
])
@pytest.mark.parametrize("sq,sk", [(4, 4), (3, 5), (5, 3)])
def test_backward_matches_finite_differences(kw, sq, sk):
    b, hq, hkv, d = 1, 2, 1, 3
    q, k, v, do = rnd(44, b, sq, hq, d), rnd(45, b, sk, hkv, d), rnd(46, b, sk, hkv, d), rnd(47, b, sq, hq, d)
    dq, dk, dv = ref.backward(q, k, v, do, **kw)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = loss(q, k, v, do, **kw)
            x[idx] = old - h
            fm = loss(q, k, v, do, **kw)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_backward_invariants():
    b, sq, sk, hq, hkv, d = 2, 6, 9, 4, 2, 5
    q, k, v, do = rnd(48, b, sq, hq, d), rnd(49, b, sk, hkv, d), rnd(50, b, sk, hkv, d), rnd(51, b, sq, hq, d)
    dq, dk, dv = ref.backward(q, k, v, do, 0.5, causal=True)
    # rows of dS sum to zero, so the key gradients of each (b, kv head) sum to zero
    np.testing.assert_allclose(dk.sum(1), 0.0, atol=1e-12)
    # P rows sum to one, so sum_j dV_j = sum of dO over the group's non-empty rows
    nonempty = ref.visible(np.arange(sq), sq, sk, True, -1, -1).any(1)
    want = do[:, nonempty].reshape(b, -1, hkv, hq // hkv, d).sum((1, 3))
    np.testing.assert_allclose(dv.sum(1), want, rtol=1e-12, atol=1e-12)


def test_fully_masked_rows_have_zero_gradients():
    q, k, v, do = rnd(52, 1, 7, 1, 3), rnd(53, 1, 3, 1, 3), rnd(54, 1, 3, 1, 3), rnd(55, 1, 7, 1, 3)
    dq, _, _ = ref.backward(q, k, v, do, 0.5, causal=True)
    assert np.all(dq[0, :4] == 0)


# ---------------------------------------------------------------- library routine


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    """Square causal masks coincide for top-left and bottom-right alignment,
    so torch's float64 CPU SDPA (and its autograd) is an independent check."""
    torch = pytest.importorskip("torch")
    b, s, hq, hkv, d = 2, 17, 4, 2, 8
    q, k, v, do = rnd(56, b, s, hq, d), rnd(57, b, s, hkv, d), rnd(58, b, s, hkv, d), rnd(59, b, s, hq, d)
    tq = torch.tensor(q.transpose(0, 2, 1, 3), requires_grad=True)
    tk = torch.tensor(np.repeat(k, 2, axis=2).transpose(0, 2, 1, 3), requires_grad=True)
    tv = torch.tensor(np.repeat(v, 2, axis=2).transpose(0, 2, 1, 3), requires_grad=True)
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.3)
    to.backward(torch.tensor(do.transpose(0, 2, 1, 3)))
    o, _ = ref.forward(q, k, v, 0.3, causal=causal)
    np.testing.assert_allclose(o, to.detach().numpy().transpose(0, 2, 1, 3), rtol=1e-12, atol=1e-13)
    dq, dk, dv = ref.backward(q, k, v, do, 0.3, causal=causal)
    np.testing.assert_allclose(dq, tq.grad.numpy().transpose(0, 2, 1, 3), rtol=1e-11, atol=1e-12)
    tdk = tk.grad.numpy().transpose(0, 2, 1, 3).reshape(b, s, hkv, 2, d).sum(3)
    tdv = tv.grad.numpy().transpose(0, 2, 1, 3).reshape(b, s, hkv, 2, d).sum(3)
    np.testing.assert_allclose(dk, tdk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tdv, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- pages' numbers


def test_standard_attention_memory_figure():
    f = facts()["standard_attention_memory"]
    assert f["N"] ** 2 * f["bytes_per_element"] == f["megabytes"] * 2 ** 20


def test_output_shape_is_query_shape():
    for shape in facts()["output_shapes"]["shapes"]:
        b, s, h, d = shape
        small = (b, min(s, 8), h if h <= 8 else 2, min(d, 8))
        q = rnd(60, *small)
        o, lse = ref.forward(q, q.copy(), q.copy(), 1.0)
        assert o.shape == small and lse.shape == (small[0], small[2], small[1])


def test_stored_output_reading_of_d():
    """D_i from the stored (rounded) O: with the exact O it is the textbook
    D_i = sum_j P_ij dP_ij (rows of P sum to one); with O rounded the
    gradients move by no more than the rounding allows."""
    q, k, v, do = rnd(62, 1, 9, 2, 8), rnd(63, 1, 11, 1, 8), rnd(64, 1, 11, 1, 8), rnd(65, 1, 9, 2, 8)
    exact = ref.backward(q, k, v, do, 0.4, causal=True)
    for dt in ("bf16", "f16"):
        got = ref.backward(q, k, v, do, 0.4, causal=True, stored_o=dt)
        np.testing.assert_array_equal(got[2], exact[2])  # dV does not involve D
        eps = 2.0 ** (-8 if dt == "bf16" else -11)
        assert np.abs(got[0] - exact[0]).max() < 50 * eps
        assert np.abs(got[0] - exact[0]).max() > 0
    np.testing.assert_array_equal(ref.round_to(np.array([1.0, 1.00390625, 1.01171875]), "bf16"),
                                  [1.0, 1.0, 1.015625])


@pytest.mark.parametrize("kw", [dict(causal=True), dict(win_l=2, win_r=1, softcap=3.0),
                                dict(causal=True, win_l=1)])
def test_probability_matrix_reproduces_forward(kw):
    """FAQ Q9 debug matrix: O = P V row by row (against the separately pinned
    forward), non-empty rows sum to 1, masked entries are exactly 0, and the
    rows that see no key (sq > sk, bottom-right causal) are all zero."""
    rng = np.random.default_rng(11)
    b, sq, sk, hq, hkv, d = 2, 7, 5, 4, 2, 8
    q, k, v = (rng.standard_normal(sh) for sh in ((b, sq, hq, d), (b, sk, hkv, d), (b, sk, hkv, d)))
    p = ref.probs(q, k, 0.4, **kw)
    o, lse = ref.forward(q, k, v, 0.4, **kw)
    g = hq // hkv
    for bi in range(b):
        for h in range(hq):
            np.testing.assert_allclose(p[bi, h] @ v[bi, :, h // g], o[bi, :, h], atol=1e-12)
    mask = ref.visible(np.arange(sq), sq, sk, kw.get("causal", False), kw.get("win_l", -1),
                       kw.get("win_r", -1))
    assert np.all(p[:, :, ~mask] == 0.0)
    nonempty = mask.any(axis=1)
    np.testing.assert_allclose(p.sum(axis=3)[:, :, nonempty], 1.0, atol=1e-12)
    assert np.all(p[:, :, ~nonempty] == 0.0)
    assert np.all(np.isneginf(lse[:, :, ~nonempty]))


def test_e4m3_format_facts():
    """OCP FP8 E4M3 (the format of FAQ Q20's FP8 tensors): bias 7, 3 mantissa
    bits, no infinities; 0x38 = 1, 0x7E = 448 (largest), 0x08 = 2^-6 (smallest
    normal), 0x01 = 2^-9 (smallest subnormal), 0x7F/0xFF = NaN."""
    from exact_attention_41_gb300 import synthetic as syn

    v = syn.e4m3_values()
    assert v[0x38] == 1.0 and v[0xB8] == -1.0 and v[0x7E] == 448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9 and v[0x00] == 0.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    finite = np.flatnonzero(~np.isnan(v))
    # every finite pattern survives a round trip (-0 keeps its sign bit)
    assert np.array_equal(syn.round_e4m3(v[finite]), finite.astype(np.uint8))
    # ties go to the even pattern, saturation at 448
    assert syn.round_e4m3(np.array([1.0625, 1.1875, 1e6, -1e6])).tolist() == [0x38, 0x3A, 0x7E, 0xFE]


def test_fp8_descale_placement():
    """Only the product descale_q * descale_k * scale enters the scores, and
    the output is linear in descale_v (FAQ Q20's descale of Q/K/V)."""
    rng = np.random.default_rng(12)
    q8, k8, v8 = (rng.standard_normal(sh) for sh in ((1, 6, 2, 8), (1, 9, 1, 8), (1, 9, 1, 8)))
    o1, l1 = ref.fp8_forward(q8, k8, v8, 2.0, 0.25, 1.0, 0.3, causal=True)
    o2, l2 = ref.fp8_forward(q8, k8, v8, 0.5, 1.0, 3.0, 0.3, causal=True)
    np.testing.assert_allclose(3.0 * o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    o3, _ = ref.forward(q8, k8, v8, 0.15, causal=True)
    np.testing.assert_allclose(o1, o3, atol=1e-12)


@pytest.mark.parametrize("kw", [dict(causal=True), dict(win_l=3, win_r=2, softcap=2.5),
                                dict(causal=True, win_l=4), dict()])
@pytest.mark.parametrize("sq,sk", [(7, 7), (5, 11), (11, 5)])
def test_forward_rows_is_dense_forward_at_samples(kw, sq, sk):
    """forward_rows (the checker of the large-shape forward parity test) must
    give exactly the dense forward's O[b, i, h] and LSE[b, h, i] for each
    (b, h, i) sample: a wrong row offset under the bottom-right mask, a
    swapped (b, h, i) order or a wrong GQA head would each fail here.  The
    dense forward is pinned by the tests above."""
    rng = np.random.default_rng(13)
    b, hq, hkv, d = 2, 6, 2, 8
    q = rng.standard_normal((b, sq, hq, d))
    k, v = rng.standard_normal((b, sk, hkv, d)), rng.standard_normal((b, sk, hkv, d))
    o, lse = ref.forward(q, k, v, 0.35, **kw)
    samples = [(int(rng.integers(b)), int(rng.integers(hq)), int(rng.integers(sq)))
               for _ in range(40)]
    samples += [(0, 0, 0), (b - 1, hq - 1, sq - 1), (1, 3, sq // 2)]
    ro, rl = ref.forward_rows(q, k, v, samples, 0.35, **kw)
    for n, (bi, h, i) in enumerate(samples):
        np.testing.assert_allclose(ro[n], o[bi, i, h], rtol=1e-13, atol=1e-14)
        if np.isneginf(lse[bi, h, i]):
            assert np.isneginf(rl[n])
        else:
            np.testing.assert_allclose(rl[n], lse[bi, h, i], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("softcap", [0.0, 3.0])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_stored_output_reading_closed_form(softcap, dt):
    """The stored-output reading of D against an independent closed form.
    With delta_i = dO_i . (O_i - round(O_i)) (O the exact output, round the
    storage rounding), using the stored O in D changes dS by P_ij delta_i, so
    the gradients move by exactly the gradient of sum_i delta_i LSE_i:
        dQ_stored - dQ_exact = d/dQ sum_i delta_i LSE_i,  same for dK,
        dV_stored = dV_exact.
    Everything on the right is computed with torch float64 autograd and
    torch's own fp16/bf16 rounding, not with the oracle."""
    torch = pytest.importorskip("torch")
    b, s, hq, hkv, d, scale = 1, 13, 4, 2, 8, 0.45
    q, k, v, do = rnd(66, b, s, hq, d), rnd(67, b, s, hkv, d), rnd(68, b, s, hkv, d), rnd(69, b, s, hq, d)
    g = hq // hkv
    tq = torch.tensor(q.transpose(0, 2, 1, 3), requires_grad=True)
    tk = torch.tensor(np.repeat(k, g, axis=2).transpose(0, 2, 1, 3), requires_grad=True)
    tv = torch.tensor(np.repeat(v, g, axis=2).transpose(0, 2, 1, 3))
    s_ = scale * tq @ tk.transpose(-1, -2)
    if softcap:
        s_ = softcap * torch.tanh(s_ / softcap)
    s_ = s_.masked_fill(~torch.ones(s, s, dtype=torch.bool).tril(), float("-inf"))
    lse = torch.logsumexp(s_, dim=-1)
    with torch.no_grad():
        o = torch.softmax(s_, dim=-1) @ tv
        o_r = o.to(torch.bfloat16 if dt == "bf16" else torch.float16).to(torch.float64)
        delta = (torch.tensor(do.transpose(0, 2, 1, 3)) * (o - o_r)).sum(-1)
    (lse * delta).sum().backward()
    corr_q = tq.grad.numpy().transpose(0, 2, 1, 3)
    corr_k = tk.grad.numpy().transpose(0, 2, 1, 3).reshape(b, s, hkv, g, d).sum(3)
    exact = ref.backward(q, k, v, do, scale, causal=True, softcap=softcap)
    got = ref.backward(q, k, v, do, scale, causal=True, softcap=softcap, stored_o=dt)
    assert np.abs(corr_q).max() > 0
    np.testing.assert_allclose(got[0] - exact[0], corr_q, rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose(got[1] - exact[1], corr_k, rtol=1e-9, atol=1e-13)
    np.testing.assert_array_equal(got[2], exact[2])
