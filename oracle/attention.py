"""Float64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library: the two
meet only through the seeded inputs of ``exact_attention_41_gb300.synthetic``.

What it computes is the plain definition, evaluated in float64 with the full
score matrix S and probability matrix P materialised (no tiling, no online
softmax, no fusion):

* Standard attention S = Q K^T * scale, P = softmax(S), O = P V
  -- "flash_attn FlashAttention完整说明" (kwkr.cn), section 一 基础定义.
* The forward keeps O and the softmax statistics (m, l); we report them as
  LSE = m + ln(l) -- same page, section 二.2 重计算 Recomputation.
* Softcap is applied to the scaled score before masking, order
  QK^T -> softcap(tanh) -> mask -> softmax -> PV -- Inference Cookbook FAQ
  ("常见问题") Q22.  Reading: s <- c * tanh(s / c), c <= 0 meaning off.
* Causal masks align to the bottom-right corner when seqlen_q != seqlen_k
  -- Inference Cookbook FAQ Q6.
* Sliding window (left, right): query i sees keys in [i - left, i + right]
  (inclusive), right = 0 being causal, -1 meaning unbounded -- Inference
  Cookbook FAQ Q21; with seqlen_q != seqlen_k the window is shifted by the
  same bottom-right offset (sk - sq) as the causal mask.
* GQA: query head h reads KV head floor(h * hkv / hq) (contiguous groups).
* Varlen: each packed sequence of cu_seqlens is an independent problem
  -- Inference Cookbook FAQ Q8.
* KV cache: the keys of batch entry b are cache[0:cache_seqlens[b]] followed
  by the s_new appended rows; the appended rows are written into the cache at
  positions cache_seqlens[b] + t, pages addressed through block_table;
  cache_seqlens itself is not changed -- Inference Cookbook FAQ Q17, Q18.
* Backward: the textbook softmax Jacobian applied to the recomputed P
  (FlashAttention完整说明 section 二.2 says only that S and P are recomputed
  from Q, K, V in the backward; the gradient itself is plain calculus).

Rows with no visible key give O = 0 and LSE = -inf (an empty sum), and
contribute nothing to the gradients.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def visible(row_ids, sq: int, sk: int, causal: bool, win_l: int, win_r: int) -> np.ndarray:
    """Boolean mask (len(row_ids), sk): may query row i attend to key j?

    Bottom-right alignment (Inference Cookbook FAQ Q6): query i sits at key
    position i + (sk - sq).  Window bounds from FAQ Q21; causal forces the
    right bound to 0.
    """
    i = np.asarray(row_ids, dtype=np.int64)[:, None]
    j = np.arange(sk, dtype=np.int64)[None, :]
    pos = i + (sk - sq)
    right = 0 if causal else win_r
    ok = np.ones((i.shape[0], sk), dtype=bool)
    if right >= 0:
        ok &= j <= pos + right
    if win_l >= 0:
        ok &= j >= pos - win_l
    return ok


def _scores(qh, kh, scale, softcap):
    """Scaled (and optionally soft-capped) scores plus the raw scaled scores."""
    s_raw = scale * (qh @ kh.T)
    if softcap > 0:
        return softcap * np.tanh(s_raw / softcap), s_raw
    return s_raw, s_raw


def _softmax_rows(s, mask):
    """Row softmax over the visible entries; returns (P, LSE)."""
    s = np.where(mask, s, NEG_INF)
    nonempty = mask.any(axis=1)
    m = np.where(nonempty, s.max(axis=1, initial=NEG_INF), 0.0)
    e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    ell = e.sum(axis=1)
    p = np.where(nonempty[:, None], e / np.where(nonempty, ell, 1.0)[:, None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(nonempty, m + np.log(np.where(nonempty, ell, 1.0)), NEG_INF)
    return p, lse


def head_forward(qh, kh, vh, row_ids, sq, sk, scale, causal=False, win_l=-1, win_r=-1,
                 softcap=0.0, return_probs=False):
    """One (batch, head) problem for the query rows ``row_ids``.

    qh: (len(row_ids), d) float64, the query rows; kh, vh: (sk, d) float64.
    Returns O (len(row_ids), d), LSE (len(row_ids),) [, P].
    """
    s, _ = _scores(qh, kh, scale, softcap)
    mask = visible(row_ids, sq, sk, causal, win_l, win_r)
    p, lse = _softmax_rows(s, mask)
    o = p @ vh
    if return_probs:
        return o, lse, p
    return o, lse


def kv_head_of(h: int, hq: int, hkv: int) -> int:
    """GQA head map: contiguous groups of hq/hkv query heads share one KV head."""
    if hq % hkv:
        raise ValueError("hq must be a multiple of hkv")
    return h // (hq // hkv)


def forward(q, k, v, scale, causal=False, win_l=-1, win_r=-1, softcap=0.0):
    """Dense attention.  q (b,sq,hq,d), k/v (b,sk,hkv,d) float64.

    Returns O (b,sq,hq,d) float64 and LSE (b,hq,sq) float64.
    """
    b, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    o = np.zeros((b, sq, hq, d))
    lse = np.zeros((b, hq, sq))
    rows = np.arange(sq)
    for bi in range(b):
        for h in range(hq):
            kv = kv_head_of(h, hq, hkv)
            o[bi, :, h], lse[bi, h] = head_forward(
                q[bi, :, h], k[bi, :, kv], v[bi, :, kv], rows, sq, sk, scale,
                causal, win_l, win_r, softcap)
    return o, lse


def forward_rows(q, k, v, samples, scale, causal=False, win_l=-1, win_r=-1, softcap=0.0):
    """O and LSE for selected (batch, head, row) triples only.

    samples: iterable of (b, h, i).  Returns O (n, d), LSE (n,).  Each row is
    the definition evaluated for that row alone (rows are independent).
    """
    b, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    samples = list(samples)
    o = np.zeros((len(samples), d))
    lse = np.zeros(len(samples))
    for n, (bi, h, i) in enumerate(samples):
        kv = kv_head_of(h, hq, hkv)
        oo, ll = head_forward(q[bi, i:i + 1, h], k[bi, :, kv], v[bi, :, kv], [i], sq, sk,
                              scale, causal, win_l, win_r, softcap)
        o[n], lse[n] = oo[0], ll[0]
    return o, lse


def probs(q, k, scale, causal=False, win_l=-1, win_r=-1, softcap=0.0):
    """The attention probability matrix P (b, hq, sq, sk) of a dense forward:
    what Inference Cookbook FAQ Q9's return_attn_probs hands back (O(N^2)
    memory, for debugging).  Row i is the softmax of the scaled, soft-capped
    scores over the keys it may see, 0 elsewhere; rows that see no key are 0.
    q (b,sq,hq,d), k (b,sk,hkv,d) float64.
    """
    b, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    p = np.zeros((b, hq, sq, sk))
    rows = np.arange(sq)
    mask = visible(rows, sq, sk, causal, win_l, win_r)
    for bi in range(b):
        for h in range(hq):
            s, _ = _scores(q[bi, :, h], k[bi, :, kv_head_of(h, hq, hkv)], scale, softcap)
            p[bi, h], _ = _softmax_rows(s, mask)
    return p


def fp8_forward(q8, k8, v8, descale_q, descale_k, descale_v, scale, causal=False, win_l=-1,
                win_r=-1, softcap=0.0):
    """FP8 forward (Inference Cookbook FAQ Q20: FP8 tensors stand for their
    values times per-tensor descale factors; the output is BF16).  q8, k8, v8
    are the E4M3 values widened to float64; the definition is the ordinary
    forward of q8*descale_q, k8*descale_k, v8*descale_v.  Returns O, LSE
    (float64; the library rounds O to bf16)."""
    return forward(q8 * descale_q, k8 * descale_k, v8 * descale_v, scale, causal, win_l, win_r,
                   softcap)


def round_to(x, dtype):
    """Round float64 values to fp16 or bf16 (round to nearest even), as the
    forward's stored output is; returns float64."""
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        f = x.astype(np.float32)
        u = f.view(np.uint32).astype(np.uint64)
        u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
        return u.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def head_backward(qh, kh, vh, doh, sq, sk, scale, causal=False, win_l=-1, win_r=-1,
                  softcap=0.0, stored_o=None):
    """Gradients of one (batch, head) problem.  Returns dq (sq,d), dk (sk,d), dv (sk,d).

    P is recomputed from Q and K (FlashAttention完整说明 section 二.2); then
      dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
      dS = P * (dP - D)  [* (1 - tanh(s_raw/c)^2) with softcap c],
      dQ = scale * dS K,  dK = scale * dS^T Q.

    stored_o: None gives the exact gradient.  "f16"/"bf16" instead takes
    D_i = dO_i . O_i with O_i the forward output rounded to that storage type,
    i.e. the output the forward saves (same page, section 二.2: the forward
    keeps only O and the softmax statistics for the backward).  The two
    differ only by that rounding; D_i = dO_i . O_i holds exactly since the
    rows of P sum to one.
    """
    s, s_raw = _scores(qh, kh, scale, softcap)
    mask = visible(np.arange(sq), sq, sk, causal, win_l, win_r)
    p, _ = _softmax_rows(s, mask)
    dv = p.T @ doh
    dp = doh @ vh.T
    if stored_o is None:
        dsum = (p * dp).sum(axis=1)
    else:
        dsum = (doh * round_to(p @ vh, stored_o)).sum(axis=1)
    ds = p * (dp - dsum[:, None])
    if softcap > 0:
        ds = ds * (1.0 - np.tanh(s_raw / softcap) ** 2)
    dq = scale * (ds @ kh)
    dk = scale * (ds.T @ qh)
    return dq, dk, dv


def backward_group(q, k, v, dout, bi, kv, scale, causal=False, win_l=-1, win_r=-1,
                   softcap=0.0, stored_o=None):
    """Gradients restricted to one (batch, KV head) group.

    Returns dq (sq, g, d) for the group's query heads h = kv*g .. kv*g+g-1,
    and dk, dv (sk, d) for that KV head (summed over the group).
    """
    _, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    g = hq // hkv
    dq = np.zeros((sq, g, d))
    dk = np.zeros((sk, d))
    dv = np.zeros((sk, d))
    for t in range(g):
        h = kv * g + t
        a, bk, bv = head_backward(q[bi, :, h], k[bi, :, kv], v[bi, :, kv], dout[bi, :, h],
                                  sq, sk, scale, causal, win_l, win_r, softcap, stored_o)
        dq[:, t] = a
        dk += bk
        dv += bv
    return dq, dk, dv


def backward(q, k, v, dout, scale, causal=False, win_l=-1, win_r=-1, softcap=0.0,
             stored_o=None):
    """Dense gradients dq (b,sq,hq,d), dk/dv (b,sk,hkv,d) in float64."""
    b, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    g = hq // hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for bi in range(b):
        for kv in range(hkv):
            a, bk, bv = backward_group(q, k, v, dout, bi, kv, scale, causal, win_l, win_r,
                                       softcap, stored_o)
            dq[bi, :, kv * g:(kv + 1) * g] = a
            dk[bi, :, kv] = bk
            dv[bi, :, kv] = bv
    return dq, dk, dv


def varlen_forward(q, k, v, cu_q, cu_k, scale, causal=False, win_l=-1, win_r=-1,
                   softcap=0.0, seqs=None):
    """Packed varlen attention (Inference Cookbook FAQ Q8).

    q (Tq,hq,d), k/v (Tk,hkv,d); sequence i owns rows cu_q[i]:cu_q[i+1] and
    keys cu_k[i]:cu_k[i+1].  Returns O (Tq,hq,d) and LSE (hq,Tq); rows of
    sequences not listed in ``seqs`` (default: all) are left as NaN.
    """
    tq, hq, d = q.shape
    o = np.full((tq, hq, d), np.nan)
    lse = np.full((hq, tq), np.nan)
    nseq = len(cu_q) - 1
    for i in (range(nseq) if seqs is None else seqs):
        q0, q1, k0, k1 = int(cu_q[i]), int(cu_q[i + 1]), int(cu_k[i]), int(cu_k[i + 1])
        oo, ll = forward(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale, causal,
                         win_l, win_r, softcap)
        o[q0:q1] = oo[0]
        lse[:, q0:q1] = ll[0]
    return o, lse


def varlen_backward(q, k, v, dout, cu_q, cu_k, scale, causal=False, win_l=-1, win_r=-1,
                    softcap=0.0, seqs=None, stored_o=None):
    """Packed varlen gradients; sequences not in ``seqs`` are left as NaN."""
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    nseq = len(cu_q) - 1
    for i in (range(nseq) if seqs is None else seqs):
        q0, q1, k0, k1 = int(cu_q[i]), int(cu_q[i + 1]), int(cu_k[i]), int(cu_k[i + 1])
        a, bk, bv = backward(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1],
                             dout[None, q0:q1], scale, causal, win_l, win_r, softcap, stored_o)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = a[0], bk[0], bv[0]
    return dq, dk, dv


def cache_positions(b: int, n: int, block_table, page_size: int):
    """(page, slot) of logical positions 0..n-1 of batch entry b.

    Paged cache (Inference Cookbook FAQ Q18): position t lives in page
    block_table[b, t // page_size] at slot t % page_size.  With no block
    table the cache is (batch, capacity, hkv, d) and the "page" is b.
    """
    t = np.arange(n)
    if block_table is None:
        return np.full(n, b), t
    return np.asarray(block_table)[b, t // page_size], t % page_size


def kvcache_forward(q, k_cache, v_cache, cache_seqlens, scale, k_new=None, v_new=None,
                    block_table=None, page_size=0, causal=False, win_l=-1, win_r=-1,
                    softcap=0.0, batches=None):
    """Decode attention against a (paged) KV cache with optional append.

    q (b,sq,hq,d); k_cache/v_cache (num_pages,page_size,hkv,d) when
    block_table is given, else (b,capacity,hkv,d); k_new/v_new (b,s_new,hkv,d)
    or None.  Returns O (b,sq,hq,d), LSE (b,hq,sq) and the caches after the
    append (copies; the inputs are not modified).  cache_seqlens is read only
    (Inference Cookbook FAQ Q17).  Batch entries not in ``batches`` are NaN.
    """
    b, sq, hq, d = q.shape
    hkv = k_cache.shape[2]
    s_new = 0 if k_new is None else k_new.shape[1]
    kc, vc = k_cache.copy(), v_cache.copy()
    o = np.full((b, sq, hq, d), np.nan)
    lse = np.full((b, hq, sq), np.nan)
    for bi in (range(b) if batches is None else batches):
        old = int(cache_seqlens[bi])
        sk = old + s_new
        pg, sl = cache_positions(bi, sk, block_table, page_size)
        if s_new:
            kc[pg[old:], sl[old:]] = k_new[bi]
            vc[pg[old:], sl[old:]] = v_new[bi]
        kseq = kc[pg, sl]  # (sk, hkv, d)
        vseq = vc[pg, sl]
        oo, ll = forward(q[bi:bi + 1], kseq[None], vseq[None], scale, causal, win_l, win_r,
                         softcap)
        o[bi], lse[bi] = oo[0], ll[0]
    return o, lse, kc, vc
