"""fp64 oracle: exact attention written out from its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring). Section names cite the
page "FlashAttention：快速且内存高效的准确注意力机制" (cloud.tencent.com.cn).

Definitions used (the page's notation where it has one):

* Scores (section "使用示例"): S = Q·Kᵀ·softmax_scale, default scale
  1/sqrt(headdim) (section "参数说明").
* Causal mask (section "2.1：更改causal标志的行为"): aligned to the
  bottom-right corner of the Sq x Sk score matrix, so query row i may attend
  key j iff j <= i + Sk - Sq. We call c(i) = i + Sk - Sq the diagonal key of row i.
* Sliding window (sections "参数说明" and "2.3：局部（即滑动窗口）注意力"):
  window_size = (left, right), -1 meaning unbounded on that side. Reading
  taken here: the window is centred on the same diagonal c(i), keys
  j in [c(i) - left, c(i) + right], inclusive; causal=True sets right = 0.
* ALiBi (sections "参数说明" and "2.4"): bias -slope * |i - j| added to the
  score; reading taken here: the distance is measured from the diagonal,
  |c(i) - j|, which equals |i - j| when Sq == Sk, and the bias is not
  multiplied by softmax_scale.
* Masked entries are -inf (exact), not the -10000 of the page's naive
  SelfAttention. A row with no live key gives O = 0 (section "2.1", last
  sentence) and, by the logsumexp of an empty set, L = -inf.
* L is the natural-log row logsumexp of S, the only statistic the backward
  uses (sections "前向传播" and "反向传播").
* Backward: the textbook derivative of softmax with the same P
  (dV = PᵀdO, dP = dO·Vᵀ, D_i = sum_j P_ij dP_ij, dS = P∘(dP - D),
  dQ = scale·dS·K, dK = scale·dSᵀ·Q).
* Split-KV decode (section "2.2：针对推理进行优化"): each split computes
  attention over its key range; a separate step merges them. Merge used here
  is the exact logsumexp merge: L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.
* Packed sequences (section "代码解读博客：FlashSelfAttention": cu_seqlens,
  "cumulative lengths of the sequences in the batch, used to index into qkv";
  section "函数重命名": flash_attn_varlen_func): sequence b is rows
  cu[b] .. cu[b+1]-1 of a (total, H, D) tensor and is attended exactly as it
  would be alone, masks placed per sequence. lse is laid out (H, total_q).
* Paged KV cache (section "2.5：分页KV缓存" names the feature only). Reading
  taken here: caches of pages (num_pages, page_size, Hk, D); key block p of
  sequence b (keys p*page_size ..) is page block_table[b, p]; the sequence has
  seqlens_k[b] keys, and decode attends them as the dense forward would.
* KV-cache decode with in-place append and rotary embedding (section "2.2",
  flash_attn_with_kvcache "performs rotary embedding and updates the KV cache
  in place"; no formula is given). Readings taken here: new rows go to
  positions cache_seqlens[b] + s; the rotary embedding is the standard one,
  each pair (x1, x2) at frequency f and position t rotated by the caller's
  table angle, (x1 cos - x2 sin, x1 sin + x2 cos), pairs (2f, 2f+1) when
  interleaved else (f, f + r/2); new keys rotate at their cache positions and
  query row i at its diagonal position i + Sk - Sq. The cache holds bf16, so a
  key written into it is the rotated key rounded to bf16 (nearest, ties to
  even); values are copied unchanged.
* Dropout (section "参数说明": dropout_p; no generator is given). Reading taken
  here: Philox4x32-10 (Salmon et al., SC 2011) draws entry (b, h, i, j) of P as
  word j % 4 of the block at counter (j // 4, i, b * H + h, offset), key = the
  two 32-bit halves of the seed; the entry is dropped when the word is below
  floor(p * 2^32), else scaled by 1 / (1 - p). O = (P o Z) V with L unchanged.
* Key/value heads (section "代码解读博客：FlashCrossAttention", kv of shape
  (B, Sk, 2, H_k, D)): k and v may have Hk heads with H a multiple of Hk.
  Reading taken here (the page gives no mapping): query head h attends
  key/value head h // (H // Hk), consecutive groups. The gradient of a shared
  key/value head is the sum of the gradients its query heads contribute.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _window(causal: bool, window_left: int, window_right: int):
    """Return (left, right) after folding causal in; -1 = unbounded."""
    wl = int(window_left)
    wr = int(window_right)
    if causal:
        wr = 0
    return wl, wr


def live_mask(Sq: int, Sk: int, causal: bool = False, window_left: int = -1,
              window_right: int = -1) -> np.ndarray:
    """Boolean (Sq, Sk) matrix: True where query row i may attend key j.

    Bottom-right alignment (section "2.1：更改causal标志的行为"): c(i) = i + Sk - Sq.
    """
    wl, wr = _window(causal, window_left, window_right)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    c = i + (Sk - Sq)
    live = np.ones((Sq, Sk), dtype=bool)
    if wr >= 0:
        live &= j <= c + wr
    if wl >= 0:
        live &= j >= c - wl
    return live


def alibi_bias(Sq: int, Sk: int, slope: float) -> np.ndarray:
    """(Sq, Sk) fp64 ALiBi bias -slope * |c(i) - j| (section "参数说明", alibi_slopes)."""
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    c = i + (Sk - Sq)
    return -float(slope) * np.abs(c - j).astype(np.float64)


def _scores(qh, kh, scale, causal, wl, wr, slope, rows=None, Sq=None):
    """Materialise S for one head: scale * q k^T (+ bias), -inf where masked.

    ``rows`` (optional) selects query rows; each row is independent.
    """
    Sq_full = qh.shape[0] if Sq is None else Sq
    Sk = kh.shape[0]
    live = live_mask(Sq_full, Sk, causal, wl, wr)
    if rows is not None:
        live = live[rows]
        qh = qh[rows]
    s = (qh @ kh.T) * scale
    if slope is not None:
        b = alibi_bias(Sq_full, Sk, slope)
        if rows is not None:
            b = b[rows]
        s = s + b
    s = np.where(live, s, NEG_INF)
    return s, live


def _softmax_rows(s: np.ndarray):
    """Row softmax and natural-log logsumexp; a row that is all -inf gives P = 0, L = -inf."""
    m = np.max(s, axis=1, keepdims=True)
    any_live = np.isfinite(m)
    m_safe = np.where(any_live, m, 0.0)
    e = np.exp(s - m_safe)  # exp(-inf) = 0 on masked entries
    z = np.sum(e, axis=1, keepdims=True)
    p = np.where(any_live, e / np.where(any_live, z, 1.0), 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(any_live, m_safe + np.log(np.where(any_live, z, 1.0)), NEG_INF)
    return p, lse[:, 0]


def head_fwd(qh, kh, vh, scale, causal=False, window_left=-1, window_right=-1,
             slope=None, rows=None, return_p=False):
    """Forward for one (batch, head): q (Sq,D), k/v (Sk,D) fp64 -> O (Sq,D), L (Sq,).

    O_i = sum_j P_ij V_j with P = softmax(S) row-wise (section "使用示例");
    rows with no live key give O = 0 and L = -inf (section "2.1").
    """
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    s, _ = _scores(qh, kh, scale, causal, window_left, window_right, slope, rows=rows)
    p, lse = _softmax_rows(s)
    o = p @ vh
    if return_p:
        return o, lse, s, p
    return o, lse


def head_bwd(doh, qh, kh, vh, scale, causal=False, window_left=-1, window_right=-1,
             slope=None, row_block=None):
    """Backward for one (batch, head) by the textbook softmax derivative.

    P is recomputed from the definition (the page's backward keeps only L,
    section "反向传播"; here P is simply rebuilt from S). ``row_block``
    bounds memory on long heads: dK and dV are then sums over row blocks of
    the same products.
    """
    doh = np.asarray(doh, dtype=np.float64)
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    Sq = qh.shape[0]
    rb = Sq if row_block is None else int(row_block)
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    for r0 in range(0, Sq, rb):
        rows = np.arange(r0, min(Sq, r0 + rb))
        s, _ = _scores(qh, kh, scale, causal, window_left, window_right, slope,
                       rows=rows, Sq=Sq)
        p, _ = _softmax_rows(s)
        do_r = doh[rows]
        dv += p.T @ do_r
        dp = do_r @ vh.T
        d = np.sum(p * dp, axis=1, keepdims=True)
        ds = p * (dp - d)
        dq[rows] = scale * (ds @ kh)
        dk += scale * (ds.T @ qh[rows])
    return dq, dk, dv


def head_partial(qh, kh, vh, key_lo, key_hi, scale, causal=False, window_left=-1,
                 window_right=-1, slope=None):
    """One split of split-KV decode (section "2.2"): attention of q over keys [key_lo, key_hi).

    The mask and bias use the global key index. Returns the split's own
    normalised output O_s (Sq,D) and logsumexp L_s (Sq,); a split with no
    live key gives O_s = 0, L_s = -inf.
    """
    qh = np.asarray(qh, dtype=np.float64)
    Sq = qh.shape[0]
    Sk = kh.shape[0]
    s, _ = _scores(qh, np.asarray(kh, dtype=np.float64), scale, causal, window_left,
                   window_right, slope, Sq=Sq)
    keep = np.zeros(Sk, dtype=bool)
    keep[key_lo:key_hi] = True
    s = np.where(keep[None, :], s, NEG_INF)
    p, lse = _softmax_rows(s)
    return p @ np.asarray(vh, dtype=np.float64), lse


def combine_partials(o_parts, l_parts):
    """Exact merge of split results: L = log sum_s exp(L_s); O = sum_s exp(L_s - L) O_s.

    o_parts: (n, Sq, D); l_parts: (n, Sq). Splits with L_s = -inf weigh 0;
    if every split is empty the row gives O = 0, L = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    m = np.max(l_parts, axis=0)
    any_live = np.isfinite(m)
    m_safe = np.where(any_live, m, 0.0)
    w = np.exp(l_parts - m_safe[None, :])
    z = np.sum(w, axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(any_live, m_safe + np.log(np.where(any_live, z, 1.0)), NEG_INF)
    wn = np.where(any_live[None, :], w / np.where(any_live, z, 1.0)[None, :], 0.0)
    o = np.einsum("sq,sqd->qd", wn, o_parts)
    return o, lse


def _slope_for(alibi_slopes, b, h):
    if alibi_slopes is None:
        return None
    a = np.asarray(alibi_slopes, dtype=np.float64)
    return float(a[h]) if a.ndim == 1 else float(a[b, h])


def _default_scale(D, scale):
    return 1.0 / math.sqrt(D) if (scale is None or scale <= 0) else float(scale)


def kv_head(h: int, H: int, Hk: int) -> int:
    """Key/value head read by query head h when k/v have Hk heads (H a multiple of Hk)."""
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"query heads {H} are not a multiple of key/value heads {Hk}")
    return h // (H // Hk)


def attention_fwd(q, k, v, scale=None, causal=False, window=(-1, -1), alibi_slopes=None):
    """Batched forward: q (B,Sq,H,D), k/v (B,Sk,Hk,D) -> O (B,Sq,H,D), L (B,H,Sq), all fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    Hk = k.shape[2]
    sc = _default_scale(D, scale)
    o = np.zeros_like(q)
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hk)
            o[b, :, h, :], lse[b, h] = head_fwd(
                q[b, :, h, :], k[b, :, g, :], v[b, :, g, :], sc, causal, window[0],
                window[1], _slope_for(alibi_slopes, b, h))
    return o, lse


def attention_bwd(dout, q, k, v, scale=None, causal=False, window=(-1, -1), alibi_slopes=None):
    """Batched backward: returns dQ, dK, dV in the layouts of q, k, v (fp64). With k/v of
    Hk < H heads, dK and dV of a key/value head sum the contributions of its query heads."""
    dout = np.asarray(dout, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    Hk = k.shape[2]
    sc = _default_scale(D, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hk)
            dqh, dkh, dvh = head_bwd(
                dout[b, :, h, :], q[b, :, h, :], k[b, :, g, :], v[b, :, g, :], sc, causal,
                window[0], window[1], _slope_for(alibi_slopes, b, h))
            dq[b, :, h, :] = dqh
            dk[b, :, g, :] += dkh
            dv[b, :, g, :] += dvh
    return dq, dk, dv


def decode_splitkv(q, k, v, num_splits, scale=None, causal=False, window=(-1, -1),
                   alibi_slopes=None):
    """Split-KV decode as the page describes it (section "2.2"): per (b,h), the
    key range is cut into ``num_splits`` contiguous chunks, each chunk's
    attention is computed on its own, then the chunks are merged.

    Returns O (B,Sq,H,D), L (B,H,Sq). By the exactness of the merge this equals
    ``attention_fwd``; the tests check that.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    sc = _default_scale(D, scale)
    bounds = [(Sk * s) // num_splits for s in range(num_splits + 1)]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hk)
            kh = np.asarray(k[b, :, g, :], dtype=np.float64)
            vh = np.asarray(v[b, :, g, :], dtype=np.float64)
            parts = [head_partial(q[b, :, h, :], kh, vh, bounds[s], bounds[s + 1], sc, causal,
                                  window[0], window[1], _slope_for(alibi_slopes, b, h))
                     for s in range(num_splits)]
            o[b, :, h, :], lse[b, h] = combine_partials([p[0] for p in parts],
                                                        [p[1] for p in parts])
    return o, lse


def _sequences(cu_seqlens_q, cu_seqlens_k):
    cq = [int(x) for x in np.asarray(cu_seqlens_q).ravel()]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).ravel()]
    if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0 or any(b < a for a, b in zip(cq, cq[1:])) or \
            any(b < a for a, b in zip(ck, ck[1:])):
        raise ValueError("cu_seqlens must be non-decreasing (B + 1,) arrays starting at 0")
    return [(cq[b], cq[b + 1], ck[b], ck[b + 1]) for b in range(len(cq) - 1)]


def attention_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale=None, causal=False, window=(-1, -1),
                         alibi_slopes=None):
    """Packed forward: q (total_q,H,D), k/v (total_k,Hk,D) -> O (total_q,H,D), L (H,total_q), fp64.
    Each sequence is the one-batch attention_fwd of its own rows (slopes of its index b)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    total_q, H, D = q.shape
    o = np.zeros_like(q)
    lse = np.full((H, total_q), -np.inf)
    for b, (q0, q1, k0, k1) in enumerate(_sequences(cu_seqlens_q, cu_seqlens_k)):
        if q1 == q0:
            continue
        slopes = None if alibi_slopes is None else _batch_slopes(alibi_slopes, b)
        if k1 == k0:  # no key at all: every row has no live key
            continue
        ob, lb = attention_fwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale, causal, window, slopes)
        o[q0:q1] = ob[0]
        lse[:, q0:q1] = lb[0]
    return o, lse


def attention_bwd_varlen(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, scale=None, causal=False, window=(-1, -1),
                         alibi_slopes=None):
    """Packed backward: dQ (total_q,H,D), dK, dV (total_k,Hk,D), fp64, sequence by sequence."""
    dout = np.asarray(dout, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, (q0, q1, k0, k1) in enumerate(_sequences(cu_seqlens_q, cu_seqlens_k)):
        if q1 == q0 or k1 == k0:
            continue
        slopes = None if alibi_slopes is None else _batch_slopes(alibi_slopes, b)
        g = attention_bwd(dout[None, q0:q1], q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale, causal,
                          window, slopes)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


def _batch_slopes(alibi_slopes, b):
    a = np.asarray(alibi_slopes, dtype=np.float64)
    return a if a.ndim == 1 else a[b]


def decode_paged(q, k_pages, v_pages, block_table, seqlens_k, scale=None, causal=False, window=(-1, -1),
                 alibi_slopes=None):
    """Decode over a paged cache: q (B,Sq,H,D), pages (num_pages,page_size,Hk,D), block_table (B,max_pages),
    seqlens_k (B,) -> O (B,Sq,H,D), L (B,H,Sq) fp64. Each sequence's keys are gathered page by page and
    attended as attention_fwd does; a sequence without keys gives O = 0, L = -inf."""
    q = np.asarray(q, dtype=np.float64)
    B, Sq, H, D = q.shape
    page_size = k_pages.shape[1]
    table = np.asarray(block_table)
    o = np.zeros_like(q)
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        n = int(seqlens_k[b])
        if n == 0:
            continue
        pages = [int(table[b, p]) for p in range((n + page_size - 1) // page_size)]
        kb = np.concatenate([np.asarray(k_pages[pg], dtype=np.float64) for pg in pages])[:n]
        vb = np.concatenate([np.asarray(v_pages[pg], dtype=np.float64) for pg in pages])[:n]
        slopes = None if alibi_slopes is None else _batch_slopes(alibi_slopes, b)
        ob, lb = attention_fwd(q[b:b + 1], kb[None], vb[None], scale, causal, window, slopes)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64: x goes through
    fp32, whose upper 16 bits are kept after adding half of the dropped range."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def rotary(x, positions, cos_tab, sin_tab, interleaved=False):
    """Rotate rows x (n, ..., D) at positions (n,) with tables (len, r/2); dims >= r unchanged.
    Positions are clamped into the tables."""
    x = np.array(x, dtype=np.float64, copy=True)
    cos_tab = np.asarray(cos_tab, dtype=np.float64)
    sin_tab = np.asarray(sin_tab, dtype=np.float64)
    half = cos_tab.shape[1]
    for n, t in enumerate(positions):
        t = min(max(int(t), 0), cos_tab.shape[0] - 1)
        for f in range(half):
            i1, i2 = (2 * f, 2 * f + 1) if interleaved else (f, f + half)
            c, s_ = cos_tab[t, f], sin_tab[t, f]
            x1, x2 = x[n, ..., i1].copy(), x[n, ..., i2].copy()
            x[n, ..., i1] = x1 * c - x2 * s_
            x[n, ..., i2] = x1 * s_ + x2 * c
    return x


def decode_kvcache(q, k_cache, v_cache, cache_seqlens, k_new=None, v_new=None, rotary_cos=None, rotary_sin=None,
                   interleaved=False, block_table=None, scale=None, causal=False, window=(-1, -1),
                   alibi_slopes=None):
    """Decode step on a cache: returns O (B,Sq,H,D), L (B,H,Sq) and the caches after the append (fp64).
    Dense caches are (B, rows, Hk, D); with block_table (B, max_pages) they are pages
    (num_pages, page_size, Hk, D). Rows past the capacity or on a page outside the cache are not written."""
    q = np.asarray(q, dtype=np.float64)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    B, Sq, H, D = q.shape
    seq = [int(x) for x in np.asarray(cache_seqlens)]
    rot = rotary_cos is not None
    if block_table is not None:
        table = np.asarray(block_table)
        page_size = kc.shape[1]
        cap = table.shape[1] * page_size

        def slot(b, pos):
            page = int(table[b, pos // page_size])
            return None if not 0 <= page < kc.shape[0] else (page, pos % page_size)
    else:
        cap = kc.shape[1]

        def slot(b, pos):
            return (b, pos)
    S_new = 0 if k_new is None else k_new.shape[1]
    for b in range(B):
        for s_ in range(S_new):
            pos = seq[b] + s_
            if not 0 <= pos < cap:
                continue
            where = slot(b, pos)
            if where is None:
                continue
            kr = np.asarray(k_new[b, s_:s_ + 1], dtype=np.float64)
            if rot:
                kr = round_bf16(rotary(kr, [pos], rotary_cos, rotary_sin, interleaved))
            kc[where] = kr[0]
            vc[where] = np.asarray(v_new[b, s_], dtype=np.float64)
    o = np.zeros_like(q)
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        n = max(0, min(seq[b] + S_new, cap))
        if n == 0:
            continue
        kb = np.stack([kc[slot(b, j)] if slot(b, j) is not None else np.zeros(kc.shape[2:]) for j in range(n)])
        vb = np.stack([vc[slot(b, j)] if slot(b, j) is not None else np.zeros(vc.shape[2:]) for j in range(n)])
        qb = q[b]
        if rot:
            qb = rotary(qb, [i + n - Sq for i in range(Sq)], rotary_cos, rotary_sin, interleaved)
        slopes = None if alibi_slopes is None else _batch_slopes(alibi_slopes, b)
        ob, lb = attention_fwd(qb[None], kb[None], vb[None], scale, causal, window, slopes)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse, kc, vc


PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57   # Philox4x32 multipliers (Salmon et al., SC 2011)
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85   # key increments between rounds


def philox4x32_10(x0, x1, x2, x3, k0, k1):
    """Philox4x32 with 10 rounds on arrays of 32-bit counters; returns the four output words (uint64 arrays
    holding 32-bit values). One round: hi0:lo0 = M0*x0, hi1:lo1 = M1*x2, then
    (x0, x1, x2, x3) <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0), then the key is bumped."""
    mask = np.uint64(0xFFFFFFFF)
    x = [np.asarray(t, dtype=np.uint64) & mask for t in (x0, x1, x2, x3)]
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * x[0]
        p1 = np.uint64(PHILOX_M1) * x[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        x = [hi1 ^ x[1] ^ k0, lo1, hi0 ^ x[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(PHILOX_W0)) & mask
        k1 = (k1 + np.uint64(PHILOX_W1)) & mask
    return x


def dropout_threshold(p):
    """Words below this are dropped: floor(p * 2^32) with p taken as fp32, at most 2^32 - 1."""
    t = int(math.floor(float(np.float32(p)) * 4294967296.0))
    return min(t, 0xFFFFFFFF)


def dropout_scale_matrix(Sq, Sk, bh, p, seed, offset):
    """Z (Sq, Sk): 1 / (1 - p) where entry (i, j) of head bh = b * H + h is kept, else 0."""
    nj4 = (Sk + 3) // 4
    j4, i = np.meshgrid(np.arange(nj4), np.arange(Sq))
    words = philox4x32_10(j4.ravel(), i.ravel(), np.full(j4.size, bh), np.full(j4.size, offset),
                          int(seed) & 0xFFFFFFFF, int(seed) >> 32)
    w = np.stack(words, axis=-1).reshape(Sq, nj4 * 4)[:, :Sk]
    keep = w >= np.uint64(dropout_threshold(p))
    return np.where(keep, 1.0 / (1.0 - float(np.float32(p))), 0.0)


def attention_fwd_dropout(q, k, v, p, seed, offset=0, scale=None, causal=False, window=(-1, -1), alibi_slopes=None):
    """Forward with dropout: O = (P o Z) V per (b, h), L as attention_fwd. Layouts as attention_fwd."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    sc = _default_scale(D, scale)
    o = np.zeros_like(q)
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hk)
            s_, _ = _scores(q[b, :, h, :], k[b, :, g, :], sc, causal, window[0], window[1],
                            _slope_for(alibi_slopes, b, h))
            prob, lse[b, h] = _softmax_rows(s_)
            z = dropout_scale_matrix(Sq, Sk, b * H + h, p, seed, offset)
            o[b, :, h, :] = (prob * z) @ v[b, :, g, :]
    return o, lse


def attention_bwd_dropout(dout, q, k, v, p, seed, offset=0, scale=None, causal=False, window=(-1, -1),
                          alibi_slopes=None):
    """Backward with dropout: dV = (P o Z)^T dO, dP = Z o (dO V^T), D_i = sum_j P_ij dP_ij,
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q (summed over a key/value head's query heads)."""
    dout = np.asarray(dout, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    sc = _default_scale(D, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hk)
            s_, _ = _scores(q[b, :, h, :], k[b, :, g, :], sc, causal, window[0], window[1],
                            _slope_for(alibi_slopes, b, h))
            prob, _ = _softmax_rows(s_)
            z = dropout_scale_matrix(Sq, Sk, b * H + h, p, seed, offset)
            do_h = dout[b, :, h, :]
            dv[b, :, g, :] += (prob * z).T @ do_h
            dp = z * (do_h @ v[b, :, g, :].T)
            dvec = np.sum(prob * dp, axis=1, keepdims=True)
            ds = prob * (dp - dvec)
            dq[b, :, h, :] = sc * ds @ k[b, :, g, :]
            dk[b, :, g, :] += sc * ds.T @ q[b, :, h, :]
    return dq, dk, dv
