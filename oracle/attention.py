"""Plain fp64 definition of (ring) softmax attention, its layouts and its gradient.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pages cited (by title and section):
  [README]   "Ring Flash Attention" README, github.com/zhuzilin/ring-flash-attention:
             the API list, the "Note that" notes and "Limits".
  [GUIJIA]   guijiagi.com, "Ring Attention：突破百万 Token 上下文的分布式注意力":
             sections "详细流程" (ring order), the ``ring_attention`` listing,
             "在线 Softmax：关键技巧" (the online-softmax update),
             "Striped Ring Attention", "Zigzag Ring Attention",
             "2. Sequence Parallelism".
  [SP]       sourcepulse.org project summary of ring-flash-attention: the
             "llama3" context-parallel variant.
  [AINEWS]   ainews.cool, ring-flash-attention long-context article,
             section "技术深度解析" (contiguous split, ring pass).
  [STRIPED]  briefgpt.xyz abstract of "Striped Attention: Faster Ring Attention
             for Causal Transformers".

Conventions (readings where the pages are silent):
  * lse is the natural log of sum_j exp(S_ij) ("softmax_lse", [README]).
  * causal means key j is allowed for query i iff j <= i in ORIGINAL token
    order, whatever layout the shards use ([GUIJIA] "Zigzag Ring Attention",
    [STRIPED]).
  * varlen: one cu_seqlens shared by q and k ([README] "Note that");
    attention is confined to each packed sequence.
  * a block with no allowed key for a row emits out = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np

LAYOUTS = ("contiguous", "zigzag", "stripe")


# --------------------------------------------------------------------------
# Layouts: which original token sits at each position of the sharded sequence
# --------------------------------------------------------------------------
def token_of_position(layout: str, n_shards: int, s: int) -> np.ndarray:
    """g[p] = original token index held at layout position p = r*L + i.

    Shards are concatenated in rank order, L = s / N tokens each.
      contiguous: shard r holds tokens [r*L, (r+1)*L)            ([AINEWS], [GUIJIA] "2. Sequence Parallelism")
      zigzag:     2N equal chunks of c = s/(2N); shard r holds chunk r then
                  chunk 2N-1-r                                     ([GUIJIA] "Zigzag Ring Attention")
      stripe:     shard r holds tokens t with t mod N == r, in order
                  (block size 1)                                   ([README] API list; [GUIJIA] "Striped Ring Attention")
    """
    N = int(n_shards)
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout!r}")
    if N < 1 or s % N:
        raise ValueError("s must be a multiple of n_shards")
    if layout == "zigzag" and s % (2 * N):
        raise ValueError("zigzag needs s to be a multiple of 2*n_shards")
    L = s // N
    g = np.empty(s, dtype=np.int64)
    for r in range(N):
        for i in range(L):
            if layout == "contiguous":
                t = r * L + i
            elif layout == "zigzag":
                c = s // (2 * N)
                t = r * c + i if i < c else (2 * N - 1 - r) * c + (i - c)
            else:
                t = i * N + r
            g[r * L + i] = t
    return g


def varlen_token_of_position(layout: str, n_shards: int, cu_seqlens) -> np.ndarray:
    """g[p] for one packed buffer of total = cu[-1] tokens split into N shards.

      contiguous: shards are contiguous slices of the packed buffer (total / N
                  tokens each; sequences may straddle shards): g[p] = p
                  ([README] API list, "the varlen versions only support passing
                  one cu_seqlens").
      zigzag:     the zigzag split applied to every sequence: sequence k
                  (L_k = cu[k+1] - cu[k] tokens, a multiple of 2N) is cut into
                  2N chunks of c_k = L_k / (2N); shard r holds, for k = 0, 1, ...
                  in turn, chunk r then chunk 2N-1-r of sequence k
                  ([README] API list, zigzag_ring_flash_attn_varlen_func;
                  [GUIJIA] "Zigzag Ring Attention").
    """
    N = int(n_shards)
    cu = [int(c) for c in cu_seqlens]
    total = cu[-1]
    if N < 1 or total % N:
        raise ValueError("the packed length must be a multiple of n_shards")
    if layout == "contiguous":
        return np.arange(total, dtype=np.int64)
    if layout != "zigzag":
        raise ValueError(f"varlen supports the contiguous and zigzag layouts, not {layout!r}")
    lens = [cu[k + 1] - cu[k] for k in range(len(cu) - 1)]
    if any(n % (2 * N) for n in lens):
        raise ValueError("zigzag varlen needs every sequence length to be a multiple of 2*n_shards")
    g = []
    for r in range(N):
        for k, n in enumerate(lens):
            c = n // (2 * N)
            g.extend(cu[k] + r * c + o for o in range(c))
            g.extend(cu[k] + (2 * N - 1 - r) * c + o for o in range(c))
    return np.asarray(g, dtype=np.int64)


def _positions(layout, n_shards, s, cu_seqlens):
    if cu_seqlens is None:
        return token_of_position(layout, n_shards, s)
    g = varlen_token_of_position(layout, n_shards, cu_seqlens)
    if len(g) != s:
        raise ValueError("cu_seqlens does not cover the sequence axis")
    return g


def permute(x, layout: str, n_shards: int, axis: int = -2, cu_seqlens=None):
    """Original order -> layout order: y[..., p, :] = x[..., g[p], :]."""
    x = np.asarray(x)
    g = _positions(layout, n_shards, x.shape[axis], cu_seqlens)
    return np.take(x, g, axis=axis)


def unpermute(y, layout: str, n_shards: int, axis: int = -2, cu_seqlens=None):
    """Layout order -> original order: x[..., g[p], :] = y[..., p, :]."""
    y = np.asarray(y)
    g = _positions(layout, n_shards, y.shape[axis], cu_seqlens)
    x = np.empty_like(y)
    idx = [slice(None)] * y.ndim
    idx[axis] = g
    x[tuple(idx)] = y
    return x


def segment_ids(cu_seqlens, s: int) -> np.ndarray:
    """seg[t] = k such that cu[k] <= t < cu[k+1] (one cu_seqlens, [README] "Note that")."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    seg = np.empty(s, dtype=np.int64)
    for k in range(len(cu) - 1):
        seg[cu[k]:cu[k + 1]] = k
    return seg


def _allowed(gq, gk, causal, segq, segk):
    """Mask of allowed (query, key) pairs, in original token indices."""
    m = np.ones((len(gq), len(gk)), dtype=bool)
    if causal:
        m &= gk[None, :] <= gq[:, None]
    if segq is not None:
        m &= segk[None, :] == segq[:, None]
    return m


def _f64(x):
    if hasattr(x, "detach"):
        import torch

        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# The definition: full (unsharded) softmax attention and its gradient
# --------------------------------------------------------------------------
def block_attention(q, k, v, gq, gk, scale, causal, segq=None, segk=None):
    """Exact attention of queries q against the keys/values k, v of one block.

    q: (m, d), k, v: (n, d) fp64; gq, gk: original token indices; segq/segk:
    segment ids (varlen) or None.  Returns (out (m, d), lse (m,)).
      S_ij = scale * <q_i, k_j> if allowed(i, j) else -inf
      lse_i = log sum_j exp(S_ij);  out_i = sum_j exp(S_ij - lse_i) v_j
    A row with no allowed key gives out = 0, lse = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = scale * (q @ k.T)
    mask = _allowed(np.asarray(gq), np.asarray(gk), causal, segq, segk)
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(S - m_safe[:, None])
    l = e.sum(axis=1)
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    P = e / np.where(has, l, 1.0)[:, None]
    out = P @ v
    return out, lse


def _kv_head(hi, h, hk):
    """Key / value head of query head hi when h query heads share hk key / value
    heads (grouped-query attention): consecutive groups of h / hk query heads
    share one, as in flash-attention's "non-equal head counts"; hk == h is plain
    multi-head attention."""
    if h % hk:
        raise ValueError(f"{h} query heads do not split into groups over {hk} key/value heads")
    return hi // (h // hk)


def attention_fwd(q, k, v, scale, causal, cu_seqlens=None, row_block=1024):
    """Full softmax attention in original token order.

    q: (b, h, s, d); k, v: (b, hk, s, d) with h a multiple of hk (query head hi
    attends with key / value head hi // (h / hk)); any float type, upcast
    exactly to fp64.  Returns out (b, h, s, d) and lse (b, h, s), fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s, d = q.shape
    hk = k.shape[1]
    t = np.arange(s)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    out = np.empty_like(q)
    lse = np.empty((b, h, s))
    for bi in range(b):
        for hi in range(h):
            for r0 in range(0, s, row_block):
                r1 = min(s, r0 + row_block)
                kend = r1 if causal else s  # keys past the block's last row are masked anyway
                kh = _kv_head(hi, h, hk)
                o, l = block_attention(q[bi, hi, r0:r1], k[bi, kh, :kend], v[bi, kh, :kend],
                                       t[r0:r1], t[:kend], scale, causal,
                                       None if seg is None else seg[r0:r1],
                                       None if seg is None else seg[:kend])
                out[bi, hi, r0:r1] = o
                lse[bi, hi, r0:r1] = l
    return out, lse


def attention_bwd(q, k, v, do, scale, causal, cu_seqlens=None, row_block=1024):
    """Analytic gradient of L = sum(dO * out) with respect to q, k, v.

      P = exp(S - lse), D_i = sum_d dO_id out_id
      dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q
    With fewer key / value heads than query heads (grouped-query attention) the
    gradient of a shared key / value head is the sum over its query heads.
    Returns dq (b, h, s, d) and dk, dv (b, hk, s, d), fp64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    b, h, s, d = q.shape
    hk = k.shape[1]
    out, lse = attention_fwd(q, k, v, scale, causal, cu_seqlens, row_block)
    t = np.arange(s)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = (do * out).sum(axis=-1)
    for bi in range(b):
        for hi in range(h):
            kh = _kv_head(hi, h, hk)
            for r0 in range(0, s, row_block):
                r1 = min(s, r0 + row_block)
                S = scale * (q[bi, hi, r0:r1] @ k[bi, kh].T)
                mask = _allowed(t[r0:r1], t, causal,
                                None if seg is None else seg[r0:r1],
                                None if seg is None else seg)
                P = np.where(mask, np.exp(S - lse[bi, hi, r0:r1, None]), 0.0)
                dv[bi, kh] += P.T @ do[bi, hi, r0:r1]
                dP = do[bi, hi, r0:r1] @ v[bi, kh].T
                dS = P * (dP - D[bi, hi, r0:r1, None])
                dq[bi, hi, r0:r1] = scale * (dS @ k[bi, kh])
                dk[bi, kh] += scale * (dS.T @ q[bi, hi, r0:r1])
    return dq, dk, dv


# --------------------------------------------------------------------------
# Sampled forms of the definition, for checks at full size
# --------------------------------------------------------------------------
def attention_rows(q, k, v, rows, scale, causal, cu_seqlens=None, do=None):
    """out_i, lse_i (and D_i, dq_i when dO is given) for selected rows of one head.

    q, k, v, do: (s, d) of one (batch, head); rows: original token indices.
    dq_i = scale * sum_j P_ij (dP_ij - D_i) k_j needs only row i.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    t = np.arange(s)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    out, lse = block_attention(q[rows], k, v, rows, t, scale, causal,
                               None if seg is None else seg[rows], seg)
    if do is None:
        return out, lse
    do = _f64(do)
    D = (do[rows] * out).sum(axis=-1)
    S = scale * (q[rows] @ k.T)
    mask = _allowed(rows, t, causal, None if seg is None else seg[rows], seg)
    P = np.where(mask, np.exp(S - lse[:, None]), 0.0)
    dP = do[rows] @ v.T
    dq = scale * ((P * (dP - D[:, None])) @ k)
    return out, lse, D, dq


def key_grads(q, k, v, do, keys, lse, D, scale, causal, cu_seqlens=None):
    """dk_j, dv_j for selected keys of one head, given lse_i and D_i of every row.

      dv_j = sum_i P_ij dO_i,  dk_j = scale * sum_i P_ij (dP_ij - D_i) q_i
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    s = q.shape[0]
    keys = np.asarray(keys, dtype=np.int64)
    t = np.arange(s)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    S = scale * (q @ k[keys].T)                       # (s, nk)
    mask = _allowed(t, keys, causal, seg, None if seg is None else seg[keys])
    P = np.where(mask, np.exp(S - np.asarray(lse)[:, None]), 0.0)
    dv = P.T @ do
    dP = do @ v[keys].T
    dS = P * (dP - np.asarray(D)[:, None])
    dk = scale * (dS.T @ q)
    return dk, dv


# --------------------------------------------------------------------------
# The ring form: per-block (out, lse) merged across shard steps
# --------------------------------------------------------------------------
def lse_merge(out_acc, lse_acc, out_blk, lse_blk):
    """Merge one block result into the running result, row by row.

    The online-softmax update of [GUIJIA] "在线 Softmax：关键技巧", with the
    running state (m, l) taken as (lse, 1) and each block as (lse_blk, 1):
      m_new = max(m_old, m_blk)
      l_new = l_old * exp(m_old - m_new) + l_blk * exp(m_blk - m_new)
      out_new = out_old * exp(m_old - m_new) * l_old / l_new
              + out_blk * exp(m_blk - m_new) * l_blk / l_new
      lse_new = m_new + log(l_new)
    A side with lse = -inf contributes nothing; both -inf gives out 0, lse -inf.
    Returns new (out, lse) arrays (inputs are not modified).
    """
    out_acc = np.array(out_acc, dtype=np.float64)
    lse_acc = np.array(lse_acc, dtype=np.float64)
    out_blk = np.asarray(out_blk, dtype=np.float64)
    lse_blk = np.asarray(lse_blk, dtype=np.float64)
    out = out_acc.copy()
    lse = lse_acc.copy()
    acc_has = np.isfinite(lse_acc)
    blk_has = np.isfinite(lse_blk)
    only_blk = blk_has & ~acc_has
    out[only_blk] = out_blk[only_blk]
    lse[only_blk] = lse_blk[only_blk]
    both = acc_has & blk_has
    m_old, m_blk = lse_acc[both], lse_blk[both]
    l_old = np.ones_like(m_old)
    l_blk = np.ones_like(m_blk)
    m_new = np.maximum(m_old, m_blk)
    a_old = np.exp(m_old - m_new)
    a_blk = np.exp(m_blk - m_new)
    l_new = l_old * a_old + l_blk * a_blk
    out[both] = (out_acc[both] * (a_old * l_old / l_new)[:, None]
                 + out_blk[both] * (a_blk * l_blk / l_new)[:, None])
    lse[both] = m_new + np.log(l_new)
    neither = ~acc_has & ~blk_has
    out[neither] = 0.0
    lse[neither] = -np.inf
    return out, lse


def ring_attention_sharded(q, k, v, layout, n_shards, scale, causal, cu_seqlens=None):
    """Simulate N ranks of the ring on one CPU, then return ORIGINAL-order results.

    Rank r holds shard r of the layout.  At ring step t = 0..N-1 it holds the
    K/V shard (r - t) mod N ([GUIJIA] "详细流程"), computes the block result
    of its Q shard against it, and merges it into its running (out, lse)
    with ``lse_merge``.  Varlen takes one global cu_seqlens over the packed
    buffer and the contiguous or zigzag layout (``varlen_token_of_position``).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s, d = q.shape
    N = int(n_shards)
    L = s // N
    g = _positions(layout, N, s, cu_seqlens)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    qs, ks, vs = (permute(x, layout, N, axis=2, cu_seqlens=cu_seqlens) for x in (q, k, v))
    out_l = np.zeros((b, h, s, d))
    lse_l = np.full((b, h, s), -np.inf)
    for bi in range(b):
        for hi in range(h):
            for r in range(N):
                rq = slice(r * L, (r + 1) * L)
                o_acc = np.zeros((L, d))
                l_acc = np.full(L, -np.inf)
                for t in range(N):
                    sk = (r - t) % N
                    rk = slice(sk * L, (sk + 1) * L)
                    ob, lb = block_attention(qs[bi, hi, rq], ks[bi, hi, rk], vs[bi, hi, rk],
                                             g[rq], g[rk], scale, causal,
                                             None if seg is None else seg[g[rq]],
                                             None if seg is None else seg[g[rk]])
                    o_acc, l_acc = lse_merge(o_acc, l_acc, ob, lb)
                out_l[bi, hi, rq] = o_acc
                lse_l[bi, hi, rq] = l_acc
    return (unpermute(out_l, layout, N, axis=2, cu_seqlens=cu_seqlens),
            unpermute(lse_l[..., None], layout, N, axis=2, cu_seqlens=cu_seqlens)[..., 0])


def llama3_rank_attention(q, k, v, rank, n_shards, scale, causal, cu_seqlens=None, do=None):
    """One rank of the llama3 context-parallel form ([SP] "llama3" variant,
    llama3_flash_attn_varlen_func): rank r holds the contiguous slice
    [r*L, (r+1)*L) of the (packed) sequence, L = s / N, and its queries attend
    to the all-gathered keys and values with the usual causal / per-sequence
    mask.  Returns out (b, h, L, d), lse (b, h, L) of the slice and, when dO of
    the slice is given, (dq of the slice, this rank's contributions to dk, dv of
    the whole sequence): the gradient of L = sum(dO * out) restricted to the
    slice's rows, i.e. the definition with dO = 0 outside the slice.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s, d = q.shape
    N = int(n_shards)
    if N < 1 or s % N or not 0 <= rank < N:
        raise ValueError("bad rank / n_shards")
    L = s // N
    rows = slice(rank * L, (rank + 1) * L)
    out, lse = attention_fwd(q, k, v, scale, causal, cu_seqlens)
    if do is None:
        return out[:, :, rows], lse[:, :, rows]
    do_full = np.zeros_like(q)
    do_full[:, :, rows] = _f64(do)
    dq, dk, dv = attention_bwd(q, k, v, do_full, scale, causal, cu_seqlens)
    return out[:, :, rows], lse[:, :, rows], dq[:, :, rows], dk, dv


def online_softmax_attention(q, k, v, scale, causal, kv_block=64, cu_seqlens=None):
    """Running-max form with unnormalised accumulation and a final divide.

    The ``ring_attention`` listing of [GUIJIA] ("详细流程" / "在线 Softmax"),
    restated for causal and varlen masks: for each key block,
      block_max = rowmax(S_blk); new_max = max(old_max, block_max)
      correction = exp(old_max - new_max); exp_sum = exp_sum * correction
      exp_sum += rowsum(exp(S_blk - new_max)); acc = acc * correction + exp(S_blk - new_max) V_blk
    and out = acc / exp_sum at the end.  Returns out (b, h, s, d) fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s, d = q.shape
    t = np.arange(s)
    seg = segment_ids(cu_seqlens, s) if cu_seqlens is not None else None
    out = np.empty_like(q)
    for bi in range(b):
        for hi in range(h):
            acc = np.zeros((s, d))
            mx = np.full((s, 1), -np.inf)
            es = np.zeros((s, 1))
            for j0 in range(0, s, kv_block):
                j1 = min(s, j0 + kv_block)
                S = scale * (q[bi, hi] @ k[bi, hi, j0:j1].T)
                mask = _allowed(t, t[j0:j1], causal, seg, None if seg is None else seg[j0:j1])
                S = np.where(mask, S, -np.inf)
                bmax = S.max(axis=1, keepdims=True)
                new = np.maximum(mx, bmax)
                new_safe = np.where(np.isfinite(new), new, 0.0)
                corr = np.where(np.isfinite(mx), np.exp(mx - new_safe), 0.0)
                es = es * corr
                e = np.exp(S - new_safe)
                es = es + e.sum(axis=1, keepdims=True)
                acc = acc * corr + e @ v[bi, hi, j0:j1]
                mx = new
            out[bi, hi] = acc / es
    return out


def causal_flops(b, h, s, d, causal=True):
    """Causal-adjusted forward FLOP count 4*b*h*s*s*d (/2 when causal)."""
    f = 4.0 * b * h * float(s) * float(s) * d
    return f / 2.0 if causal else f

