// Tile walks over the (Q shard, KV shard) pairs of the ring, shared by the
// forward, the dQ pass and the dK/dV pass.
//
// The ring order is the pages' (guijiagi.com "Ring Attention：突破百万 Token
// 上下文的分布式注意力", "详细流程"): at step t, Q shard r meets KV shard
// (r - t) mod N, and KV shard s meets Q shard (s + t) mod N.  The original
// token of a local position is increasing inside every shard for all layouts,
// so for causal masking the allowed keys of a row are a prefix of each KV
// shard (within its sequence, for varlen), the allowed queries of a key a
// suffix of each Q shard, and a tile is empty, full or partial by its corners.
// Varlen takes one cu_seqlens over the packed buffer with the contiguous
// layout (shards are slices of the packed buffer) or the zigzag layout applied
// to every sequence (sequence k at local [cu[k]/N, cu[k+1]/N) of every shard).
// P is FwdParamsT or BwdParamsT (N, L, layout, causal, cu, n_seqs and kVarlen).
#pragma once

#include "ra_internal.h"

namespace ra {

// cu_seqlens of a varlen call; nullptr (known at compile time) in batched kernels.
template <class P>
__device__ __forceinline__ const int* cu_of(const P& p) {
  return P::kVarlen ? p.cu : nullptr;
}

template <class P>
__device__ __forceinline__ bool vz(const P& p) {
  return cu_of(p) != nullptr && p.layout == LAYOUT_ZIGZAG;
}

// Original token of local position i of shard r.
template <class P>
__device__ __forceinline__ int tok(const P& p, int r, int i) {
  if (vz(p)) return vz_token(p.cu, p.n_seqs, p.N, r, i);
  return token_of(p.layout, p.N, p.L, r, i);
}

// Heavy-first order of query tiles for the batched causal zigzag layout.
// Chunk c of the 2N (tokens [c C, (c+1) C)) sits in shard c (c < N) or
// 2N-1-c, and a query tile of a later chunk sees more keys.  Rank k of a grid
// of 2N * tpc tiles (tpc per chunk) is mapped to (shard, local tile) so that
// every head's heaviest tiles start first and the lightest end the grid (the
// plain reversed order left the heaviest chunk, in shard 0, to the end).
__device__ __forceinline__ void zigzag_heavy_first(int k, int N, int tpc, int& shard, int& tile) {
  const int ch = 2 * N - 1 - k / tpc;
  const int t = tpc - 1 - k % tpc;
  shard = ch < N ? ch : 2 * N - 1 - ch;
  tile = (ch < N ? 0 : tpc) + t;
}

// Query rows [i0, i0 + rows) of Q shard r; the valid ones end at i_last.
struct QRange {
  int r, i0, i_last;
  int gq_lo, gq_hi;    // original token indices of the first / last valid row
  // varlen: the keys any row may see.  Contiguous: tokens [key_lo, key_hi].
  // Zigzag: local positions from key_lo in every shard up to, when causal, the
  // last row's offset zo in its sequence (first local position zb, chunk zc),
  // else up to key_hi.  Set once per CTA, so kv_range is integer compares.
  int key_lo, key_hi, zb, zc, zo;
};

// Searches of cu_seqlens: the first and last valid positions are the same in
// every lane, and (varlen) every thread of the CTA calls this, so the
// searches run warp-wide (segment_of_warp).
template <class P>
__device__ __forceinline__ void ends_and_segments(const P& p, int r, int ilo, int ihi, int& g_lo, int& g_hi, int& sa,
                                                  int& sz) {
  sa = sz = 0;
  if (vz(p)) {
    // local position i of any shard holds sequence k for cu[k] <= i N < cu[k+1]
    sa = segment_of_warp(p.cu, p.n_seqs, ilo * p.N);
    sz = segment_of_warp(p.cu, p.n_seqs, ihi * p.N, sa);
    g_lo = vz_token_in(__ldg(p.cu + sa), __ldg(p.cu + sa + 1), p.N, r, ilo);
    g_hi = vz_token_in(__ldg(p.cu + sz), __ldg(p.cu + sz + 1), p.N, r, ihi);
    return;
  }
  g_lo = token_of(p.layout, p.N, p.L, r, ilo);
  g_hi = token_of(p.layout, p.N, p.L, r, ihi);
  if (cu_of(p)) {
    sa = segment_of_warp(p.cu, p.n_seqs, g_lo);
    sz = segment_of_warp(p.cu, p.n_seqs, g_hi, sa);
  }
}

template <class P>
__device__ __forceinline__ void make_qrange(const P& p, int r, int i0, int rows, QRange& q) {
  q.r = r;
  q.i0 = i0;
  q.i_last = min(i0 + rows, p.L) - 1;
  const int ilo = min(i0, p.L - 1);
  int sa, sz;
  ends_and_segments(p, r, ilo, max(q.i_last, ilo), q.gq_lo, q.gq_hi, sa, sz);
  q.key_lo = q.key_hi = q.zb = q.zc = q.zo = 0;
  if (vz(p)) {
    const int cz = __ldg(p.cu + sz), cz1 = __ldg(p.cu + sz + 1);
    q.key_lo = __ldg(p.cu + sa) / p.N;
    q.key_hi = cz1 / p.N - 1;
    q.zb = cz / p.N;
    q.zc = (cz1 - cz) / (2 * p.N);
    q.zo = q.gq_hi - cz;
  } else if (cu_of(p)) {
    q.key_lo = __ldg(p.cu + sa);
    q.key_hi = p.causal ? q.gq_hi : __ldg(p.cu + sz + 1) - 1;
  }
}

// Key-tile range [lo, hi) of KV shard s that can hold a key allowed for some row of q.
template <class P>
__device__ __forceinline__ void kv_range(const P& p, const QRange& q, int s, int nkt, int& lo, int& hi) {
  if (cu_of(p)) {
    int jlo, jhi;  // local key positions of shard s, inclusive
    if (vz(p)) {
      // keys of the rows' sequences up to the last row's token (local order is token order)
      jlo = q.key_lo;
      jhi = p.causal ? vz_prefix_end(q.zb, q.zc, p.N, s, q.zo) - 1 : q.key_hi;
    } else {
      const int base = s * p.L;
      jlo = q.key_lo - base;
      jhi = q.key_hi - base;
    }
    if (jlo < 0) jlo = 0;
    if (jhi > p.L - 1) jhi = p.L - 1;
    if (jlo > jhi) {
      lo = hi = 0;
      return;
    }
    lo = jlo / kTileN;
    hi = jhi / kTileN + 1;
    return;
  }
  lo = 0;
  if (!p.causal) {
    hi = nkt;
    return;
  }
  // the allowed keys of the largest row token are a prefix of the shard and
  // cover every other row's keys
  const int jm = last_local_at_or_before(p.layout, p.N, p.L, s, q.gq_hi);
  hi = jm < 0 ? 0 : jm / kTileN + 1;
}

// True when every (valid row of q, key) pair of key tile kt of shard s is
// allowed (batched calls; varlen rows use RowWin).
template <class P>
__device__ __forceinline__ bool kv_tile_full(const P& p, const QRange& q, int s, int kt) {
  static_assert(!P::kVarlen, "varlen rows use RowWin");
  const int j0 = kt * kTileN;
  if (j0 + kTileN > p.L || q.i0 >= p.L) return false;
  return !p.causal || q.gq_lo >= token_of(p.layout, p.N, p.L, s, j0 + kTileN - 1);
}

// Calls f(s, kt) for every key tile the rows of q meet at ring steps [t0, t1).
template <class P, class F>
__device__ __forceinline__ void walk_kv_tiles(const P& p, const QRange& q, int nkt, int t0, int t1, F&& f) {
  for (int t = t0; t < t1; ++t) {
    int s = q.r - t;
    if (s < 0) s += p.N;
    int lo, hi;
    kv_range(p, q, s, nkt, lo, hi);
    for (int kt = lo; kt < hi; ++kt)
      if (!f(s, kt)) return;
  }
}

// Allowed key columns [c_lo, c_hi) of a query row (token gq) in key tile kt
// of shard s (batched calls).
template <class P>
__device__ __forceinline__ void row_key_window(const P& p, int gq, int s, int kt, int& c_lo, int& c_hi) {
  static_assert(!P::kVarlen, "varlen rows use RowWin");
  const int j0 = kt * kTileN;
  const int jlim = min(kTileN, p.L - j0);
  c_lo = 0;
  c_hi = jlim;
  if (p.causal) {
    const int jm = last_local_at_or_before(p.layout, p.N, p.L, s, gq);
    c_hi = min(jlim, jm - j0 + 1);
  }
}

// Key rows [j0, j0 + rows) of KV shard s (rows = 128, or 256 for the key
// tiles of a CTA pair, whose query walk is the union of its two tiles').
struct KRange {
  int s, j0, j_last;
  int gk_lo, gk_hi;
  // varlen: the queries any key may serve.  Contiguous: tokens [qry_lo, qry_hi].
  // Zigzag: local positions up to qry_hi in every shard, from (causal) the
  // first local position past offset zo of the first key's sequence (first
  // local position zb, chunk zc), else from qry_lo.
  int qry_lo, qry_hi, zb, zc, zo;
};

template <class P>
__device__ __forceinline__ void make_krange(const P& p, int s, int j0, KRange& k, int rows = kTileN) {
  k.s = s;
  k.j0 = j0;
  k.j_last = min(j0 + rows, p.L) - 1;
  int sa, sz;
  ends_and_segments(p, s, j0, k.j_last, k.gk_lo, k.gk_hi, sa, sz);
  k.qry_lo = k.qry_hi = k.zb = k.zc = k.zo = 0;
  if (vz(p)) {
    const int ca = __ldg(p.cu + sa), ca1 = __ldg(p.cu + sa + 1);
    k.qry_lo = ca / p.N;
    k.qry_hi = __ldg(p.cu + sz + 1) / p.N - 1;
    k.zb = ca / p.N;
    k.zc = (ca1 - ca) / (2 * p.N);
    k.zo = k.gk_lo - 1 - ca;
  } else if (cu_of(p)) {
    k.qry_lo = p.causal ? k.gk_lo : __ldg(p.cu + sa);
    k.qry_hi = __ldg(p.cu + sz + 1) - 1;
  }
}

// Query-tile range [lo, hi) (tiles of QT rows) of Q shard r that holds a query some key of k serves.
template <int QT, class P>
__device__ __forceinline__ void q_range(const P& p, const KRange& k, int r, int nqt, int& lo, int& hi) {
  if (cu_of(p)) {
    int ilo, ihi;  // local query positions of shard r, inclusive
    if (vz(p)) {
      // queries of the keys' sequences from the first key's token on
      ilo = p.causal ? vz_prefix_end(k.zb, k.zc, p.N, r, k.zo) : k.qry_lo;
      ihi = k.qry_hi;
    } else {
      const int base = r * p.L;
      ilo = k.qry_lo - base;
      ihi = k.qry_hi - base;
    }
    if (ilo < 0) ilo = 0;
    if (ihi > p.L - 1) ihi = p.L - 1;
    if (ilo > ihi) {
      lo = hi = 0;
      return;
    }
    lo = ilo / QT;
    hi = ihi / QT + 1;
    return;
  }
  hi = nqt;
  if (!p.causal) {
    lo = 0;
    return;
  }
  // first local query of shard r whose token is >= the tile's first key token
  const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, k.gk_lo - 1) + 1;
  lo = imin >= p.L ? nqt : imin / QT;
}

// True when every (key of k, valid query) pair of query tile qt (QT rows) of
// shard r is allowed (batched calls; varlen rows use RowWin).
template <int QT, class P>
__device__ __forceinline__ bool q_tile_full(const P& p, const KRange& k, int r, int qt) {
  static_assert(!P::kVarlen, "varlen rows use RowWin");
  const int i0 = qt * QT;
  if (i0 + QT > p.L || k.j0 + kTileN > p.L) return false;
  return !p.causal || token_of(p.layout, p.N, p.L, r, i0) >= k.gk_hi;
}

// Calls f(r, qt) for every query tile (QT rows) the keys of k serve, in ring
// order (only Q shard p.r_only when it is set).
template <int QT, class P, class F>
__device__ __forceinline__ void walk_q_tiles(const P& p, const KRange& k, int nqt, F&& f) {
  for (int t = 0; t < p.N; ++t) {
    int r = k.s + t;
    if (r >= p.N) r -= p.N;
    if (p.r_only >= 0 && r != p.r_only) continue;
    int lo, hi;
    q_range<QT>(p, k, r, nqt, lo, hi);
    for (int qt = lo; qt < hi; ++qt)
      if (!f(r, qt)) return;
  }
}

// walk_q_tiles over every query head that shares key / value head hk
// (grouped-query attention: heads hk * G .. hk * G + G - 1; G = 1 is plain
// multi-head attention): calls f(hq, r, qt) in head order, then ring order.
template <int QT, class P, class F>
__device__ __forceinline__ void walk_group_q_tiles(const P& p, const KRange& k, int nqt, int hk, F&& f) {
  bool go = true;
  for (int g = 0; g < p.G && go; ++g) {
    const int hq = hk * p.G + g;
    walk_q_tiles<QT>(p, k, nqt, [&](int r, int qt) {
      go = f(hq, r, qt);
      return go;
    });
  }
}

// Allowed query columns [c_lo, c_hi) of a key row (token gk) in query tile
// qt (QT rows) of shard r (batched calls).
template <int QT, class P>
__device__ __forceinline__ void key_query_window(const P& p, bool valid_k, int gk, int r, int qt, int& c_lo,
                                                 int& c_hi) {
  static_assert(!P::kVarlen, "varlen rows use RowWin");
  c_lo = c_hi = 0;
  if (!valid_k) return;
  const int i0 = qt * QT;
  const int ilim = min(QT, p.L - i0);
  c_hi = ilim;
  if (p.causal) {
    const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, gk - 1) + 1;
    c_lo = max(0, imin - i0);
  }
}

// One varlen row's window: the local positions of a shard that the row may
// meet (a query row: keys of its sequence at or before it; a key row: queries
// of its sequence at or after it).  Set up once per row, with one warp-wide
// search of cu_seqlens; per shard and tile only integer arithmetic follows.
struct RowWin {
  int a, b;         // contiguous: allowed tokens [a, b); zigzag: allowed offsets (a, b] in the sequence
  int base, c;      // zigzag: the sequence's first local position (every shard) and its chunk length
  int cur, lo, hi;  // shard `cur` allows local positions [lo, hi)
};

// Window of the row at local position i of shard r; returns its token.
// Called by full warps with i not decreasing along the lanes (padding rows
// pass the last valid position).  key_row: the dK/dV side.
template <class P>
__device__ __forceinline__ int make_row_win(const P& p, int r, int i, bool key_row, RowWin& w) {
  static_assert(P::kVarlen, "batched rows use the tile classification");
  int g, ck, ck1;
  if (vz(p)) {
    const int k = segment_of_lanes(p.cu, p.n_seqs, i * p.N);
    ck = __ldg(p.cu + k);
    ck1 = __ldg(p.cu + k + 1);
    g = vz_token_in(ck, ck1, p.N, r, i);
    const int o = g - ck, last = ck1 - ck - 1;
    w.base = ck / p.N;
    w.c = (ck1 - ck) / (2 * p.N);
    w.a = key_row && p.causal ? o - 1 : -1;
    w.b = !key_row && p.causal ? o : last;
  } else {
    g = r * p.L + i;
    const int k = segment_of_lanes(p.cu, p.n_seqs, g);
    ck = __ldg(p.cu + k);
    ck1 = __ldg(p.cu + k + 1);
    w.a = key_row && p.causal ? g : ck;
    w.b = !key_row && p.causal ? g + 1 : ck1;
    w.base = w.c = 0;
  }
  w.cur = -1;
  w.lo = w.hi = 0;
  return g;
}

// Allowed columns [c_lo, c_hi) of the row in the tile of `tlen` positions
// starting at local position t0 of shard s.
template <class P>
__device__ __forceinline__ void row_win_cols(const P& p, RowWin& w, int s, int t0, int tlen, int& c_lo, int& c_hi) {
  if (s != w.cur) {
    w.cur = s;
    if (vz(p)) {
      w.lo = vz_prefix_end(w.base, w.c, p.N, s, w.a);
      w.hi = vz_prefix_end(w.base, w.c, p.N, s, w.b);
    } else {
      w.lo = w.a - s * p.L;
      w.hi = w.b - s * p.L;
    }
  }
  const int lim = min(tlen, p.L - t0);
  const int lo = w.lo - t0, hi = w.hi - t0;
  c_lo = lo < 0 ? 0 : (lo > tlen ? tlen : lo);
  c_hi = hi < 0 ? 0 : (hi > lim ? lim : hi);
}

}  // namespace ra
