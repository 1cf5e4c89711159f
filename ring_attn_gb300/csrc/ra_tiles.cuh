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

// Query rows [i0, i0 + rows) of Q shard r; the valid ones end at i_last.
struct QRange {
  int r, i0, i_last;
  int gq_lo, gq_hi;    // original token indices of the first / last valid row
  int key_lo, key_hi;  // contiguous varlen: keys any row may see (inclusive)
  int seg_lo, seg_hi;  // varlen: segments of the first / last valid row
  int seg_single;      // varlen: the segment of every valid row, or -1
};

template <class P>
__device__ __forceinline__ void make_qrange(const P& p, int r, int i0, int rows, QRange& q) {
  q.r = r;
  q.i0 = i0;
  q.i_last = min(i0 + rows, p.L) - 1;
  const int ilo = min(i0, p.L - 1);
  q.gq_lo = tok(p, r, ilo);
  q.gq_hi = tok(p, r, max(q.i_last, ilo));
  q.key_lo = q.key_hi = 0;
  q.seg_lo = q.seg_hi = 0;
  q.seg_single = -1;
  if (cu_of(p)) {
    const int sa = segment_of(p.cu, p.n_seqs, q.gq_lo);
    const int sz = segment_of(p.cu, p.n_seqs, q.gq_hi);
    q.key_lo = __ldg(p.cu + sa);
    q.key_hi = p.causal ? q.gq_hi : __ldg(p.cu + sz + 1) - 1;
    q.seg_lo = sa;
    q.seg_hi = sz;
    q.seg_single = sa == sz ? sa : -1;
  }
}

// Key-tile range [lo, hi) of KV shard s that can hold a key allowed for some row of q.
template <class P>
__device__ __forceinline__ void kv_range(const P& p, const QRange& q, int s, int nkt, int& lo, int& hi) {
  if (cu_of(p)) {
    int jlo, jhi;  // local key positions of shard s, inclusive
    if (vz(p)) {
      // keys of the rows' sequences up to the last row's token (local order is token order)
      const int ca = __ldg(p.cu + q.seg_lo), cz = __ldg(p.cu + q.seg_hi), cz1 = __ldg(p.cu + q.seg_hi + 1);
      jlo = ca / p.N;
      jhi = p.causal ? vz_last_le(cz, cz1, p.N, s, q.gq_hi) : cz1 / p.N - 1;
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

// True when every (valid row of q, key) pair of key tile kt of shard s is allowed.
template <class P>
__device__ __forceinline__ bool kv_tile_full(const P& p, const QRange& q, int s, int kt) {
  const int j0 = kt * kTileN;
  if (j0 + kTileN > p.L || q.i0 >= p.L) return false;
  if (cu_of(p)) {
    if (q.seg_single < 0) return false;
    const int slo = __ldg(p.cu + q.seg_single), shi = __ldg(p.cu + q.seg_single + 1);
    if (vz(p)) {
      if (j0 < slo / p.N || j0 + kTileN > shi / p.N) return false;
      return !p.causal || q.gq_lo >= vz_token_in(slo, shi, p.N, s, j0 + kTileN - 1);
    }
    const int base = s * p.L + j0;
    if (base < slo || base + kTileN > shi) return false;
    return !p.causal || q.gq_lo >= base + kTileN - 1;
  }
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

// Per-row bounds for the varlen windows below: the row's key bounds in
// tokens [rk_lo, rk_hi) for the contiguous layout (the causal bound folded
// in), or its sequence [cu[k], cu[k+1]) for the zigzag layout.
template <class P>
__device__ __forceinline__ void row_key_bounds(const P& p, int gq, int& rk_lo, int& rk_hi) {
  const int sg = segment_of(p.cu, p.n_seqs, gq);
  rk_lo = __ldg(p.cu + sg);
  rk_hi = (p.causal && !vz(p)) ? gq + 1 : __ldg(p.cu + sg + 1);
}

// Allowed key columns [c_lo, c_hi) of a query row (token gq, varlen bounds
// [rk_lo, rk_hi) from row_key_bounds) in key tile kt of shard s.
template <class P>
__device__ __forceinline__ void row_key_window(const P& p, int gq, int rk_lo, int rk_hi, int s, int kt, int& c_lo,
                                               int& c_hi) {
  const int j0 = kt * kTileN;
  const int jlim = min(kTileN, p.L - j0);
  c_lo = 0;
  c_hi = jlim;
  if (cu_of(p)) {
    int lo, hi;  // allowed local keys [lo, hi) of shard s, relative to the tile
    if (vz(p)) {
      lo = rk_lo / p.N - j0;
      hi = (p.causal ? vz_last_le(rk_lo, rk_hi, p.N, s, gq) + 1 : rk_hi / p.N) - j0;
    } else {
      const int base = s * p.L + j0;
      lo = rk_lo - base;
      hi = rk_hi - base;
    }
    c_lo = lo < 0 ? 0 : (lo > kTileN ? kTileN : lo);
    c_hi = hi < 0 ? 0 : (hi > jlim ? jlim : hi);
  } else if (p.causal) {
    const int jm = last_local_at_or_before(p.layout, p.N, p.L, s, gq);
    c_hi = min(jlim, jm - j0 + 1);
  }
}

// Key rows [j0, j0 + 128) of KV shard s.
struct KRange {
  int s, j0, j_last;
  int gk_lo, gk_hi;
  int qry_lo, qry_hi;  // contiguous varlen: queries any key of the tile may serve (inclusive)
  int seg_lo, seg_hi;  // varlen: segments of the first / last valid key
  int seg_single;
};

template <class P>
__device__ __forceinline__ void make_krange(const P& p, int s, int j0, KRange& k) {
  k.s = s;
  k.j0 = j0;
  k.j_last = min(j0 + kTileN, p.L) - 1;
  k.gk_lo = tok(p, s, j0);
  k.gk_hi = tok(p, s, k.j_last);
  k.qry_lo = k.qry_hi = 0;
  k.seg_lo = k.seg_hi = 0;
  k.seg_single = -1;
  if (cu_of(p)) {
    const int sa = segment_of(p.cu, p.n_seqs, k.gk_lo);
    const int sz = segment_of(p.cu, p.n_seqs, k.gk_hi);
    k.qry_lo = p.causal ? k.gk_lo : __ldg(p.cu + sa);
    k.qry_hi = __ldg(p.cu + sz + 1) - 1;
    k.seg_lo = sa;
    k.seg_hi = sz;
    k.seg_single = sa == sz ? sa : -1;
  }
}

// Query-tile range [lo, hi) (tiles of QT rows) of Q shard r that holds a query some key of k serves.
template <int QT, class P>
__device__ __forceinline__ void q_range(const P& p, const KRange& k, int r, int nqt, int& lo, int& hi) {
  if (cu_of(p)) {
    int ilo, ihi;  // local query positions of shard r, inclusive
    if (vz(p)) {
      // queries of the keys' sequences from the first key's token on
      const int ca = __ldg(p.cu + k.seg_lo), ca1 = __ldg(p.cu + k.seg_lo + 1);
      ilo = p.causal ? vz_last_le(ca, ca1, p.N, r, k.gk_lo - 1) + 1 : ca / p.N;
      ihi = __ldg(p.cu + k.seg_hi + 1) / p.N - 1;
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

// True when every (key of k, valid query) pair of query tile qt (QT rows) of shard r is allowed.
template <int QT, class P>
__device__ __forceinline__ bool q_tile_full(const P& p, const KRange& k, int r, int qt) {
  const int i0 = qt * QT;
  if (i0 + QT > p.L || k.j0 + kTileN > p.L) return false;
  if (cu_of(p)) {
    if (k.seg_single < 0) return false;
    const int slo = __ldg(p.cu + k.seg_single), shi = __ldg(p.cu + k.seg_single + 1);
    if (vz(p)) {
      if (i0 < slo / p.N || i0 + QT > shi / p.N) return false;
      return !p.causal || vz_token_in(slo, shi, p.N, r, i0) >= k.gk_hi;
    }
    const int base = r * p.L + i0;
    if (base < slo || base + QT > shi) return false;
    return !p.causal || base >= k.gk_hi;
  }
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

// Per-key bounds for key_query_window: the queries a key serves in tokens
// [rq_lo, rq_hi) for the contiguous layout (the causal bound folded in), or
// its sequence [cu[k], cu[k+1]) for the zigzag layout.
template <class P>
__device__ __forceinline__ void key_query_bounds(const P& p, int gk, int& rq_lo, int& rq_hi) {
  const int sg = segment_of(p.cu, p.n_seqs, gk);
  rq_lo = (p.causal && !vz(p)) ? gk : __ldg(p.cu + sg);
  rq_hi = __ldg(p.cu + sg + 1);
}

// Allowed query columns [c_lo, c_hi) of a key row (token gk, varlen bounds
// [rq_lo, rq_hi) from key_query_bounds) in query tile qt (QT rows) of shard r.
template <int QT, class P>
__device__ __forceinline__ void key_query_window(const P& p, bool valid_k, int gk, int rq_lo, int rq_hi, int r, int qt,
                                                 int& c_lo, int& c_hi) {
  c_lo = c_hi = 0;
  if (!valid_k) return;
  const int i0 = qt * QT;
  const int ilim = min(QT, p.L - i0);
  c_hi = ilim;
  if (cu_of(p)) {
    int lo, hi;  // allowed local queries [lo, hi) of shard r, relative to the tile
    if (vz(p)) {
      lo = (p.causal ? vz_last_le(rq_lo, rq_hi, p.N, r, gk - 1) + 1 : rq_lo / p.N) - i0;
      hi = rq_hi / p.N - i0;
    } else {
      const int base = r * p.L + i0;
      lo = rq_lo - base;
      hi = rq_hi - base;
    }
    c_lo = lo < 0 ? 0 : (lo > QT ? QT : lo);
    c_hi = hi < 0 ? 0 : (hi > ilim ? ilim : hi);
  } else if (p.causal) {
    const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, gk - 1) + 1;
    c_lo = max(0, imin - i0);
  }
}

}  // namespace ra
