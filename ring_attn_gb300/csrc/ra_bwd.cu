// Ring-attention backward on sm_103a.
//
// One CTA owns a 128-row key tile of KV shard s and meets the query shards in
// ring order r = (s + t) mod N, t = 0..N-1 (the path the K/V block and its
// gradient accumulators travel on the ring: guijiagi.com "Ring Attention：
// 突破百万 Token 上下文的分布式注意力", "详细流程").  For every query tile it
// recomputes the probabilities from the saved log-sum-exp ("Ring Flash
// Attention" README: "use the softmax_lse output") and applies the gradient
// of exact attention:
//   P^T = exp(S^T - lse),  dV += P^T dO,  dP^T = V dO^T,
//   dS^T = P^T * (dP^T - D),  dK += scale dS^T Q,  dQ += scale dS K,
// with D = rowsum(dO * O) computed beforehand.  dK and dV live in tensor
// memory for the CTA's whole life; dQ partial tiles are added in fp32 into a
// workspace accumulator.
//
// Warps (384 threads):
//   0      TMA producer: K and V once, then Q and dO per query tile
//   1      MMA issuer (one thread)
//   2      TMEM allocation (512 columns)
//   4-7    one thread per key row: P^T and dS^T (bf16, 128B-swizzled smem),
//          then the dK / dV epilogue
//   8-11   one thread per query row: reads the dQ tile from TMEM and adds it
//          to the fp32 accumulator
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D);
// the dQ tile reuses [0, D) once S^T has been consumed.
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBox = 128 * 128;

template <int D>
struct BwdLayout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kPT = kDO + kTile;      // P^T: 128 key rows x 128 queries (2 boxes)
  static constexpr int kDST = kPT + 2 * kBox;  // dS^T: same shape
  static constexpr int kLse = kDST + 2 * kBox; // 2 x 128 fp32 (log2 units)
  static constexpr int kDv = kLse + 1024;      // 2 x 128 fp32
  static constexpr int kBar = kDv + 1024;
  static constexpr int kNumBars = 10;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 256 + D, kTmemDQ = 0;
};

enum BwdBar {
  C_KV_FULL = 0,
  C_QDO_FULL,
  C_QDO_EMPTY,
  C_S_FULL,
  C_P_FULL,
  C_DQ_FULL,
  C_DQ_FREE,
  C_TEARDOWN,
  C_STATS_READY  // 2: per-tile lse / D staged in shared memory
};

struct KTile {
  int b, h, s, j0, j_last;
  long long gk_lo, gk_hi;
  long long qry_lo, qry_hi;  // varlen: queries any key of the tile may serve (inclusive)
  int seg_single;
};

__device__ __forceinline__ void q_range(const BwdParams& p, const KTile& k, int r, int& lo, int& hi) {
  const int nqt = p.n_qtiles;
  if (p.cu) {
    const long long base = (long long)r * p.L;
    long long ilo = k.qry_lo - base, ihi = k.qry_hi - base;
    if (ilo < 0) ilo = 0;
    if (ihi > p.L - 1) ihi = p.L - 1;
    if (ilo > ihi) {
      lo = hi = 0;
      return;
    }
    lo = (int)(ilo / kTileM);
    hi = (int)(ihi / kTileM) + 1;
    return;
  }
  hi = nqt;
  if (!p.causal) {
    lo = 0;
    return;
  }
  // first local query of shard r whose token is >= the tile's first key token
  const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, k.gk_lo - 1) + 1;
  lo = imin >= p.L ? nqt : imin / kTileM;
}

__device__ __forceinline__ bool qtile_full(const BwdParams& p, const KTile& k, int r, int qt) {
  const int i0 = qt * kTileM;
  if (i0 + kTileM > p.L || k.j0 + kTileN > p.L) return false;
  if (p.cu) {
    if (k.seg_single < 0) return false;
    const long long base = (long long)r * p.L + i0;
    const long long slo = __ldg(p.cu + k.seg_single), shi = __ldg(p.cu + k.seg_single + 1);
    if (base < slo || base + kTileM > shi) return false;
    return !p.causal || base >= k.gk_hi;
  }
  return !p.causal || token_of(p.layout, p.N, p.L, r, i0) >= k.gk_hi;
}

template <class F>
__device__ __forceinline__ void walk_qtiles(const BwdParams& p, const KTile& k, F&& f) {
  for (int t = 0; t < p.N; ++t) {
    int r = k.s + t;
    if (r >= p.N) r -= p.N;
    int lo, hi;
    q_range(p, k, r, lo, hi);
    for (int qt = lo; qt < hi; ++qt)
      if (!f(r, qt)) return;
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    ring_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using LY = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  KTile k;
  k.b = blockIdx.y / p.H;
  k.h = blockIdx.y % p.H;
  k.s = blockIdx.x / p.n_ktiles;
  k.j0 = (blockIdx.x % p.n_ktiles) * kTileN;
  k.j_last = min(k.j0 + kTileN, p.L) - 1;
  k.gk_lo = token_of(p.layout, p.N, p.L, k.s, k.j0);
  k.gk_hi = token_of(p.layout, p.N, p.L, k.s, k.j_last);
  k.qry_lo = k.qry_hi = 0;
  k.seg_single = -1;
  if (p.cu) {
    const int sa = segment_of(p.cu, p.n_seqs, k.gk_lo);
    const int sz = segment_of(p.cu, p.n_seqs, k.gk_hi);
    k.qry_lo = p.causal ? k.gk_lo : (long long)__ldg(p.cu + sa);
    k.qry_hi = (long long)__ldg(p.cu + sz + 1) - 1;
    k.seg_single = sa == sz ? sa : -1;
  }
  int n_tiles = 0;
  walk_qtiles(p, k, [&](int, int) {
    ++n_tiles;
    return true;
  });

  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C_KV_FULL), 1);
    mbar_init(BAR(C_QDO_FULL), 1);
    mbar_init(BAR(C_QDO_EMPTY), 1);
    mbar_init(BAR(C_S_FULL), 1);
    mbar_init(BAR(C_P_FULL), 128);
    mbar_init(BAR(C_DQ_FULL), 1);
    mbar_init(BAR(C_DQ_FREE), 128);
    mbar_init(BAR(C_TEARDOWN), 1);
    mbar_init(BAR(C_STATS_READY), 128);
    mbar_init(BAR(C_STATS_READY + 1), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      const int krow = k.s * p.L + k.j0;
      mbar_expect_tx(BAR(C_KV_FULL), 2 * LY::kTile);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_4d(sb + LY::kK + c * kBox, &tmK, BAR(C_KV_FULL), c * 64, krow, k.h, k.b);
        tma_load_4d(sb + LY::kV + c * kBox, &tmV, BAR(C_KV_FULL), c * 64, krow, k.h, k.b);
      }
      int i = 0;
      walk_qtiles(p, k, [&](int r, int qt) {
        if (i > 0 && !wait_one(BAR(C_QDO_EMPTY), (i - 1) & 1, abort_flag, p.ctl, 31)) return false;
        const int qrow = r * p.L + qt * kTileM;
        mbar_expect_tx(BAR(C_QDO_FULL), 2 * LY::kTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sb + LY::kQ + c * kBox, &tmQ, BAR(C_QDO_FULL), c * 64, qrow, k.h, k.b);
          tma_load_4d(sb + LY::kDO + c * kBox, &tmDO, BAR(C_QDO_FULL), c * 64, qrow, k.h, k.b);
        }
        ++i;
        return true;
      });
      drain_one(BAR(C_KV_FULL), 0, p.ctl, 40);
      if (i > 0) drain_one(BAR(C_QDO_FULL), (i - 1) & 1, p.ctl, 41);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileM, 0, 0);  // S^T, dP^T: K-major A and B
      constexpr uint32_t kIdKV = idesc_bf16_f32(128, D, 0, 1);      // dV, dK: K-major A, MN-major B
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 1, 1);       // dQ: MN-major A and B
      bool ok = wait_one(BAR(C_KV_FULL), 0, abort_flag, p.ctl, 32);
      int i = 0;
      if (ok) {
        walk_qtiles(p, k, [&](int, int) {
          if (!wait_one(BAR(C_QDO_FULL), i & 1, abort_flag, p.ctl, 33) ||
              (i > 0 && !wait_one(BAR(C_DQ_FREE), (i - 1) & 1, abort_flag, p.ctl, 34))) {
            ok = false;
            return false;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            // S^T = K Q^T (A = K tile, B = Q tile; both K-major over d)
            mma_bf16_ss(tmem + LY::kTmemS, sdesc_sw128(sb + LY::kK + off, 16, 1024),
                        sdesc_sw128(sb + LY::kQ + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            // dP^T = V dO^T
            mma_bf16_ss(tmem + LY::kTmemDP, sdesc_sw128(sb + LY::kV + off, 16, 1024),
                        sdesc_sw128(sb + LY::kDO + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C_S_FULL));
          if (!wait_one(BAR(C_P_FULL), i & 1, abort_flag, p.ctl, 35)) {
            ok = false;
            return false;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;  // K-major A: 16 queries = 32 bytes
            const uint32_t boff = kk * 2048;                        // MN-major B: 16 query rows
            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
            // dV += P^T dO
            mma_bf16_ss(tmem + LY::kTmemDV, sdesc_sw128(sb + LY::kPT + aoff, 16, 1024),
                        sdesc_sw128(sb + LY::kDO + boff, kBox, 1024), kIdKV, acc);
            // dK += dS^T Q (the softmax scale is applied in the epilogue)
            mma_bf16_ss(tmem + LY::kTmemDK, sdesc_sw128(sb + LY::kDST + aoff, 16, 1024),
                        sdesc_sw128(sb + LY::kQ + boff, kBox, 1024), kIdKV, acc);
          }
          if (i + 1 < n_tiles) mma_commit(BAR(C_QDO_EMPTY));
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            // dQ = dS K: A = dS (queries contiguous in the dS^T tile: MN-major), B = K (MN-major)
            mma_bf16_ss(tmem + LY::kTmemDQ, sdesc_sw128(sb + LY::kDST + kk * 2048, kBox, 1024),
                        sdesc_sw128(sb + LY::kK + kk * 2048, kBox, 1024), kIdQ, kk > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C_DQ_FULL));
          ++i;
          return true;
        });
      }
      mma_commit(BAR(C_TEARDOWN));
      drain_one(BAR(C_TEARDOWN), 0, p.ctl, 42);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ P^T / dS^T per key row
    const int tid = threadIdx.x - 128;  // 0..127
    const int jr = tid;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int j = k.j0 + jr;
    const bool valid_k = j < p.L;
    const long long gk = token_of(p.layout, p.N, p.L, k.s, valid_k ? j : k.j_last);
    long long rq_lo = 0, rq_hi = 0;  // varlen: queries [rq_lo, rq_hi) this key serves
    if (p.cu) {
      const int sg = segment_of(p.cu, p.n_seqs, gk);
      rq_lo = p.causal ? gk : (long long)__ldg(p.cu + sg);
      rq_hi = __ldg(p.cu + sg + 1);
    }
    float* lse_s = reinterpret_cast<float*>(sp + LY::kLse);
    float* d_s = reinterpret_cast<float*>(sp + LY::kDv);
    const float* lse_bh = p.lse + (long long)k.b * p.l_sb + (long long)k.h * p.l_sh;
    const float* D_bh = p.Dsum + ((long long)k.b * p.H + k.h) * p.S;
    bool ok = true;
    int i = 0;
    walk_qtiles(p, k, [&](int r, int qt) {
      const int i0 = qt * kTileM;
      const int buf = i & 1;
      {
        const int qi = i0 + tid;
        const bool qv = qi < p.L;
        const long long pos = (long long)r * p.L + qi;
        lse_s[buf * 128 + tid] = qv ? lse_bh[pos * p.l_ss] * 1.4426950408889634f : INFINITY;
        d_s[buf * 128 + tid] = qv ? D_bh[pos] : 0.f;
      }
      // all 128 rows staged (a bounded wait, unlike bar.sync, so an abort cannot strand a warp)
      mbar_arrive(BAR(C_STATS_READY + buf));
      if (!wait_warp(BAR(C_STATS_READY + buf), (i >> 1) & 1, abort_flag, p.ctl, 43) ||
          !wait_warp(BAR(C_S_FULL), i & 1, abort_flag, p.ctl, 36)) {
        ok = false;
        return false;
      }
      // P^T / dS^T buffers are free once the previous tile's dQ MMA (their last reader) is done
      if (i > 0 && !wait_warp(BAR(C_DQ_FULL), (i - 1) & 1, abort_flag, p.ctl, 37)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      int c_lo = 0, c_hi = 0;
      if (valid_k) {
        const int ilim = min(kTileM, p.L - i0);
        c_hi = ilim;
        if (p.cu) {
          const long long base = (long long)r * p.L + i0;
          const long long lo = rq_lo - base, hi = rq_hi - base;
          c_lo = (int)(lo < 0 ? 0 : (lo > kTileM ? kTileM : lo));
          c_hi = (int)(hi < 0 ? 0 : (hi > ilim ? ilim : hi));
        } else if (p.causal) {
          const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, gk - 1) + 1;
          c_lo = max(0, imin - i0);
        }
      }
      const bool full = qtile_full(p, k, r, qt);
      const float* ls = lse_s + buf * 128;
      const float* dsv = d_s + buf * 128;
      uint8_t* pt = sp + LY::kPT;
      uint8_t* dst = sp + LY::kDST;
#pragma unroll
      for (int ch = 0; ch < kTileM / 32; ++ch) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tl + LY::kTmemS + ch * 32, sr);
        tmem_ld32(tl + LY::kTmemDP + ch * 32, dr);
        tmem_ld_wait(sr);
        tmem_ld_wait(dr);
        float pv[32], dv[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = ch * 32 + c;
          float pp = fast_exp2(__uint_as_float(sr[c]) * p.scale_log2 - ls[col]);
          if (!full) pp = (col >= c_lo && col < c_hi) ? pp : 0.f;
          pv[c] = pp;
          dv[c] = pp * (__uint_as_float(dr[c]) - dsv[col]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k16 = ch * 4 + u;
          const uint32_t off = (k16 >> 3) * kBox + sw128_offset(jr, k16 & 7);
          uint4 a, b2;
          a.x = pack_bf16x2(pv[8 * u + 0], pv[8 * u + 1]);
          a.y = pack_bf16x2(pv[8 * u + 2], pv[8 * u + 3]);
          a.z = pack_bf16x2(pv[8 * u + 4], pv[8 * u + 5]);
          a.w = pack_bf16x2(pv[8 * u + 6], pv[8 * u + 7]);
          b2.x = pack_bf16x2(dv[8 * u + 0], dv[8 * u + 1]);
          b2.y = pack_bf16x2(dv[8 * u + 2], dv[8 * u + 3]);
          b2.z = pack_bf16x2(dv[8 * u + 4], dv[8 * u + 5]);
          b2.w = pack_bf16x2(dv[8 * u + 6], dv[8 * u + 7]);
          *reinterpret_cast<uint4*>(pt + off) = a;
          *reinterpret_cast<uint4*>(dst + off) = b2;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(C_P_FULL));
      ++i;
      return true;
    });
    // ---------------- epilogue: dV, dK rows (bf16)
    const long long prow = (long long)k.s * p.L + j;
    __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + (long long)k.b * p.v_sb +
                         (long long)k.h * p.v_sh + prow * p.v_ss;
    __nv_bfloat16* dkp = reinterpret_cast<__nv_bfloat16*>(p.dk) + (long long)k.b * p.k_sb +
                         (long long)k.h * p.k_sh + prow * p.k_ss;
    if (n_tiles > 0) {
      if (ok && wait_warp(BAR(C_DQ_FULL), (n_tiles - 1) & 1, abort_flag, p.ctl, 38)) {
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t col0 = part == 0 ? LY::kTmemDV : LY::kTmemDK;
          const float mul = part == 0 ? 1.f : p.scale;
          __nv_bfloat16* outp = part == 0 ? dvp : dkp;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tl + col0 + c * 32, o);
            tmem_ld_wait(o);
            if (valid_k) {
              uint4* d4 = reinterpret_cast<uint4*>(outp + c * 32);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * mul, __uint_as_float(o[8 * u + 1]) * mul);
                v.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * mul, __uint_as_float(o[8 * u + 3]) * mul);
                v.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * mul, __uint_as_float(o[8 * u + 5]) * mul);
                v.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * mul, __uint_as_float(o[8 * u + 7]) * mul);
                d4[u] = v;
              }
            }
          }
        }
      }
    } else if (valid_k) {
      for (int u = 0; u < D / 8; ++u) {
        reinterpret_cast<uint4*>(dvp)[u] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(dkp)[u] = make_uint4(0, 0, 0, 0);
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ accumulation
    const int qr = (warp - 8) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float* acc_bh = p.dq_acc + ((long long)k.b * p.H + k.h) * (long long)p.S * D;
    int i = 0;
    walk_qtiles(p, k, [&](int r, int qt) {
      if (!wait_warp(BAR(C_DQ_FULL), i & 1, abort_flag, p.ctl, 39)) return false;
      tc_fence_after();
      const int qi = qt * kTileM + qr;
      const bool qv = qi < p.L;
      float* dst = acc_bh + ((long long)r * p.L + qi) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + LY::kTmemDQ + c * 32, o);
        tmem_ld_wait(o);
        if (qv) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float4 v = make_float4(__uint_as_float(o[4 * u]) * p.scale, __uint_as_float(o[4 * u + 1]) * p.scale,
                                   __uint_as_float(o[4 * u + 2]) * p.scale, __uint_as_float(o[4 * u + 3]) * p.scale);
            atomicAdd(reinterpret_cast<float4*>(dst + c * 32 + 4 * u), v);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(C_DQ_FREE));
      ++i;
      return true;
    });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
  using LY = BwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(ring_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(p.N * p.n_ktiles), (unsigned)(p.B * p.H));
  ring_bwd_kernel<D><<<grid, 384, LY::kAlloc, st>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_smem_bytes(int D) { return D == 64 ? BwdLayout<64>::kAlloc : BwdLayout<128>::kAlloc; }

cudaError_t launch_bwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
  if (D == 64) return launch_bwd_t<64>(tq, tk, tv, tdo, p, st);
  return launch_bwd_t<128>(tq, tk, tv, tdo, p, st);
}

}  // namespace ra
