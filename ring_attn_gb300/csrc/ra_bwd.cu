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
// memory for the CTA's whole life; dQ tiles are added in fp32 into a
// workspace accumulator.
//
// Warpgroups (384 threads; per-warpgroup register budgets via setmaxnreg):
//   0  warp 0: TMA producer (K and V once; Q, dO and the tile's lse / D rows
//      into a 2-stage ring); warp 1: MMA issuer; warp 2: TMEM allocation.
//   1  one thread per key row: P^T (written as packed bf16 over its own S^T
//      columns, the A operand of dV += P^T dO straight from TMEM), then
//      dS^T (bf16, 128B-swizzled shared memory, the A operand of dK and dQ),
//      and the dK / dV epilogue.
//   2  loads the dQ tile from TMEM, frees those columns, and adds scale * dQ
//      into the fp32 accumulator.  At d = 128 the tile is computed transposed,
//      dQ^T = K^T dS^T, so TMEM lane = head-dim index and each warp's atomic
//      add covers 128 contiguous bytes of one query row (one L2 transaction
//      instead of 32); at d = 64 one thread per query row adds float4s.
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).
// The dQ tile reuses [128, 256) once dP^T has been consumed.  MMA order per
// query tile i:  S^T(i), dP^T(i) [after dQ(i-1) is read out], then, once P^T
// and dS^T are ready, dQ(i) first (its read-out then overlaps the next MMAs),
// dV(i), dK(i).  S^T(i+1) may overwrite P^T(i) because the MMAs of one thread
// execute in issue order.
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBox = 128 * 128;
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 72;
constexpr int kRegsSm = 232;
constexpr int kRegsDq = 200;
static_assert(128 * (kRegsCtl + kRegsSm + kRegsDq) <= kThreads * kLaunchRegs, "register split exceeds the launch");
constexpr int kStatWin = kTileM;  // lse2 / D floats staged per query tile

template <int D>
struct BwdLayout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;          // 2 stages
  static constexpr int kDO = kQ + 2 * kTile;     // 2 stages
  static constexpr int kDST = kDO + 2 * kTile;   // dS^T: 128 key rows x 128 queries (2 boxes)
  static constexpr int kStats = kDST + 2 * kBox; // 2 stages x (lse2, D) windows
  static constexpr int kStatBytes = kStatWin * 4;
  static constexpr int kBar = kStats + 2 * 2 * kStatBytes;
  static constexpr int kNumBars = 12;  // 11 used
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16;      // the dynamic base is 1024-aligned (checked)
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 256 + D, kTmemDQ = 128;
};

enum BwdBar {
  C_KV_FULL = 0,
  C_QDO_FULL = 1,   // 2
  C_QDO_EMPTY = 3,  // 2
  C_S_FULL = 5,
  C_DP_FULL = 6,
  C_P_FULL = 7,
  C_DQ_FULL = 8,
  C_DQ_FREE = 9,
  C_TEARDOWN = 10,
  C_KV_DONE = 11    // every dV / dK MMA has completed
};

struct KTile {
  int b, h, s, j0, j_last;
  int gk_lo, gk_hi;
  int qry_lo, qry_hi;  // varlen: queries any key of the tile may serve (inclusive)
  int seg_single;
};

__device__ __forceinline__ void q_range(const BwdParams& p, const KTile& k, int r, int& lo, int& hi) {
  const int nqt = p.n_qtiles;
  if (p.cu) {
    const int base = r * p.L;
    int ilo = k.qry_lo - base, ihi = k.qry_hi - base;
    if (ilo < 0) ilo = 0;
    if (ihi > p.L - 1) ihi = p.L - 1;
    if (ilo > ihi) {
      lo = hi = 0;
      return;
    }
    lo = ilo / kTileM;
    hi = ihi / kTileM + 1;
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
    const int base = r * p.L + i0;
    const int slo = __ldg(p.cu + k.seg_single), shi = __ldg(p.cu + k.seg_single + 1);
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
__global__ void __launch_bounds__(kThreads, 1)
    ring_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using LY = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sb = smem_u32(smem_raw);
  if (sb & 1023u) {  // the 128B-swizzled tiles need a 1024-aligned base
    if (threadIdx.x == 0) record_error(p.ctl, DEV_BAD_SMEM, 50);
    return;
  }
  uint8_t* sp = smem_raw;
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
    k.qry_lo = p.causal ? k.gk_lo : __ldg(p.cu + sa);
    k.qry_hi = __ldg(p.cu + sz + 1) - 1;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C_QDO_FULL + i), 1);
      mbar_init(BAR(C_QDO_EMPTY + i), 1);
    }
    mbar_init(BAR(C_S_FULL), 1);
    mbar_init(BAR(C_DP_FULL), 1);
    mbar_init(BAR(C_P_FULL), 4);   // one elected arrival per key-row warp
    mbar_init(BAR(C_DQ_FULL), 1);
    mbar_init(BAR(C_DQ_FREE), 4);  // one elected arrival per query-row warp
    mbar_init(BAR(C_TEARDOWN), 1);
    mbar_init(BAR(C_KV_DONE), 1);
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
  const long long stat_bh = ((long long)k.b * p.H + k.h) * p.N * p.stat_L;  // statistics row of (b, h, shard 0)

  if (warp < 4) {
    regs_dec<kRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && n_tiles > 0) {
        int issued[2] = {0, 0};
        const int krow = k.s * p.L + k.j0;
        mbar_expect_tx(BAR(C_KV_FULL), 2 * LY::kTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sb + LY::kK + c * kBox, &tmK, BAR(C_KV_FULL), c * 64, krow, k.h, k.b);
          tma_load_4d(sb + LY::kV + c * kBox, &tmV, BAR(C_KV_FULL), c * 64, krow, k.h, k.b);
        }
        int i = 0;
        walk_qtiles(p, k, [&](int r, int qt) {
          const int st = i & 1;
          if (i >= 2 && !wait_one(BAR(C_QDO_EMPTY + st), ((i >> 1) - 1) & 1, abort_flag, p.ctl, 31)) return false;
          const int qrow = r * p.L + qt * kTileM;
          // lse2 / D of the tile's 128 query rows: 512-byte aligned in the padded layout
          const long long e0 = stat_bh + (long long)r * p.stat_L + qt * kTileM;
          mbar_expect_tx(BAR(C_QDO_FULL + st), 2 * LY::kTile + 2 * LY::kStatBytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(sb + LY::kQ + st * LY::kTile + c * kBox, &tmQ, BAR(C_QDO_FULL + st), c * 64, qrow, k.h, k.b);
            tma_load_4d(sb + LY::kDO + st * LY::kTile + c * kBox, &tmDO, BAR(C_QDO_FULL + st), c * 64, qrow, k.h,
                        k.b);
          }
          bulk_load(sb + LY::kStats + (st * 2 + 0) * LY::kStatBytes, p.lse2 + e0, LY::kStatBytes,
                    BAR(C_QDO_FULL + st));
          bulk_load(sb + LY::kStats + (st * 2 + 1) * LY::kStatBytes, p.Dsum + e0, LY::kStatBytes,
                    BAR(C_QDO_FULL + st));
          ++issued[st];
          ++i;
          return true;
        });
        drain_one(BAR(C_KV_FULL), 0, p.ctl, 40);
        for (int st = 0; st < 2; ++st)
          if (issued[st]) drain_one(BAR(C_QDO_FULL + st), (issued[st] - 1) & 1, p.ctl, 41);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && n_tiles > 0) {
        constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileM, 0, 0);  // S^T, dP^T: K-major A and B
        constexpr uint32_t kIdKV = idesc_bf16_f32(128, D, 0, 1);      // dV, dK: K-major A, MN-major B
        constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 1, 1);       // dQ: MN-major A and B
        constexpr uint32_t kIdQT = idesc_bf16_f32(D, kTileM, 1, 1);   // dQ^T: MN-major A and B
        bool ok = wait_one(BAR(C_KV_FULL), 0, abort_flag, p.ctl, 32);
        int i = 0;
        if (ok) {
          walk_qtiles(p, k, [&](int, int) {
            const int st = i & 1;
            const uint32_t qb = sb + LY::kQ + st * LY::kTile, ob = sb + LY::kDO + st * LY::kTile;
            if (!wait_one(BAR(C_QDO_FULL + st), (i >> 1) & 1, abort_flag, p.ctl, 33)) {
              ok = false;
              return false;
            }
            tc_fence_after();
            // S^T = K Q^T (its columns held P^T(i-1), already read by dV(i-1), issued earlier)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
              mma_bf16_ss(tmem + LY::kTmemS, sdesc_sw128(sb + LY::kK + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024),
                          kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C_S_FULL));
            // dP^T = V dO^T, once dQ(i-1) has left those columns
            if (i > 0 && !wait_one(BAR(C_DQ_FREE), (i - 1) & 1, abort_flag, p.ctl, 34)) {
              ok = false;
              return false;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
              mma_bf16_ss(tmem + LY::kTmemDP, sdesc_sw128(sb + LY::kV + off, 16, 1024),
                          sdesc_sw128(ob + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C_DP_FULL));
            if (!wait_one(BAR(C_P_FULL), i & 1, abort_flag, p.ctl, 35)) {
              ok = false;
              return false;
            }
            tc_fence_after();
            if constexpr (D == 128) {
#pragma unroll
              for (int kk = 0; kk < kTileN / 16; ++kk) {
                // dQ^T = K^T dS^T: A = K^T (head dim contiguous: MN-major), B = dS^T (queries contiguous: MN-major)
                mma_bf16_ss(tmem + LY::kTmemDQ, sdesc_sw128(sb + LY::kK + kk * 2048, kBox, 1024),
                            sdesc_sw128(sb + LY::kDST + kk * 2048, kBox, 1024), kIdQT, kk > 0 ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < kTileN / 16; ++kk) {
                // dQ = dS K: A = dS (queries contiguous in dS^T: MN-major), B = K (MN-major)
                mma_bf16_ss(tmem + LY::kTmemDQ, sdesc_sw128(sb + LY::kDST + kk * 2048, kBox, 1024),
                            sdesc_sw128(sb + LY::kK + kk * 2048, kBox, 1024), kIdQ, kk > 0 ? 1u : 0u);
              }
            }
            mma_commit(BAR(C_DQ_FULL));
#pragma unroll
            for (int kk = 0; kk < kTileM / 16; ++kk) {
              const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
              // dV += P^T dO: A = P^T from TMEM (8 packed columns per 16 queries), B = dO MN-major
              mma_bf16_ts(tmem + LY::kTmemDV, tmem + LY::kTmemS + kk * 8, sdesc_sw128(ob + kk * 2048, kBox, 1024),
                          kIdKV, acc);
              // dK += dS^T Q: A = dS^T K-major (16 queries = 32 bytes), B = Q MN-major
              mma_bf16_ss(tmem + LY::kTmemDK, sdesc_sw128(sb + LY::kDST + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                          sdesc_sw128(qb + kk * 2048, kBox, 1024), kIdKV, acc);
            }
            if (i + 2 < n_tiles) mma_commit(BAR(C_QDO_EMPTY + st));
            if (i + 1 == n_tiles) mma_commit(BAR(C_KV_DONE));
            ++i;
            return true;
          });
        }
        mma_commit(BAR(C_TEARDOWN));
        drain_one(BAR(C_TEARDOWN), 0, p.ctl, 42);
      }
      __syncwarp();
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T / dS^T per key row
    regs_inc<kRegsSm>();
    const int jr = threadIdx.x - 128;  // 0..127
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int j = k.j0 + jr;
    const bool valid_k = j < p.L;
    const int gk = token_of(p.layout, p.N, p.L, k.s, valid_k ? j : k.j_last);
    int rq_lo = 0, rq_hi = 0;  // varlen: queries [rq_lo, rq_hi) this key serves
    if (p.cu) {
      const int sg = segment_of(p.cu, p.n_seqs, gk);
      rq_lo = p.causal ? gk : __ldg(p.cu + sg);
      rq_hi = __ldg(p.cu + sg + 1);
    }
    uint8_t* dst = sp + LY::kDST;
    bool ok = true;
    int i = 0;
    walk_qtiles(p, k, [&](int r, int qt) {
      const int i0 = qt * kTileM;
      const int st = i & 1;
      // allowed query columns [c_lo, c_hi) of this key row
      int c_lo = 0, c_hi = 0;
      if (valid_k) {
        const int ilim = min(kTileM, p.L - i0);
        c_hi = ilim;
        if (p.cu) {
          const int base = r * p.L + i0;
          const int lo = rq_lo - base, hi = rq_hi - base;
          c_lo = lo < 0 ? 0 : (lo > kTileM ? kTileM : lo);
          c_hi = hi < 0 ? 0 : (hi > ilim ? ilim : hi);
        } else if (p.causal) {
          const int imin = last_local_at_or_before(p.layout, p.N, p.L, r, gk - 1) + 1;
          c_lo = max(0, imin - i0);
        }
      }
      // partial tiles mask columns outside [c_lo, c_hi); padding query rows have
      // lse2 = +inf and D = 0, so they give P = 0 and dS = 0 without a mask
      const bool masked = !qtile_full(p, k, r, qt) && (c_lo > 0 || c_hi < kTileM);
      const float4* ls4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 0) * LY::kStatBytes);
      const float4* ds4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 1) * LY::kStatBytes);
      // the stage's Q / dO / statistics landed before S^T(i) was issued; waiting on
      // the stage barrier too orders this thread's reads after that arrival
      if (!wait_warp(BAR(C_S_FULL), i & 1, abort_flag, p.ctl, 36) ||
          !wait_warp(BAR(C_QDO_FULL + st), (i >> 1) & 1, abort_flag, p.ctl, 44)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      uint32_t v[kTileM];
      tmem_ld32(tl + LY::kTmemS + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
      tmem_ld32(tl + LY::kTmemS + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld32(tl + LY::kTmemS + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld32(tl + LY::kTmemS + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 0));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 96));
      // P^T = exp2(S^T * scale * log2 e - lse2)
#pragma unroll
      for (int c4 = 0; c4 < kTileM / 4; ++c4) {
        const float4 l = ls4[c4];
        v[4 * c4 + 0] = __float_as_uint(fast_exp2(fmaf(__uint_as_float(v[4 * c4 + 0]), p.scale_log2, -l.x)));
        v[4 * c4 + 1] = __float_as_uint(fast_exp2(fmaf(__uint_as_float(v[4 * c4 + 1]), p.scale_log2, -l.y)));
        v[4 * c4 + 2] = __float_as_uint(fast_exp2(fmaf(__uint_as_float(v[4 * c4 + 2]), p.scale_log2, -l.z)));
        v[4 * c4 + 3] = __float_as_uint(fast_exp2(fmaf(__uint_as_float(v[4 * c4 + 3]), p.scale_log2, -l.w)));
      }
      if (masked) {
#pragma unroll
        for (int c = 0; c < kTileM; ++c) v[c] = (c >= c_lo && c < c_hi) ? v[c] : 0u;
      }
      // P^T as bf16 pairs over the first 64 S^T columns (already read): the A operand of dV
#pragma unroll
      for (int c32 = 0; c32 < kTileM / 32; ++c32) {
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(v[c32 * 32 + 2 * u]), __uint_as_float(v[c32 * 32 + 2 * u + 1]));
        tmem_st16(tl + LY::kTmemS + c32 * 16, pk);
      }
      if (!wait_warp(BAR(C_DP_FULL), i & 1, abort_flag, p.ctl, 37)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      // dS^T = P^T * (dP^T - D), 64 columns per TMEM round trip, into the swizzled smem tile
#pragma unroll
      for (int h64 = 0; h64 < 2; ++h64) {
        uint32_t dr[64];
        tmem_ld32(tl + LY::kTmemDP + h64 * 64, *reinterpret_cast<uint32_t(*)[32]>(dr + 0));
        tmem_ld32(tl + LY::kTmemDP + h64 * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(dr + 0));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(dr + 32));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c0 = h64 * 64 + u * 8;
          const float4 d0 = ds4[c0 / 4], d1 = ds4[c0 / 4 + 1];
          const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[c0 + e]) * (__uint_as_float(dr[u * 8 + e]) - dd[e]);
          uint4 w;
          w.x = pack_bf16x2(x[0], x[1]);
          w.y = pack_bf16x2(x[2], x[3]);
          w.z = pack_bf16x2(x[4], x[5]);
          w.w = pack_bf16x2(x[6], x[7]);
          const int k16 = c0 / 8;
          *reinterpret_cast<uint4*>(dst + (k16 >> 3) * kBox + sw128_offset(jr, k16 & 7)) = w;
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(BAR(C_P_FULL));
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
      if (ok && wait_warp(BAR(C_KV_DONE), 0, abort_flag, p.ctl, 38)) {
        tc_fence_after();
#pragma unroll 1
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
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * mul, __uint_as_float(o[8 * u + 1]) * mul);
                w.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * mul, __uint_as_float(o[8 * u + 3]) * mul);
                w.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * mul, __uint_as_float(o[8 * u + 5]) * mul);
                w.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * mul, __uint_as_float(o[8 * u + 7]) * mul);
                d4[u] = w;
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
  } else {
    // ------------------------------------------------------------ dQ accumulation
    regs_inc<kRegsDq>();
    const int rl = (warp - 8) * 32 + lane;  // TMEM lane: head-dim index (d = 128) or query row
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float* acc_bh = p.dq_acc + ((long long)k.b * p.H + k.h) * (long long)p.S * D;
    int i = 0;
    walk_qtiles(p, k, [&](int r, int qt) {
      if (!wait_warp(BAR(C_DQ_FULL), i & 1, abort_flag, p.ctl, 39)) return false;
      tc_fence_after();
      uint32_t o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + LY::kTmemDQ + c * 32, *reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
      // the columns are free as soon as they are in registers
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C_DQ_FREE));
      const int i0 = qt * kTileM;
      const int nvalid = min(kTileM, p.L - i0);
      float* rowp = acc_bh + ((long long)r * p.L + i0) * D;
      if constexpr (D == 128) {
        // lane rl holds dQ^T[rl][0..127]: for each query row the warp adds 32 consecutive floats
#pragma unroll
        for (int c = 0; c < kTileM; ++c)
          if (c < nvalid) atomicAdd(rowp + (long long)c * D + rl, __uint_as_float(o[c]) * p.scale);
      } else {
        if (rl < nvalid) {
          float* dst = rowp + (long long)rl * D;
#pragma unroll
          for (int u = 0; u < D / 4; ++u) {
            const float4 w = make_float4(__uint_as_float(o[4 * u]) * p.scale, __uint_as_float(o[4 * u + 1]) * p.scale,
                                         __uint_as_float(o[4 * u + 2]) * p.scale,
                                         __uint_as_float(o[4 * u + 3]) * p.scale);
            atomicAdd(reinterpret_cast<float4*>(dst + 4 * u), w);
          }
        }
      }
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
  // the register split inside the kernel is only safe with the launch allocation it was sized for
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, ring_bwd_kernel<D>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(ring_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(p.N * p.n_ktiles), (unsigned)(p.B * p.H));
  ring_bwd_kernel<D><<<grid, kThreads, LY::kAlloc, st>>>(tq, tk, tv, tdo, p);
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
