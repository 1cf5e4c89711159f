// The dQ pass of the ring-attention backward as a persistent kernel.
//
// The work is that of ring_dq_kernel (ra_bwd.cu): per 128-row query tile of Q
// shard r, walk the KV shards (r - t) mod N in ring order (guijiagi.com "Ring
// Attention：突破百万 Token 上下文的分布式注意力", "详细流程") and, with P
// recomputed from the saved log-sum-exp ("Ring Flash Attention" README: "use
// the softmax_lse output"), accumulate dQ = scale * sum_j dS_j K_j in tensor
// memory, dS = P * (dO V^T - D).
//
// Here a CTA does not end with its query tile.  The grid is launched as before
// (one CTA per query tile, in the same order); a running CTA asks the hardware
// (cluster launch control) to cancel the launch of a CTA that has not started
// and takes over its query tile.  The hardware's order and load balance stay,
// and the set-up of the next tile overlaps the current one: its Q and dO are
// loaded and copied into tensor memory while the current tile's last key tiles
// run, its first S and dP MMAs issue while the current tile's dQ is written out,
// and the K / V rings and the S / dP hand-over run on across tiles.  With short
// tiles (packed varlen sequences: ~16 key tiles, ~26 us) a one-tile CTA spends
// ~22 % of its life in that set-up, a tail and the gap to the next CTA.
//
// Warps: 0 scheduler and TMA producer (Q, dO once per tile, K into a 3-stage
// ring), 3 TMA producer (V into a 2-stage ring), 1 MMA, 2 TMEM; warpgroups 1 and
// 2: one query row each, key columns [0, 64) and [64, 128).  TMEM: S [0,128),
// dP [128,256), Q [256, 256+D/2), dO [256+D/2, 256+D), dQ [384, 384+D).  The
// query tiles reach the other roles through a two-slot queue in shared memory.
#include "ra_bwd_common.cuh"

namespace ra {
namespace {

using bwd::kBox;
using bwd::pcol;

constexpr int kThreads = 384;

template <int D>
struct DqpLayout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kK = kDO + kTile;
  static constexpr int kV = kK + kKStages * kTile;
  static constexpr int kBar = kV + kVStages * kTile;
  static constexpr int kNumBars = 26;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, abort flag, 2 item slots, CLC response
  static constexpr int kItems = kMisc + 16;          // 2 x (bx, by)
  static constexpr int kClc = kItems + 16;           // 16-byte aligned response
  static constexpr int kAlloc = kClc + 16 + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemQ = 256, kTmemDO = 256 + D / 2, kTmemDQ = 384;
  static_assert(kClc % 16 == 0, "the cluster-launch-control response must be 16-byte aligned");
};

enum DqpBar {
  G_QDO_FULL = 0,
  G_K_FULL = 1,    // 3
  G_K_EMPTY = 4,   // 3
  G_V_FULL = 7,    // 2
  G_V_EMPTY = 9,   // 2
  G_S_FULL = 11,
  G_S_READ = 12,   // 8 elected arrivals
  G_DP_FULL = 13,
  G_DS_FULL = 14,  // 8
  G_QDO_TMEM = 15, // 8: a tile's Q and dO are in TMEM (their smem buffers are free)
  G_DQ_DONE = 16,
  G_DQ_FREE = 17,  // 8: the tile's dQ has left TMEM
  G_ITEM_FULL = 18,   // 2
  G_ITEM_EMPTY = 20,  // 2, 10 elected arrivals (warps 1, 3 and the 8 elementwise warps)
  G_CLC = 22,
  G_TEARDOWN = 23
};
constexpr uint32_t kItemReaders = 10;

// Query tile of a launch index (bx of grid width gx): shard r, first row i0.
// Causal grids start from the heavy (late) tiles, by chunk for the batched
// zigzag split; the same order as the one-tile-per-CTA kernel.
template <bool VL>
__device__ __forceinline__ void dq_item(const BwdParamsT<VL>& p, int bx, int gx, int& r, int& i0) {
  if (!VL && p.causal && p.layout == LAYOUT_ZIGZAG && p.r_only < 0 && p.L % (2 * kTileM) == 0) {
    int qt;
    zigzag_heavy_first(bx, p.N, p.n_qtiles / 2, r, qt);
    i0 = qt * kTileM;
  } else {
    const int x = p.causal ? gx - 1 - bx : bx;
    r = p.r_only >= 0 ? p.r_only : x / p.n_qtiles;
    i0 = (x % p.n_qtiles) * kTileM;
  }
}

// Per tile: shard, rows, key-tile count.  Called by whole warps (varlen searches are warp-wide).
template <bool VL>
struct DqItem {
  int b, h, r, i0, n_tiles;
  QRange qr;
};

template <bool VL>
__device__ __forceinline__ void dq_item_setup(const BwdParamsT<VL>& p, int bx, int by, DqItem<VL>& it) {
  it.b = by / p.H;
  it.h = by % p.H;
  dq_item(p, bx, (int)gridDim.x, it.r, it.i0);
  make_qrange(p, it.r, it.i0, kTileM, it.qr);
  const int nkt = (p.L + kTileN - 1) / kTileN;
  int n = 0;
  walk_kv_tiles(p, it.qr, nkt, 0, p.N, [&](int, int) {
    ++n;
    return true;
  });
  it.n_tiles = n;
}

// A role's wait for query tile k in the queue; returns (bx, by) with bx < 0 at the end.
__device__ __forceinline__ bool take_item(uint32_t full_bar, const volatile int* slot, int k, volatile int* abort_flag,
                                          const DevCtl& ctl, int site, int& bx, int& by) {
  if (!wait_warp(full_bar, (uint32_t)(k >> 1) & 1u, abort_flag, ctl, site)) return false;
  bx = slot[0];
  by = slot[1];
  return true;
}

template <int D, bool VL>
__global__ void __launch_bounds__(kThreads, 1)
    ring_dq_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                           const BwdParamsT<VL> p) {
  using LY = DqpLayout<D>;
  constexpr int KS = LY::kKStages, VS = LY::kVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkt = (p.L + kTileN - 1) / kTileN;

  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);
  volatile int* items = reinterpret_cast<volatile int*>(sp + LY::kItems);  // slot s: items[2 s], items[2 s + 1]
  const uint32_t clc_resp = sb + LY::kClc;
  if (threadIdx.x == 0) {
    mbar_init(BAR(G_QDO_FULL), 1);
    for (int i = 0; i < KS; ++i) {
      mbar_init(BAR(G_K_FULL + i), 1);
      mbar_init(BAR(G_K_EMPTY + i), 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(BAR(G_V_FULL + i), 1);
      mbar_init(BAR(G_V_EMPTY + i), 1);
    }
    mbar_init(BAR(G_S_FULL), 1);
    mbar_init(BAR(G_S_READ), 8);
    mbar_init(BAR(G_DP_FULL), 1);
    mbar_init(BAR(G_DS_FULL), 8);
    mbar_init(BAR(G_QDO_TMEM), 8);
    mbar_init(BAR(G_DQ_DONE), 1);
    mbar_init(BAR(G_DQ_FREE), 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(G_ITEM_FULL + i), 1);
      mbar_init(BAR(G_ITEM_EMPTY + i), kItemReaders);
    }
    mbar_init(BAR(G_CLC), 1);
    mbar_init(BAR(G_TEARDOWN), 1);
    *abort_flag = 0;
    // the launch's own query tile is the first in the queue
    items[0] = (int)blockIdx.x;
    items[1] = (int)blockIdx.y;
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
  if (threadIdx.x == 0) mbar_arrive(BAR(G_ITEM_FULL));
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer (Q, dO, K)
    int k = 0, kl = 0, jk = 0;  // tiles taken, tiles with key tiles (Q / dO loads), K tiles issued
    int issued_k[KS] = {};
    bool clc_live = true, ok = true;
    int bx = (int)blockIdx.x, by = (int)blockIdx.y;
    while (ok) {
      DqItem<VL> it;
      dq_item_setup(p, bx, by, it);
      int nbx = -1, nby = 0;
      if (lane == 0) {
        // ask for the next query tile now: the answer is in by the time this one's loads are issued
        if (clc_live) {
          mbar_expect_tx(BAR(G_CLC), 16);
          clc_try_cancel(clc_resp, BAR(G_CLC));
        }
        if (it.n_tiles > 0) {
          // the Q / dO buffers are free once the previous tile's rows are in TMEM
          if (kl > 0 && !wait_one(BAR(G_QDO_TMEM), (uint32_t)(kl - 1) & 1u, abort_flag, p.ctl, 100)) ok = false;
          if (ok) {
            const int qrow = it.r * p.L + it.i0 - p.q_base;
            mbar_expect_tx(BAR(G_QDO_FULL), 2 * LY::kTile);
            for (int c = 0; c < D / 64; ++c)
              if (in_bounds(tma_coords_ok(TmaExtent{D, p.q_rows, p.H, p.B}, c * 64, qrow, it.h, it.b), p.ctl, 40)) {
                tma_load_4d(sb + LY::kQ + c * kBox, &tmQ, BAR(G_QDO_FULL), c * 64, qrow, it.h, it.b);
                tma_load_4d(sb + LY::kDO + c * kBox, &tmDO, BAR(G_QDO_FULL), c * 64, qrow, it.h, it.b);
              }
            ++kl;
          }
        }
        // publish the next tile (or the end) once the slot's previous reading is released
        if (clc_live) {
          // always take the answer: it must not land after the CTA has left
          drain_one(BAR(G_CLC), (uint32_t)k & 1u, p.ctl, 101);
          if (!clc_query(clc_resp, nbx, nby)) {
            clc_live = false;
            nbx = -1;
          }
        }
        if (!ok) nbx = -1;
        const int ns = (k + 1) & 1;
        if (k + 1 >= 2 && !wait_one(BAR(G_ITEM_EMPTY + ns), (uint32_t)((k + 1) / 2 - 1) & 1u, abort_flag, p.ctl, 102)) {
          nbx = -1;
          ok = false;
        }
        items[2 * ns] = nbx;
        items[2 * ns + 1] = nby;
        mbar_arrive(BAR(G_ITEM_FULL + ns));
        // the tile's K tiles into the ring (stages and phases run on across tiles)
        if (ok && it.n_tiles > 0) {
          walk_kv_tiles(p, it.qr, nkt, 0, p.N, [&](int s, int kt) {
            const int st = jk % KS;
            if (jk >= KS && !wait_one(BAR(G_K_EMPTY + st), (uint32_t)(jk / KS - 1) & 1u, abort_flag, p.ctl, 103)) {
              ok = false;
              return false;
            }
            mbar_expect_tx(BAR(G_K_FULL + st), LY::kTile);
            for (int c = 0; c < D / 64; ++c)
              if (in_bounds(tma_coords_ok(TmaExtent{D, p.S, p.H, p.B}, c * 64, s * p.L + kt * kTileN, it.h, it.b),
                            p.ctl, 41))
                tma_load_4d(sb + LY::kK + st * LY::kTile + c * kBox, &tmK, BAR(G_K_FULL + st), c * 64,
                            s * p.L + kt * kTileN, it.h, it.b);
            ++issued_k[st];
            ++jk;
            return true;
          });
        }
      }
      nbx = __shfl_sync(0xffffffffu, nbx, 0);
      nby = __shfl_sync(0xffffffffu, nby, 0);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++k;
      if (nbx < 0) break;
      bx = nbx;
      by = nby;
    }
    if (lane == 0) {
      // every issued copy lands before the CTA may exit
      if (kl > 0) drain_one(BAR(G_QDO_FULL), (uint32_t)(kl - 1) & 1u, p.ctl, 104);
      for (int st = 0; st < KS; ++st)
        if (issued_k[st]) drain_one(BAR(G_K_FULL + st), (uint32_t)(issued_k[st] - 1) & 1u, p.ctl, 104);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ TMA producer (V)
    int k = 0, jv = 0;
    int issued_v[VS] = {};
    bool ok = true;
    while (ok) {
      int bx, by;
      if (!take_item(BAR(G_ITEM_FULL + (k & 1)), items + 2 * (k & 1), k, abort_flag, p.ctl, 105, bx, by)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(G_ITEM_EMPTY + (k & 1)));
      ++k;
      if (bx < 0) break;
      DqItem<VL> it;
      dq_item_setup(p, bx, by, it);
      if (lane == 0 && it.n_tiles > 0) {
        walk_kv_tiles(p, it.qr, nkt, 0, p.N, [&](int s, int kt) {
          const int st = jv % VS;
          if (jv >= VS && !wait_one(BAR(G_V_EMPTY + st), (uint32_t)(jv / VS - 1) & 1u, abort_flag, p.ctl, 106)) {
            ok = false;
            return false;
          }
          mbar_expect_tx(BAR(G_V_FULL + st), LY::kTile);
          for (int c = 0; c < D / 64; ++c)
            if (in_bounds(tma_coords_ok(TmaExtent{D, p.S, p.H, p.B}, c * 64, s * p.L + kt * kTileN, it.h, it.b),
                          p.ctl, 42))
              tma_load_4d(sb + LY::kV + st * LY::kTile + c * kBox, &tmV, BAR(G_V_FULL + st), c * 64,
                          s * p.L + kt * kTileN, it.h, it.b);
          ++issued_v[st];
          ++jv;
          return true;
        });
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0)
      for (int st = 0; st < VS; ++st)
        if (issued_v[st]) drain_one(BAR(G_V_FULL + st), (uint32_t)(issued_v[st] - 1) & 1u, p.ctl, 107);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileN, 0, 0);  // S = Q K^T, dP = dO V^T: TMEM A, K-major B
    constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 0, 1);       // dQ += dS K: TMEM A, MN-major B
    int k = 0, kl = 0, jt = 0;  // tiles taken, tiles with key tiles, key tiles over all tiles
    bool ok = true;
    // X = A B^T over D with A (Q or dO) packed in TMEM, 16 head-dim columns = 8 TMEM columns per step
    auto issue_t = [&](uint32_t dcol, uint32_t acol, uint32_t bt) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
        mma_bf16_ts(tmem + dcol, tmem + acol + 8 * kk, sdesc_sw128(bt + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
      }
    };
    // S of the CTA's key tile g (over all its query tiles), once S of g - 1 is read
    auto issue_s = [&](int g) -> bool {
      const int ks = g % KS;
      if (!wait_one(BAR(G_K_FULL + ks), (uint32_t)(g / KS) & 1u, abort_flag, p.ctl, 108)) return false;
      if (g > 0 && !wait_one(BAR(G_S_READ), (uint32_t)(g - 1) & 1u, abort_flag, p.ctl, 109)) return false;
      tc_fence_after();
      issue_t(LY::kTmemS, LY::kTmemQ, sb + LY::kK + ks * LY::kTile);
      mma_commit(BAR(G_S_FULL));
      return true;
    };
    // dP(g) overwrites dS(g - 1), which the dQ MMA issued before it has read
    auto issue_dp = [&](int g) -> bool {
      const int vs = g % VS;
      if (!wait_one(BAR(G_V_FULL + vs), (uint32_t)(g / VS) & 1u, abort_flag, p.ctl, 110)) return false;
      tc_fence_after();
      issue_t(LY::kTmemDP, LY::kTmemDO, sb + LY::kV + vs * LY::kTile);
      mma_commit(BAR(G_DP_FULL));
      mma_commit(BAR(G_V_EMPTY + vs));  // the ring runs on into the next query tiles
      return true;
    };
    auto issue_dq = [&](int g, bool first) -> bool {
      if (!wait_one(BAR(G_DS_FULL), (uint32_t)g & 1u, abort_flag, p.ctl, 111)) return false;
      tc_fence_after();
      const uint32_t kb = sb + LY::kK + (g % KS) * LY::kTile;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_bf16_ts(tmem + LY::kTmemDQ, tmem + LY::kTmemDP + pcol(kk), sdesc_sw128(kb + kk * 2048, kBox, 1024), kIdQ,
                    (!first || kk > 0) ? 1u : 0u);
      mma_commit(BAR(G_K_EMPTY + g % KS));
      return true;
    };
    while (ok) {
      int bx, by;
      if (!take_item(BAR(G_ITEM_FULL + (k & 1)), items + 2 * (k & 1), k, abort_flag, p.ctl, 112, bx, by)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(G_ITEM_EMPTY + (k & 1)));
      ++k;
      if (bx < 0) break;
      DqItem<VL> it;
      dq_item_setup(p, bx, by, it);
      const int n = it.n_tiles;
      if (lane == 0 && n > 0) {
        // the tile's Q and dO are in TMEM (which also means the last tile's S and dP are done)
        ok = wait_one(BAR(G_QDO_TMEM), (uint32_t)kl & 1u, abort_flag, p.ctl, 113);
        if (ok) {
          tc_fence_after();
          ok = issue_s(jt) && issue_dp(jt);
        }
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n) ok = issue_s(jt + j + 1);
          // the first dQ MMA of a tile overwrites the accumulator: the last tile's dQ must have left it
          if (ok && j == 0 && kl > 0) {
            ok = wait_one(BAR(G_DQ_FREE), (uint32_t)(kl - 1) & 1u, abort_flag, p.ctl, 114);
            tc_fence_after();
          }
          ok = ok && issue_dq(jt + j, j == 0);
          if (ok && j + 1 < n) ok = issue_dp(jt + j + 1);
        }
        if (ok) mma_commit(BAR(G_DQ_DONE));
        ++kl;
      }
      jt += n;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      mma_commit(BAR(G_TEARDOWN));
      drain_one(BAR(G_TEARDOWN), 0, p.ctl, 115);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P and dS, half a query row per thread
    const int half = (warp - 4) >> 2;  // key columns [64 half, 64 half + 64)
    const int row = ((warp - 4) & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
    const int* rmap = VL ? p.row_map : nullptr;  // varlen in original order: rows of the caller's layout
    int k = 0, kl = 0, jt = 0;
    bool ok = true;
    // the previous tile's dQ rows leave TMEM after this tile's Q and dO went in
    bool pend = false;
    long long pend_row = 0;  // row of dq, -1 when the row is padding
    __nv_bfloat16* pend_base = nullptr;
    auto epilogue = [&]() -> bool {
      if (!wait_warp(BAR(G_DQ_DONE), (uint32_t)(kl - 1) & 1u, abort_flag, p.ctl, 116)) return false;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + LY::kTmemDQ + half * (D / 2) + 32 * c, o);
        tmem_ld_wait(o);
        if (pend_row >= 0) {
          const long long dr = rmap ? (long long)__ldg(rmap + pend_row) : pend_row;
          uint4* dst = reinterpret_cast<uint4*>(pend_base + dr * p.q_ss + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * p.scale, __uint_as_float(o[8 * u + 1]) * p.scale);
            w.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * p.scale, __uint_as_float(o[8 * u + 3]) * p.scale);
            w.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * p.scale, __uint_as_float(o[8 * u + 5]) * p.scale);
            w.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * p.scale, __uint_as_float(o[8 * u + 7]) * p.scale);
            dst[u] = w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(G_DQ_FREE));
      return true;
    };
    while (ok) {
      int bx, by;
      if (!take_item(BAR(G_ITEM_FULL + (k & 1)), items + 2 * (k & 1), k, abort_flag, p.ctl, 117, bx, by)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(G_ITEM_EMPTY + (k & 1)));
      ++k;
      if (bx < 0) break;
      DqItem<VL> it;
      dq_item_setup(p, bx, by, it);
      const int i = it.i0 + row;
      const bool valid = i < p.L;
      RowWin win;
      int gq = 0;
      if constexpr (VL)
        make_row_win(p, it.r, min(i, p.L - 1), false, win);
      else
        gq = tok(p, it.r, valid ? i : max(it.qr.i_last, 0));
      const long long qrow = (long long)it.r * p.L + i - p.q_base;
      __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.dq) + (long long)it.b * p.q_sb +
                            (long long)it.h * p.q_sh + half * (D / 2);
      const bool store_ok = valid && in_bounds(qrow >= 0 && qrow < p.q_rows, p.ctl, 43);
      if (it.n_tiles > 0) {
        // this row's statistics, negated (padding rows: -lse2 = -inf, -D = 0, so P = dS = 0)
        const long long srow = (((long long)it.b * p.H + it.h) * p.stat_N + (it.r - p.stat_r0)) * p.stat_L + i;
        const uint64_t nl2 = f32x2(__ldg(p.nlse2 + srow), __ldg(p.nlse2 + srow));
        const uint64_t nD2 = f32x2(__ldg(p.nD + srow), __ldg(p.nD + srow));
        // Q (warpgroup 1) or dO (warpgroup 2) of the row into TMEM as packed bf16
        if (!wait_warp(BAR(G_QDO_FULL), (uint32_t)kl & 1u, abort_flag, p.ctl, 118)) break;
        const uint8_t* src = sp + (half == 0 ? LY::kQ : LY::kDO);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + c * kBox + row * 128 + ((q ^ (row & 7)) << 4));
            w[4 * q] = x.x;
            w[4 * q + 1] = x.y;
            w[4 * q + 2] = x.z;
            w[4 * q + 3] = x.w;
          }
          tmem_st32(tl + (half == 0 ? LY::kTmemQ : LY::kTmemDO) + 32 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(G_QDO_TMEM));
        if (pend) {
          if (!epilogue()) break;
          pend = false;
        }
        int j = 0;
        walk_kv_tiles(p, it.qr, nkt, 0, p.N, [&](int s, int kt) {
          const int g = jt + j;
          int c_lo = 0, c_hi = kTileN;
          if constexpr (VL)
            row_win_cols(p, win, s, kt * kTileN, kTileN, c_lo, c_hi);
          else if (!kv_tile_full(p, it.qr, s, kt))
            row_key_window(p, gq, s, kt, c_lo, c_hi);
          c_lo -= 64 * half;
          c_hi -= 64 * half;
          const bool masked = c_lo > 0 || c_hi < 64;
          if (!wait_warp(BAR(G_S_FULL), (uint32_t)g & 1u, abort_flag, p.ctl, 119)) {
            ok = false;
            return false;
          }
          tc_fence_after();
          uint32_t v[64];
          bwd::tmem_ld64(tl + LY::kTmemS + 64 * half, v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(G_S_READ));
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), sc2, nl2), x0, x1);
            v[c] = __float_as_uint(fast_exp2(x0));
            v[c + 1] = __float_as_uint(fast_exp2(x1));
          }
          if (masked) {
            const uint64_t mw = bit_window64(c_lo, c_hi);
#pragma unroll
            for (int c = 0; c < 64; ++c) v[c] = ((mw >> c) & 1ull) ? v[c] : 0u;
          }
          if (!wait_warp(BAR(G_DP_FULL), (uint32_t)g & 1u, abort_flag, p.ctl, 120)) {
            ok = false;
            return false;
          }
          tc_fence_after();
          // dS = P * (dP - D), packed over the first 32 of this thread's 64 dP columns
          const uint32_t tdp = tl + LY::kTmemDP + 64 * half;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t d[32];
            tmem_ld32(tdp + 32 * hh, d);
            tmem_ld_wait(d);
            uint32_t pk[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int c = 32 * hh + 2 * u;
              float s0, s1;
              f32x2_split(mul_f32x2(f32x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                    add_f32x2(f32x2(__uint_as_float(d[2 * u]), __uint_as_float(d[2 * u + 1])), nD2)),
                          s0, s1);
              pk[u] = pack_bf16x2(s0, s1);
            }
            tmem_st16(tdp + 16 * hh, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(G_DS_FULL));
          ++j;
          return true;
        });
        if (!ok) break;
        pend = true;
        pend_row = store_ok ? qrow : -1;
        pend_base = base;
        ++kl;
      } else {
        if (pend) {
          if (!epilogue()) break;
          pend = false;
        }
        if (store_ok) {  // no key tile at all: dq = 0
          __nv_bfloat16* dst = base + (rmap ? (long long)__ldg(rmap + qrow) : qrow) * p.q_ss;
          for (int u = 0; u < D / 16; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
        }
      }
      jt += it.n_tiles;
    }
    if (ok && pend) epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool VL>
cudaError_t launch_v(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                     const BwdParams& p, cudaStream_t st) {
  BwdParamsT<VL> pv;
  static_cast<BwdParams&>(pv) = p;
  cudaError_t e = configure_kernel<ring_dq_persist_kernel<D, VL>>(0, DqpLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.r_only >= 0 ? 1 : p.N) * p.n_qtiles), (unsigned)(p.B * p.H));
  ring_dq_persist_kernel<D, VL><<<grid, kThreads, DqpLayout<D>::kAlloc, st>>>(tq, tk, tv, tdo, pv);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                     const BwdParams& p, cudaStream_t st) {
  return p.cu ? launch_v<D, true>(tq, tk, tv, tdo, p, st) : launch_v<D, false>(tq, tk, tv, tdo, p, st);
}

}  // namespace

cudaError_t launch_dq_persist(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
  if (D == 64) return launch_t<64>(tq, tk, tv, tdo, p, st);
  return launch_t<128>(tq, tk, tv, tdo, p, st);
}

}  // namespace ra
