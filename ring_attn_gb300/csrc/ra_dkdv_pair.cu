// dK / dV of the ring-attention backward with CTA pairs (tcgen05 cta_group::2),
// head_dim 128.
//
// The work is that of the one-CTA dK / dV kernel in ra_bwd.cu: per 128-row key
// tile of KV shard s, walk the query tiles of the shards (s + t) mod N in ring
// order (guijiagi.com "Ring Attention：突破百万 Token 上下文的分布式注意力",
// "详细流程"), and with P recomputed from the saved log-sum-exp ("Ring Flash
// Attention" README: "use the softmax_lse output") accumulate
//   S^T = K Q^T,  dP^T = V dO^T,  P^T = exp(S^T - lse),  dS^T = P^T (dP^T - D),
//   dV += P^T dO,  dK += dS^T Q
// in tensor memory.  Here two CTAs on the two SMs of a pair take two adjacent
// key tiles of the same shard and walk the same query tiles, and one thread of
// the even CTA issues every MMA at M = 256 for both.  Each CTA keeps its own
// 128 key rows of A (K, V, or P^T / dS^T in tensor memory) and supplies half of
// the B operand (the query tile's Q or dO), so per MMA an SM reads 6 KB of
// shared memory instead of 8 KB (S^T, dP^T) and 2 KB instead of 4 KB (dK, dV):
// the two shared-memory-fed GEMMs of the one-CTA kernel issue below the tensor
// rate because both operands stream from shared memory.
//
// The B halves.  For S^T and dP^T (N = the 128 queries) CTA c supplies query
// rows [64c, 64c + 64) over all of d; for dK and dV (N = d) it supplies head
// dims [64c, 64c + 64) over all 128 query rows.  Both halves must sit at the
// same shared-memory offsets in the two CTAs, so every Q and dO stage holds four
// 64 x 64 swizzled blocks:
//   X  = rows [64c, 64c + 64) x d [0, 64)      (S^T: K steps 0-3)
//   X2 = rows [64c, 64c + 64) x d [64, 128)    (S^T: K steps 4-7)
//   Y  = rows [0, 64)   x d [64c, 64c + 64)    (dK: query steps 0-3)
//   Y2 = rows [64, 128) x d [64c, 64c + 64)    (dK: query steps 4-7)
// (in the even CTA X and Y hold the same block, loaded twice).
//
// Synchronisation.  Both CTAs load their own K, V, Q, dO blocks; the copies
// signal the even CTA's full barriers (the cta_group::2 form of the tiled
// copy), where the even CTA's producer expects both CTAs' bytes.  Each CTA
// loads the query tile's statistics for its own elementwise warps into its
// own memory.  MMA completions are committed to the barriers of both CTAs
// (multicast), and the elementwise warps of both CTAs arrive on the even CTA's
// "S^T read" and "P^T, dS^T written" barriers.  Every wait is bounded; a
// timeout raises the abort flag of both CTAs.
#include "ra_bwd_common.cuh"

namespace ra {
namespace {

using bwd::kBox;
using bwd::pcol;
using bwd::stat_rows_ok;
using bwd::store_rows_bf16;
using bwd::tmem_ld64;

constexpr int kThreads = 384;
constexpr int kSub = 64 * 128;  // one 64-row x 64-column swizzled block of bf16: 8 KB
constexpr uint16_t kBoth = 3;   // multicast mask: both CTAs of the pair

struct PairLayout {
  static constexpr int D = 128;
  static constexpr int kTile = 2 * kBox;          // 128 rows x 128 columns: 32 KB
  static constexpr int kK = 0;                    // this CTA's 128 key rows, two 64-column boxes
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;           // 2 stages of [X | X2 | Y | Y2]
  static constexpr int kDO = kQ + 2 * kTile;      // 2 stages
  static constexpr int kStats = kDO + 2 * kTile;  // 2 stages x (-lse2, -D), 128 floats each
  static constexpr int kBar = kStats + 2 * 2 * 512;
  static constexpr int kNumBars = 17;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  static constexpr int kX = 0, kX2 = kSub, kY = 2 * kSub;  // blocks of a stage (Y2 = Y + kSub)
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 384;
  static_assert(8 * 32 * D * 2 <= kStats, "output row slots exceed the operand buffers");
};

// Register split (as in the one-CTA kernel): launch allocation kThreads x 168,
// control warpgroup 72, elementwise warpgroups 216; checked at launch.
constexpr int kPairLaunchRegs = 168;
constexpr int kPairRegsLow = 72;
constexpr int kPairRegsHigh = 216;
static_assert(128 * kPairRegsLow + 256 * kPairRegsHigh <= kThreads * kPairLaunchRegs, "register split exceeds the launch");

enum PairBar {
  P_KV_FULL = 0,    // even CTA: K and V of both CTAs
  P_Q_FULL = 1,     // 2, even CTA: a Q stage of both CTAs
  P_DO_FULL = 3,    // 2, even CTA: a dO stage of both CTAs
  P_ST_FULL = 5,    // 2, each CTA: its copy of the tile's -lse2 and -D
  P_Q_EMPTY = 7,    // 2, each CTA: the MMAs that read a Q stage are done
  P_DO_EMPTY = 9,   // 2
  P_S_FULL = 11,    // each CTA
  P_S_READ = 12,    // even CTA: S^T in registers, 16 elected arrivals (8 per CTA)
  P_DP_FULL = 13,   // each CTA
  P_PS_FULL = 14,   // even CTA: P^T and dS^T in tensor memory, 16 elected arrivals
  P_KV_DONE = 15,   // each CTA: every MMA done
  P_TEARDOWN = 16   // each CTA
};

// The four blocks of one Q or dO stage of CTA `c` for the query tile at row qrow
// (e: the tensor's extents, for the debug bounds checks).
__device__ __forceinline__ void load_stage(uint32_t dst, const CUtensorMap* map, uint32_t bar, int qrow, int c, int h,
                                           int b, const TmaExtent& e, const DevCtl& ctl) {
  // rows qrow .. qrow + 64 and head-dim columns 0 and 64 cover all four copies
  if (!in_bounds(tma_coords_ok(e, 0, qrow, h, b) && tma_coords_ok(e, 64, qrow + 64, h, b), ctl, 20)) return;
  tma_load_4d_pair(dst + PairLayout::kX, map, bar, 0, qrow + 64 * c, h, b);
  tma_load_4d_pair(dst + PairLayout::kX2, map, bar, 64, qrow + 64 * c, h, b);
  tma_load_4d_pair(dst + PairLayout::kY, map, bar, 64 * c, qrow, h, b);
  tma_load_4d_pair(dst + PairLayout::kY + kSub, map, bar, 64 * c, qrow + 64, h, b);
}

// blockIdx.x = 2 * (shard * n_pairs + pair) + rank in the pair; blockIdx.y = b * H + h.
template <bool VL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    ring_dkdv_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                          const BwdParamsT<VL> p) {
  using LY = PairLayout;
  constexpr int D = LY::D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();  // 0: the CTA whose thread issues the MMAs
  const int b = blockIdx.y / p.H, h = blockIdx.y % p.H;
  const int n_pairs = (p.n_ktiles + 1) >> 1;
  const int pg = (int)blockIdx.x >> 1;
  const int s = pg / n_pairs;
  const int j0_pair = (pg % n_pairs) * 2 * kTileN;
  const int j0 = j0_pair + crank * kTileN;  // this CTA's key rows [j0, j0 + 128)

  // Both CTAs walk the query tiles of the pair's 256 key rows (the union of
  // what the two tiles meet), in the same order.
  KRange kp;
  make_krange(p, s, j0_pair, kp, 2 * kTileN);
  int n_tiles = 0;
  walk_q_tiles<kTileM>(p, kp, p.n_qtiles, [&](int, int) {
    ++n_tiles;
    return true;
  });

  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const uint32_t lead0 = mapa_shared(bar0, 0);  // the even CTA's barriers
  auto LBAR = [lead0](int i) -> uint32_t { return lead0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  const uint32_t peer_abort = mapa_shared(smem_u32(sp + LY::kMisc + 4), (uint32_t)(crank ^ 1));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);
  if (threadIdx.x == 0) {
    mbar_init(BAR(P_KV_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(P_Q_FULL + i), 1);
      mbar_init(BAR(P_DO_FULL + i), 1);
      mbar_init(BAR(P_ST_FULL + i), 1);
      mbar_init(BAR(P_Q_EMPTY + i), 1);
      mbar_init(BAR(P_DO_EMPTY + i), 1);
    }
    mbar_init(BAR(P_S_FULL), 1);
    mbar_init(BAR(P_S_READ), 16);
    mbar_init(BAR(P_DP_FULL), 1);
    mbar_init(BAR(P_PS_FULL), 16);
    mbar_init(BAR(P_KV_DONE), 1);
    mbar_init(BAR(P_TEARDOWN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {  // collective with warp 2 of the other CTA
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any copy or arrival crosses over
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long stat_bh = ((long long)b * p.H + h) * p.stat_N * p.stat_L;

  if (warp < 4) {
    regs_dec<kPairRegsLow>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (both CTAs)
      if (lane == 0 && n_tiles > 0) {
        int issued[2] = {0, 0};
        const int krow = s * p.L + j0;
        if (crank == 0) mbar_expect_tx(BAR(P_KV_FULL), 4 * LY::kTile);  // K and V of both CTAs
        const TmaExtent ek{D, p.S, p.H, p.B}, eq{D, p.q_rows, p.H, p.B};
        for (int c = 0; c < D / 64; ++c)
          for (int hr = 0; hr < 2; ++hr)
            if (in_bounds(tma_coords_ok(ek, c * 64, krow + 64 * hr, h, b), p.ctl, 21)) {
              tma_load_4d_pair(sb + LY::kK + c * kBox + hr * kSub, &tmK, LBAR(P_KV_FULL), c * 64, krow + 64 * hr, h, b);
              tma_load_4d_pair(sb + LY::kV + c * kBox + hr * kSub, &tmV, LBAR(P_KV_FULL), c * 64, krow + 64 * hr, h, b);
            }
        int i = 0;
        walk_q_tiles<kTileM>(p, kp, p.n_qtiles, [&](int r, int qt) {
          const int st = i & 1;
          const uint32_t par = ((i >> 1) - 1) & 1;
          const int qrow = r * p.L + qt * kTileM - p.q_base;
          if (i >= 2 && !wait_one_pair(BAR(P_Q_EMPTY + st), par, abort_flag, peer_abort, p.ctl, 81)) return false;
          // -lse2 / -D of the tile's 128 query rows: 512-byte aligned in the padded layout
          const long long e0 = stat_bh + (long long)(r - p.stat_r0) * p.stat_L + qt * kTileM;
          mbar_expect_tx(BAR(P_ST_FULL + st), 2 * 512);
          if (in_bounds(stat_rows_ok(p, e0), p.ctl, 22)) {
            bulk_load(sb + LY::kStats + (st * 2 + 0) * 512, p.nlse2 + e0, 512, BAR(P_ST_FULL + st));
            bulk_load(sb + LY::kStats + (st * 2 + 1) * 512, p.nD + e0, 512, BAR(P_ST_FULL + st));
          }
          if (crank == 0) mbar_expect_tx(BAR(P_Q_FULL + st), 2 * LY::kTile);
          load_stage(sb + LY::kQ + st * LY::kTile, &tmQ, LBAR(P_Q_FULL + st), qrow, crank, h, b, eq, p.ctl);
          if (i >= 2 && !wait_one_pair(BAR(P_DO_EMPTY + st), par, abort_flag, peer_abort, p.ctl, 82)) {
            drain_one_pair(BAR(P_ST_FULL + st), (i >> 1) & 1, p.ctl, 83);
            if (crank == 0) drain_one_pair(BAR(P_Q_FULL + st), (i >> 1) & 1, p.ctl, 83);
            return false;
          }
          if (crank == 0) mbar_expect_tx(BAR(P_DO_FULL + st), 2 * LY::kTile);
          load_stage(sb + LY::kDO + st * LY::kTile, &tmDO, LBAR(P_DO_FULL + st), qrow, crank, h, b, eq, p.ctl);
          ++issued[st];
          ++i;
          return true;
        });
        // the even CTA's full barriers collect both CTAs' copies: once they
        // complete, nothing is in flight into either CTA's memory
        if (crank == 0) drain_one_pair(BAR(P_KV_FULL), 0, p.ctl, 84);
        for (int st = 0; st < 2; ++st)
          if (issued[st]) {
            drain_one_pair(BAR(P_ST_FULL + st), (issued[st] - 1) & 1, p.ctl, 85);
            if (crank == 0) {
              drain_one_pair(BAR(P_Q_FULL + st), (issued[st] - 1) & 1, p.ctl, 85);
              drain_one_pair(BAR(P_DO_FULL + st), (issued[st] - 1) & 1, p.ctl, 85);
            }
          }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      if (lane == 0 && crank == 0 && n_tiles > 0) {
        constexpr uint32_t kIdS = idesc_bf16_f32(256, kTileM, 0, 0);  // S^T, dP^T: K-major A and B
        constexpr uint32_t kIdKV = idesc_bf16_f32(256, D, 0, 1);      // dV, dK: TMEM A, MN-major B
        // X^T = A B^T over d: A (K or V, 128 rows per CTA) and B (64 query rows per CTA) K-major
        auto issue_t = [&](uint32_t dcol, uint32_t a, uint32_t bst) {
          // descriptors built once and stepped by the K offset
          const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(bst, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
            const uint32_t boff = (kk >> 2) * kSub + (kk & 3) * 32;  // block X, then X2
            mma_bf16_ss_pair(tmem + dcol, sdesc_add(da, aoff), sdesc_add(db, boff), kIdS, kk > 0 ? 1u : 0u);
          }
        };
        bool ok = wait_one_pair(BAR(P_KV_FULL), 0, abort_flag, peer_abort, p.ctl, 86) &&
                  wait_one_pair(BAR(P_Q_FULL), 0, abort_flag, peer_abort, p.ctl, 87);
        if (ok) {
          tc_fence_after();
          issue_t(LY::kTmemS, sb + LY::kK, sb + LY::kQ);
          mma_commit_pair(BAR(P_S_FULL), kBoth);
          ok = wait_one_pair(BAR(P_DO_FULL), 0, abort_flag, peer_abort, p.ctl, 88);
          if (ok) {
            tc_fence_after();
            issue_t(LY::kTmemDP, sb + LY::kV, sb + LY::kDO);
            mma_commit_pair(BAR(P_DP_FULL), kBoth);
          }
        }
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int st = i & 1, st1 = (i + 1) & 1;
          const uint32_t par1 = ((i + 1) >> 1) & 1;
          if (i + 1 < n_tiles) {
            // S^T(i+1) once both CTAs hold S^T(i) in registers
            if (!wait_one_pair(BAR(P_Q_FULL + st1), par1, abort_flag, peer_abort, p.ctl, 87) ||
                !wait_one_pair(BAR(P_S_READ), i & 1, abort_flag, peer_abort, p.ctl, 89)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_t(LY::kTmemS, sb + LY::kK, sb + LY::kQ + st1 * LY::kTile);
            mma_commit_pair(BAR(P_S_FULL), kBoth);
          }
          if (!wait_one_pair(BAR(P_PS_FULL), i & 1, abort_flag, peer_abort, p.ctl, 90)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dK += dS^T Q, then dV += P^T dO: A from the packed dP^T columns of
          // each CTA, B = blocks Y, Y2 (this CTA's 64 head dims), 16 query rows per step
          const uint64_t dqy = sdesc_sw128(sb + LY::kQ + st * LY::kTile + LY::kY, kSub, 1024);
          const uint64_t doy = sdesc_sw128(sb + LY::kDO + st * LY::kTile + LY::kY, kSub, 1024);
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_bf16_ts_pair(tmem + LY::kTmemDK, tmem + LY::kTmemDP + pcol(kk) + 32,
                             sdesc_add(dqy, kk * 2048), kIdKV, (i > 0 || kk > 0) ? 1u : 0u);
          if (i + 2 < n_tiles) mma_commit_pair(BAR(P_Q_EMPTY + st), kBoth);
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk)
            mma_bf16_ts_pair(tmem + LY::kTmemDV, tmem + LY::kTmemDP + pcol(kk), sdesc_add(doy, kk * 2048), kIdKV,
                             (i > 0 || kk > 0) ? 1u : 0u);
          if (i + 2 < n_tiles) mma_commit_pair(BAR(P_DO_EMPTY + st), kBoth);
          if (i + 1 == n_tiles) {
            mma_commit_pair(BAR(P_KV_DONE), kBoth);
          } else {
            // dP^T(i+1) overwrites the packed operands that the dK / dV MMAs above read first
            if (!wait_one_pair(BAR(P_DO_FULL + st1), par1, abort_flag, peer_abort, p.ctl, 88)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_t(LY::kTmemDP, sb + LY::kV, sb + LY::kDO + st1 * LY::kTile);
            mma_commit_pair(BAR(P_DP_FULL), kBoth);
          }
        }
        mma_commit_pair(BAR(P_TEARDOWN), kBoth);
        drain_one_pair(BAR(P_TEARDOWN), 0, p.ctl, 91);
      } else if (lane == 0 && n_tiles > 0) {
        // the odd CTA: the even CTA's last commit also lands here; take it before leaving
        drain_one_pair(BAR(P_TEARDOWN), 0, p.ctl, 92);
      }
      __syncwarp();
    }
  } else {
    regs_inc<kPairRegsHigh>();
    // ---------------------------------------------------------- P^T and dS^T, half a key row per thread
    const int half = (warp - 4) >> 2;  // query columns [64 half, 64 half + 64)
    const int jr = ((warp - 4) & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int j = j0 + jr;
    const bool valid_k = j < p.L;
    const uint32_t s_read = LBAR(P_S_READ), ps_full = LBAR(P_PS_FULL);
    RowWin win;
    KRange ko;  // this CTA's own 128 key rows: the batched tile classification
    int gk = 0;
    if constexpr (VL) {
      make_row_win(p, s, min(j, p.L - 1), true, win);
    } else {
      make_krange(p, s, j0, ko);
      gk = tok(p, s, valid_k ? j : p.L - 1);
    }
    bool ok = true;
    int i = 0;
    walk_q_tiles<kTileM>(p, kp, p.n_qtiles, [&](int r, int qt) {
      const int st = i & 1;
      // padding query rows have -lse2 = -inf and -D = 0 (P = 0, dS = 0) without a mask;
      // tiles of the pair's walk that this CTA's keys do not meet are masked whole
      int c_lo = 0, c_hi = kTileM;
      if constexpr (VL) {
        row_win_cols(p, win, r, qt * kTileM, kTileM, c_lo, c_hi);
        if (!valid_k) c_lo = c_hi = 0;
      } else if (!q_tile_full<kTileM>(p, ko, r, qt)) {
        key_query_window<kTileM>(p, valid_k, gk, r, qt, c_lo, c_hi);
      }
      c_lo -= 64 * half;
      c_hi -= 64 * half;
      const bool masked = c_lo > 0 || c_hi < 64;
      const float4* ls4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 0) * 512) + 16 * half;
      const float4* ds4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 1) * 512) + 16 * half;
      if (!wait_warp_pair(BAR(P_S_FULL), i & 1, abort_flag, peer_abort, p.ctl, 93) ||
          !wait_warp_pair(BAR(P_ST_FULL + st), (i >> 1) & 1, abort_flag, peer_abort, p.ctl, 94)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld64(tl + LY::kTmemS + 64 * half, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(s_read);
      const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l = ls4[c4];
        float x0, x1, x2, x3;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1])), sc2, f32x2(l.x, l.y)),
                    x0, x1);
        f32x2_split(
            fma_f32x2(f32x2(__uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3])), sc2, f32x2(l.z, l.w)),
            x2, x3);
        v[4 * c4 + 0] = __float_as_uint(fast_exp2(x0));
        v[4 * c4 + 1] = __float_as_uint(fast_exp2(x1));
        v[4 * c4 + 2] = __float_as_uint(fast_exp2(x2));
        v[4 * c4 + 3] = __float_as_uint(fast_exp2(x3));
      }
      if (masked) {
        const uint64_t mw = bit_window64(c_lo, c_hi);
#pragma unroll
        for (int c = 0; c < 64; ++c) v[c] = ((mw >> c) & 1ull) ? v[c] : 0u;
      }
      if (!wait_warp_pair(BAR(P_DP_FULL), i & 1, abort_flag, peer_abort, p.ctl, 95)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      // dS^T = P^T * (dP^T - D); the thread's 64 dP^T columns then hold P^T packed
      // in [0, 32) and dS^T packed in [32, 64)
      const uint32_t tdp = tl + LY::kTmemDP + 64 * half;
      uint32_t ps[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t d[32];
        tmem_ld32(tdp + 32 * hh, d);
        tmem_ld_wait(d);
        uint32_t pp[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 dd = ds4[8 * hh + c4];
          const int c = 32 * hh + 4 * c4;
          const float p0 = __uint_as_float(v[c]), p1 = __uint_as_float(v[c + 1]);
          const float p2 = __uint_as_float(v[c + 2]), p3 = __uint_as_float(v[c + 3]);
          pp[2 * c4] = pack_bf16x2(p0, p1);
          pp[2 * c4 + 1] = pack_bf16x2(p2, p3);
          float s0, s1, s2, s3;
          f32x2_split(mul_f32x2(f32x2(p0, p1), add_f32x2(f32x2(__uint_as_float(d[4 * c4]), __uint_as_float(d[4 * c4 + 1])),
                                                         f32x2(dd.x, dd.y))),
                      s0, s1);
          f32x2_split(mul_f32x2(f32x2(p2, p3), add_f32x2(f32x2(__uint_as_float(d[4 * c4 + 2]),
                                                                __uint_as_float(d[4 * c4 + 3])),
                                                         f32x2(dd.z, dd.w))),
                      s2, s3);
          ps[16 * hh + 2 * c4] = pack_bf16x2(s0, s1);
          ps[16 * hh + 2 * c4 + 1] = pack_bf16x2(s2, s3);
        }
        tmem_st16(tdp + 16 * hh, pp);
      }
      tmem_st16(tdp + 32, *reinterpret_cast<uint32_t(*)[16]>(ps));
      tmem_st16(tdp + 48, *reinterpret_cast<uint32_t(*)[16]>(ps + 16));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(ps_full);
      ++i;
      return true;
    });
    // ---------------- epilogue: warpgroup 1 writes the dV rows, warpgroup 2 the dK rows
    const long long prow = (long long)s * p.L + j;
    const int* rmap = VL ? p.row_map : nullptr;  // varlen in original order: rows of the caller's layout
    __nv_bfloat16* base = half == 0 ? reinterpret_cast<__nv_bfloat16*>(p.dv) + (long long)b * p.v_sb +
                                          (long long)h * p.v_sh
                                    : reinterpret_cast<__nv_bfloat16*>(p.dk) + (long long)b * p.k_sb +
                                          (long long)h * p.k_sh;
    const long long pitch = half == 0 ? p.v_ss : p.k_ss;
    if (n_tiles > 0) {
      if (ok && wait_warp_pair(BAR(P_KV_DONE), 0, abort_flag, peer_abort, p.ctl, 96)) {
        tc_fence_after();
        // every MMA of the pair is done: this CTA's K / V buffers hold the warps' row slots
        fence_proxy_async_smem();
        const int j_w = j - lane;  // the warp's first key row
        const int nvalid = min(max(p.L - j_w, 0), 32);
        const long long row_w = (long long)s * p.L + j_w;  // the warp's first row of dk / dv
        if (in_bounds(nvalid == 0 || (row_w >= 0 && row_w + nvalid <= p.S), p.ctl, 23))
          store_rows_bf16<D / 32>(tl + (half == 0 ? LY::kTmemDV : LY::kTmemDK), half == 0 ? 1.f : p.scale,
                                  sp + (warp - 4) * (32 * D * 2), base, pitch, row_w, nvalid, rmap);
      }
    } else if (valid_k && in_bounds(prow >= 0 && prow < p.S, p.ctl, 24)) {
      __nv_bfloat16* dst = base + (rmap ? (long long)__ldg(rmap + prow) : prow) * pitch;
      for (int u = 0; u < D / 8; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no copy, MMA or arrival of either CTA is still aimed at the other
  if (warp == 2) {  // collective with warp 2 of the other CTA
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool VL>
cudaError_t launch_v(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                     const BwdParams& p, cudaStream_t st) {
  BwdParamsT<VL> pv;
  static_cast<BwdParams&>(pv) = p;
  // the register split inside the kernel is only safe with the launch allocation it was sized for
  cudaError_t e = configure_kernel<ring_dkdv_pair_kernel<VL>>(kPairLaunchRegs, PairLayout::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_pairs = (p.n_ktiles + 1) / 2;
  dim3 grid((unsigned)(2 * p.N * n_pairs), (unsigned)(p.B * p.H));
  ring_dkdv_pair_kernel<VL><<<grid, kThreads, PairLayout::kAlloc, st>>>(tq, tk, tv, tdo, pv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dkdv_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
  return p.cu ? launch_v<true>(tq, tk, tv, tdo, p, st) : launch_v<false>(tq, tk, tv, tdo, p, st);
}

}  // namespace ra
