// Ring-attention backward on sm_103a, as two kernels with no atomics.
//
// The gradient of exact attention, with P recomputed from the saved
// log-sum-exp ("Ring Flash Attention" README: "use the softmax_lse output")
// and D = rowsum(dO * O) computed beforehand:
//   P = exp(S - lse),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ = scale dS K,   dK = scale dS^T Q.
// Both kernels walk the ring (guijiagi.com "Ring Attention：突破百万 Token
// 上下文的分布式注意力", "详细流程"):
//   ring_dkdv_kernel  one CTA per 128-row key tile of KV shard s, meeting the
//                     query shards (s + t) mod N (the path the K/V block and its
//                     gradient accumulators travel); dK and dV accumulate in
//                     tensor memory for the CTA's whole life.
//   ring_dq_kernel    one CTA per 128-row query tile of Q shard r, meeting the
//                     KV shards (r - t) mod N like the forward; dQ accumulates in
//                     tensor memory and is written once, in bf16.
// The dQ pass recomputes S and dP (two extra GEMMs) instead of adding fp32
// partial dQ tiles into memory from every key tile, whose traffic (64 KB per
// tile pair) is bounded by the GPU's reduction bandwidth.  The results are
// deterministic.
//
// Each tile row is split between two threads (query or key columns [0, 64) and
// [64, 128)); ra_bwd_common.cuh describes the packed TMEM operands this gives.
#include "ra_bwd_common.cuh"

namespace ra {
namespace {

using bwd::kBox;
using bwd::pcol;
using bwd::stat_rows_ok;
using bwd::store_rows_bf16;
using bwd::tmem_ld64;
constexpr int kThreads = 384;

// ======================================================================== dK / dV
// Warps: 0 TMA (K, V once; Q with the query tile's -lse2 / -D, and dO, into two
// 2-stage rings filled onto the Q stage's barrier), 1 MMA, 2 TMEM; warpgroups
// 1 and 2: one key row each, query columns [0, 64) and [64, 128).  TMEM: S^T
// [0,128), dP^T [128,256), dV [256, 256+D), dK [256+D, 256+2D).  A thread
// reads its 64 S^T columns,
// writes P^T as packed bf16 over the first 32 of them (the A operand of
// dV += P^T dO) and signals; once dP^T is ready it writes dS^T packed over the
// first 32 of its own 64 dP^T columns (the A operand of dK += dS^T Q).  Per
// query tile i the MMA thread issues
//   dV(i) [once P^T(i) is in TMEM], S^T(i+1), dK(i) [once dS^T(i) is in TMEM],
//   dP^T(i+1)
// so the next tile's exponentials overlap dK(i) and dP^T(i+1), and its dS^T
// overlaps dV(i+1) and S^T(i+2): each hand-off has two MMA groups of slack.
template <int D>
struct DkdvLayout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;          // 2 stages
  static constexpr int kDO = kQ + 2 * kTile;     // 2 stages
  static constexpr int kStats = kDO + 2 * kTile; // 2 stages (with Q) x (-lse2, -D), 128 floats each
  static constexpr int kBar = kStats + 2 * 2 * 512;
  static constexpr int kNumBars = 15;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 256 + D;
  static_assert(8 * 32 * D * 2 <= kStats, "output row slots exceed the operand buffers");
};

// Register split of the dK / dV kernel: the control warpgroup (TMA, MMA, TMEM)
// gives registers to the two elementwise warpgroups.  The launch allocation is
// kThreads * kDkdvLaunchRegs; the launcher checks the compiled kernel against it.
constexpr int kDkdvLaunchRegs = 168;
constexpr int kDkdvRegsLow = 72;
constexpr int kDkdvRegsHigh = 216;
static_assert(128 * kDkdvRegsLow + 256 * kDkdvRegsHigh <= kThreads * kDkdvLaunchRegs, "register split exceeds the launch");

enum DkdvBar {
  E_KV_FULL = 0,
  E_Q_FULL = 1,     // 2: Q, dO, -lse2 and -D of a query tile
  E_Q_EMPTY = 3,    // 2
  // 5..6: unused (dO lands on the Q stage's barrier)
  E_DO_EMPTY = 7,   // 2
  E_S_FULL = 9,
  E_P_FULL = 10,    // P^T packed over the S^T columns: 8 elected arrivals
  E_DP_FULL = 11,
  E_DS_FULL = 12,   // dS^T packed over the dP^T columns: 8 elected arrivals
  E_KV_DONE = 13,
  E_TEARDOWN = 14
};

// VL: varlen instantiation (FwdParamsT / BwdParamsT carry it as kVarlen).
template <int D, bool VL>
__global__ void __launch_bounds__(kThreads, 1)
    ring_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const BwdParamsT<VL> p) {
  using LY = DkdvLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // one key / value head; with grouped-query attention its G query heads share it
  const int b = blockIdx.y / p.Hk, hk = blockIdx.y % p.Hk;

  const int ks = (int)blockIdx.x / p.n_ktiles, kj0 = ((int)blockIdx.x % p.n_ktiles) * kTileN;
  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);
  if (threadIdx.x == 0) {
    mbar_init(BAR(E_KV_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(E_Q_FULL + i), 1);
      mbar_init(BAR(E_Q_EMPTY + i), 1);
      mbar_init(BAR(E_DO_EMPTY + i), 1);
    }
    mbar_init(BAR(E_S_FULL), 1);
    mbar_init(BAR(E_P_FULL), 8);
    mbar_init(BAR(E_DP_FULL), 1);
    mbar_init(BAR(E_DS_FULL), 8);
    mbar_init(BAR(E_KV_DONE), 1);
    mbar_init(BAR(E_TEARDOWN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    // the key tile's K and V depend on nothing the walk below computes: issued
    // first, their latency overlaps the CTA's set-up
    const int krow = ks * p.L + kj0;
    mbar_expect_tx(BAR(E_KV_FULL), 2 * LY::kTile);
    for (int c = 0; c < D / 64; ++c)
      if (!(p.ctl.debug_flags & DBG_SKIP_KV_LOAD) &&
          in_bounds(tma_coords_ok(TmaExtent{D, p.S, p.Hk, p.B}, c * 64, krow, hk, b), p.ctl, 10)) {
        tma_load_4d(sb + LY::kK + c * kBox, &tmK, BAR(E_KV_FULL), c * 64, krow, hk, b);
        tma_load_4d(sb + LY::kV + c * kBox, &tmV, BAR(E_KV_FULL), c * 64, krow, hk, b);
      }
  }
  KRange k;
  make_krange(p, ks, kj0, k);
  int n_tiles = 0;  // over all query heads of the group (every head meets the same tiles)
  walk_q_tiles<kTileM>(p, k, p.n_qtiles, [&](int, int) {
    ++n_tiles;
    return true;
  });
  n_tiles *= p.G;
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    regs_dec<kDkdvRegsLow>();
    if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      int issued[2] = {0, 0};
      int i = 0;
      auto load = [&](int h, int r, int qt) {
        const int st = i & 1;
        const uint32_t par = ((i >> 1) - 1) & 1;
        const int qrow = r * p.L + qt * kTileM - p.q_base;
        const long long stat_bh = ((long long)b * p.H + h) * p.stat_N * p.stat_L;  // (b, h, first shard)
        // dV frees the dO stage two MMA groups before dK frees the Q stage: dO
        // goes first, onto the same barrier (its bytes added without an arrival)
        if (i >= 2 && !wait_one(BAR(E_DO_EMPTY + st), par, abort_flag, p.ctl, 39)) return false;
        const bool rows_ok = in_bounds(tma_coords_ok(TmaExtent{D, p.q_rows, p.H, p.B}, 0, qrow, h, b), p.ctl, 11);
        mbar_add_tx(BAR(E_Q_FULL + st), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          if (rows_ok)
            tma_load_4d(sb + LY::kDO + st * LY::kTile + c * kBox, &tmDO, BAR(E_Q_FULL + st), c * 64, qrow, h, b);
        if (i >= 2 && !wait_one(BAR(E_Q_EMPTY + st), par, abort_flag, p.ctl, 31)) {
          // the phase then completes once dO has landed, and the drain below waits for it
          mbar_arrive(BAR(E_Q_FULL + st));
          ++issued[st];
          return false;
        }
        // -lse2 / -D of the tile's 128 query rows: 512-byte aligned in the padded layout
        const long long e0 = stat_bh + (long long)(r - p.stat_r0) * p.stat_L + qt * kTileM;
        mbar_expect_tx(BAR(E_Q_FULL + st), LY::kTile + 2 * 512);
        for (int c = 0; c < D / 64; ++c)
          if (rows_ok)
            tma_load_4d(sb + LY::kQ + st * LY::kTile + c * kBox, &tmQ, BAR(E_Q_FULL + st), c * 64, qrow, h, b);
        if (in_bounds(stat_rows_ok(p, e0), p.ctl, 12)) {
          bulk_load(sb + LY::kStats + (st * 2 + 0) * 512, p.nlse2 + e0, 512, BAR(E_Q_FULL + st));
          bulk_load(sb + LY::kStats + (st * 2 + 1) * 512, p.nD + e0, 512, BAR(E_Q_FULL + st));
        }
        ++issued[st];
        ++i;
        return true;
      };
      // (one head per key head kept apart: the producer runs on few registers)
      if (p.G == 1)
        walk_q_tiles<kTileM>(p, k, p.n_qtiles, [&](int r, int qt) { return load(hk, r, qt); });
      else
        walk_group_q_tiles<kTileM>(p, k, p.n_qtiles, hk, load);
      for (int st = 0; st < 2; ++st)
        if (issued[st]) drain_one(BAR(E_Q_FULL + st), (issued[st] - 1) & 1, p.ctl, 41);
    }
    if (lane == 0) drain_one(BAR(E_KV_FULL), 0, p.ctl, 40);  // issued at entry
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileM, 0, 0);  // S^T, dP^T: K-major A and B
      constexpr uint32_t kIdKV = idesc_bf16_f32(128, D, 0, 1);      // dV, dK: TMEM A, MN-major B
      // X^T = A B^T over D: A (K or V) and B (Q or dO tile) K-major in shared memory
      auto issue_t = [&](uint32_t dcol, uint32_t a, uint32_t bq) {
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(bq, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + dcol, sdesc_add(da, off), sdesc_add(db, off), kIdS, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = wait_one(BAR(E_KV_FULL), 0, abort_flag, p.ctl, 32) &&
                wait_one(BAR(E_Q_FULL), 0, abort_flag, p.ctl, 33);
      if (ok) {
        tc_fence_after();
        issue_t(LY::kTmemS, sb + LY::kK, sb + LY::kQ);
        mma_commit(BAR(E_S_FULL));
        issue_t(LY::kTmemDP, sb + LY::kV, sb + LY::kDO);
        mma_commit(BAR(E_DP_FULL));
      }
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i & 1, st1 = (i + 1) & 1;
        const uint32_t par1 = ((i + 1) >> 1) & 1;
        // dV += P^T dO once P^T(i) is packed over the S^T columns
        if (!wait_one(BAR(E_P_FULL), i & 1, abort_flag, p.ctl, 45)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dob = sdesc_sw128(sb + LY::kDO + st * LY::kTile, kBox, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)
          mma_bf16_ts(tmem + LY::kTmemDV, tmem + LY::kTmemS + pcol(kk), sdesc_add(dob, kk * 2048), kIdKV,
                      (i > 0 || kk > 0) ? 1u : 0u);
        if (i + 2 < n_tiles) mma_commit(BAR(E_DO_EMPTY + st));
        if (i + 1 < n_tiles) {
          // S^T(i+1) overwrites the P^T(i) the dV MMAs above read first
          if (!wait_one(BAR(E_Q_FULL + st1), par1, abort_flag, p.ctl, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_t(LY::kTmemS, sb + LY::kK, sb + LY::kQ + st1 * LY::kTile);
          mma_commit(BAR(E_S_FULL));
        }
        // dK += dS^T Q once dS^T(i) is packed over the dP^T columns
        if (!wait_one(BAR(E_DS_FULL), i & 1, abort_flag, p.ctl, 35)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dqb = sdesc_sw128(sb + LY::kQ + st * LY::kTile, kBox, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)
          mma_bf16_ts(tmem + LY::kTmemDK, tmem + LY::kTmemDP + pcol(kk), sdesc_add(dqb, kk * 2048), kIdKV,
                      (i > 0 || kk > 0) ? 1u : 0u);
        if (i + 2 < n_tiles) mma_commit(BAR(E_Q_EMPTY + st));
        if (i + 1 == n_tiles) {
          mma_commit(BAR(E_KV_DONE));
        } else {
          // dP^T(i+1) overwrites the dS^T(i) the dK MMAs above read first (dO(i+1)
          // landed with Q(i+1), waited for before S^T(i+1))
          issue_t(LY::kTmemDP, sb + LY::kV, sb + LY::kDO + st1 * LY::kTile);
          mma_commit(BAR(E_DP_FULL));
        }
      }
      mma_commit(BAR(E_TEARDOWN));
      drain_one(BAR(E_TEARDOWN), 0, p.ctl, 42);
    }
    __syncwarp();
    }
  } else {
    regs_inc<kDkdvRegsHigh>();
    // ------------------------------------------------------------ P^T and dS^T, half a key row per thread
    const int half = (warp - 4) >> 2;  // query columns [64 half, 64 half + 64)
    const int jr = ((warp - 4) & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int j = k.j0 + jr;
    const bool valid_k = j < p.L;
    // batched: tiles classified per key tile, masks per row on partial tiles;
    // varlen: every key row's query window, set up once
    RowWin win;
    int gk = 0;
    if constexpr (VL)
      make_row_win(p, k.s, min(j, p.L - 1), true, win);
    else
      gk = tok(p, k.s, valid_k ? j : k.j_last);
    bool ok = true;
    int i = 0;
    auto tile = [&](int r, int qt) {
      const int st = i & 1;
      // padding query rows have -lse2 = -inf and -D = 0 (P = 0, dS = 0) without a mask
      int c_lo = 0, c_hi = kTileM;
      if constexpr (VL) {
        row_win_cols(p, win, r, qt * kTileM, kTileM, c_lo, c_hi);
        if (!valid_k) c_lo = c_hi = 0;
      } else if (!q_tile_full<kTileM>(p, k, r, qt)) {
        key_query_window<kTileM>(p, valid_k, gk, r, qt, c_lo, c_hi);
      }
      c_lo -= 64 * half;
      c_hi -= 64 * half;
      const bool masked = c_lo > 0 || c_hi < 64;
      const float4* ls4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 0) * 512) + 16 * half;
      const float4* ds4 = reinterpret_cast<const float4*>(sp + LY::kStats + (st * 2 + 1) * 512) + 16 * half;
      // waiting on the stage barrier orders this thread's statistics reads after the copy landed
      if (!wait_warp(BAR(E_S_FULL), i & 1, abort_flag, p.ctl, 36) ||
          !wait_warp(BAR(E_Q_FULL + st), (i >> 1) & 1, abort_flag, p.ctl, 44)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld64(tl + LY::kTmemS + 64 * half, v);
      // P^T = exp2(s * scale - lse2), s * scale - lse2 two lanes per instruction
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
      // P^T packed over the first 32 of the thread's 64 S^T columns (column m:
      // queries 2m, 2m + 1), the A operand of dV += P^T dO; the MMA thread then
      // computes the next tile's S^T over it
      {
        const uint32_t ts = tl + LY::kTmemS + 64 * half;
        uint32_t pp[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pp[c] = pack_bf16x2(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
        tmem_st16(ts, *reinterpret_cast<uint32_t(*)[16]>(pp));
        tmem_st16(ts + 16, *reinterpret_cast<uint32_t(*)[16]>(pp + 16));
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(E_P_FULL));
      if (!wait_warp(BAR(E_DP_FULL), i & 1, abort_flag, p.ctl, 37)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      // dS^T = P^T * (dP^T - D), 32 dP^T columns at a time, packed over the first
      // 32 of the thread's 64 dP^T columns (a packed half is stored once the
      // columns under it are read): the A operand of dK += dS^T Q
      const uint32_t tdp = tl + LY::kTmemDP + 64 * half;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t d[32];
        tmem_ld32(tdp + 32 * hh, d);
        tmem_ld_wait(d);
        uint32_t ps[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 dd = ds4[8 * hh + c4];
          const int c = 32 * hh + 4 * c4;
          const float p0 = __uint_as_float(v[c]), p1 = __uint_as_float(v[c + 1]);
          const float p2 = __uint_as_float(v[c + 2]), p3 = __uint_as_float(v[c + 3]);
          // dS^T = P^T * (dP^T + (-D)), two lanes per instruction
          float s0, s1, s2, s3;
          f32x2_split(mul_f32x2(f32x2(p0, p1), add_f32x2(f32x2(__uint_as_float(d[4 * c4]), __uint_as_float(d[4 * c4 + 1])),
                                                         f32x2(dd.x, dd.y))),
                      s0, s1);
          f32x2_split(mul_f32x2(f32x2(p2, p3), add_f32x2(f32x2(__uint_as_float(d[4 * c4 + 2]),
                                                                __uint_as_float(d[4 * c4 + 3])),
                                                         f32x2(dd.z, dd.w))),
                      s2, s3);
          ps[2 * c4] = pack_bf16x2(s0, s1);
          ps[2 * c4 + 1] = pack_bf16x2(s2, s3);
        }
        tmem_st16(tdp + 16 * hh, ps);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(E_DS_FULL));
      ++i;
      return true;
    };
    // every query head of the group meets the same tiles; the walk does not depend on the head
    for (int g = 0; ok && g < p.G; ++g) walk_q_tiles<kTileM>(p, k, p.n_qtiles, tile);
    // ---------------- epilogue: warpgroup 1 writes the dV rows, warpgroup 2 the dK rows
    const long long prow = (long long)k.s * p.L + j;
    const int* rmap = VL ? p.row_map : nullptr;  // varlen in original order: rows of the caller's layout
    __nv_bfloat16* base = half == 0 ? reinterpret_cast<__nv_bfloat16*>(p.dv) + (long long)b * p.v_sb +
                                          (long long)hk * p.v_sh
                                    : reinterpret_cast<__nv_bfloat16*>(p.dk) + (long long)b * p.k_sb +
                                          (long long)hk * p.k_sh;
    const long long pitch = half == 0 ? p.v_ss : p.k_ss;
    if (n_tiles > 0) {
      if (ok && wait_warp(BAR(E_KV_DONE), 0, abort_flag, p.ctl, 38)) {
        tc_fence_after();
        // every MMA is done: the operand buffers hold the warps' row slots
        fence_proxy_async_smem();
        const int j_w = j - lane;  // the warp's first key row
        const int nvalid = min(max(p.L - j_w, 0), 32);
        const long long row_w = (long long)k.s * p.L + j_w;  // the warp's first row of dk / dv
        if (in_bounds(nvalid == 0 || (row_w >= 0 && row_w + nvalid <= p.S), p.ctl, 14))
          store_rows_bf16<D / 32>(tl + (half == 0 ? LY::kTmemDV : LY::kTmemDK), half == 0 ? 1.f : p.scale,
                                  sp + (warp - 4) * (32 * D * 2), base, pitch, row_w, nvalid, rmap);
      }
    } else if (valid_k && in_bounds(prow >= 0 && prow < p.S, p.ctl, 15)) {
      __nv_bfloat16* dst = base + (rmap ? (long long)__ldg(rmap + prow) : prow) * pitch;
      for (int u = 0; u < D / 8; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================== dQ
// Warps: 0 TMA (Q, dO once, then each key tile's K into a 3-stage ring and V
// into a 2-stage ring, both completing on the V stage's barrier, so the MMA
// thread waits once per key tile), 1 MMA, 2 TMEM, 3 idle; warpgroups 1 and 2:
// one query row each, key columns [0, 64) and [64, 128).  Q and dO are the
// same for every key tile, so
// the softmax threads copy them once into tensor memory (packed bf16) and the
// S and dP MMAs take them from there: shared memory then feeds only the K and V
// operands.  TMEM: S [0,128), dP [128,256), Q [256, 256+D/2), dO [256+D/2, 256+D),
// dQ [384, 384+D).  A thread reads its 64 S columns into registers and releases
// them at once; it writes dS as packed bf16 over the first 32 of its own 64 dP
// columns, the A operand of dQ += dS K.  Per key tile j the MMA thread issues
//   S(j+1) [once S(j) is read], dQ += dS(j) K(j) [once dS(j) is in TMEM], dP(j+1)
// so S of the next tile and the exponentials of the current one overlap.
template <int D>
struct DqLayout {
  static constexpr int kTile = (D / 64) * kBox;
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kK = kDO + kTile;
  static constexpr int kV = kK + kKStages * kTile;
  static constexpr int kBar = kV + kVStages * kTile;
  static constexpr int kNumBars = 18;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemQ = 256, kTmemDO = 256 + D / 2, kTmemDQ = 384;
  static_assert(8 * 32 * D <= kBar, "output row slots exceed the operand buffers");
};

enum DqBar {
  F_QDO_FULL = 0,
  // 1..3: unused (K lands on the V stage's barrier)
  F_K_EMPTY = 4,   // 3
  F_V_FULL = 7,    // 2
  F_V_EMPTY = 9,   // 2
  F_S_FULL = 11,
  F_S_READ = 12,   // S in registers: 8 elected arrivals
  F_DP_FULL = 13,
  F_DS_FULL = 14,  // dS in TMEM: 8 elected arrivals
  F_QDO_TMEM = 15, // Q and dO copied into TMEM: 8 elected arrivals
  F_DQ_DONE = 16,
  F_TEARDOWN = 17
};

template <int D, bool VL>
__global__ void __launch_bounds__(kThreads, 1)
    ring_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const BwdParamsT<VL> p) {
  using LY = DqLayout<D>;
  constexpr int KS = LY::kKStages, VS = LY::kVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.y / p.H, h = blockIdx.y % p.H;
  const int hk = h / p.G;  // the key / value head of query head h (grouped-query attention)
  // causal: the later query tiles carry more work, start them first (the
  // batched zigzag split by chunk, so that every head's heaviest tiles lead)
  int r, i0;
  if (!VL && p.causal && p.layout == LAYOUT_ZIGZAG && p.r_only < 0 && p.L % (2 * kTileM) == 0) {
    int qt;
    zigzag_heavy_first((int)blockIdx.x, p.N, p.n_qtiles / 2, r, qt);
    i0 = qt * kTileM;
  } else {
    const int x = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    r = p.r_only >= 0 ? p.r_only : x / p.n_qtiles;
    i0 = (x % p.n_qtiles) * kTileM;
  }
  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);
  if (threadIdx.x == 0) {
    mbar_init(BAR(F_QDO_FULL), 1);
    for (int i = 0; i < KS; ++i) {
      mbar_init(BAR(F_K_EMPTY + i), 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(BAR(F_V_FULL + i), 1);
      mbar_init(BAR(F_V_EMPTY + i), 1);
    }
    mbar_init(BAR(F_S_FULL), 1);
    mbar_init(BAR(F_S_READ), 8);
    mbar_init(BAR(F_DP_FULL), 1);
    mbar_init(BAR(F_DS_FULL), 8);
    mbar_init(BAR(F_QDO_TMEM), 8);
    mbar_init(BAR(F_DQ_DONE), 1);
    mbar_init(BAR(F_TEARDOWN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    // the tile's Q and dO depend on nothing the tile walk below computes:
    // issued first, their latency overlaps the CTA's set-up
    const int qrow = r * p.L + i0 - p.q_base;
    mbar_expect_tx(BAR(F_QDO_FULL), 2 * LY::kTile);
    for (int c = 0; c < D / 64; ++c)
      if (!(p.ctl.debug_flags & DBG_SKIP_QDO_LOAD) &&
          in_bounds(tma_coords_ok(TmaExtent{D, p.q_rows, p.H, p.B}, c * 64, qrow, h, b), p.ctl, 16)) {
        tma_load_4d(sb + LY::kQ + c * kBox, &tmQ, BAR(F_QDO_FULL), c * 64, qrow, h, b);
        tma_load_4d(sb + LY::kDO + c * kBox, &tmDO, BAR(F_QDO_FULL), c * 64, qrow, h, b);
      }
  }
  QRange qr;
  make_qrange(p, r, i0, kTileM, qr);
  const int nkt = (p.L + kTileN - 1) / kTileN;
  int n_tiles = 0;
  walk_kv_tiles(p, qr, nkt, 0, p.N, [&](int, int) {
    ++n_tiles;
    return true;
  });

  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    if (warp == 0 && lane == 0 && n_tiles > 0) {
      // K(j) and V(j) land on one barrier (the V stage's): the MMA thread
      // waits once per key tile
      int issued[2] = {0, 0};
      int j = 0;
      walk_kv_tiles(p, qr, nkt, 0, p.N, [&](int s, int kt) {
        const int sk = j % KS, sv = j % VS;
        if (j >= KS && !wait_one(BAR(F_K_EMPTY + sk), (j / KS - 1) & 1, abort_flag, p.ctl, 51)) return false;
        if (j >= VS && !wait_one(BAR(F_V_EMPTY + sv), (j / VS - 1) & 1, abort_flag, p.ctl, 52)) return false;
        mbar_expect_tx(BAR(F_V_FULL + sv), 2 * LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          if (in_bounds(tma_coords_ok(TmaExtent{D, p.S, p.Hk, p.B}, c * 64, s * p.L + kt * kTileN, hk, b), p.ctl,
                        17)) {
            tma_load_4d(sb + LY::kK + sk * LY::kTile + c * kBox, &tmK, BAR(F_V_FULL + sv), c * 64,
                        s * p.L + kt * kTileN, hk, b);
            tma_load_4d(sb + LY::kV + sv * LY::kTile + c * kBox, &tmV, BAR(F_V_FULL + sv), c * 64,
                        s * p.L + kt * kTileN, hk, b);
          }
        ++issued[sv];
        ++j;
        return true;
      });
      for (int st = 0; st < VS; ++st)
        if (issued[st]) drain_one(BAR(F_V_FULL + st), (issued[st] - 1) & 1, p.ctl, 54);
    }
    if (threadIdx.x == 0) drain_one(BAR(F_QDO_FULL), 0, p.ctl, 53);  // issued at entry
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileN, 0, 0);  // S = Q K^T, dP = dO V^T: TMEM A, K-major B
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 0, 1);       // dQ += dS K: TMEM A, MN-major B
      bool ok = wait_one(BAR(F_QDO_TMEM), 0, abort_flag, p.ctl, 55);
      // X = A B^T over D with A (Q or dO) packed in TMEM, 16 head-dim columns = 8 TMEM columns per step
      auto issue_t = [&](uint32_t dcol, uint32_t acol, uint32_t bt) {
        const uint64_t db = sdesc_sw128(bt, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ts(tmem + dcol, tmem + acol + 8 * kk, sdesc_add(db, off), kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_s = [&](int j) -> bool {
        const int ks = j % KS;
        if (!wait_one(BAR(F_V_FULL + j % VS), (j / VS) & 1, abort_flag, p.ctl, 56)) return false;
        if (j > 0 && !wait_one(BAR(F_S_READ), (j - 1) & 1, abort_flag, p.ctl, 57)) return false;
        tc_fence_after();
        issue_t(LY::kTmemS, LY::kTmemQ, sb + LY::kK + ks * LY::kTile);
        mma_commit(BAR(F_S_FULL));
        return true;
      };
      // dP(j) overwrites dS(j-1), which the dQ MMA issued before it has read
      auto issue_dp = [&](int j) -> bool {
        const int vs = j % VS;  // V(j) landed with K(j), waited for before S(j)
        issue_t(LY::kTmemDP, LY::kTmemDO, sb + LY::kV + vs * LY::kTile);
        mma_commit(BAR(F_DP_FULL));
        if (j + VS < n_tiles) mma_commit(BAR(F_V_EMPTY + vs));
        return true;
      };
      auto issue_dq = [&](int j) -> bool {
        if (!wait_one(BAR(F_DS_FULL), j & 1, abort_flag, p.ctl, 59)) return false;
        tc_fence_after();
        const uint64_t dkb = sdesc_sw128(sb + LY::kK + (j % KS) * LY::kTile, kBox, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // A = dS (16 keys = 8 packed columns of the dP region), B = K with 16 key rows per step
          mma_bf16_ts(tmem + LY::kTmemDQ, tmem + LY::kTmemDP + pcol(kk), sdesc_add(dkb, kk * 2048),
                      kIdQ, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (j + KS < n_tiles) mma_commit(BAR(F_K_EMPTY + j % KS));
        return true;
      };
      if (ok) {
        tc_fence_after();
        ok = issue_s(0) && issue_dp(0);
        for (int j = 0; ok && j < n_tiles; ++j) {
          if (j + 1 < n_tiles) ok = issue_s(j + 1);
          ok = ok && issue_dq(j);
          if (ok && j + 1 < n_tiles) ok = issue_dp(j + 1);
        }
        if (ok) mma_commit(BAR(F_DQ_DONE));
      }
      mma_commit(BAR(F_TEARDOWN));
      drain_one(BAR(F_TEARDOWN), 0, p.ctl, 60);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P and dS, half a query row per thread
    const int half = (warp - 4) >> 2;  // key columns [64 half, 64 half + 64)
    const int row = ((warp - 4) & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int i = i0 + row;
    const bool valid = i < p.L;
    // batched: tiles classified per query tile; varlen: every row's key window, set up once
    RowWin win;
    int gq = 0;
    if constexpr (VL)
      make_row_win(p, r, min(i, p.L - 1), false, win);
    else
      gq = tok(p, r, valid ? i : max(qr.i_last, 0));
    // this row's statistics, negated (padding rows: -lse2 = -inf, -D = 0, so P = dS = 0)
    const long long srow = (((long long)b * p.H + h) * p.stat_N + (r - p.stat_r0)) * p.stat_L + i;
    const uint64_t nl2 = f32x2(__ldg(p.nlse2 + srow), __ldg(p.nlse2 + srow));
    const uint64_t nD2 = f32x2(__ldg(p.nD + srow), __ldg(p.nD + srow));
    const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
    // warpgroup 1 copies the row's Q, warpgroup 2 its dO, into tensor memory as
    // packed bf16 (column m: head-dim elements 2m, 2m + 1) for the S and dP MMAs
    bool ok = n_tiles == 0 || wait_warp(BAR(F_QDO_FULL), 0, abort_flag, p.ctl, 64);
    if (ok && n_tiles > 0) {
      const uint8_t* src = sp + (half == 0 ? LY::kQ : LY::kDO);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          // 128-byte swizzle: 16-byte chunk q of row `row` sits at chunk q ^ (row & 7)
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
      if (lane == 0) mbar_arrive(BAR(F_QDO_TMEM));
    }
    int j = 0;
    if (ok) walk_kv_tiles(p, qr, nkt, 0, p.N, [&](int s, int kt) {
      int c_lo = 0, c_hi = kTileN;
      if constexpr (VL)
        row_win_cols(p, win, s, kt * kTileN, kTileN, c_lo, c_hi);
      else if (!kv_tile_full(p, qr, s, kt))
        row_key_window(p, gq, s, kt, c_lo, c_hi);
      c_lo -= 64 * half;
      c_hi -= 64 * half;
      const bool masked = c_lo > 0 || c_hi < 64;
      if (!wait_warp(BAR(F_S_FULL), j & 1, abort_flag, p.ctl, 61)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld64(tl + LY::kTmemS + 64 * half, v);
      // S is in registers: the MMA thread may compute the next tile's S over it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(F_S_READ));
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        // P = exp2(s * scale - lse2), s * scale - lse2 two lanes per instruction
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
      if (!wait_warp(BAR(F_DP_FULL), j & 1, abort_flag, p.ctl, 62)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      // dS = P * (dP - D), 32 dP columns at a time, packed (column m: keys 2m, 2m + 1)
      // over the first 32 of this thread's 64 dP columns once they are read
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
          // dS = P * (dP + (-D)), two lanes per instruction
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
      if (lane == 0) mbar_arrive(BAR(F_DS_FULL));
      ++j;
      return true;
    });
    // ---------------- epilogue: dQ = scale * (dS K), half the head dim per thread
    const int* rmap = VL ? p.row_map : nullptr;  // varlen in original order: rows of the caller's layout
    __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(p.dq) + (long long)b * p.q_sb + (long long)h * p.q_sh +
                          half * (D / 2);
    const long long qrow = (long long)r * p.L + i - p.q_base;
    if (n_tiles > 0) {
      if (ok && wait_warp(BAR(F_DQ_DONE), 0, abort_flag, p.ctl, 63)) {
        tc_fence_after();
        // every MMA is done: the operand buffers hold the warps' row slots
        fence_proxy_async_smem();
        const int i_w = i - lane;  // the warp's first query row
        const int nvalid = min(max(p.L - i_w, 0), 32);
        const long long row_w = (long long)r * p.L + i_w - p.q_base;  // the warp's first row of dq
        if (in_bounds(nvalid == 0 || (row_w >= 0 && row_w + nvalid <= p.q_rows), p.ctl, 18))
          store_rows_bf16<D / 64>(tl + LY::kTmemDQ + half * (D / 2), p.scale, sp + (warp - 4) * (32 * D), base,
                                  p.q_ss, row_w, nvalid, rmap);
      }
    } else if (valid && in_bounds(qrow < p.q_rows, p.ctl, 19)) {
      __nv_bfloat16* dst = base + (rmap ? (long long)__ldg(rmap + qrow) : qrow) * p.q_ss;
      for (int u = 0; u < D / 16; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool VL>
cudaError_t launch_bwd_v(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, int which, cudaStream_t st) {
  BwdParamsT<VL> pv;
  static_cast<BwdParams&>(pv) = p;
  if (which == 0) {
    // the register split inside the kernel is only safe with the launch allocation it was sized for
    cudaError_t e = configure_kernel<ring_dkdv_kernel<D, VL>>(kDkdvLaunchRegs, DkdvLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.N * p.n_ktiles), (unsigned)(p.B * p.Hk));
    ring_dkdv_kernel<D, VL><<<grid, kThreads, DkdvLayout<D>::kAlloc, st>>>(tq, tk, tv, tdo, pv);
  } else {
    cudaError_t e = configure_kernel<ring_dq_kernel<D, VL>>(0, DqLayout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((p.r_only >= 0 ? 1 : p.N) * p.n_qtiles), (unsigned)(p.B * p.H));
    ring_dq_kernel<D, VL><<<grid, kThreads, DqLayout<D>::kAlloc, st>>>(tq, tk, tv, tdo, pv);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, int which, cudaStream_t st) {
  return p.cu ? launch_bwd_v<D, true>(tq, tk, tv, tdo, p, which, st)
              : launch_bwd_v<D, false>(tq, tk, tv, tdo, p, which, st);
}

}  // namespace

cudaError_t launch_bwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int which, cudaStream_t st) {
  if (D == 64) return launch_bwd_t<64>(tq, tk, tv, tdo, p, which, st);
  return launch_bwd_t<128>(tq, tk, tv, tdo, p, which, st);
}

}  // namespace ra
