// Ring-attention forward on sm_103a: blockwise exact attention of query tiles
// against every key tile of the KV shards they meet on the ring, with the
// online-softmax merge held in fp32 across all ring steps.
//
// Method (cited by page title and section):
//   * ring order: at step t the Q shard r meets KV shard (r - t) mod N
//     (guijiagi.com "Ring Attention：突破百万 Token 上下文的分布式注意力", "详细流程");
//   * online softmax across blocks: running max m and sum l, the accumulator
//     rescaled by exp(m_old - m_new) (same page, "在线 Softmax：关键技巧");
//   * the accumulator stays fp32 across blocks, never bf16 per block
//     ("Ring Flash Attention" README, "Limits");
//   * tiles of 128 tokens, scores never materialised in HBM (same page,
//     "Ring Attention + Flash Attention"; ainews.cool article "技术深度解析").
//
// Kernel structure: one CTA owns two 128-row query tiles (Q0, Q1: 256
// consecutive rows of one shard) and 12 warps.
//   warp 0      TMA producer: Q0 and Q1 once, then per key tile K into a
//               3-stage ring (freed when both S MMAs of a tile complete) and V
//               into a 2-stage ring (freed when both PV MMAs complete), the two
//               completing on the V stage's barrier, so the MMA thread waits
//               once per key tile for both (K, whose stage frees first, is
//               issued first).  Warp 3 is idle.
//   warp 1      MMA issuer (one thread).  Per key tile j it issues
//                 PV0(j-1), S0(j), PV1(j-1), S1(j)
//               (PV0(j-1) does not wait for K(j)),
//               so the tensor core works on one query tile while the other
//               tile's softmax runs (ping-pong).  S_t = Q_t K^T lands in TMEM
//               columns [128 t, 128 t + 128); O_t in [256 + 128 t, ...).
//   warp 2      allocates / frees the 512 TMEM columns.
//   warps 4-7   softmax of Q0, warps 8-11 softmax of Q1: one thread per query
//               row (its TMEM lane).  A thread reads its 128 scores, masks
//               partial tiles, updates the running max (O is rescaled in TMEM
//               only when the max grows by more than 2^8), and writes P as
//               packed bf16 over the first 64 columns of its own S tile, which
//               the PV MMA then reads as its A operand straight from TMEM.
// The commit that signals S_t(j) also covers PV_t(j-1) (commits track every
// earlier MMA of the issuing thread), so a softmax thread may rescale O_t as
// soon as its S tile is ready.  Empty key tiles are never loaded; only
// partial tiles are masked element by element.
#include "ra_tiles.cuh"

namespace ra {
namespace {

constexpr int kBox = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 bytes) = 16 KB
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kQTiles = 2;       // query tiles per CTA
constexpr int kRowsPerCta = kQTiles * kTileM;
constexpr int kThreads = 384;
// Register split: the producer / MMA warpgroup gives registers to the two
// softmax warpgroups, which hold a whole 128-score row each.  The launch
// allocation is kThreads * kLaunchRegs, and 128 * kRegsLow + 256 * kRegsHigh
// must not exceed it (checked by the launcher against the compiled kernel).
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 216;
// Suspend-time hint (ns) of every barrier wait in this kernel: a thread whose
// phase is not complete sleeps until it completes (or 2 us pass) instead of
// re-polling at the system's default interval.  Measured on the benchmark
// workload: forward -4 %, whole fwd+bwd step -0.7 % (the step runs at the
// power cap); the backward kernels measured slower with hints and keep the
// default.
constexpr uint32_t kWaitHint = 2000;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kLaunchRegs, "register split exceeds the launch");

template <int D>
struct FwdLayout {
  static constexpr int kTile = (D / 64) * kBox;      // one Q/K/V tile (128 rows x D)
  static constexpr int kQ = 0;                       // Q0, Q1
  static constexpr int kK = kQ + kQTiles * kTile;    // kKStages stages
  static constexpr int kV = kK + kKStages * kTile;   // kVStages stages
  static constexpr int kBar = kV + kVStages * kTile;
  static constexpr int kNumBars = 17;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;       // slack to align the base to 1024 bytes
  // the epilogue's row slots (8 warps x 32 rows, fp32 at most) reuse the Q / K / V buffers
  static_assert(8 * 32 * D * 4 <= kBar, "output slots exceed the operand buffers");
  static constexpr uint32_t kTmemS = 0;              // + 128 t
  static constexpr uint32_t kTmemO = 256;            // + 128 t
};

enum FwdBar {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // kKStages (unused: K lands on the V stage's barrier)
  B_K_EMPTY = 4,   // kKStages
  B_V_FULL = 7,    // kVStages
  B_V_EMPTY = 9,   // kVStages
  B_S_FULL = 11,   // kQTiles
  B_P_FULL = 13,   // kQTiles
  B_O_DONE = 15,
  B_TEARDOWN = 16
};

// The CTA's key tiles, in ring order (all ring steps, or the one the step mode asks for).
template <class P, class F>
__device__ __forceinline__ void walk_tiles(const P& p, const QRange& q, int nkt, F&& f) {
  const int t0 = p.step < 0 ? 0 : p.step;
  const int t1 = p.step < 0 ? p.N : p.step + 1;
  walk_kv_tiles(p, q, nkt, t0, t1, f);
}

// VL: varlen instantiation (FwdParamsT / BwdParamsT carry it as kVarlen).
template <int D, bool VL>
__global__ void __launch_bounds__(kThreads, 1)
    ring_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParamsT<VL> p) {
  using LY = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int b = blockIdx.y / p.H;
  const int h = blockIdx.y % p.H;
  // causal: the later query rows carry more work, start them first (the
  // batched zigzag split by chunk, so that every head's heaviest tiles lead)
  const int n_pairs = (p.L + kRowsPerCta - 1) / kRowsPerCta;
  int r, i0;
  if (!VL && p.causal && p.layout == LAYOUT_ZIGZAG && p.r_only < 0 && p.L % (2 * kRowsPerCta) == 0) {
    int pr;
    zigzag_heavy_first((int)blockIdx.x, p.N, n_pairs / 2, r, pr);
    i0 = pr * kRowsPerCta;
  } else {
    const int x = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    r = p.r_only >= 0 ? p.r_only : x / n_pairs;
    i0 = (x % n_pairs) * kRowsPerCta;
  }
  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);

  bool q_issued = false;  // by thread 0, the Q / K producer
  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q_FULL), 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(BAR(B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(BAR(B_V_FULL + i), 1);
      mbar_init(BAR(B_V_EMPTY + i), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(BAR(B_S_FULL + t), 1);
      mbar_init(BAR(B_P_FULL + t), 4);  // one elected arrival per softmax warp
    }
    mbar_init(BAR(B_O_DONE), 1);
    mbar_init(BAR(B_TEARDOWN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    // the CTA's Q tiles depend on nothing the tile walk below computes: issued
    // first, their latency overlaps the CTA's set-up
    if (!(p.ctl.debug_flags & DBG_SKIP_Q_LOAD)) {
      const int prow0 = r * p.L + i0 - p.q_base;
      mbar_expect_tx(BAR(B_Q_FULL), kQTiles * LY::kTile);
      for (int t = 0; t < kQTiles; ++t)
        for (int c = 0; c < D / 64; ++c)
          if (in_bounds(tma_coords_ok(TmaExtent{D, p.q_rows, p.H, p.B}, c * 64, prow0 + t * kTileM, h, b), p.ctl, 1))
            tma_load_4d(sb + LY::kQ + t * LY::kTile + c * kBox, &tmQ, BAR(B_Q_FULL), c * 64, prow0 + t * kTileM, h,
                        b);
      q_issued = true;
    }
  }
  QRange cta;  // both query tiles together: decides which key tiles are visited
  make_qrange(p, r, i0, kRowsPerCta, cta);
  const int nkt = (p.L + kTileN - 1) / kTileN;
  int n_tiles = 0;
  walk_tiles(p, cta, nkt, [&](int, int) {
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
  if (warp < 4) {
    // ------------------------------------------------------------ control warpgroup
    regs_dec<kRegsLow>();
    if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producer (warp 0)
    if (warp == 0 && lane == 0 && n_tiles > 0) {
      // K(j) and V(j) land on one barrier (the V stage's), so that the MMA
      // thread waits once per key tile
      int issued[kVStages] = {};
      int j = 0;
      walk_tiles(p, cta, nkt, [&](int s, int kt) {
        const int sk = j % kKStages, sv = j % kVStages;
        // K's stage frees about two key tiles before V's: K goes first, its
        // bytes added to the V stage's phase without an arrival, once that
        // phase is the one of tile j (the phase of tile j - 2 has completed)
        if (j >= kKStages &&
            !wait_one<kWaitHint>(BAR(B_K_EMPTY + sk), (j / kKStages - 1) & 1, abort_flag, p.ctl, 1))
          return false;
        if (j >= kVStages &&
            !wait_one<kWaitHint>(BAR(B_V_FULL + sv), (j / kVStages - 1) & 1, abort_flag, p.ctl, 6))
          return false;
        const int hk = (int)(blockIdx.y % p.H) / p.G;
        const int krow = s * p.L + kt * kTileN;
        const bool rows_ok = in_bounds(tma_coords_ok(TmaExtent{D, p.S, p.Hk, p.B}, 0, krow, hk, b), p.ctl, 2);
        mbar_add_tx(BAR(B_V_FULL + sv), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          if (rows_ok) tma_load_4d(sb + LY::kK + sk * LY::kTile + c * kBox, &tmK, BAR(B_V_FULL + sv), c * 64, krow, hk, b);
        if (j >= kVStages &&
            !wait_one<kWaitHint>(BAR(B_V_EMPTY + sv), (j / kVStages - 1) & 1, abort_flag, p.ctl, 10)) {
          // the phase then completes once K has landed, and the drain below waits for it
          mbar_arrive(BAR(B_V_FULL + sv));
          ++issued[sv];
          return false;
        }
        mbar_expect_tx(BAR(B_V_FULL + sv), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          if (rows_ok) tma_load_4d(sb + LY::kV + sv * LY::kTile + c * kBox, &tmV, BAR(B_V_FULL + sv), c * 64, krow, hk, b);
        ++issued[sv];
        ++j;
        return true;
      });
      for (int st = 0; st < kVStages; ++st)
        if (issued[st]) drain_one(BAR(B_V_FULL + st), (issued[st] - 1) & 1, p.ctl, 21);
    }
    if (threadIdx.x == 0 && q_issued) drain_one(BAR(B_Q_FULL), 0, p.ctl, 20);
    __syncwarp();
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileN, 0, 0);  // A = Q, B = K: both K-major
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);      // A = P (TMEM), B = V: MN-major
      bool ok = wait_one<kWaitHint>(BAR(B_Q_FULL), 0, abort_flag, p.ctl, 2);
      auto issue_s = [&](int t, int j) {
        // descriptors built once and stepped (low words only: this thread runs on few registers)
        constexpr uint32_t kHi = sdesc_sw128_hi(1024);
        const uint32_t lk = sdesc_sw128_lo(sb + LY::kK + (j % kKStages) * LY::kTile, 16);
        const uint32_t lq = sdesc_sw128_lo(sb + LY::kQ + t * LY::kTile, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBox + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + LY::kTmemS + t * 128, sdesc_words(lq + off, kHi), sdesc_words(lk + off, kHi), kIdS,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(B_S_FULL + t));
      };
      auto issue_pv = [&](int t, int i) -> bool {
        if (!wait_one<kWaitHint>(BAR(B_P_FULL + t), i & 1, abort_flag, p.ctl, 3)) return false;
        tc_fence_after();
        const uint32_t lv = sdesc_sw128_lo(sb + LY::kV + (i % kVStages) * LY::kTile, kBox);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // A = P: 16 keys = 8 packed columns of the S_t tile; B = V: 16 key rows = 2048 bytes
          mma_bf16_ts(tmem + LY::kTmemO + t * 128, tmem + LY::kTmemS + t * 128 + kk * 8,
                      sdesc_words(lv + kk * 128, sdesc_sw128_hi(1024)), kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        if (t == kQTiles - 1 && i + kVStages < n_tiles) mma_commit(BAR(B_V_EMPTY + i % kVStages));
        return true;
      };
      int j = 0;
      if (ok) {
        tc_fence_after();
        walk_tiles(p, cta, nkt, [&](int, int) {
          for (int t = 0; t < kQTiles; ++t) {
            // PV_t(j-1) reads P_t from the S_t columns, so it goes first; S_t(j) then overwrites them
            if (j >= 1 && !issue_pv(t, j - 1)) {
              ok = false;
              return false;
            }
            if (t == 0) {
              if (!wait_one<kWaitHint>(BAR(B_V_FULL + j % kVStages), (j / kVStages) & 1, abort_flag, p.ctl, 5)) {
                ok = false;
                return false;
              }
              tc_fence_after();
            }
            issue_s(t, j);
          }
          if (j + kKStages < n_tiles) mma_commit(BAR(B_K_EMPTY + j % kKStages));
          ++j;
          return true;
        });
        if (ok && j >= 1)
          for (int t = 0; t < kQTiles && ok; ++t) ok = issue_pv(t, j - 1);
        if (ok) mma_commit(BAR(B_O_DONE));
      }
      // every issued MMA completes before the CTA frees TMEM
      mma_commit(BAR(B_TEARDOWN));
      drain_one(BAR(B_TEARDOWN), 0, p.ctl, 23);
    }
    __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    regs_inc<kRegsHigh>();
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    const int row = ((warp - 4) & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = tl + LY::kTmemS + t * 128;
    const uint32_t tO = tl + LY::kTmemO + t * 128;
    const int i = i0 + t * kTileM + row;
    bool valid = i < p.L;
    // batched: tiles classified per query tile, masks per row on partial tiles;
    // varlen: every row's key window, set up once (padding rows take the last valid row's)
    QRange qt;
    RowWin win;
    int gq = 0;
    if constexpr (VL) {
      make_row_win(p, r, min(i, p.L - 1), false, win);
    } else {
      make_qrange(p, r, i0 + t * kTileM, kTileM, qt);
      gq = tok(p, r, valid ? i : max(qt.i_last, 0));
    }
    float m_run = -INFINITY;  // running max, in log2 units (scores * scale * log2 e)
    float l_run = 0.f;        // running sum of exp2(x - m_run)
    bool ok = true;
    int j = 0;
    walk_tiles(p, cta, nkt, [&](int s, int kt) {
      // column window [c_lo, c_hi) of allowed keys for this row (all 128 when the tile is full)
      int c_lo = 0, c_hi = kTileN;
      if constexpr (VL)
        row_win_cols(p, win, s, kt * kTileN, kTileN, c_lo, c_hi);
      else if (!kv_tile_full(p, qt, s, kt))
        row_key_window(p, gq, s, kt, c_lo, c_hi);
      const bool masked = c_lo > 0 || c_hi < kTileN;
      if (!wait_warp<kWaitHint>(BAR(B_S_FULL + t), j & 1, abort_flag, p.ctl, 7)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      // all 128 scores of the row in registers, in two halves: the row max of the
      // first half runs while the second half is loading
      uint32_t v[kTileN];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 0));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      float mc[4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (hh == 1) {
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 64));
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 96));
        }
        if (masked) {
          const uint64_t mw = bit_window64(c_lo - 64 * hh, c_hi - 64 * hh);
#pragma unroll
          for (int u = 0; u < 64; ++u)
            v[64 * hh + u] = ((mw >> u) & 1ull) ? v[64 * hh + u] : __float_as_uint(-INFINITY);
        }
        // four chains of three-input maxima over the 64 scores of this half
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c0 = 64 * hh + 16 * q;
          float m = hh == 0 ? __uint_as_float(v[c0]) : fmaxf(mc[q], __uint_as_float(v[c0]));
#pragma unroll
          for (int c = c0 + 1; c < c0 + 15; c += 2) m = fmax3f(m, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
          mc[q] = fmaxf(m, __uint_as_float(v[c0 + 15]));
        }
      }
      // raw scores: the scale is > 0, so max(s) * scale = max(s * scale)
      const float mx = fmax3f(mc[0], mc[1], fmaxf(mc[2], mc[3])) * p.scale_log2;
      float alpha = 1.f;
      if (mx > -INFINITY) {
        if (m_run == -INFINITY) {
          m_run = mx;  // nothing accumulated yet for this row
        } else if (mx > m_run + 8.f) {
          alpha = fast_exp2(m_run - mx);
          m_run = mx;
        }
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // P = exp2(s * scale - m) and the row sum; P goes as bf16 pairs over the
      // first 64 columns of this tile's S columns (column 16 c32 + u holds keys
      // 32 c32 + 2u and 32 c32 + 2u + 1); the scores are already in registers.
      // s * scale - m and the sums run two lanes per instruction (f32x2).
      const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2), nm2 = f32x2(-m_use, -m_use);
      uint64_t acc[4] = {0, 0, 0, 0};  // four pairs of partial row sums (+0.0f bits)
#pragma unroll
      for (int c32 = 0; c32 < kTileN / 32; ++c32) {
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int c = c32 * 32 + 2 * u;
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), sc2, nm2), x0, x1);
          const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
          acc[u & 3] = add_f32x2(acc[u & 3], f32x2(e0, e1));
          pk[u] = pack_bf16x2(e0, e1);
        }
        tmem_st16(tS + c32 * 16, pk);
      }
      float s0, s1;
      f32x2_split(add_f32x2(add_f32x2(acc[0], acc[1]), add_f32x2(acc[2], acc[3])), s0, s1);
      l_run = l_run * alpha + (s0 + s1);
      // O_t is stable here (the commit behind S_FULL covers PV_t(j-1)) and PV_t(j)
      // waits for P_FULL, so the rescale fits between them
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_P_FULL + t));
      ++j;
      return true;
    });

    const long long qpos = (long long)(r * p.L + i - p.q_base);  // row of q / out / lse
    if (valid && !in_bounds(qpos >= 0 && qpos < p.q_rows, p.ctl, 3)) valid = false;  // skip this row's stores
    // varlen computed in original order: out / lse rows of the caller's layout order
    const int* rmap = VL ? p.row_map : nullptr;
    const long long opos = rmap && valid ? (long long)__ldg(rmap + qpos) : qpos;
    float* lse_ptr = p.lse + (long long)b * p.l_sb + (long long)h * p.l_sh + opos * p.l_ss;
    if (n_tiles > 0) {
      if (ok && wait_warp<kWaitHint>(BAR(B_O_DONE), 0, abort_flag, p.ctl, 9)) {
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        if constexpr (!VL) {
          // long CTAs: one row per thread, straight to global memory
          const long long orow = (long long)b * p.o_sb + (long long)h * p.o_sh + qpos * p.o_ss;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
            if (valid) {
              if (p.out_f32) {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow + c * 32);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                       __uint_as_float(o[4 * k + 2]) * inv_l, __uint_as_float(o[4 * k + 3]) * inv_l);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow + c * 32);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  uint4 v;
                  v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
                  v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
                  v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
                  v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
                  dst[k] = v;
                }
              }
            }
          }
        } else {
          fence_proxy_async_smem();
          // varlen (short CTAs, where the epilogue weighs): O leaves through
          // shared memory (every MMA is done, so the operand buffers are
          // free).  Each thread writes its row into its warp's slot (16-byte
          // pieces, the piece index XOR the row's low bits, so the 32 lanes
          // spread over the banks), then the warp stores whole rows with
          // consecutive lanes on consecutive pieces of a row.
          const int esz = p.out_f32 ? 4 : 2;
          const int nch = D * esz / 16;  // 16-byte pieces per row: 8, 16 or 32
          uint8_t* slot = sp + (warp - 4) * (32 * D * 4);
          uint8_t* mine = slot + lane * nch * 16;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
            if (p.out_f32) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4*>(mine + (((c * 8 + k) ^ (lane & 7)) << 4)) =
                    make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                __uint_as_float(o[4 * k + 2]) * inv_l, __uint_as_float(o[4 * k + 3]) * inv_l);
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
                v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
                v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
                v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
                *reinterpret_cast<uint4*>(mine + (((c * 4 + k) ^ (lane & 7)) << 4)) = v;
              }
            }
          }
          __syncwarp();
          const int rows_per = 32 / nch, lr = lane / nch, pc = lane % nch;
          const int i_w = i0 + t * kTileM + (warp & 3) * 32;  // local position of the warp's first row
          for (int R0 = 0; R0 < 32; R0 += rows_per) {
            const int R = R0 + lr;
            const uint4 val = *reinterpret_cast<const uint4*>(slot + R * nch * 16 + ((pc ^ (R & 7)) << 4));
            const long long q_row = (long long)(r * p.L + i_w + R - p.q_base);
            if (i_w + R < p.L && in_bounds(q_row >= 0 && q_row < p.q_rows, p.ctl, 4)) {
              const long long o_row = rmap ? (long long)__ldg(rmap + q_row) : q_row;
              const long long e = (long long)b * p.o_sb + (long long)h * p.o_sh + o_row * p.o_ss;
              *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.out) + e * esz + pc * 16) = val;
            }
          }
        }
        if (valid) *lse_ptr = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
    } else if (valid) {
      // no key tile at all (a single ring step can be empty): out = 0, lse = -inf
      const long long orow = (long long)b * p.o_sb + (long long)h * p.o_sh + opos * p.o_ss;
      if (p.out_f32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow);
        for (int k = 0; k < D / 4; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow);
        for (int k = 0; k < D / 8; ++k) dst[k] = make_uint4(0, 0, 0, 0);
      }
      *lse_ptr = -INFINITY;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool VL>
cudaError_t launch_fwd_v(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t st) {
  using LY = FwdLayout<D>;
  // the register split inside the kernel is only safe with the launch
  // allocation it was sized for
  cudaError_t e = configure_kernel<ring_fwd_kernel<D, VL>>(kLaunchRegs, LY::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_pairs = (p.L + kRowsPerCta - 1) / kRowsPerCta;
  dim3 grid((unsigned)((p.r_only >= 0 ? 1 : p.N) * n_pairs), (unsigned)(p.B * p.H));
  FwdParamsT<VL> pv;
  static_cast<FwdParams&>(pv) = p;
  ring_fwd_kernel<D, VL><<<grid, kThreads, LY::kAlloc, st>>>(tq, tk, tv, pv);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t st) {
  return p.cu ? launch_fwd_v<D, true>(tq, tk, tv, p, st) : launch_fwd_v<D, false>(tq, tk, tv, p, st);
}

}  // namespace

size_t fwd_smem_bytes(int D) { return D == 64 ? FwdLayout<64>::kAlloc : FwdLayout<128>::kAlloc; }

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t st) {
  if (D == 64) return launch_fwd_t<64>(tq, tk, tv, p, st);
  return launch_fwd_t<128>(tq, tk, tv, p, st);
}

}  // namespace ra
