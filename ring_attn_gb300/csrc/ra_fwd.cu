// Ring-attention forward on sm_103a: blockwise exact attention of one 128-row
// query tile against every key tile of the KV shards it meets on the ring,
// with the online-softmax merge held in fp32 across all ring steps.
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
// Kernel structure (one CTA per query tile, 8 warps):
//   warp 0     TMA producer: Q once, then K tiles into a 3-stage ring (freed
//              when S = Q K^T completes) and V tiles into a 2-stage ring
//              (freed when O += P V completes), so loads run ahead of use.
//   warp 1     MMA issuer (one thread): S = Q K^T into a double-buffered TMEM
//              tile, then O += P V into the TMEM output accumulator.
//   warp 2     allocates / frees 512 TMEM columns.
//   warps 4-7  softmax: one thread per query row (the TMEM lane of that row).
//              It reads its S row from TMEM, masks, updates the running max
//              (rescaling O only when the max grows by more than 2^8), writes
//              P as bf16 into a 128B-swizzled shared tile for the PV MMA, and
//              finally normalises O and writes out and lse.
// Empty key tiles (causal / varlen) are never loaded; only partial tiles are
// masked element by element.
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBox = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 bytes) = 16 KB

constexpr int kKStages = 3;  // K tiles are released as soon as S = Q K^T completes
constexpr int kVStages = 2;  // V tiles are released when O += P V completes

template <int D>
struct FwdLayout {
  static constexpr int kTile = (D / 64) * kBox;  // one Q/K/V tile (128 rows x D)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;              // kKStages stages
  static constexpr int kV = kK + kKStages * kTile;   // kVStages stages
  static constexpr int kP = kV + kVStages * kTile;   // P tile: 2 boxes (128 key columns)
  static constexpr int kBar = kP + 2 * kBox;
  static constexpr int kNumBars = 18;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;   // slack to align the base to 1024 bytes
  static constexpr uint32_t kTmemO = 256;        // S buffers at columns 0 and 128
};

enum FwdBar {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // kKStages
  B_K_EMPTY = 4,   // kKStages
  B_V_FULL = 7,    // kVStages
  B_V_EMPTY = 9,   // kVStages
  B_S_FULL = 11,   // 2
  B_S_FREE = 13,   // 2
  B_P_FULL = 15,
  B_PV_DONE = 16,
  B_TEARDOWN = 17
};

struct QTile {
  int b, h, r, i0, i_last;
  long long gq_lo, gq_hi;    // original token indices of the first / last valid row
  long long key_lo, key_hi;  // varlen: keys any row of the tile may see (inclusive)
  int seg_single;            // varlen: the segment of every valid row, or -1
};

// Key-tile range [lo, hi) of KV shard s that can hold an allowed key.
__device__ __forceinline__ void kv_range(const FwdParams& p, const QTile& q, int s, int nkt, int& lo, int& hi) {
  if (p.cu) {
    const long long base = (long long)s * p.L;
    long long jlo = q.key_lo - base, jhi = q.key_hi - base;
    if (jlo < 0) jlo = 0;
    if (jhi > p.L - 1) jhi = p.L - 1;
    if (jlo > jhi) {
      lo = hi = 0;
      return;
    }
    lo = (int)(jlo / kTileN);
    hi = (int)(jhi / kTileN) + 1;
    return;
  }
  lo = 0;
  if (!p.causal) {
    hi = nkt;
    return;
  }
  // token_of is increasing inside a shard, so the allowed keys of the tile's
  // last (largest-token) row are a prefix of the shard.
  const int jm = last_local_at_or_before(p.layout, p.N, p.L, s, q.gq_hi);
  hi = jm < 0 ? 0 : jm / kTileN + 1;
}

// True when every (valid row, key) pair of the tile is allowed: no masking needed.
__device__ __forceinline__ bool tile_full(const FwdParams& p, const QTile& q, int s, int kt) {
  const int j0 = kt * kTileN;
  if (j0 + kTileN > p.L) return false;
  if (p.cu) {
    if (q.seg_single < 0) return false;
    const long long base = (long long)s * p.L + j0;
    const long long slo = __ldg(p.cu + q.seg_single), shi = __ldg(p.cu + q.seg_single + 1);
    if (base < slo || base + kTileN > shi) return false;
    return !p.causal || q.gq_lo >= base + kTileN - 1;
  }
  return !p.causal || q.gq_lo >= token_of(p.layout, p.N, p.L, s, j0 + kTileN - 1);
}

// Calls f(s, kt) for every key tile the query tile meets, in ring order.
template <class F>
__device__ __forceinline__ void walk_tiles(const FwdParams& p, const QTile& q, int nkt, F&& f) {
  const int t0 = p.step < 0 ? 0 : p.step;
  const int t1 = p.step < 0 ? p.N : p.step + 1;
  for (int t = t0; t < t1; ++t) {
    int s = q.r - t;
    if (s < 0) s += p.N;
    int lo, hi;
    kv_range(p, q, s, nkt, lo, hi);
    for (int kt = lo; kt < hi; ++kt)
      if (!f(s, kt)) return;
  }
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    ring_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using LY = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sp = smem_raw + (sb - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  QTile q;
  q.b = blockIdx.y / p.H;
  q.h = blockIdx.y % p.H;
  // causal: the later query tiles carry more work, start them first
  const int x = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  q.r = x / p.n_qtiles;
  q.i0 = (x % p.n_qtiles) * kTileM;
  q.i_last = min(q.i0 + kTileM, p.L) - 1;
  q.gq_lo = token_of(p.layout, p.N, p.L, q.r, q.i0);
  q.gq_hi = token_of(p.layout, p.N, p.L, q.r, q.i_last);
  q.key_lo = q.key_hi = 0;
  q.seg_single = -1;
  if (p.cu) {
    const int sa = segment_of(p.cu, p.n_seqs, q.gq_lo);
    const int sz = segment_of(p.cu, p.n_seqs, q.gq_hi);
    q.key_lo = __ldg(p.cu + sa);
    q.key_hi = p.causal ? q.gq_hi : (long long)__ldg(p.cu + sz + 1) - 1;
    q.seg_single = sa == sz ? sa : -1;
  }
  const int nkt = (p.L + kTileN - 1) / kTileN;
  int n_tiles = 0;
  walk_tiles(p, q, nkt, [&](int, int) {
    ++n_tiles;
    return true;
  });

  const uint32_t bar0 = sb + LY::kBar;
  auto BAR = [bar0](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + LY::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sp + LY::kMisc);

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q_FULL), 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(BAR(B_K_FULL + i), 1);
      mbar_init(BAR(B_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(BAR(B_V_FULL + i), 1);
      mbar_init(BAR(B_V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_S_FULL + i), 1);
      mbar_init(BAR(B_S_FREE + i), 4);  // one elected arrival per softmax warp
    }
    mbar_init(BAR(B_P_FULL), 4);
    mbar_init(BAR(B_PV_DONE), 1);
    mbar_init(BAR(B_TEARDOWN), 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      bool q_issued = false;
      int k_issued[kKStages] = {}, v_issued[kVStages] = {};
      const int prow0 = q.r * p.L + q.i0;
      if (!(p.ctl.debug_flags & DBG_SKIP_Q_LOAD)) {
        mbar_expect_tx(BAR(B_Q_FULL), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sb + LY::kQ + c * kBox, &tmQ, BAR(B_Q_FULL), c * 64, prow0, q.h, q.b);
        q_issued = true;
      }
      int j = 0;
      walk_tiles(p, q, nkt, [&](int s, int kt) {
        const int ks = j % kKStages, vs = j % kVStages;
        const int row = s * p.L + kt * kTileN;
        // use number u of a stage waits for the release of use u - 1
        if (j >= kKStages && !wait_one(BAR(B_K_EMPTY + ks), (j / kKStages - 1) & 1, abort_flag, p.ctl, 1))
          return false;
        mbar_expect_tx(BAR(B_K_FULL + ks), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sb + LY::kK + ks * LY::kTile + c * kBox, &tmK, BAR(B_K_FULL + ks), c * 64, row, q.h, q.b);
        ++k_issued[ks];
        if (j >= kVStages && !wait_one(BAR(B_V_EMPTY + vs), (j / kVStages - 1) & 1, abort_flag, p.ctl, 10))
          return false;
        mbar_expect_tx(BAR(B_V_FULL + vs), LY::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sb + LY::kV + vs * LY::kTile + c * kBox, &tmV, BAR(B_V_FULL + vs), c * 64, row, q.h, q.b);
        ++v_issued[vs];
        ++j;
        return true;
      });
      // every issued copy lands before the CTA may exit
      if (q_issued) drain_one(BAR(B_Q_FULL), 0, p.ctl, 20);
      for (int st = 0; st < kKStages; ++st)
        if (k_issued[st]) drain_one(BAR(B_K_FULL + st), (k_issued[st] - 1) & 1, p.ctl, 21);
      for (int st = 0; st < kVStages; ++st)
        if (v_issued[st]) drain_one(BAR(B_V_FULL + st), (v_issued[st] - 1) & 1, p.ctl, 22);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTileN, 0, 0);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);
      bool ok = wait_one(BAR(B_Q_FULL), 0, abort_flag, p.ctl, 2);
      auto issue_pv = [&](int i) -> bool {
        const int vs = i % kVStages;
        if (!wait_one(BAR(B_P_FULL), i & 1, abort_flag, p.ctl, 3)) return false;
        if (!wait_one(BAR(B_V_FULL + vs), (i / kVStages) & 1, abort_flag, p.ctl, 4)) return false;
        tc_fence_after();
        const uint32_t vb = sb + LY::kV + vs * LY::kTile;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // A = P (K-major, 128 query rows x 128 keys); B = V (MN-major: key rows, D columns)
          const uint64_t a = sdesc_sw128(sb + LY::kP + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, kBox, 1024);
          mma_bf16_ss(tmem + LY::kTmemO, a, bd, kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR(B_PV_DONE));
        if (i + kVStages < n_tiles) mma_commit(BAR(B_V_EMPTY + vs));
        return true;
      };
      int j = 0;
      if (ok) {
        tc_fence_after();
        walk_tiles(p, q, nkt, [&](int, int) {
          const int st = j & 1, ks = j % kKStages;
          if (!wait_one(BAR(B_K_FULL + ks), (j / kKStages) & 1, abort_flag, p.ctl, 5) ||
              (j >= 2 && !wait_one(BAR(B_S_FREE + st), ((j >> 1) - 1) & 1, abort_flag, p.ctl, 6))) {
            ok = false;
            return false;
          }
          tc_fence_after();
          const uint32_t kb = sb + LY::kK + ks * LY::kTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // A = Q, B = K, both K-major (D contiguous)
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            mma_bf16_ss(tmem + st * 128, sdesc_sw128(sb + LY::kQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                        kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(BAR(B_S_FULL + st));
          if (j + kKStages < n_tiles) mma_commit(BAR(B_K_EMPTY + ks));
          if (j >= 1 && !issue_pv(j - 1)) {
            ok = false;
            return false;
          }
          ++j;
          return true;
        });
        if (ok && j >= 1) issue_pv(j - 1);
      }
      // every issued MMA completes before the CTA frees TMEM
      mma_commit(BAR(B_TEARDOWN));
      drain_one(BAR(B_TEARDOWN), 0, p.ctl, 23);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int row = (warp - 4) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int i = q.i0 + row;
    const bool valid = i < p.L;
    const long long gq = token_of(p.layout, p.N, p.L, q.r, valid ? i : q.i_last);
    long long rk_lo = 0, rk_hi = 0;  // varlen: this row's allowed keys [rk_lo, rk_hi)
    if (p.cu) {
      const int sg = segment_of(p.cu, p.n_seqs, gq);
      rk_lo = __ldg(p.cu + sg);
      rk_hi = p.causal ? gq + 1 : (long long)__ldg(p.cu + sg + 1);
    }
    float m_run = -INFINITY;  // running max, in log2 units (scores * scale * log2 e)
    float l_run = 0.f;        // running sum of exp2(x - m_run)
    bool ok = true;
    int j = 0;
    walk_tiles(p, q, nkt, [&](int s, int kt) {
      const int st = j & 1;
      if (!wait_warp(BAR(B_S_FULL + st), (j >> 1) & 1, abort_flag, p.ctl, 7)) {
        ok = false;
        return false;
      }
      tc_fence_after();
      float x[kTileN];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t sa = tl + (uint32_t)(st * 128);
        tmem_ld32(sa + 0, r0);
        tmem_ld32(sa + 32, r1);
        tmem_ld32(sa + 64, r2);
        tmem_ld32(sa + 96, r3);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        tmem_ld_wait(r2);
        tmem_ld_wait(r3);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]);
          x[32 + c] = __uint_as_float(r1[c]);
          x[64 + c] = __uint_as_float(r2[c]);
          x[96 + c] = __uint_as_float(r3[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_S_FREE + st));
      if (!tile_full(p, q, s, kt)) {
        const int j0 = kt * kTileN;
        const int jlim = min(kTileN, p.L - j0);
        int c_lo = 0, c_hi = jlim;
        if (p.cu) {
          const long long base = (long long)s * p.L + j0;
          const long long lo = rk_lo - base, hi = rk_hi - base;
          c_lo = (int)(lo < 0 ? 0 : (lo > kTileN ? kTileN : lo));
          c_hi = (int)(hi < 0 ? 0 : (hi > jlim ? jlim : hi));
        } else if (p.causal) {
          const int jm = last_local_at_or_before(p.layout, p.N, p.L, s, gq);
          c_hi = min(jlim, jm - j0 + 1);
        }
#pragma unroll
        for (int c = 0; c < kTileN; ++c) x[c] = (c >= c_lo && c < c_hi) ? x[c] : -INFINITY;
      }
      float m0 = x[0], m1 = x[1], m2 = x[2], m3 = x[3];
#pragma unroll
      for (int c = 4; c < kTileN; c += 4) {
        m0 = fmaxf(m0, x[c]);
        m1 = fmaxf(m1, x[c + 1]);
        m2 = fmaxf(m2, x[c + 2]);
        m3 = fmaxf(m3, x[c + 3]);
      }
      // raw scores: the scale is > 0, so max(s) * scale = max(s * scale)
      const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * p.scale_log2;
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
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int c = 0; c < kTileN; c += 4) {
        x[c] = fast_exp2(fmaf(x[c], p.scale_log2, -m_use));
        x[c + 1] = fast_exp2(fmaf(x[c + 1], p.scale_log2, -m_use));
        x[c + 2] = fast_exp2(fmaf(x[c + 2], p.scale_log2, -m_use));
        x[c + 3] = fast_exp2(fmaf(x[c + 3], p.scale_log2, -m_use));
        s0 += x[c];
        s1 += x[c + 1];
        s2 += x[c + 2];
        s3 += x[c + 3];
      }
      l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
      if (j > 0) {
        // the previous PV has finished: P's buffer is free and O is stable
        if (!wait_warp(BAR(B_PV_DONE), (j - 1) & 1, abort_flag, p.ctl, 8)) {
          ok = false;
          return false;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tl + LY::kTmemO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(tl + LY::kTmemO + c * 32, o);
          }
          tmem_st_wait();
        }
      }
      uint8_t* pb = sp + LY::kP;
#pragma unroll
      for (int k = 0; k < kTileN / 8; ++k) {
        uint4 v;
        v.x = pack_bf16x2(x[8 * k + 0], x[8 * k + 1]);
        v.y = pack_bf16x2(x[8 * k + 2], x[8 * k + 3]);
        v.z = pack_bf16x2(x[8 * k + 4], x[8 * k + 5]);
        v.w = pack_bf16x2(x[8 * k + 6], x[8 * k + 7]);
        *reinterpret_cast<uint4*>(pb + (k >> 3) * kBox + sw128_offset(row, k & 7)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_P_FULL));
      ++j;
      return true;
    });

    const long long orow = (long long)q.b * p.o_sb + (long long)q.h * p.o_sh + (long long)(q.r * p.L + i) * p.o_ss;
    float* lse_ptr = p.lse + (long long)q.b * p.l_sb + (long long)q.h * p.l_sh + (long long)(q.r * p.L + i) * p.l_ss;
    if (n_tiles > 0) {
      if (ok && wait_warp(BAR(B_PV_DONE), (n_tiles - 1) & 1, abort_flag, p.ctl, 9)) {
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + LY::kTmemO + c * 32, o);
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
        if (valid) *lse_ptr = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      }
    } else if (valid) {
      // no key tile at all (a single ring step can be empty): out = 0, lse = -inf
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

template <int D>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         cudaStream_t st) {
  using LY = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(ring_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(p.N * p.n_qtiles), (unsigned)(p.B * p.H));
  ring_fwd_kernel<D><<<grid, 256, LY::kAlloc, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) { return D == 64 ? FwdLayout<64>::kAlloc : FwdLayout<128>::kAlloc; }

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t st) {
  if (D == 64) return launch_fwd_t<64>(tq, tk, tv, p, st);
  return launch_fwd_t<128>(tq, tk, tv, p, st);
}

}  // namespace ra
