// Memory-bound kernels of the ring-attention path: shard-layout permutation,
// the standalone LSE merge and the backward preprocess D = rowsum(dO * O).  All are grid-stride loops with
// 16-byte accesses, sized to a multiple of the SM count.
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreads = 256;

int grid_for(long long work_items, int per_block) {
  long long blocks = (work_items + per_block - 1) / per_block;
  long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

// ------------------------------------------------------------------ permutation
// A "row" is the packed run of elements after the sequence dimension, moved as
// vpr vectors V (16 bytes when the row allows it).  blockIdx.y walks the outer
// index (decoded once per block); blockIdx.x walks the layout positions with
// rows_per_block rows per block and turn, vpr threads per row, so a row costs
// its layout map and two multiply-adds.  When a row is one vector per thread,
// each thread moves UNROLL rows per turn, all loads before the stores
// (streaming cache hints: every byte is read and written once).
template <typename V, int UNROLL>
__global__ void __launch_bounds__(kThreads) permute_kernel(PermuteArgs a, int vpr, int rows_per_block) {
  const int rloc = threadIdx.x / vpr, v = threadIdx.x % vpr;
  if (rloc >= rows_per_block) return;
  const int L = a.s / a.N;
  const int pstride = (int)gridDim.x * rows_per_block;
  for (long long o = blockIdx.y; o < a.n_outer; o += gridDim.y) {
    const long long o2 = o % a.outer_shape[2];
    const long long o01 = o / a.outer_shape[2];
    const long long o1 = o01 % a.outer_shape[1];
    const long long o0 = o01 / a.outer_shape[1];
    const char* sbase = reinterpret_cast<const char*>(a.src) +
                        (o0 * a.src_outer_stride[0] + o1 * a.src_outer_stride[1] + o2 * a.src_outer_stride[2]) *
                            a.esize;
    char* dbase = reinterpret_cast<char*>(a.dst) +
                  (o0 * a.dst_outer_stride[0] + o1 * a.dst_outer_stride[1] + o2 * a.dst_outer_stride[2]) * a.esize;
    for (int p0 = (int)blockIdx.x * rows_per_block + rloc; p0 < a.s; p0 += UNROLL * pstride) {
      const V* src[UNROLL];
      V* dst[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int p = p0 + u * pstride;  // layout position
        src[u] = nullptr;
        dst[u] = nullptr;
        if (p >= a.s) continue;
        // original token at layout position p
        const int g = a.gmap != nullptr ? __ldg(a.gmap + p)
                      : a.cu == nullptr ? token_of(a.layout, a.N, L, p / L, p % L)
                      : a.layout == LAYOUT_ZIGZAG ? vz_token(a.cu, a.n_seqs, a.N, p / L, p % L)
                                                  : p;
        if (kDebugBounds && (g < 0 || g >= a.s)) {  // the layout map left the sequence
          record_error(a.ctl, DEV_BOUNDS, 0x80 | 30);
          continue;
        }
        const long long src_pos = a.inverse ? p : g;
        const long long dst_pos = a.inverse ? g : p;
        src[u] = reinterpret_cast<const V*>(sbase + src_pos * a.src_seq_stride * a.esize);
        dst[u] = reinterpret_cast<V*>(dbase + dst_pos * a.dst_seq_stride * a.esize);
      }
      if (a.vpr_total == vpr) {
        V val[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
          if (src[u]) val[u] = __ldcs(src[u] + v);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
          if (dst[u]) __stcs(dst[u] + v, val[u]);
      } else {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
          if (src[u])
            for (int k = v; k < a.vpr_total; k += vpr) dst[u][k] = __ldg(src[u] + k);
      }
    }
  }
}

// ------------------------------------------------------------------ LSE merge
// A group of d/VEC threads (a power of two dividing 32, so a group sits inside
// one warp) owns a row, VEC (4, 8 or 16) consecutive columns per thread:
//   lse_new = max(a, b) + log1p(exp(-|a - b|)),  w = exp(lse_blk - lse_new),
//   out_acc += w * (out_blk - out_acc).
// Each thread handles UNROLL rows per loop turn and issues every load before
// using any, so that enough bytes are in flight to keep HBM busy; the row data
// is read and written once, with streaming cache hints.  Loop control is
// warp-uniform: every lane of a row has read the old lse_acc (before
// __syncwarp) before the row's first lane overwrites it.
template <bool BLK_F32, int VEC, int UNROLL>
__global__ void __launch_bounds__(kThreads) lse_merge_kernel(MergeArgs a) {
  constexpr int NV = VEC / 4;  // float4 of out_acc per thread
  const long long per_row = a.d / VEC;
  const long long total = a.rows * per_row;
  const long long step = (long long)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (long long base = (long long)blockIdx.x * blockDim.x + threadIdx.x - lane; base < total;
       base += UNROLL * step) {
    float* oa[UNROLL];
    float* la[UNROLL];
    float A[UNROLL], B[UNROLL];
    float4 ob[UNROLL][NV], oc[UNROLL][NV];
    bool live[UNROLL];
    bool first[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long t = base + u * step + lane;
      live[u] = t < total;
      const long long c = live[u] ? (t & (per_row - 1)) : 0;  // per_row is a power of two
      first[u] = c == 0;
      long long rw = live[u] ? (t >> a.qshift) : 0;
      long long i0 = 0, i1 = 0, i2 = rw;
      if (!a.flat) {
        i2 = rw % a.n2;
        rw /= a.n2;
        i1 = rw % a.n1;
        i0 = rw / a.n1;
      }
      oa[u] = a.out_acc + i0 * a.oa_s0 + i1 * a.oa_s1 + i2 * a.oa_s2 + VEC * c;
      la[u] = a.lse_acc + i0 * a.la_s0 + i1 * a.la_s1 + i2 * a.la_s2;
      const float* lb = a.lse_blk + i0 * a.lb_s0 + i1 * a.lb_s1 + i2 * a.lb_s2;
      const long long bofs = i0 * a.ob_s0 + i1 * a.ob_s1 + i2 * a.ob_s2 + VEC * c;
      A[u] = live[u] ? *la[u] : 0.f;
      B[u] = live[u] ? __ldg(lb) : -INFINITY;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        oc[u][k] = live[u] ? __ldcs(reinterpret_cast<const float4*>(oa[u]) + k) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (BLK_F32) {
#pragma unroll
        for (int k = 0; k < NV; ++k)
          ob[u][k] = live[u] ? __ldcs(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.out_blk) + bofs) + k)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (VEC % 8 == 0) {
#pragma unroll
        for (int k8 = 0; k8 < VEC / 8; ++k8) {
          const uint4 raw = live[u] ? __ldcs(reinterpret_cast<const uint4*>(
                                          reinterpret_cast<const __nv_bfloat16*>(a.out_blk) + bofs) + k8)
                                    : make_uint4(0u, 0u, 0u, 0u);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
          ob[u][2 * k8] = make_float4(__low2float(h[0]), __high2float(h[0]), __low2float(h[1]), __high2float(h[1]));
          ob[u][2 * k8 + 1] =
              make_float4(__low2float(h[2]), __high2float(h[2]), __low2float(h[3]), __high2float(h[3]));
        }
      } else {
        const uint2 raw = live[u] ? __ldcs(reinterpret_cast<const uint2*>(
                                        reinterpret_cast<const __nv_bfloat16*>(a.out_blk) + bofs))
                                  : make_uint2(0u, 0u);
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        ob[u][0] = make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (!live[u]) continue;
      float4 r[NV];
      float lse_new;
      if (B[u] == -INFINITY) {
        // empty block: unchanged, except that an empty accumulator is normalised to out = 0
        if (A[u] != -INFINITY) continue;
#pragma unroll
        for (int k = 0; k < NV; ++k) r[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        lse_new = -INFINITY;
      } else if (A[u] == -INFINITY) {
#pragma unroll
        for (int k = 0; k < NV; ++k) r[k] = ob[u][k];  // empty accumulator: take the block
        lse_new = B[u];
      } else {
        lse_new = fmaxf(A[u], B[u]) + log1pf(expf(-fabsf(A[u] - B[u])));
        const float w = expf(B[u] - lse_new);
#pragma unroll
        for (int k = 0; k < NV; ++k)
          r[k] = make_float4(oc[u][k].x + w * (ob[u][k].x - oc[u][k].x), oc[u][k].y + w * (ob[u][k].y - oc[u][k].y),
                             oc[u][k].z + w * (ob[u][k].z - oc[u][k].z), oc[u][k].w + w * (ob[u][k].w - oc[u][k].w));
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) __stcs(reinterpret_cast<float4*>(oa[u]) + k, r[k]);
      if (first[u]) *la[u] = lse_new;
    }
  }
}

// ------------------------------------------------------------------ backward preprocess
// Per query row: -D = -sum_d dO * O and -lse2 = -lse * log2(e), stored per shard
// with each shard's rows padded to stat_L (padding: -D = 0, -lse2 = -inf, so a
// padded column contributes P = 0 and dS = 0).  The statistics rows are taken
// in order, (b, h, shard, row), kPreUnroll * rows_per_block consecutive rows
// per block and turn (they never straddle a shard: stat_L is a multiple of
// 128), so each turn reads contiguous runs of dO and O; d/8 threads per row (8
// bf16 each), every load of the turn issued before the first use; one
// persistent wave of blocks strides over the turns.
constexpr int kPreUnroll = 4;

__global__ void __launch_bounds__(kThreads, 4) bwd_pre_kernel(View4 dout, View4 out, LseView lse, float* nD,
                                                               float* nlse2, int N, int stat_L, DevCtl ctl,
                                                               const int* out_row) {
  const int tpr = dout.d / 8;  // threads per row; divides 32, so a row's threads share a warp
  const int rows_per_block = kThreads / tpr;
  const int rows_per_turn = kPreUnroll * rows_per_block;
  const int rloc = threadIdx.x / tpr, part = threadIdx.x % tpr;
  const int L = dout.s / N;
  const long long n_rows = (long long)dout.b * dout.h * N * stat_L;
  for (long long row0 = (long long)blockIdx.x * rows_per_turn; row0 < n_rows;
       row0 += (long long)gridDim.x * rows_per_turn) {
    const long long bhr = row0 / stat_L;
    const int i0 = (int)(row0 - bhr * stat_L);
    const int r = (int)(bhr % N);
    const long long bh = bhr / N;
    const long long h = bh % dout.h, b = bh / dout.h;
    const __nv_bfloat16* dsrc = reinterpret_cast<const __nv_bfloat16*>(dout.data) + b * dout.sb + h * dout.sh;
    const __nv_bfloat16* osrc = reinterpret_cast<const __nv_bfloat16*>(out.data) + b * out.sb + h * out.sh;
    const float* lsrc = lse.data + b * lse.sb + h * lse.sh;
    uint4 x[kPreUnroll], y[kPreUnroll];
    float l[kPreUnroll];
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const int i = i0 + u * rows_per_block + rloc;
      const long long p = (long long)r * L + i;  // layout position
      bool real = i < L && in_bounds(p < dout.s, ctl, 31);
      // out and lse of position p: row out_row[p] of the caller's layout order, or p
      const long long po = real && out_row ? (long long)__ldg(out_row + p) : p;
      real = real && in_bounds(po >= 0 && po < out.s, ctl, 32);
      x[u] = real ? __ldcs(reinterpret_cast<const uint4*>(dsrc + p * dout.ss) + part) : make_uint4(0, 0, 0, 0);
      y[u] = real ? __ldcs(reinterpret_cast<const uint4*>(osrc + po * out.ss) + part) : make_uint4(0, 0, 0, 0);
      l[u] = real && part == 0 ? __ldcs(lsrc + po * lse.ss) : INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const __nv_bfloat162* xv = reinterpret_cast<const __nv_bfloat162*>(&x[u]);
      const __nv_bfloat162* yv = reinterpret_cast<const __nv_bfloat162*>(&y[u]);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 a2 = __bfloat1622float2(xv[k]);
        const float2 c2 = __bfloat1622float2(yv[k]);
        acc = fmaf(a2.x, c2.x, acc);
        acc = fmaf(a2.y, c2.y, acc);
      }
      for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (part == 0) {
        const long long row = row0 + u * rows_per_block + rloc;
        nD[row] = -acc;
        nlse2[row] = l[u] * -1.4426950408889634f;  // padding rows: +inf * -log2(e) = -inf
      }
    }
  }
}

// One thread per layout position: the search of cu_seqlens that the permute
// kernel would repeat for every row of every tensor is done once per call.
__global__ void __launch_bounds__(kThreads) zigzag_varlen_map_kernel(const int* cu, int n_seqs, int N, int L, int total,
                                                                     int* map, int* inv) {
  for (int p = blockIdx.x * kThreads + threadIdx.x; p < total; p += gridDim.x * kThreads) {
    const int g = vz_token(cu, n_seqs, N, p / L, p % L);
    map[p] = g;
    if (inv) inv[g] = p;
  }
}

}  // namespace

cudaError_t launch_zigzag_varlen_map(const int* cu, int n_seqs, int N, int total, int* map, int* inv,
                                     cudaStream_t st) {
  if (N < 1 || total < 1 || total % N) return cudaErrorInvalidValue;
  zigzag_varlen_map_kernel<<<grid_for(total, kThreads), kThreads, 0, st>>>(cu, n_seqs, N, total / N, total, map,
                                                                           inv);
  return cudaGetLastError();
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

constexpr int kPermuteUnroll = 4;

cudaError_t launch_permute(const PermuteArgs& a_in, cudaStream_t st) {
  PermuteArgs a = a_in;
  const long long row_bytes = a.inner * a.esize;
  const bool vec16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(a.src) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.dst) % 16 == 0) && (a.src_seq_stride * a.esize) % 16 == 0 &&
                     (a.dst_seq_stride * a.esize) % 16 == 0 && (a.src_outer_stride[0] * a.esize) % 16 == 0 &&
                     (a.src_outer_stride[1] * a.esize) % 16 == 0 && (a.src_outer_stride[2] * a.esize) % 16 == 0 &&
                     (a.dst_outer_stride[0] * a.esize) % 16 == 0 && (a.dst_outer_stride[1] * a.esize) % 16 == 0 &&
                     (a.dst_outer_stride[2] * a.esize) % 16 == 0;
  const long long vpr_total = vec16 ? row_bytes / 16 : a.inner;
  if (vpr_total > (1LL << 30)) return cudaErrorInvalidValue;
  a.vpr_total = (int)vpr_total;
  const int vpr = (int)(vpr_total < kThreads ? vpr_total : kThreads);  // threads per row
  const int rows_per_block = kThreads / vpr;
  // about 16 blocks per SM in total, split between the outer
  // index (y) and the positions (x)
  const long long gy = a.n_outer < 65535 ? a.n_outer : 65535;
  long long gx = ((long long)num_sms() * 16 + gy - 1) / gy;
  const long long need_x = (a.s + rows_per_block - 1) / rows_per_block;
  if (gx > need_x) gx = need_x;
  if (gx < 1) gx = 1;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  if (vec16)
    permute_kernel<uint4, kPermuteUnroll><<<grid, kThreads, 0, st>>>(a, vpr, rows_per_block);
  else if (a.esize == 4)
    permute_kernel<uint32_t, kPermuteUnroll><<<grid, kThreads, 0, st>>>(a, vpr, rows_per_block);
  else
    permute_kernel<uint16_t, kPermuteUnroll><<<grid, kThreads, 0, st>>>(a, vpr, rows_per_block);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t st) {
  const long long total = a.rows * (a.d / 4);
  // two rows in flight per thread: measured faster than four on the benchmark
  // shape (occupancy beats per-thread depth)
  if (a.vec == 16) {
    lse_merge_kernel<false, 16, 2><<<grid_for(a.rows * (a.d / 16), kThreads), kThreads, 0, st>>>(a);
  } else if (a.vec == 8) {
    const long long items = a.rows * (a.d / 8);
    if (a.blk_f32)
      lse_merge_kernel<true, 8, 2><<<grid_for(items, kThreads), kThreads, 0, st>>>(a);
    else
      lse_merge_kernel<false, 8, 2><<<grid_for(items, kThreads), kThreads, 0, st>>>(a);
  } else if (a.blk_f32) {
    lse_merge_kernel<true, 4, 2><<<grid_for(total, kThreads), kThreads, 0, st>>>(a);
  } else {
    lse_merge_kernel<false, 4, 2><<<grid_for(total, kThreads), kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const View4& dout, const View4& out, const LseView& lse, float* nD, float* nlse2, int N,
                           int stat_L, const DevCtl& ctl, const int* out_row, cudaStream_t st) {
  const int rows_per_turn = kPreUnroll * (kThreads / (dout.d / 8));
  if (stat_L % rows_per_turn != 0) return cudaErrorInvalidValue;  // a turn must not straddle a shard
  const long long turns = (long long)dout.b * dout.h * N * stat_L / rows_per_turn;
  static int per_sm[64] = {0};  // resident blocks per SM, per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!per_sm[dev]) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_pre_kernel, kThreads, 0) != cudaSuccess || n < 1) n = 1;
    per_sm[dev] = n;
  }
  long long blocks = (long long)num_sms() * per_sm[dev];  // one full wave
  if (blocks > turns) blocks = turns;
  if (blocks < 1) blocks = 1;
  bwd_pre_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(dout, out, lse, nD, nlse2, N, stat_L, ctl, out_row);
  return cudaGetLastError();
}


}  // namespace ra
