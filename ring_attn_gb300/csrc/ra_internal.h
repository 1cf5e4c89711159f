// Parameters shared between the C-ABI host code and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ra_device.cuh"

namespace ra {

constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // key rows per tile

struct FwdParams {
  int B, H, N, L, S;        // batch, query heads, shards, tokens per shard, total tokens
  int Hk, G;                // key / value heads; query heads per key / value head (H = G * Hk)
  int layout, causal;
  int step;                 // -1: fused ring over all N steps; else one ring step
  int n_qtiles;             // ceil(L / 128)
  float scale_log2;         // softmax_scale * log2(e)
  void* out;                // bf16 (fused) or bf16/fp32 (step mode)
  long long o_sb, o_sh, o_ss;
  int out_f32;
  float* lse;
  long long l_sb, l_sh, l_ss;
  const int* cu;            // varlen cu_seqlens (device) or nullptr
  int n_seqs;
  int q_base;               // token row of q / out / lse row 0 (one rank's slice: r_only * L, else 0)
  int r_only;               // -1: every Q shard; else only this one (a llama3 rank)
  int q_rows;               // rows of q / out / lse: S, or L for one llama3 rank (bounds checks)
  const int* row_map;       // varlen: row of out / lse for each (original-order) row, or nullptr (the same row)
  DevCtl ctl;
};

struct BwdParams {
  int B, H, N, L, S;        // batch, query heads, shards, tokens per shard, total tokens
  int Hk, G;                // key / value heads; query heads per key / value head (H = G * Hk)
  int layout, causal;
  int n_qtiles, n_ktiles;   // tiles per shard
  int stat_L;               // per-shard rows of the statistics arrays: n_qtiles * 128
  float scale;              // softmax scale
  float scale_log2;
  const float* nlse2;       // -lse * log2(e), (b, h, shard, stat_L); padding rows hold -inf
  const float* nD;          // -rowsum(dO * O), same layout; padding rows hold 0
  void* dq;                 // bf16 outputs
  void* dk;
  void* dv;
  long long q_sb, q_sh, q_ss;   // strides of dq
  long long k_sb, k_sh, k_ss;   // strides of dk
  long long v_sb, v_sh, v_ss;   // strides of dv
  const int* cu;
  int n_seqs;
  int q_base;               // token row of q / dO / out / dq row 0 (one rank's slice: r_only * L, else 0)
  int r_only;               // -1: every Q shard; else only this one (a llama3 rank)
  int stat_N, stat_r0;      // the statistics hold shards [stat_r0, stat_r0 + stat_N)
  int q_rows;               // rows of q / dO / out / dq: S, or L for one llama3 rank (bounds checks)
  const int* row_map;       // varlen: row of dq / dk / dv for each (original-order) row, or nullptr (the same row)
  DevCtl ctl;
};

// The kernel parameters with a compile-time varlen flag: the batched kernels
// are instantiated with kVarlen = false, so every varlen branch folds away.
template <bool VL>
struct FwdParamsT : FwdParams {
  static constexpr bool kVarlen = VL;
};
template <bool VL>
struct BwdParamsT : BwdParams {
  static constexpr bool kVarlen = VL;
};

// Strided 4-D view of a tensor whose last dimension is contiguous.
struct View4 {
  void* data;
  long long sb, sh, ss;     // element strides of dims 0..2
  int b, h, s, d;
};

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t st);
size_t fwd_smem_bytes(int D);

// which = 0: the dK / dV kernel; 1: the dQ kernel.
cudaError_t launch_bwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int which, cudaStream_t st);

// The dK / dV kernel on CTA pairs (cta_group::2), head_dim 128 only.  The four
// tensor maps have 64 x 64 boxes (64 head dims by 64 rows).
cudaError_t launch_dkdv_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st);

// Per query row: -D = -rowsum(dO * O) and -lse2 = -lse * log2(e), stored per
// shard with the rows padded to stat_L (padding rows get 0 and -inf); negated so
// that the backward adds them in packed f32x2 arithmetic.
struct LseView {
  const float* data;
  long long sb, sh, ss;
};
// out_row: null, or out and lse rows by position (out and lse of position p
// are row out_row[p] of their tensors; dout is read at p)
cudaError_t launch_bwd_pre(const View4& dout, const View4& out, const LseView& lse, float* nD, float* nlse2, int N,
                           int stat_L, const DevCtl& ctl, const int* out_row, cudaStream_t st);

struct MergeArgs {
  float* out_acc;        // rows x d, row stride (elements)
  float* lse_acc;
  const void* out_blk;
  const float* lse_blk;
  int blk_f32;
  long long rows, d;
  // 3 outer dims (rows = o0 * o1 * o2) with their strides
  long long n0, n1, n2;
  long long oa_s0, oa_s1, oa_s2;
  long long la_s0, la_s1, la_s2;
  long long ob_s0, ob_s1, ob_s2;
  long long lb_s0, lb_s1, lb_s2;
  int flat;              // the three row dims collapse to one stride per tensor (the *_s2 strides)
  int vec;               // columns per thread: 16 or 8, or 4 when the row layout does not allow 8
  int qshift;            // log2(d / vec)
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t st);

struct PermuteArgs {
  const void* src;
  void* dst;
  int esize;                // bytes per element
  long long inner;          // elements per row (packed dims after seq)
  long long n_outer;        // product of dims before seq
  long long outer_shape[3]; // up to 3 outer dims (unused = 1)
  long long src_outer_stride[3], dst_outer_stride[3];
  long long src_seq_stride, dst_seq_stride;
  int s, layout, N;
  int inverse;              // 0: dst[p] = src[g(p)]; 1: dst[g(p)] = src[p]
  int vpr_total;            // vectors per row (set by the launcher)
  const int* cu;            // varlen cu_seqlens (device) or nullptr
  int n_seqs;
  const int* gmap;          // optional: gmap[p] = original token at layout position p (replaces the search)
  DevCtl ctl;               // error word (debug bounds checks)
};
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t st);

// map[p] = original token at layout position p of the zigzag varlen split of
// one packed buffer of `total` tokens (N shards, cu_seqlens with n_seqs entries + 1).
// With inv non-null also inv[map[p]] = p (the layout position of each original token).
cudaError_t launch_zigzag_varlen_map(const int* cu, int n_seqs, int N, int total, int* map, int* inv,
                                     cudaStream_t st);

int num_sms();

// One-time set-up of a kernel on the current device, cached per kernel and
// device: checks the compiled register count when the kernel's register split
// depends on it (want_regs > 0) and raises its dynamic shared-memory limit.
// Later calls on the device return the cached result without touching the driver.
template <auto Kernel>
cudaError_t configure_kernel(int want_regs, int smem_bytes) {
  static int state[64] = {0};  // per device: 0 not yet, 1 ready, else the cudaError_t + 1000
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int s = __atomic_load_n(&state[dev], __ATOMIC_ACQUIRE);
  if (s == 1) return cudaSuccess;
  if (s > 1) return static_cast<cudaError_t>(s - 1000);
  if (want_regs > 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, Kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != want_regs) {
      __atomic_store_n(&state[dev], 1000 + (int)cudaErrorInvalidConfiguration, __ATOMIC_RELEASE);
      return cudaErrorInvalidConfiguration;
    }
  }
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  __atomic_store_n(&state[dev], 1, __ATOMIC_RELEASE);
  return cudaSuccess;
}

}  // namespace ra
