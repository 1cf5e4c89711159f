// Pieces shared by the backward kernels (ra_bwd.cu: the one-CTA dK / dV and
// dQ kernels; ra_dkdv_pair.cu: the CTA-pair dK / dV kernel).
//
// In the backward the per-element work needs no row reduction (lse and D are
// known), so each row is split between two threads: warpgroup 1 takes columns
// [0, 64) and warpgroup 2 columns [64, 128) of every tile row.  A thread writes
// its bf16 results over the first 32 of its own 64 fp32 columns, so the packed
// operand of a tile sits at TMEM columns [0, 32) and [64, 96) of the region,
// and the 16-column K step kk of a TMEM A operand starts at column pcol(kk).
#pragma once

#include "ra_tiles.cuh"

namespace ra {
namespace bwd {

constexpr int kBox = 128 * 128;  // bytes of one swizzled box: 128 rows of 64 bf16
// first TMEM column of K step kk of a packed operand: 8 kk (kk < 4) or 64 + 8 (kk - 4)
static __device__ __forceinline__ uint32_t pcol(int kk) { return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4); }

// 64 fp32 TMEM columns of this thread's lane into v (one wait).
static __device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 0));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
}

// The warp's 32 output row segments (lane l: N32 * 32 columns of row l, from
// TMEM, times mul, as bf16) leave through a shared-memory slot of 32 * N32 * 64
// bytes: each lane writes its segment there (16-byte pieces, the piece index
// XOR the row's low bits, so the lanes spread over the banks), then the warp
// stores whole segments with consecutive lanes on consecutive pieces.  Rows
// [0, nvalid) are written: row l goes to row row0 + l of base (pitch `stride`),
// or, with a row map, to row rmap[row0 + l] (a varlen call computed in
// original order that writes its results in the caller's layout order).
template <int N32>
static __device__ __forceinline__ void store_rows_bf16(uint32_t taddr, float mul, uint8_t* slot, __nv_bfloat16* base,
                                                       long long stride, long long row0, int nvalid,
                                                       const int* rmap) {
  constexpr int kPieces = 4 * N32;                      // 16-byte pieces per segment
  constexpr int kSwz = kPieces < 8 ? kPieces - 1 : 7;  // XOR mask on the piece index
  const int lane = threadIdx.x & 31;
  uint8_t* mine = slot + lane * kPieces * 16;
#pragma unroll
  for (int c = 0; c < N32; ++c) {
    uint32_t o[32];
    tmem_ld32(taddr + c * 32, o);
    tmem_ld_wait(o);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * mul, __uint_as_float(o[8 * u + 1]) * mul);
      w.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * mul, __uint_as_float(o[8 * u + 3]) * mul);
      w.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * mul, __uint_as_float(o[8 * u + 5]) * mul);
      w.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * mul, __uint_as_float(o[8 * u + 7]) * mul);
      *reinterpret_cast<uint4*>(mine + (((c * 4 + u) ^ (lane & kSwz)) << 4)) = w;
    }
  }
  __syncwarp();
  constexpr int kRowsPer = 32 / kPieces;  // segments per warp-wide store
  const int pc = lane % kPieces;
#pragma unroll 1
  for (int r0 = 0; r0 < 32; r0 += kRowsPer) {
    const int row = r0 + lane / kPieces;
    const uint4 v = *reinterpret_cast<const uint4*>(slot + row * kPieces * 16 + ((pc ^ (row & kSwz)) << 4));
    if (row < nvalid) {
      const long long dr = rmap ? (long long)__ldg(rmap + row0 + row) : row0 + row;
      *reinterpret_cast<uint4*>(base + dr * stride + pc * 8) = v;
    }
  }
}

// The 128 statistics rows of a query tile starting at row e0 lie inside the
// statistics arrays and start 512-byte aligned (the bulk copies need 16).
template <class P>
static __device__ __forceinline__ bool stat_rows_ok(const P& p, long long e0) {
  return e0 >= 0 && (e0 & 127) == 0 && e0 + 128 <= (long long)p.B * p.H * p.stat_N * p.stat_L;
}

}  // namespace bwd
}  // namespace ra
