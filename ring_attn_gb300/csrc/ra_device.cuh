// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 MMA / TMEM access, shared-memory operand
// descriptors, and the shard-layout index maps.
//
// Every wait in this library is bounded: past a time limit (globaltimer) the
// waiting warp records RA_ERR_TIMEOUT in the device error word, raises the
// CTA's abort flag in shared memory and returns false, so that every role
// leaves its loop and the CTA frees its tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ra {

// ------------------------------------------------------------------ errors
enum : int { DEV_OK = 0, DEV_TIMEOUT = 6, DEV_BAD_SMEM = 7, DEV_BOUNDS = 7 };

struct DevCtl {
  int* err_word;          // first error code wins (atomicCAS from 0)
  int* err_info;          // site | (block << 8) of the first failure
  unsigned long long wait_limit_ns;
  int debug_flags;        // bounded-wait tests: the forward (bit 0), dK/dV (bit 1) or dQ (bit 2) kernel skips its entry load
};

enum : int { DBG_SKIP_Q_LOAD = 1, DBG_SKIP_KV_LOAD = 2, DBG_SKIP_QDO_LOAD = 4 };

__device__ __forceinline__ void record_error(const DevCtl& c, int code, int site) {
  if (atomicCAS(c.err_word, 0, code) == 0) {
    atomicExch(c.err_info, site | (int)((blockIdx.x + blockIdx.y * gridDim.x) << 8));
  }
}

// ------------------------------------------------------------------ debug bounds checks
// Built with RA_DEBUG_BOUNDS (the library's debug variant), every tiled copy,
// statistics copy and global row store first checks its coordinates against
// the tensor's extents; a failed check records DEV_BOUNDS (RA_ERR_DEVICE)
// with the site in the error word and skips the access (the kernel's bounded
// waits then end the CTA).  Without the flag the checks compile away.
#ifdef RA_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

__device__ __forceinline__ bool in_bounds(bool ok, const DevCtl& c, int site) {
  if (kDebugBounds && !ok) {
    record_error(c, DEV_BOUNDS, 0x80 | site);
    return false;
  }
  return true;
}

// Extents of a (b, h, rows, d) tensor as its TMA map sees it.
struct TmaExtent {
  int d, rows, h, b;
};

// A 64-column tiled copy starting at (c0, c1, c2, c3): 16-byte aligned column
// start inside the row, a start row inside the tensor or at most one 128-row
// tile past its end (that copy reads the zero fill), head and batch inside.
__device__ __forceinline__ bool tma_coords_ok(const TmaExtent& e, int c0, int c1, int c2, int c3) {
  return c0 >= 0 && (c0 & 63) == 0 && c0 + 64 <= e.d && c1 >= 0 && c1 < e.rows + 128 && c2 >= 0 && c2 < e.h &&
         c3 >= 0 && c3 < e.b;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Raises the phase's expected transaction bytes without arriving (the phase
// still needs its arrivals).
__device__ __forceinline__ void mbar_add_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test with a suspend-time hint: a thread whose phase is not complete
// may stay suspended up to hint_ns nanoseconds (it resumes as soon as the
// phase completes) instead of the system's default limit.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
template <uint32_t H>
__device__ __forceinline__ bool mbar_try_wait_h(uint32_t bar, uint32_t parity) {
  return H ? mbar_try_wait_hint(bar, parity, H) : mbar_try_wait(bar, parity);
}

// One thread waits.  Returns false when the CTA aborts (own timeout or another role's).
// H: suspend-time hint of each test in nanoseconds (0: the system's default).
template <uint32_t H = 0>
static __device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int* abort_flag, const DevCtl& c,
                                      int site) {
  if (mbar_try_wait_h<H>(bar, parity)) return true;
  unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_h<H>(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > c.wait_limit_ns) {
        *abort_flag = 1;
        record_error(c, DEV_TIMEOUT, site);
        return false;
      }
    }
  }
}

// A whole converged warp waits; the result is the same on every lane.
template <uint32_t H = 0>
static __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, const DevCtl& c,
                                       int site) {
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    bool done = mbar_try_wait_h<H>(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 15u) == 15u) {
      int stop = 0;
      if (lane_id() == 0) {
        if (*abort_flag) {
          stop = 1;
        } else {
          unsigned long long now = globaltimer();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > c.wait_limit_ns) {
            *abort_flag = 1;
            record_error(c, DEV_TIMEOUT, site);
            stop = 1;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

// Per-warpgroup register budgets (all four warps of a warpgroup execute these).
// The sum over warpgroups must not exceed the block's launch allocation, or
// setmaxnreg.inc would wait forever: launchers check the kernel's register
// count before using a split.
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier among a subset of warps (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-D tiled load (coordinates innermost first) into shared memory; completion
// is signalled as transaction bytes on the mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (MMA reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, fp32 accumulate.  A (M x K,
// K-major) sits in tensor memory: row m in lane m, two consecutive bf16 K
// elements per 32-bit column (the lower K index in the low half).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on the mbarrier when every previously issued MMA of this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// ------------------------------------------------------------------ CTA pairs (cta_group::2)
// A cluster of two CTAs on two SMs runs one M = 256 MMA: each CTA holds 128
// rows of A and half of B's N columns at the same shared-memory offsets, and
// each CTA's tensor memory holds its 128 rows of D.  One thread of the even
// CTA issues the MMAs; every tcgen05 instruction of such a kernel uses
// cta_group::2 (the assembler refuses a mix).  Allocation and deallocation
// are collective: one warp of each CTA of the pair executes them.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier anywhere in the cluster (addr from mapa_shared).  The
// pair kernels hand over tensor-memory contents and copy completions only,
// which the tcgen05 fences and the barriers' own transaction accounting
// order, so CTA-scope release suffices: cluster scope would put a memory
// barrier into every arrival (and, on the waiting side, every poll).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void st_shared_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Every thread of both CTAs: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at offset `bar` of every CTA in cta_mask when
// the issuing thread's earlier MMAs have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// Tiled load into this CTA's shared memory whose completion (transaction
// bytes) is signalled on an mbarrier of either CTA of the pair (bar from
// mapa_shared).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1, int c2,
                                                 int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Instruction descriptor for kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn: 0 = K-major, 1 = MN-major operand in shared memory.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((uint32_t)a_mn << 15)        // A major
         | ((uint32_t)b_mn << 16)        // B major
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA's
// SWIZZLE_128B writes: 8 rows of 128 B form a 1024-byte atom, and the 16-byte
// chunk c of row r sits at chunk c ^ (r & 7)).
//   K-major operand:  rows = M (or N) at 128 B pitch, SBO = 1024 (next 8 rows);
//                     the start address advances 32 B per 16-element K step.
//   MN-major operand: rows = K at 128 B pitch holding 64 consecutive MN elements;
//                     SBO = 1024 (next 8 K rows), LBO = offset of the next 64-wide
//                     MN block; the start advances 2048 B per 16-row K step.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// The descriptor of sdesc_sw128(saddr + bytes, ...) from that of saddr: the
// start address field holds saddr / 16 in its low 14 bits, and every shared
// memory address (< 256 KB) keeps the sum inside them, so the MMA loops step
// a descriptor with one add instead of rebuilding it.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }
// The same descriptor as two 32-bit words, for loops short of registers: the
// high word is a constant of the stride (SBO), the low word holds the address
// and LBO and steps by bytes / 16.
__device__ __forceinline__ uint32_t sdesc_sw128_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_sw128_hi(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint64_t sdesc_words(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }

// Byte offset of 16-byte chunk `chunk` of row `row` inside a 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

#define RA_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])
#define RA_P8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), \
                 "+r"(r[i + 6]), "+r"(r[i + 7])
#define RA_I8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                 "r"(r[i + 6]), "r"(r[i + 7])

// Lane (32*quadrant + laneid) reads 32 consecutive 32-bit columns starting at taddr's column.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : RA_R8(0), RA_R8(8), RA_R8(16), RA_R8(24)
      : "r"(taddr)
      : "memory");
}
// Wait for outstanding tcgen05.ld; the registers are threaded through so that
// no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : RA_P8(0), RA_P8(8), RA_P8(16), RA_P8(24) : : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      RA_I8(0), RA_I8(8), RA_I8(16), RA_I8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Lane (32*quadrant + laneid) writes 16 consecutive 32-bit columns starting at taddr's column.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      RA_I8(0), RA_I8(8)
      : "memory");
}

#undef RA_R8
#undef RA_P8
#undef RA_I8

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// max of three floats in one instruction (sm_100 and later)
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic of sm_100.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bits [lo, hi) of a 64-bit word (lo and hi clamped to [0, 64]; none when
// lo >= hi): a row's allowed columns of a 64-column half tile, so masking a
// column is one bit test and one select.
__device__ __forceinline__ uint64_t bit_window64(int lo, int hi) {
  lo = min(max(lo, 0), 64);
  hi = min(max(hi, 0), 64);
  const uint64_t below_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
  const uint64_t below_lo = lo >= 64 ? ~0ull : ((1ull << lo) - 1ull);
  return below_hi & ~below_lo;
}

// ------------------------------------------------------------------ layouts
// Original token index of local position i in shard r (L tokens per shard).
// 32-bit: the host validates s <= 2^30, so every token index fits.
enum : int { LAYOUT_CONTIGUOUS = 0, LAYOUT_ZIGZAG = 1, LAYOUT_STRIPE = 2 };

__host__ __device__ __forceinline__ int token_of(int layout, int N, int L, int r, int i) {
  if (layout == LAYOUT_STRIPE) return i * N + r;
  if (layout == LAYOUT_ZIGZAG) {
    const int c = L >> 1;
    return i < c ? r * c + i : (2 * N - 1 - r) * c + (i - c);
  }
  return r * L + i;
}

// Largest local index j of shard s with token_of(s, j) <= g, or -1.
__host__ __device__ __forceinline__ int last_local_at_or_before(int layout, int N, int L, int s, int g) {
  if (layout == LAYOUT_STRIPE) {
    if (g < s) return -1;
    const int j = (g - s) / N;
    return j < L - 1 ? j : L - 1;
  }
  if (layout == LAYOUT_ZIGZAG) {
    const int c = L >> 1;
    const int hi0 = (2 * N - 1 - s) * c;
    if (g >= hi0) {
      const int j = c + (g - hi0);
      return j < L - 1 ? j : L - 1;
    }
    const int lo0 = s * c;
    if (g >= lo0) {
      const int j = g - lo0;
      return j < c - 1 ? j : c - 1;
    }
    return -1;
  }
  const int j = g - s * L;
  if (j < 0) return -1;
  return j < L - 1 ? j : L - 1;
}

// Segment index k with cu[k] <= t < cu[k+1] (binary search, n_seqs >= 1).
__device__ __forceinline__ int segment_of(const int* __restrict__ cu, int n_seqs, int t) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// segment_of for a target that is the same in every lane of a full warp,
// with the answer known to be >= lo: the 32 lanes probe 32 evenly spaced
// entries at a time, so each round of loads narrows the range 32-fold.
__device__ __forceinline__ int segment_of_warp(const int* __restrict__ cu, int n_seqs, int t, int lo = 0) {
  const int lane = threadIdx.x & 31;
  int hi = n_seqs - 1;
  while (lo < hi) {
    const int step = (hi - lo + 32) >> 5;  // ceil((hi - lo + 1) / 32)
    const int idx = lo + lane * step;
    const bool le = idx <= hi && __ldg(cu + idx) <= t;
    // lane 0 probes lo, where cu[lo] <= t holds already
    const unsigned m = __ballot_sync(0xffffffffu, le) | 1u;
    lo += (31 - __clz(m)) * step;
    hi = min(hi, lo + step - 1);
  }
  return lo;
}

// segment_of for targets that do not decrease with the lane index, in a full
// warp: two warp searches bound the lanes' segments, and a lane searches
// between them only when the warp spans more than one sequence.
__device__ __forceinline__ int segment_of_lanes(const int* __restrict__ cu, int n_seqs, int t) {
  const int k0 = segment_of_warp(cu, n_seqs, __shfl_sync(0xffffffffu, t, 0));
  const int t31 = __shfl_sync(0xffffffffu, t, 31);
  if (t31 < __ldg(cu + k0 + 1)) return k0;
  int lo = k0, hi = segment_of_warp(cu, n_seqs, t31, k0);
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Zigzag varlen: sequence k (tokens [cu_k, cu_k1), a multiple of 2N) is cut
// into 2N chunks of c = (cu_k1 - cu_k) / 2N tokens; every shard holds chunk r
// then chunk 2N-1-r of each sequence in turn, so sequence k occupies local
// positions [cu_k / N, cu_k1 / N) of every shard, in increasing token order.
__device__ __forceinline__ int vz_token_in(int cu_k, int cu_k1, int N, int r, int i) {
  const int c = (cu_k1 - cu_k) / (2 * N);
  const int o = i - cu_k / N;
  return cu_k + (o < c ? r * c + o : (2 * N - 1 - r) * c + (o - c));
}

__device__ __forceinline__ int vz_token(const int* __restrict__ cu, int n_seqs, int N, int r, int i) {
  const int k = segment_of(cu, n_seqs, i * N);  // cu[k] / N <= i < cu[k+1] / N
  return vz_token_in(__ldg(cu + k), __ldg(cu + k + 1), N, r, i);
}

// One past the largest local index of shard s holding a token of a zigzag
// sequence (local start base, chunk length c) whose offset in the sequence
// is <= o; base when there is none.  Integer compares only: base and c are
// computed once per sequence.
__device__ __forceinline__ int vz_prefix_end(int base, int c, int N, int s, int o) {
  if (o < s * c) return base;
  if (o < (s + 1) * c) return base + (o - s * c) + 1;
  if (o < (2 * N - 1 - s) * c) return base + c;
  if (o < (2 * N - s) * c) return base + c + (o - (2 * N - 1 - s) * c) + 1;
  return base + 2 * c;
}

}  // namespace ra

namespace ra {
// Wait that ignores the abort flag (bounded by time only): used at teardown to
// let copies and MMAs already in flight land before the CTA exits.
static __device__ __forceinline__ void drain_one(uint32_t bar, uint32_t parity, const DevCtl& c, int site) {
  unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > c.wait_limit_ns) {
      record_error(c, DEV_TIMEOUT, site);
      return;
    }
  }
}
}  // namespace ra

namespace ra {
// Bounded waits of a CTA pair: a timeout raises the abort flag of both CTAs
// (peer_abort: the other CTA's flag, from mapa_shared), so that the partner
// leaves its loops at once instead of timing out too.
static __device__ __forceinline__ bool wait_one_pair(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                     uint32_t peer_abort, const DevCtl& c, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > c.wait_limit_ns) {
        *abort_flag = 1;
        st_shared_cluster(peer_abort, 1u);
        record_error(c, DEV_TIMEOUT, site);
        return false;
      }
    }
  }
}

static __device__ __forceinline__ bool wait_warp_pair(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                      uint32_t peer_abort, const DevCtl& c, int site) {
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 15u) == 15u) {
      int stop = 0;
      if (lane_id() == 0) {
        if (*abort_flag) {
          stop = 1;
        } else {
          unsigned long long now = globaltimer();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > c.wait_limit_ns) {
            *abort_flag = 1;
            st_shared_cluster(peer_abort, 1u);
            record_error(c, DEV_TIMEOUT, site);
            stop = 1;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

static __device__ __forceinline__ void drain_one_pair(uint32_t bar, uint32_t parity, const DevCtl& c, int site) {
  unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > c.wait_limit_ns) {
      record_error(c, DEV_TIMEOUT, site);
      return;
    }
  }
}
}  // namespace ra
