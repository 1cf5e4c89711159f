/*
 * ringattn.h: C ABI of the GB300 (sm_103a) blockwise ring-attention library.
 *
 * What the library computes: exact softmax attention of every local Q shard
 * against every K/V shard of a sequence split into N shards, each block giving
 * its output and its log-sum-exp, with the partial results merged across the
 * ring steps by the online-softmax rule.  On one GPU the "ring" is a loop over
 * (Q shard, KV shard) pairs in HBM.
 *
 * Pages that define the operations (cited by title and section):
 *   [README]  "Ring Flash Attention" README, github.com/zhuzilin/ring-flash-attention:
 *             the API list (ring / zigzag / stripe, varlen with one cu_seqlens),
 *             "The main idea is to use the softmax_lse output", "Limits" (fp32
 *             accumulation across blocks).
 *   [GUIJIA]  guijiagi.com "Ring Attention：突破百万 Token 上下文的分布式注意力":
 *             "详细流程" (ring order), "在线 Softmax：关键技巧" (merge rule),
 *             "Striped Ring Attention", "Zigzag Ring Attention",
 *             "2. 显存预分配" (caller-preallocated buffers).
 *   [AINEWS]  ainews.cool ring-flash-attention article, "技术深度解析".
 *   [STRIPED] briefgpt.xyz abstract of "Striped Attention" (causal imbalance).
 *   [SP]      sourcepulse.org project summary of ring-flash-attention ("llama3"
 *             context parallelism).
 *
 * Conventions shared by every call
 *   - Tensors are described by ra_tensor: a DEVICE pointer, a dtype, and up to
 *     four dimensions with ELEMENT strides.  The last dimension must be
 *     contiguous (stride 1) unless a call says otherwise.
 *   - Sequence tensors are in LAYOUT ORDER: the N shards concatenated along the
 *     sequence axis, i.e. what the N ranks of the ring would hold.  Use
 *     ring_attn_permute / ring_attn_unpermute to move between original token
 *     order and layout order.
 *   - Ownership: the caller allocates every tensor and the workspace; the
 *     library never allocates or frees device memory and keeps no pointer
 *     after a call returns ([GUIJIA] "2. 显存预分配").
 *   - Streams: every call is asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).
 *   - Errors: argument errors are returned synchronously before any launch;
 *     a failed launch returns RA_ERR_CUDA.  Device-side failures (a bounded
 *     wait that ran out) are reported by ring_attn_check_device_error.  On
 *     any error the outputs are unspecified.
 *   - Layout constraints for attention calls: head_dim d in {64, 128}; q, k,
 *     v (and out, dout, dq, dk, dv) have the same shape, except that k and v
 *     (and dk, dv) may have hk heads where hk divides q's h (grouped-query
 *     attention: query head i attends with key / value head i / (h / hk),
 *     integer division; the pages only use hk = h, and every call below that
 *     says "(b, h, s, d)" for k or v accepts hk in place of h); every stride
 *     but the last is a multiple of 8 elements and every base pointer is
 *     16-byte aligned (TMA tiles), else RA_ERR_ALIGNMENT.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shard layouts ([README] API list; [GUIJIA] "Striped Ring Attention",
 * "Zigzag Ring Attention"; [AINEWS] contiguous blocks).  With L = s / N:
 *   CONTIGUOUS: shard r holds original tokens [r*L, (r+1)*L).
 *   ZIGZAG:     2N chunks of c = s / (2N); shard r holds chunk r then chunk 2N-1-r.
 *   STRIPE:     shard r holds tokens t with t mod N == r, in increasing order. */
typedef enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_ZIGZAG = 1, RA_LAYOUT_STRIPE = 2 } ra_layout;

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1, /* bad pointer, shape, dtype, layout, scale or size */
  RA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head_dim 96) */
  RA_ERR_ALIGNMENT = 3,   /* stride or base pointer unusable for TMA tiles */
  RA_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than ring_attn_workspace_size */
  RA_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  RA_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out (see check_device_error) */
  RA_ERR_DEVICE = 7,      /* other device-side error (e.g. misaligned shared memory) */
  RA_ERR_SCRATCH_LIMIT = 8 /* the problem needs more than the library's static scratch holds */
} ra_status;

typedef enum { RA_BF16 = 0, RA_FP32 = 1 } ra_dtype;

typedef struct {
  void* data;        /* device pointer */
  int32_t dtype;     /* ra_dtype */
  int32_t ndim;      /* 1..4 */
  int64_t shape[4];
  int64_t stride[4]; /* in elements */
} ra_tensor;

typedef enum { RA_OP_FWD = 0, RA_OP_BWD = 1 } ra_op;

/* ring_attn_fwd: the ring forward with the LSE merge fused in fp32.
 *   q, k, v: (b, h, s, d) bf16, layout order.  out: (b, h, s, d) bf16, layout
 *   order.  lse: (b, h, s) fp32, natural log, layout order.
 *   For each Q shard r the kernel visits KV shards (r - t) mod N for ring steps
 *   t = 0..N-1 ([GUIJIA] "详细流程"), computes each block with tcgen05 MMAs,
 *   and folds it into a running fp32 (max, sum, output) state, which is the
 *   merge of [GUIJIA] "在线 Softmax：关键技巧" kept in fp32 across blocks
 *   ([README] "Limits").  causal: key allowed iff its original token index
 *   <= the query's.  softmax_scale: finite and > 0 (usually 1/sqrt(d)).
 *   workspace: may be NULL (the forward needs none). */
ra_status ring_attn_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v, int32_t layout,
                        int32_t n_shards, int32_t causal, float softmax_scale, ra_tensor* out, ra_tensor* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ring_attn_fwd_step: one ring step on its own, every block emitting its own
 * result, as one rank of the ring does per step ([README] "use the
 * softmax_lse output").  For every Q shard r, attends to KV shard (r - step)
 * mod N only, and writes the normalised block output out_blk (b, h, s, d),
 * bf16 or fp32, and lse_blk (b, h, s) fp32.  A row with no allowed key gets
 * out_blk = 0 and lse_blk = -inf.  Combine the N steps with lse_merge. */
ra_status ring_attn_fwd_step(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v, int32_t layout,
                             int32_t n_shards, int32_t causal, float softmax_scale, int32_t step,
                             ra_tensor* out_blk, ra_tensor* lse_blk, void* stream);

/* lse_merge: out_acc, lse_acc <- merge(out_acc, lse_acc, out_blk, lse_blk),
 * row by row, in place ([GUIJIA] "在线 Softmax：关键技巧", with each side's
 * (max, sum) taken as (lse, 1)):
 *   lse_new = max(a, b) + log1p(exp(-|a - b|)),  w = exp(lse_blk - lse_new),
 *   out_acc += w * (out_blk - out_acc).
 * lse_blk = -inf leaves the row unchanged; lse_acc = -inf takes the block;
 * both -inf give out_acc = 0, lse_acc = -inf.
 *   out_acc: (..., rows, d) fp32; lse_acc: (..., rows) fp32; out_blk: same
 *   shape as out_acc, bf16 or fp32; lse_blk: same shape as lse_acc.  2-D to
 *   4-D; d contiguous, d a multiple of 4, rows 16-byte aligned. */
ra_status lse_merge(ra_tensor* out_acc, ra_tensor* lse_acc, const ra_tensor* out_blk, const ra_tensor* lse_blk,
                    void* stream);

/* ring_attn_bwd: gradients of exact attention given the forward's out and lse.
 *   dout, q, k, v, out: (b, h, s, d) bf16 layout order; lse: (b, h, s) fp32.
 *   dq, dk, dv: (b, h, s, d) bf16 outputs, layout order.
 *   With P = exp(S - lse) recomputed from the saved lse:
 *   D = rowsum(dO * O), dV = P^T dO, dS = P * (dO V^T - D), dQ = scale dS K,
 *   dK = scale dS^T Q.  One kernel per key tile keeps dK and dV in tensor
 *   memory while it meets the query tiles in ring order; one kernel per query
 *   tile recomputes S and dP and keeps dQ in tensor memory.  No atomics: the
 *   results are deterministic.  With grouped key / value heads (hk < h), dK
 *   and dV of a key / value head sum over its h / hk query heads, all met by
 *   the same key-tile kernel in head order.
 *   workspace: at least ring_attn_workspace_size(RA_OP_BWD, b, h, s, d, n_shards)
 *   bytes (h: q's head count), 256-byte aligned, owned by the caller, need not
 *   be initialised. */
ra_status ring_attn_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                        const ra_tensor* out, const ra_tensor* lse, int32_t layout, int32_t n_shards,
                        int32_t causal, float softmax_scale, ra_tensor* dq, ra_tensor* dk, ra_tensor* dv,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ring_attn_bwd_static_scratch: ring_attn_bwd without a caller workspace.
 * The pages have no counterpart: it is a library convenience for callers that
 * cannot hand over device memory, e.g. an integration point whose signature
 * has no workspace argument, or a process whose device memory is already
 * fully reserved by another allocator, so that allocating at that point would
 * fail.  It allocates nothing: the per-row statistics (-D and -lse * log2(e))
 * live in one array of RA_STATIC_SCRATCH_BYTES bytes that the library holds
 * in device memory on every device that loads it, until the process exits (a
 * file-scope __device__ array).
 *   Arguments, layouts and results are those of ring_attn_bwd.
 *   Limit: ring_attn_workspace_size(RA_OP_BWD, b, h, s, d, n_shards) must not
 *   exceed RA_STATIC_SCRATCH_BYTES (16 MiB: up to 2,097,152 query rows after
 *   padding each shard to a multiple of 128, e.g. b = 1, h = 32, s = 65536),
 *   else RA_ERR_SCRATCH_LIMIT is returned before any launch.
 *   Set-up: the first call on each device looks up the array's device address
 *   with that device current (cudaGetSymbolAddress, which loads the library's
 *   device code if it is not loaded yet); make that first call before any
 *   stream capture begins.  Later calls on the device reuse the address, so
 *   do not call it again on a device after cudaDeviceReset in the same
 *   process: the cached address would be stale.
 *   Errors: every argument error of ring_attn_bwd is reported first, with the
 *   same status; only a valid problem that is too large gets
 *   RA_ERR_SCRATCH_LIMIT.
 *   The array keeps the last call's contents; nothing in it needs to start at
 *   zero, because every call writes all of it that it reads before reading it.
 *   Races: every call on a device shares the array.  Calls ordered on one
 *   stream are safe; two calls that can run on the GPU at the same time
 *   (different streams without ordering between them, or other host threads)
 *   race on it and give wrong gradients. */
#define RA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
ra_status ring_attn_bwd_static_scratch(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k,
                                       const ra_tensor* v, const ra_tensor* out, const ra_tensor* lse,
                                       int32_t layout, int32_t n_shards, int32_t causal, float softmax_scale,
                                       ra_tensor* dq, ra_tensor* dk, ra_tensor* dv, void* stream);

/* Varlen (packed) forms ([README] API list, "the varlen versions only support
 * passing one cu_seqlens").  q, k, v, out: 3-D (total, h, d) or (h, total, d)
 * bf16, given by strides (dimension 0 of shape is the one whose size is
 * `total` when shape[0] == total, else dimension 1 must be total); lse:
 * (h, total) fp32.  cu_seqlens_dev / cu_seqlens_host: the same int32 array of
 * n_seqs + 1 prefix sums (0 = cu[0] <= cu[1] <= ... <= cu[n_seqs] = total);
 * the host copy is validated before launch, the device copy is read by the
 * kernels.  Attention is confined to each sequence.  Tensors are in layout
 * order (ring_attn_varlen_permute):
 *   RA_LAYOUT_CONTIGUOUS: shards are contiguous slices of the packed buffer
 *     (total / N tokens each; sequences may straddle shards);
 *   RA_LAYOUT_ZIGZAG: the zigzag split of every sequence ([README] API list,
 *     zigzag_ring_flash_attn_varlen_func): sequence k, whose length must be a
 *     multiple of 2N, is cut into 2N chunks and shard r holds chunk r then
 *     chunk 2N-1-r of each sequence in turn, so sequence k occupies positions
 *     [cu[k]/N, cu[k+1]/N) of every shard.
 * Other layouts return RA_ERR_UNSUPPORTED; a zigzag length that is not a
 * multiple of 2N returns RA_ERR_INVALID_ARG.
 * Workspace.  The forward needs none and the backward needs
 * ring_attn_varlen_workspace_size(RA_OP_BWD, ..., RA_LAYOUT_CONTIGUOUS, N)
 * bytes (its per-row statistics).  For RA_LAYOUT_ZIGZAG a workspace of at
 * least ring_attn_varlen_workspace_size(op, total, h, d, RA_LAYOUT_ZIGZAG, N)
 * bytes (256-byte aligned) makes the call run in original token order: it
 * copies its tensor-core operands (q, k, v; in the backward dO, q, k, v) out
 * of the zigzag order into the workspace and runs the contiguous-layout
 * kernels there, which read out and lse and write every result row straight
 * through the token map, in the caller's zigzag order.  On one GPU the
 * zigzag split is only a storage order, and with short sequences its 2N chunks
 * put several sequences into every 128-row tile, so most of the tiles' work
 * would be masked.  With a smaller (or no) workspace the zigzag kernels run on
 * the zigzag order directly.  Both give the same results up to fp32 summation
 * order. */
ra_status ring_attn_varlen_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                               const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                               int32_t max_seqlen, int32_t layout, int32_t n_shards, int32_t causal,
                               float softmax_scale, ra_tensor* out, ra_tensor* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

ra_status ring_attn_varlen_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                               const ra_tensor* out, const ra_tensor* lse, const int32_t* cu_seqlens_dev,
                               const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t max_seqlen, int32_t layout,
                               int32_t n_shards, int32_t causal, float softmax_scale, ra_tensor* dq, ra_tensor* dk,
                               ra_tensor* dv, void* workspace, size_t workspace_bytes, void* stream);

/* llama3 context-parallel form, one rank ([SP]: the "llama3" context
 * parallelism variant, llama3_flash_attn_varlen_func): rank r of N holds the contiguous
 * slice [r*L, (r+1)*L) of the packed buffer (L = total / N) and its queries
 * attend to the all-gathered keys and values, with one cu_seqlens over the
 * whole packed buffer.  q, out, dout, dq: (L, h, d) or (h, L, d), the rank's
 * rows; k, v, dk, dv: (total, h, d) or (h, total, d); lse: (h, L) fp32.
 * The forward gives the rank's out and lse (the rows of full varlen
 * attention).  The backward gives dq of the rank's rows and the rank's
 * contribution to dk and dv of every key: the gradient of sum(dO * out) over
 * the rank's rows only (summing the N ranks' contributions gives the full
 * gradient).  workspace: ring_attn_workspace_size(RA_OP_BWD, 1, h, L, d, 1)
 * bytes.  Errors as for the varlen calls; rank outside [0, N) or total not a
 * multiple of N is RA_ERR_INVALID_ARG. */
ra_status ring_attn_llama3_varlen_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                                      const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                                      int32_t max_seqlen, int32_t rank, int32_t n_shards, int32_t causal,
                                      float softmax_scale, ra_tensor* out, ra_tensor* lse, void* stream);
ra_status ring_attn_llama3_varlen_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k,
                                      const ra_tensor* v, const ra_tensor* out, const ra_tensor* lse,
                                      const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                                      int32_t max_seqlen, int32_t rank, int32_t n_shards, int32_t causal,
                                      float softmax_scale, ra_tensor* dq, ra_tensor* dk, ra_tensor* dv,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ring_attn_permute: original token order -> layout order along seq_dim:
 *   y[..., p, ...] = x[..., g(p), ...], g(p) = original token at layout position p.
 * ring_attn_unpermute: the inverse, x[..., g(p), ...] = y[..., p, ...].
 *   x, y: same shape, 1-D to 4-D, bf16 or fp32 (same dtype); the dimensions
 *   after seq_dim must be packed (row-major contiguous).  A bit copy.
 *   x and y must not overlap in memory (no in-place permutation: rows are
 *   gathered by many blocks at once); overlapping byte ranges get
 *   RA_ERR_INVALID_ARG before any launch. */
ra_status ring_attn_permute(const ra_tensor* x, ra_tensor* y, int32_t layout, int32_t n_shards, int32_t seq_dim,
                            void* stream);
ra_status ring_attn_unpermute(const ra_tensor* y, ra_tensor* x, int32_t layout, int32_t n_shards, int32_t seq_dim,
                              void* stream);

/* Varlen forms of the two above for one packed buffer of total tokens
 * (cu_seqlens as in the varlen calls; x.shape[seq_dim] == total):
 * RA_LAYOUT_CONTIGUOUS is the identity (a copy), RA_LAYOUT_ZIGZAG the
 * per-sequence zigzag split described above the varlen calls. */
ra_status ring_attn_varlen_permute(const ra_tensor* x, ra_tensor* y, const int32_t* cu_seqlens_dev,
                                   const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t layout, int32_t n_shards,
                                   int32_t seq_dim, void* stream);
ra_status ring_attn_varlen_unpermute(const ra_tensor* y, ra_tensor* x, const int32_t* cu_seqlens_dev,
                                     const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t layout, int32_t n_shards,
                                     int32_t seq_dim, void* stream);

/* Workspace bytes of a varlen call (see the varlen calls above): RA_OP_FWD: 0
 * for RA_LAYOUT_CONTIGUOUS, and for RA_LAYOUT_ZIGZAG the original-order copies
 * of q, k, v (3 * total * h * d bf16); RA_OP_BWD: the per-row statistics, plus
 * for RA_LAYOUT_ZIGZAG the copies of dO, q, k, v (4 tensors; out and lse are
 * read where they are); zigzag also takes 2 * total int32 for the token map
 * between layout and original order and its inverse.
 * Each part 256-byte aligned.  0 on bad sizes (head_dim other than 64 or 128,
 * total not a multiple of n_shards, another layout). */
size_t ring_attn_varlen_workspace_size(int32_t op, int64_t total, int64_t h, int64_t d, int32_t layout,
                                       int32_t n_shards);

/* Workspace bytes needed by `op` (ra_op) for (b, h, s, d) split into n_shards
 * shards; 0 for RA_OP_FWD.  RA_OP_BWD: -D = -rowsum(dO*O) and -lse*log2(e) per
 * query row, each laid out per shard with the shard's rows padded to a
 * multiple of 128 (b*h*n_shards*ceil(s/n_shards/128)*128 floats each), each
 * part 256-byte aligned.  Varlen calls use b = 1, s = total.  0 on bad sizes. */
size_t ring_attn_workspace_size(int32_t op, int64_t b, int64_t h, int64_t s, int64_t d, int32_t n_shards);

/* Synchronises `stream`, then reads and clears this device's error word.
 * Returns RA_OK, RA_ERR_TIMEOUT (a bounded wait ran out: the kernel gave up
 * and returned) or RA_ERR_DEVICE; RA_ERR_CUDA if the synchronisation failed.
 * *info (optional) gets the failing wait site and block. */
ra_status ring_attn_check_device_error(void* stream, int32_t* info);

/* Knobs (process-wide).  RA_KNOB_WAIT_LIMIT_NS: the bounded-wait limit in ns
 * (default 4e9).  RA_KNOB_DEBUG_FLAGS: bit 0 makes the forward's TMA producer
 * skip the Q tile load, bit 1 the one-CTA dK / dV kernel skip its K / V load,
 * bit 2 the dQ kernel skip its Q / dO load, so that every consumer's bounded
 * wait runs out: tests of the timeout path that hang nothing.  RA_KNOB_DKDV_PAIR: 1 runs the
 * backward's dK / dV pass at head_dim 128 on CTA pairs (two SMs share each
 * M = 256 tensor-core MMA, halving each SM's operand reads from shared memory);
 * 0 (default) runs the one-CTA kernel, which head_dim 64 always uses.  Both
 * give the same results up to fp32 summation order. */
typedef enum { RA_KNOB_WAIT_LIMIT_NS = 0, RA_KNOB_DEBUG_FLAGS = 1, RA_KNOB_DKDV_PAIR = 2 } ra_knob;
ra_status ring_attn_set_knob(int32_t knob, int64_t value);

/* Per-kernel timing (process-wide, off by default; one device per process).
 * While enabled, the library brackets every kernel it launches with CUDA
 * events recorded on the launch stream.  ring_attn_timing_read synchronises
 * the recorded events of `kernel` (ra_kernel), returns the summed device
 * milliseconds and the number of launches since the last read, and resets
 * them.  Disabling drops anything not yet read. */
typedef enum {
  RA_KERNEL_FWD = 0,       /* ring forward (fused merge, or one ring step) */
  RA_KERNEL_BWD = 1,       /* ring backward: the dK / dV kernel */
  RA_KERNEL_BWD_PRE = 2,   /* D = rowsum(dO * O) and lse * log2(e) per query row */
  RA_KERNEL_BWD_DQ = 3,    /* ring backward: the dQ kernel */
  RA_KERNEL_PERMUTE = 4,   /* permute / unpermute */
  RA_KERNEL_LSE_MERGE = 5,
  RA_KERNEL_COUNT = 6
} ra_kernel;
ra_status ring_attn_timing_enable(int32_t on);
ra_status ring_attn_timing_read(int32_t kernel, double* total_ms, int64_t* launches);

const char* ra_status_string(int32_t status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t ring_attn_version(void);

/* 1 in the debug variant of the library (libringattn_dbg.so, compiled with
 * RA_DEBUG_BOUNDS), else 0.  In that variant every kernel checks each tiled
 * copy's coordinates, each statistics copy and each global row store against
 * the tensors' extents before making it; a violation skips the access and
 * records RA_ERR_DEVICE, with the site in the low byte of check_device_error's
 * info (0x80 | site), instead of touching memory outside a tensor. */
int32_t ring_attn_debug_bounds(void);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
