// C-ABI entry points: argument validation, TMA tensor maps, workspace layout
// and kernel launches.  Every argument error is returned before any launch.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <utility>
#include <vector>

#include "../../include/ringattn.h"
#include "ra_internal.h"

namespace {

using namespace ra;

__device__ int g_dev_err[2];  // [0] error code, [1] site | block << 8

std::mutex g_mu;
unsigned long long g_wait_limit_ns = 4000000000ull;
int g_debug_flags = 0;
int g_dkdv_pair = 0;  // head_dim 128: 1 runs the dK / dV pass on CTA pairs
int* g_err_ptr[64] = {nullptr};

ra_status dev_ctl(DevCtl* c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess || !p) return RA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  c->err_word = g_err_ptr[dev];
  c->err_info = g_err_ptr[dev] + 1;
  c->wait_limit_ns = g_wait_limit_ns;
  c->debug_flags = g_debug_flags;
  return RA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// (b, h, s, d) view of a bf16 tensor with element strides.
struct Bhsd {
  void* data;
  long long b, h, s, d;
  long long sb, sh, ss;
};

// TMA map over (d, s, h, b) with boxes of 64 head dims by box_rows rows and 128-byte swizzle.
ra_status make_tmap(const Bhsd& t, CUtensorMap* m, int box_rows = kTileM) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return RA_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)t.d, (cuuint64_t)t.s, (cuuint64_t)t.h, (cuuint64_t)t.b};
  long long sb = t.b > 1 ? t.sb : t.sh * t.h;  // any legal stride for a size-1 dimension
  if (sb <= 0) sb = 8;
  long long sh = t.h > 1 ? t.sh : (t.ss * t.s > 0 ? t.ss * t.s : 8);
  cuuint64_t strides[3] = {(cuuint64_t)(t.ss * 2), (cuuint64_t)(sh * 2), (cuuint64_t)(sb * 2)};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.data, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RA_OK : RA_ERR_ALIGNMENT;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks a bf16 (b, h, s, d) tensor usable by the tiled kernels.
ra_status check_bhsd(const ra_tensor* t, Bhsd* v) {
  if (!t || !t->data) return RA_ERR_INVALID_ARG;
  if (t->ndim != 4 || t->dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (t->shape[i] < 1) return RA_ERR_INVALID_ARG;
  if (t->stride[3] != 1) return RA_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (t->stride[i] <= 0 || t->stride[i] % 8 != 0) return RA_ERR_ALIGNMENT;
  if (!aligned(t->data, 16)) return RA_ERR_ALIGNMENT;
  *v = Bhsd{t->data, t->shape[0], t->shape[1], t->shape[2], t->shape[3], t->stride[0], t->stride[1], t->stride[2]};
  return RA_OK;
}

// Varlen tensors: (total, h, d) or (h, total, d), bf16, as a b = 1 view.
ra_status check_thd(const ra_tensor* t, long long total, Bhsd* v) {
  if (!t || !t->data) return RA_ERR_INVALID_ARG;
  if (t->ndim != 3 || t->dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  if (t->stride[2] != 1) return RA_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if (t->shape[i] < 1) return RA_ERR_INVALID_ARG;
  long long h, ss, sh;
  if (t->shape[0] == total) {
    h = t->shape[1];
    ss = t->stride[0];
    sh = t->stride[1];
  } else if (t->shape[1] == total) {
    h = t->shape[0];
    ss = t->stride[1];
    sh = t->stride[0];
  } else {
    return RA_ERR_INVALID_ARG;
  }
  if (ss <= 0 || sh <= 0 || ss % 8 || sh % 8) return RA_ERR_ALIGNMENT;
  if (!aligned(t->data, 16)) return RA_ERR_ALIGNMENT;
  *v = Bhsd{t->data, 1, h, total, t->shape[2], 0, sh, ss};
  return RA_OK;
}

bool same_shape(const Bhsd& a, const Bhsd& b) { return a.b == b.b && a.h == b.h && a.s == b.s && a.d == b.d; }

// k / v against q: the same batch and head dim, and (grouped-query attention)
// a head count that divides q's; s_ratio = k rows per q row (1, or N for one
// llama3 rank holding L = S / N query rows).
bool kv_matches_q(const Bhsd& q, const Bhsd& k, long long s_ratio) {
  return q.b == k.b && q.d == k.d && k.h >= 1 && q.h % k.h == 0 && q.s * s_ratio == k.s;
}

ra_status check_layout(int32_t layout, int32_t n_shards, long long s) {
  if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_STRIPE) return RA_ERR_INVALID_ARG;
  if (n_shards < 1 || s % n_shards != 0) return RA_ERR_INVALID_ARG;
  if (layout == RA_LAYOUT_ZIGZAG && s % (2LL * n_shards) != 0) return RA_ERR_INVALID_ARG;
  return RA_OK;
}

ra_status check_scale(float sc) { return (isfinite(sc) && sc > 0.f) ? RA_OK : RA_ERR_INVALID_ARG; }

ra_status check_lse(const ra_tensor* t, long long b, long long h, long long s, long long* sb, long long* sh,
                    long long* ss) {
  if (!t || !t->data || t->dtype != RA_FP32 || !aligned(t->data, 4)) return RA_ERR_INVALID_ARG;
  if (t->ndim == 3) {
    if (t->shape[0] != b || t->shape[1] != h || t->shape[2] != s) return RA_ERR_INVALID_ARG;
    *sb = t->stride[0];
    *sh = t->stride[1];
    *ss = t->stride[2];
    return RA_OK;
  }
  if (t->ndim == 2 && b == 1) {  // varlen: (h, total)
    if (t->shape[0] != h || t->shape[1] != s) return RA_ERR_INVALID_ARG;
    *sb = 0;
    *sh = t->stride[0];
    *ss = t->stride[1];
    return RA_OK;
  }
  return RA_ERR_INVALID_ARG;
}

ra_status cuda_status(cudaError_t e) { return e == cudaSuccess ? RA_OK : RA_ERR_CUDA; }

// ------------------------------------------------------------------ kernel timing
// Event pairs are pooled per kernel kind and reused after each read.
struct TimingSlot {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pool;
  size_t used = 0;
};
bool g_timing_on = false;
TimingSlot g_timing[RA_KERNEL_COUNT];

// Brackets one launch with events when timing is on.
struct TimedLaunch {
  int kind;
  cudaStream_t st;
  cudaEvent_t stop = nullptr;
  TimedLaunch(int k, cudaStream_t s) : kind(k), st(s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_timing_on) return;
    TimingSlot& t = g_timing[kind];
    if (t.used == t.pool.size()) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess) return;
      if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(a);
        return;
      }
      t.pool.emplace_back(a, b);
    }
    auto& pr = t.pool[t.used++];
    cudaEventRecord(pr.first, st);
    stop = pr.second;
  }
  ~TimedLaunch() {
    if (stop) cudaEventRecord(stop, st);
  }
};

#define RA_TRY(x)                    \
  do {                               \
    ra_status _s = (x);              \
    if (_s != RA_OK) return _s;      \
  } while (0)

// Shared forward: fused ring (step < 0) or one ring step.
// The argument checks of every backward entry point, made before anything
// touches the device or the workspace.
ra_status bwd_check_args(const Bhsd& dout, const Bhsd& q, const Bhsd& k, const Bhsd& v, const Bhsd& out,
                         int32_t layout, int32_t n_shards, int32_t causal, float scale, const Bhsd& dq,
                         const Bhsd& dk, const Bhsd& dv, int32_t rank) {
  if (!same_shape(k, v) || !same_shape(k, dk) || !same_shape(k, dv) || !same_shape(q, out) ||
      !same_shape(q, dout) || !same_shape(q, dq))
    return RA_ERR_INVALID_ARG;
  if (rank < 0 && !kv_matches_q(q, k, 1)) return RA_ERR_INVALID_ARG;
  if (rank >= 0 && (rank >= n_shards || !kv_matches_q(q, k, n_shards))) return RA_ERR_INVALID_ARG;
  if (q.d != 64 && q.d != 128) return RA_ERR_UNSUPPORTED;
  RA_TRY(check_layout(layout, n_shards, k.s));
  RA_TRY(check_scale(scale));
  if (causal != 0 && causal != 1) return RA_ERR_INVALID_ARG;
  if (k.s > (1LL << 30) || q.b * q.h > 65535) return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

// rank >= 0: one rank of the llama3 form: q and o hold that rank's L = S / N
// rows (the contiguous slice [rank*L, (rank+1)*L)), k and v all S rows.
ra_status fwd_common(const Bhsd& q, const Bhsd& k, const Bhsd& v, int32_t layout, int32_t n_shards, int32_t causal,
                     float scale, int32_t step, const Bhsd& o, int out_f32, float* lse, long long lsb, long long lsh,
                     long long lss, const int32_t* cu_dev, int32_t n_seqs, void* stream, int32_t rank = -1,
                     const int* row_map = nullptr) {
  if (!same_shape(k, v) || !same_shape(q, o)) return RA_ERR_INVALID_ARG;
  if (rank < 0 && !kv_matches_q(q, k, 1)) return RA_ERR_INVALID_ARG;
  if (rank >= 0 && (rank >= n_shards || !kv_matches_q(q, k, n_shards))) return RA_ERR_INVALID_ARG;
  if (q.d != 64 && q.d != 128) return RA_ERR_UNSUPPORTED;
  RA_TRY(check_layout(layout, n_shards, k.s));
  RA_TRY(check_scale(scale));
  if (causal != 0 && causal != 1) return RA_ERR_INVALID_ARG;
  if (k.s > (1LL << 30) || q.b * q.h > 65535) return RA_ERR_UNSUPPORTED;
  if (o.ss % (out_f32 ? 4 : 8) || o.sh % (out_f32 ? 4 : 8) || (o.b > 1 && o.sb % (out_f32 ? 4 : 8)))
    return RA_ERR_ALIGNMENT;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = (int)q.b;
  p.H = (int)q.h;
  p.Hk = (int)k.h;
  p.G = (int)(q.h / k.h);
  p.N = n_shards;
  p.S = (int)k.s;
  p.L = (int)(k.s / n_shards);
  p.r_only = rank;
  p.q_base = rank >= 0 ? rank * p.L : 0;
  p.q_rows = (int)q.s;
  p.row_map = row_map;
  p.layout = layout;
  p.causal = causal;
  p.step = step;
  p.n_qtiles = (p.L + kTileM - 1) / kTileM;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = o.data;
  p.o_sb = o.sb;
  p.o_sh = o.sh;
  p.o_ss = o.ss;
  p.out_f32 = out_f32;
  p.lse = lse;
  p.l_sb = lsb;
  p.l_sh = lsh;
  p.l_ss = lss;
  p.cu = cu_dev;
  p.n_seqs = n_seqs;
  RA_TRY(dev_ctl(&p.ctl));
  CUtensorMap tq, tk, tv;
  RA_TRY(make_tmap(q, &tq));
  RA_TRY(make_tmap(k, &tk));
  RA_TRY(make_tmap(v, &tv));
  TimedLaunch tl(RA_KERNEL_FWD, static_cast<cudaStream_t>(stream));
  return cuda_status(launch_fwd((int)q.d, tq, tk, tv, p, static_cast<cudaStream_t>(stream)));
}

// Workspace: -D and -lse2, each laid out per shard with rows padded to a
// multiple of 128, each part 256-byte aligned.
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
long long stat_rows_per_shard(long long s, int n_shards) {
  const long long L = s / n_shards;
  return (L + kTileM - 1) / kTileM * kTileM;
}
size_t bwd_ws_bytes(long long b, long long h, long long s, int n_shards) {
  return 2 * round256((size_t)b * h * n_shards * stat_rows_per_shard(s, n_shards) * sizeof(float));
}

// rank >= 0: one rank of the llama3 form: q, out, dout, dq hold that rank's
// L = S / N rows, k, v, dk, dv all S rows (dk, dv get this rank's contribution),
// and the statistics cover the rank's rows only.
ra_status bwd_common(const Bhsd& dout, const Bhsd& q, const Bhsd& k, const Bhsd& v, const Bhsd& out,
                     const float* lse, long long lsb, long long lsh, long long lss, int32_t layout, int32_t n_shards,
                     int32_t causal, float scale, const Bhsd& dq, const Bhsd& dk, const Bhsd& dv, void* ws,
                     size_t ws_bytes, const int32_t* cu_dev, int32_t n_seqs, void* stream, int32_t rank = -1,
                     const int* row_map = nullptr) {
  RA_TRY(bwd_check_args(dout, q, k, v, out, layout, n_shards, causal, scale, dq, dk, dv, rank));
  const int stat_N = rank >= 0 ? 1 : n_shards;  // shards whose rows the statistics hold
  if (!ws || !aligned(ws, 256) || ws_bytes < bwd_ws_bytes(q.b, q.h, q.s, stat_N)) return RA_ERR_WORKSPACE;
  const int stat_L = (int)stat_rows_per_shard(q.s, stat_N);
  const size_t stats = round256((size_t)q.b * q.h * stat_N * stat_L * sizeof(float));
  float* nD = static_cast<float*>(ws);
  float* nlse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + stats);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  View4 vdo{dout.data, dout.sb, dout.sh, dout.ss, (int)dout.b, (int)dout.h, (int)dout.s, (int)dout.d};
  View4 vo{out.data, out.sb, out.sh, out.ss, (int)out.b, (int)out.h, (int)out.s, (int)out.d};

  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = (int)q.b;
  p.H = (int)q.h;
  p.Hk = (int)k.h;
  p.G = (int)(q.h / k.h);
  p.N = n_shards;
  p.S = (int)k.s;
  p.L = (int)(k.s / n_shards);
  p.layout = layout;
  p.causal = causal;
  p.n_qtiles = (p.L + kTileM - 1) / kTileM;
  p.n_ktiles = (p.L + kTileN - 1) / kTileN;
  p.r_only = rank;
  p.q_base = rank >= 0 ? rank * p.L : 0;
  p.q_rows = (int)q.s;
  p.row_map = row_map;
  p.stat_N = stat_N;
  p.stat_r0 = rank >= 0 ? rank : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.stat_L = stat_L;
  p.nlse2 = nlse2;
  p.nD = nD;
  p.dq = dq.data;
  p.dk = dk.data;
  p.dv = dv.data;
  p.q_sb = dq.sb;
  p.q_sh = dq.sh;
  p.q_ss = dq.ss;
  p.k_sb = dk.sb;
  p.k_sh = dk.sh;
  p.k_ss = dk.ss;
  p.v_sb = dv.sb;
  p.v_sh = dv.sh;
  p.v_ss = dv.ss;
  p.cu = cu_dev;
  p.n_seqs = n_seqs;
  RA_TRY(dev_ctl(&p.ctl));
  CUtensorMap tq, tk, tv, tdo;
  RA_TRY(make_tmap(q, &tq));
  RA_TRY(make_tmap(k, &tk));
  RA_TRY(make_tmap(v, &tv));
  RA_TRY(make_tmap(dout, &tdo));
  {
    TimedLaunch tl(RA_KERNEL_BWD_PRE, st);
    // with a row map (varlen in original order), out and lse stay in the
    // caller's layout order and are read through it
    RA_TRY(cuda_status(
        launch_bwd_pre(vdo, vo, LseView{lse, lsb, lsh, lss}, nD, nlse2, stat_N, stat_L, p.ctl, row_map, st)));
  }
  if (q.d == 128 && q.h == k.h && __atomic_load_n(&g_dkdv_pair, __ATOMIC_RELAXED)) {
    CUtensorMap pq, pk, pv, pdo;  // 64-row boxes: the pair kernel loads 64 x 64 blocks
    RA_TRY(make_tmap(q, &pq, 64));
    RA_TRY(make_tmap(k, &pk, 64));
    RA_TRY(make_tmap(v, &pv, 64));
    RA_TRY(make_tmap(dout, &pdo, 64));
    TimedLaunch tl(RA_KERNEL_BWD, st);
    RA_TRY(cuda_status(launch_dkdv_pair(pq, pk, pv, pdo, p, st)));
  } else {
    TimedLaunch tl(RA_KERNEL_BWD, st);
    RA_TRY(cuda_status(launch_bwd((int)q.d, tq, tk, tv, tdo, p, 0, st)));
  }
  TimedLaunch tl(RA_KERNEL_BWD_DQ, st);
  return cuda_status(launch_bwd((int)q.d, tq, tk, tv, tdo, p, 1, st));
}

// Scratch of ring_attn_bwd_static_scratch: one array per device, its device
// address looked up once per device (with that device current) and cached.
void* g_scratch_ptr[64] = {nullptr};

ra_status static_scratch(void** out);

// Varlen layouts: contiguous slices of the packed buffer, or the zigzag split
// of every sequence (each length a multiple of 2 * n_shards).
ra_status check_varlen_layout(int32_t layout, int32_t n_shards, const int32_t* cu_host, int32_t n_seqs) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG) return RA_ERR_UNSUPPORTED;
  if (n_shards < 1) return RA_ERR_INVALID_ARG;
  if (layout == RA_LAYOUT_ZIGZAG)
    for (int32_t i = 0; i < n_seqs; ++i)
      if ((cu_host[i + 1] - cu_host[i]) % (2 * n_shards) != 0) return RA_ERR_INVALID_ARG;
  return RA_OK;
}

ra_status check_cu(const int32_t* cu_dev, const int32_t* cu_host, int32_t n_seqs, int32_t max_seqlen,
                   long long* total) {
  if (!cu_dev || !cu_host || n_seqs < 1) return RA_ERR_INVALID_ARG;
  if (!aligned(cu_dev, 4)) return RA_ERR_ALIGNMENT;
  if (cu_host[0] != 0) return RA_ERR_INVALID_ARG;
  int32_t mx = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    if (cu_host[i + 1] < cu_host[i]) return RA_ERR_INVALID_ARG;
    const int32_t len = cu_host[i + 1] - cu_host[i];
    if (len > mx) mx = len;
  }
  if (max_seqlen < mx) return RA_ERR_INVALID_ARG;
  *total = cu_host[n_seqs];
  if (*total < 1) return RA_ERR_INVALID_ARG;
  return RA_OK;
}

// ---------------------------------------------------------------- zigzag varlen in original order
// On one GPU the zigzag split of every sequence is only a storage order.  With
// a large enough caller workspace the zigzag varlen calls copy their inputs
// into it in original order and run the contiguous-layout kernels there (tiles
// then hold whole runs of one sequence instead of the 2N short chunks of
// several), which write each output row straight to its row of the caller's
// zigzag order through the inverse token map.
size_t zz_tensor_bytes(long long total, long long h, long long d) { return round256((size_t)total * h * d * 2); }
size_t zz_map_bytes(long long total) { return round256((size_t)total * 4); }
// The outputs are written straight into the caller's layout-order rows (the
// kernels take the inverse map), so only inputs are copied.
// forward: q, k, v in original order (h, total, d), the map and its inverse
size_t zz_fwd_bytes(long long total, long long h, long long d) {
  return 3 * zz_tensor_bytes(total, h, d) + 2 * zz_map_bytes(total);
}
// backward: the statistics, then dO, q, k, v, the map and its inverse (out and
// lse are only read by the statistics pass, through the map, where they are)
size_t zz_bwd_bytes(long long total, long long h, long long d, int n_shards) {
  return bwd_ws_bytes(1, h, total, n_shards) + 4 * zz_tensor_bytes(total, h, d) + 2 * zz_map_bytes(total);
}

// A contiguous (h, total, d) bf16 view at p.
Bhsd zz_view(void* p, long long total, long long h, long long d) {
  return Bhsd{p, 1, h, total, d, 0, total * d, d};
}

// Permutes one (1, h, total, d) view (or an (h, total) fp32 lse when d == 0)
// between zigzag layout order and original order: inverse = 1 reads layout
// order (src) and writes original order (dst).
ra_status zz_permute(const void* src, long long s_sh, long long s_ss, void* dst, long long d_sh, long long d_ss,
                     long long h, long long total, long long d, int inverse, const int32_t* cu_dev, int32_t n_seqs,
                     int32_t n_shards, const int* gmap, cudaStream_t st) {
  PermuteArgs a;
  memset(&a, 0, sizeof(a));
  a.src = src;
  a.dst = dst;
  a.esize = d > 0 ? 2 : 4;
  a.inner = d > 0 ? d : 1;
  for (int i = 0; i < 3; ++i) a.outer_shape[i] = 1;
  a.outer_shape[2] = h;
  a.src_outer_stride[2] = s_sh;
  a.dst_outer_stride[2] = d_sh;
  a.n_outer = h;
  a.src_seq_stride = s_ss;
  a.dst_seq_stride = d_ss;
  a.s = (int)total;
  a.layout = RA_LAYOUT_ZIGZAG;
  a.N = n_shards;
  a.inverse = inverse;
  a.cu = cu_dev;
  a.n_seqs = n_seqs;
  a.gmap = gmap;
  RA_TRY(dev_ctl(&a.ctl));
  TimedLaunch tl(RA_KERNEL_PERMUTE, st);
  return cuda_status(launch_permute(a, st));
}

// The copies of one call share the token map, computed once into the workspace.
struct ZzCtx {
  const int32_t* cu;
  int32_t n, N;
  cudaStream_t st;
  const int* map;  // layout position -> original token
  const int* inv;  // original token -> layout position
};
// map (total int32) then its inverse (the next 256-aligned total int32) at w
ra_status zz_map(ZzCtx& z, char* w, long long total) {
  z.map = reinterpret_cast<const int*>(w);
  z.inv = reinterpret_cast<const int*>(w + zz_map_bytes(total));
  TimedLaunch tl(RA_KERNEL_PERMUTE, z.st);
  return cuda_status(launch_zigzag_varlen_map(z.cu, z.n, z.N, (int)total, reinterpret_cast<int*>(w),
                                              reinterpret_cast<int*>(w + zz_map_bytes(total)), z.st));
}
ra_status zz_in(const ZzCtx& z, const Bhsd& x, void* dst) {
  return zz_permute(x.data, x.sh, x.ss, dst, x.s * x.d, x.d, x.h, x.s, x.d, 1, z.cu, z.n, z.N, z.map, z.st);
}

}  // namespace

// Statistics of ring_attn_bwd_static_scratch (-D, then -lse * log2(e)).  The
// library never allocates it: it is part of the loaded device image.  In host
// code this name is only a stand-in; static_scratch gives the device address.
static __device__ __align__(256) unsigned char g_bwd_scratch[RA_STATIC_SCRATCH_BYTES];

namespace {

ra_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return RA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}

}  // namespace

extern "C" {

ra_status ring_attn_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v, int32_t layout,
                        int32_t n_shards, int32_t causal, float softmax_scale, ra_tensor* out, ra_tensor* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  Bhsd vq, vk, vv, vo;
  RA_TRY(check_bhsd(q, &vq));
  RA_TRY(check_bhsd(k, &vk));
  RA_TRY(check_bhsd(v, &vv));
  RA_TRY(check_bhsd(out, &vo));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, vq.b, vq.h, vq.s, &lsb, &lsh, &lss));
  return fwd_common(vq, vk, vv, layout, n_shards, causal, softmax_scale, -1, vo, 0, static_cast<float*>(lse->data),
                    lsb, lsh, lss, nullptr, 0, stream);
}

ra_status ring_attn_fwd_step(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v, int32_t layout,
                             int32_t n_shards, int32_t causal, float softmax_scale, int32_t step,
                             ra_tensor* out_blk, ra_tensor* lse_blk, void* stream) {
  Bhsd vq, vk, vv;
  RA_TRY(check_bhsd(q, &vq));
  RA_TRY(check_bhsd(k, &vk));
  RA_TRY(check_bhsd(v, &vv));
  if (n_shards < 1 || step < 0 || step >= n_shards) return RA_ERR_INVALID_ARG;
  if (!out_blk || !out_blk->data || out_blk->ndim != 4) return RA_ERR_INVALID_ARG;
  const int f32 = out_blk->dtype == RA_FP32;
  if (!f32 && out_blk->dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  if (out_blk->stride[3] != 1 || !aligned(out_blk->data, 16)) return RA_ERR_ALIGNMENT;
  Bhsd vo{out_blk->data, out_blk->shape[0], out_blk->shape[1], out_blk->shape[2], out_blk->shape[3],
          out_blk->stride[0], out_blk->stride[1], out_blk->stride[2]};
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse_blk, vq.b, vq.h, vq.s, &lsb, &lsh, &lss));
  return fwd_common(vq, vk, vv, layout, n_shards, causal, softmax_scale, step, vo, f32,
                    static_cast<float*>(lse_blk->data), lsb, lsh, lss, nullptr, 0, stream);
}

ra_status lse_merge(ra_tensor* out_acc, ra_tensor* lse_acc, const ra_tensor* out_blk, const ra_tensor* lse_blk,
                    void* stream) {
  if (!out_acc || !lse_acc || !out_blk || !lse_blk) return RA_ERR_INVALID_ARG;
  if (!out_acc->data || !lse_acc->data || !out_blk->data || !lse_blk->data) return RA_ERR_INVALID_ARG;
  const int nd = out_acc->ndim;
  if (nd < 2 || nd > 4 || out_blk->ndim != nd || lse_acc->ndim != nd - 1 || lse_blk->ndim != nd - 1)
    return RA_ERR_INVALID_ARG;
  if (out_acc->dtype != RA_FP32 || lse_acc->dtype != RA_FP32 || lse_blk->dtype != RA_FP32) return RA_ERR_INVALID_ARG;
  if (out_blk->dtype != RA_FP32 && out_blk->dtype != RA_BF16) return RA_ERR_INVALID_ARG;
  for (int i = 0; i < nd; ++i) {
    if (out_acc->shape[i] < 1 || out_blk->shape[i] != out_acc->shape[i]) return RA_ERR_INVALID_ARG;
    if (i < nd - 1 && (lse_acc->shape[i] != out_acc->shape[i] || lse_blk->shape[i] != out_acc->shape[i]))
      return RA_ERR_INVALID_ARG;
  }
  const long long d = out_acc->shape[nd - 1];
  if (d % 4 != 0 || 32 % (d / 4) != 0) return RA_ERR_UNSUPPORTED;
  if (out_acc->stride[nd - 1] != 1 || out_blk->stride[nd - 1] != 1) return RA_ERR_ALIGNMENT;
  const int bs = out_blk->dtype == RA_FP32 ? 16 : 8;  // bytes per 4 elements
  if (!aligned(out_acc->data, 16) || !aligned(out_blk->data, bs) || !aligned(lse_acc->data, 4) ||
      !aligned(lse_blk->data, 4))
    return RA_ERR_ALIGNMENT;
  MergeArgs a;
  memset(&a, 0, sizeof(a));
  long long n[3] = {1, 1, 1}, oa[3] = {0, 0, 0}, la[3] = {0, 0, 0}, ob[3] = {0, 0, 0}, lb[3] = {0, 0, 0};
  const int outer = nd - 1;  // 1..3 row dimensions, right-aligned into 3 slots
  for (int i = 0; i < outer; ++i) {
    const int slot = 3 - outer + i;
    n[slot] = out_acc->shape[i];
    oa[slot] = out_acc->stride[i];
    ob[slot] = out_blk->stride[i];
    la[slot] = lse_acc->stride[i];
    lb[slot] = lse_blk->stride[i];
    if (oa[slot] % 4 || ob[slot] % 4) return RA_ERR_ALIGNMENT;
  }
  a.out_acc = static_cast<float*>(out_acc->data);
  a.lse_acc = static_cast<float*>(lse_acc->data);
  a.out_blk = out_blk->data;
  a.lse_blk = static_cast<const float*>(lse_blk->data);
  a.blk_f32 = out_blk->dtype == RA_FP32;
  a.d = d;
  a.n0 = n[0];
  a.n1 = n[1];
  a.n2 = n[2];
  a.rows = n[0] * n[1] * n[2];
  a.oa_s0 = oa[0];
  a.oa_s1 = oa[1];
  a.oa_s2 = oa[2];
  a.la_s0 = la[0];
  a.la_s1 = la[1];
  a.la_s2 = la[2];
  a.ob_s0 = ob[0];
  a.ob_s1 = ob[1];
  a.ob_s2 = ob[2];
  a.lb_s0 = lb[0];
  a.lb_s1 = lb[1];
  a.lb_s2 = lb[2];
  // rows that collapse to one stride per tensor are indexed without divisions:
  // walk the non-unit row dims from the inside out, each must step by the
  // previous dim's extent; the innermost non-unit stride is the row stride
  auto row_stride = [&](const long long* st, long long* out) {
    long long stride = 0, expect = -1;
    for (int i = 2; i >= 0; --i) {
      if (n[i] == 1) continue;
      if (expect < 0) {
        stride = st[i];
      } else if (st[i] != expect) {
        return false;
      }
      expect = st[i] * n[i];
    }
    *out = stride;
    return true;
  };
  long long f_oa, f_ob, f_la, f_lb;
  a.flat = row_stride(oa, &f_oa) && row_stride(ob, &f_ob) && row_stride(la, &f_la) && row_stride(lb, &f_lb);
  if (a.flat) {  // the kernel then reads only the *_s2 strides
    a.oa_s2 = f_oa;
    a.ob_s2 = f_ob;
    a.la_s2 = f_la;
    a.lb_s2 = f_lb;
  }
  // 8 columns per thread (two 16-byte fp32 accesses, one 16-byte bf16 access)
  // when every row start allows it
  const bool v8 = d % 8 == 0 && 32 % (d / 8) == 0 && oa[0] % 8 == 0 && oa[1] % 8 == 0 && oa[2] % 8 == 0 &&
                  ob[0] % 8 == 0 && ob[1] % 8 == 0 && ob[2] % 8 == 0 && aligned(out_blk->data, 16);
  // 16 columns (four 16-byte fp32 accesses, two 16-byte bf16 accesses) for a bf16 block
  const bool v16 = v8 && !a.blk_f32 && d % 16 == 0 && 32 % (d / 16) == 0;
  a.vec = v16 ? 16 : (v8 ? 8 : 4);
  a.qshift = 0;
  while ((1LL << a.qshift) < d / a.vec) ++a.qshift;
  TimedLaunch tl(RA_KERNEL_LSE_MERGE, static_cast<cudaStream_t>(stream));
  return cuda_status(launch_lse_merge(a, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                        const ra_tensor* out, const ra_tensor* lse, int32_t layout, int32_t n_shards,
                        int32_t causal, float softmax_scale, ra_tensor* dq, ra_tensor* dk, ra_tensor* dv,
                        void* workspace, size_t workspace_bytes, void* stream) {
  Bhsd vdo, vq, vk, vv, vo, vdq, vdk, vdv;
  RA_TRY(check_bhsd(dout, &vdo));
  RA_TRY(check_bhsd(q, &vq));
  RA_TRY(check_bhsd(k, &vk));
  RA_TRY(check_bhsd(v, &vv));
  RA_TRY(check_bhsd(out, &vo));
  RA_TRY(check_bhsd(dq, &vdq));
  RA_TRY(check_bhsd(dk, &vdk));
  RA_TRY(check_bhsd(dv, &vdv));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, vq.b, vq.h, vq.s, &lsb, &lsh, &lss));
  return bwd_common(vdo, vq, vk, vv, vo, static_cast<const float*>(lse->data), lsb, lsh, lss, layout, n_shards,
                    causal, softmax_scale, vdq, vdk, vdv, workspace, workspace_bytes, nullptr, 0, stream);
}

ra_status ring_attn_bwd_static_scratch(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k,
                                       const ra_tensor* v, const ra_tensor* out, const ra_tensor* lse,
                                       int32_t layout, int32_t n_shards, int32_t causal, float softmax_scale,
                                       ra_tensor* dq, ra_tensor* dk, ra_tensor* dv, void* stream) {
  Bhsd vdo, vq, vk, vv, vo, vdq, vdk, vdv;
  RA_TRY(check_bhsd(dout, &vdo));
  RA_TRY(check_bhsd(q, &vq));
  RA_TRY(check_bhsd(k, &vk));
  RA_TRY(check_bhsd(v, &vv));
  RA_TRY(check_bhsd(out, &vo));
  RA_TRY(check_bhsd(dq, &vdq));
  RA_TRY(check_bhsd(dk, &vdk));
  RA_TRY(check_bhsd(dv, &vdv));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, vq.b, vq.h, vq.s, &lsb, &lsh, &lss));
  // Every argument check of ring_attn_bwd comes first, so a bad argument gets
  // the same status from both calls; only then the size of the array.
  RA_TRY(bwd_check_args(vdo, vq, vk, vv, vo, layout, n_shards, causal, softmax_scale, vdq, vdk, vdv, -1));
  if (bwd_ws_bytes(vq.b, vq.h, vq.s, n_shards) > RA_STATIC_SCRATCH_BYTES) return RA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  RA_TRY(static_scratch(&scratch));
  return bwd_common(vdo, vq, vk, vv, vo, static_cast<const float*>(lse->data), lsb, lsh, lss, layout, n_shards,
                    causal, softmax_scale, vdq, vdk, vdv, scratch, RA_STATIC_SCRATCH_BYTES, nullptr, 0, stream);
}

ra_status ring_attn_varlen_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                               const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                               int32_t max_seqlen, int32_t layout, int32_t n_shards, int32_t causal,
                               float softmax_scale, ra_tensor* out, ra_tensor* lse, void* workspace,
                               size_t workspace_bytes, void* stream) {
  long long total = 0;
  RA_TRY(check_cu(cu_seqlens_dev, cu_seqlens_host, n_seqs, max_seqlen, &total));
  RA_TRY(check_varlen_layout(layout, n_shards, cu_seqlens_host, n_seqs));
  Bhsd vq, vk, vv, vo;
  RA_TRY(check_thd(q, total, &vq));
  RA_TRY(check_thd(k, total, &vk));
  RA_TRY(check_thd(v, total, &vv));
  RA_TRY(check_thd(out, total, &vo));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, 1, vq.h, total, &lsb, &lsh, &lss));
  if (layout == RA_LAYOUT_ZIGZAG && workspace && workspace_bytes >= zz_fwd_bytes(total, vq.h, vq.d)) {
    // original-order path: the same checks as the kernels' before any launch
    if (!kv_matches_q(vq, vk, 1) || !same_shape(vk, vv) || !same_shape(vq, vo)) return RA_ERR_INVALID_ARG;
    if (vq.d != 64 && vq.d != 128) return RA_ERR_UNSUPPORTED;
    RA_TRY(check_scale(softmax_scale));
    if (causal != 0 && causal != 1) return RA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return RA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(workspace);
    const size_t T = zz_tensor_bytes(total, vq.h, vq.d);
    // (k and v may have fewer heads than q: their copies use the first part of each T)
    const Bhsd q2 = zz_view(w, total, vq.h, vq.d), k2 = zz_view(w + T, total, vk.h, vq.d),
               v2 = zz_view(w + 2 * T, total, vk.h, vq.d);
    ZzCtx z{cu_seqlens_dev, n_seqs, n_shards, st, nullptr, nullptr};
    RA_TRY(zz_map(z, w + 3 * T, total));
    RA_TRY(zz_in(z, vq, q2.data));
    RA_TRY(zz_in(z, vk, k2.data));
    RA_TRY(zz_in(z, vv, v2.data));
    return fwd_common(q2, k2, v2, RA_LAYOUT_CONTIGUOUS, n_shards, causal, softmax_scale, -1, vo, 0,
                      static_cast<float*>(lse->data), lsb, lsh, lss, cu_seqlens_dev, n_seqs, stream, -1, z.inv);
  }
  return fwd_common(vq, vk, vv, layout, n_shards, causal, softmax_scale, -1, vo, 0,
                    static_cast<float*>(lse->data), lsb, lsh, lss, cu_seqlens_dev, n_seqs, stream);
}

ra_status ring_attn_varlen_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                               const ra_tensor* out, const ra_tensor* lse, const int32_t* cu_seqlens_dev,
                               const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t max_seqlen,
                               int32_t layout, int32_t n_shards, int32_t causal, float softmax_scale, ra_tensor* dq,
                               ra_tensor* dk, ra_tensor* dv, void* workspace, size_t workspace_bytes, void* stream) {
  long long total = 0;
  RA_TRY(check_cu(cu_seqlens_dev, cu_seqlens_host, n_seqs, max_seqlen, &total));
  RA_TRY(check_varlen_layout(layout, n_shards, cu_seqlens_host, n_seqs));
  Bhsd vdo, vq, vk, vv, vo, vdq, vdk, vdv;
  RA_TRY(check_thd(dout, total, &vdo));
  RA_TRY(check_thd(q, total, &vq));
  RA_TRY(check_thd(k, total, &vk));
  RA_TRY(check_thd(v, total, &vv));
  RA_TRY(check_thd(out, total, &vo));
  RA_TRY(check_thd(dq, total, &vdq));
  RA_TRY(check_thd(dk, total, &vdk));
  RA_TRY(check_thd(dv, total, &vdv));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, 1, vq.h, total, &lsb, &lsh, &lss));
  if (layout == RA_LAYOUT_ZIGZAG && workspace && workspace_bytes >= zz_bwd_bytes(total, vq.h, vq.d, n_shards)) {
    // original-order path: the same checks as the kernels' before any launch
    RA_TRY(bwd_check_args(vdo, vq, vk, vv, vo, layout, n_shards, causal, softmax_scale, vdq, vdk, vdv, -1));
    if (!aligned(workspace, 256)) return RA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t SB = bwd_ws_bytes(1, vq.h, total, n_shards), T = zz_tensor_bytes(total, vq.h, vq.d);
    char* w = static_cast<char*>(workspace) + SB;
    const long long h = vq.h, d = vq.d;
    const long long hk = vk.h;  // k and v may have fewer heads than q
    const Bhsd do2 = zz_view(w, total, h, d), q2 = zz_view(w + T, total, h, d), k2 = zz_view(w + 2 * T, total, hk, d),
               v2 = zz_view(w + 3 * T, total, hk, d);
    ZzCtx z{cu_seqlens_dev, n_seqs, n_shards, st, nullptr, nullptr};
    RA_TRY(zz_map(z, w + 4 * T, total));
    RA_TRY(zz_in(z, vdo, do2.data));
    RA_TRY(zz_in(z, vq, q2.data));
    RA_TRY(zz_in(z, vk, k2.data));
    RA_TRY(zz_in(z, vv, v2.data));
    // out and lse stay in the caller's zigzag order: the statistics pass reads
    // them through the inverse map
    return bwd_common(do2, q2, k2, v2, vo, static_cast<const float*>(lse->data), lsb, lsh, lss, RA_LAYOUT_CONTIGUOUS,
                      n_shards, causal, softmax_scale, vdq, vdk, vdv, workspace, SB, cu_seqlens_dev, n_seqs, stream, -1,
                      z.inv);
  }
  return bwd_common(vdo, vq, vk, vv, vo, static_cast<const float*>(lse->data), lsb, lsh, lss, layout, n_shards,
                    causal, softmax_scale, vdq, vdk, vdv, workspace, workspace_bytes, cu_seqlens_dev, n_seqs,
                    stream);
}

// One rank of the llama3 form: shapes of the local (L rows) and full (total rows) tensors.
static ra_status llama3_shapes(const int32_t* cu_dev, const int32_t* cu_host, int32_t n_seqs, int32_t max_seqlen,
                               int32_t rank, int32_t n_shards, long long* total, long long* L) {
  RA_TRY(check_cu(cu_dev, cu_host, n_seqs, max_seqlen, total));
  if (n_shards < 1 || rank < 0 || rank >= n_shards || *total % n_shards) return RA_ERR_INVALID_ARG;
  *L = *total / n_shards;
  return RA_OK;
}

ra_status ring_attn_llama3_varlen_fwd(const ra_tensor* q, const ra_tensor* k, const ra_tensor* v,
                                      const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                                      int32_t max_seqlen, int32_t rank, int32_t n_shards, int32_t causal,
                                      float softmax_scale, ra_tensor* out, ra_tensor* lse, void* stream) {
  long long total = 0, L = 0;
  RA_TRY(llama3_shapes(cu_seqlens_dev, cu_seqlens_host, n_seqs, max_seqlen, rank, n_shards, &total, &L));
  Bhsd vq, vk, vv, vo;
  RA_TRY(check_thd(q, L, &vq));
  RA_TRY(check_thd(k, total, &vk));
  RA_TRY(check_thd(v, total, &vv));
  RA_TRY(check_thd(out, L, &vo));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, 1, vq.h, L, &lsb, &lsh, &lss));
  return fwd_common(vq, vk, vv, RA_LAYOUT_CONTIGUOUS, n_shards, causal, softmax_scale, -1, vo, 0,
                    static_cast<float*>(lse->data), lsb, lsh, lss, cu_seqlens_dev, n_seqs, stream, rank);
}

ra_status ring_attn_llama3_varlen_bwd(const ra_tensor* dout, const ra_tensor* q, const ra_tensor* k,
                                      const ra_tensor* v, const ra_tensor* out, const ra_tensor* lse,
                                      const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_host, int32_t n_seqs,
                                      int32_t max_seqlen, int32_t rank, int32_t n_shards, int32_t causal,
                                      float softmax_scale, ra_tensor* dq, ra_tensor* dk, ra_tensor* dv,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  long long total = 0, L = 0;
  RA_TRY(llama3_shapes(cu_seqlens_dev, cu_seqlens_host, n_seqs, max_seqlen, rank, n_shards, &total, &L));
  Bhsd vdo, vq, vk, vv, vo, vdq, vdk, vdv;
  RA_TRY(check_thd(dout, L, &vdo));
  RA_TRY(check_thd(q, L, &vq));
  RA_TRY(check_thd(k, total, &vk));
  RA_TRY(check_thd(v, total, &vv));
  RA_TRY(check_thd(out, L, &vo));
  RA_TRY(check_thd(dq, L, &vdq));
  RA_TRY(check_thd(dk, total, &vdk));
  RA_TRY(check_thd(dv, total, &vdv));
  long long lsb, lsh, lss;
  RA_TRY(check_lse(lse, 1, vq.h, L, &lsb, &lsh, &lss));
  return bwd_common(vdo, vq, vk, vv, vo, static_cast<const float*>(lse->data), lsb, lsh, lss, RA_LAYOUT_CONTIGUOUS,
                    n_shards, causal, softmax_scale, vdq, vdk, vdv, workspace, workspace_bytes, cu_seqlens_dev, n_seqs,
                    stream, rank);
}

// Byte span [first, last] that a tensor's strides can reach (negative strides
// are refused by the callers' packing checks, but are handled here anyway).
static void byte_span(const ra_tensor* t, int es, uintptr_t* lo, uintptr_t* hi) {
  long long mn = 0, mx = 0;
  for (int i = 0; i < t->ndim; ++i) {
    const long long reach = (t->shape[i] - 1) * t->stride[i];
    if (reach < 0) mn += reach; else mx += reach;
  }
  const uintptr_t base = reinterpret_cast<uintptr_t>(t->data);
  *lo = base + (uintptr_t)(mn * es);
  *hi = base + (uintptr_t)(mx * es) + (uintptr_t)(es - 1);
}

static bool ranges_overlap(const ra_tensor* a, const ra_tensor* b, int es) {
  uintptr_t alo, ahi, blo, bhi;
  byte_span(a, es, &alo, &ahi);
  byte_span(b, es, &blo, &bhi);
  return alo <= bhi && blo <= ahi;
}

static ra_status permute_common(const ra_tensor* src, ra_tensor* dst, int32_t layout, int32_t n_shards,
                                int32_t seq_dim, int inverse, const int32_t* cu_dev, int32_t n_seqs, void* stream) {
  if (!src || !dst || !src->data || !dst->data) return RA_ERR_INVALID_ARG;
  const int nd = src->ndim;
  if (nd < 1 || nd > 4 || dst->ndim != nd || src->dtype != dst->dtype) return RA_ERR_INVALID_ARG;
  if (src->dtype != RA_BF16 && src->dtype != RA_FP32) return RA_ERR_INVALID_ARG;
  if (seq_dim < 0 || seq_dim >= nd) return RA_ERR_INVALID_ARG;
  for (int i = 0; i < nd; ++i)
    if (src->shape[i] < 1 || dst->shape[i] != src->shape[i]) return RA_ERR_INVALID_ARG;
  const long long s = src->shape[seq_dim];
  RA_TRY(check_layout(layout, n_shards, s));
  if (s > (1LL << 30)) return RA_ERR_UNSUPPORTED;
  // dimensions after seq_dim must be packed in both tensors
  long long inner = 1;
  for (int i = nd - 1; i > seq_dim; --i) {
    if (src->stride[i] != inner || dst->stride[i] != inner) return RA_ERR_INVALID_ARG;
    inner *= src->shape[i];
  }
  const int es = src->dtype == RA_FP32 ? 4 : 2;
  if (!aligned(src->data, es) || !aligned(dst->data, es)) return RA_ERR_ALIGNMENT;
  // Rows are gathered by many blocks at once, so a destination that overlaps
  // the source would be read after other blocks overwrote it: refuse it.
  if (ranges_overlap(src, dst, es)) return RA_ERR_INVALID_ARG;
  PermuteArgs a;
  memset(&a, 0, sizeof(a));
  a.src = src->data;
  a.dst = dst->data;
  a.esize = es;
  a.inner = inner;
  for (int i = 0; i < 3; ++i) {
    a.outer_shape[i] = 1;
    a.src_outer_stride[i] = 0;
    a.dst_outer_stride[i] = 0;
  }
  for (int i = 0; i < seq_dim; ++i) {  // right-align the outer dims into 3 slots
    const int slot = 3 - seq_dim + i;
    a.outer_shape[slot] = src->shape[i];
    a.src_outer_stride[slot] = src->stride[i];
    a.dst_outer_stride[slot] = dst->stride[i];
  }
  a.n_outer = a.outer_shape[0] * a.outer_shape[1] * a.outer_shape[2];
  a.src_seq_stride = src->stride[seq_dim];
  a.dst_seq_stride = dst->stride[seq_dim];
  a.s = (int)s;
  a.layout = layout;
  a.N = n_shards;
  a.inverse = inverse;
  a.cu = cu_dev;
  a.n_seqs = n_seqs;
  RA_TRY(dev_ctl(&a.ctl));
  TimedLaunch tl(RA_KERNEL_PERMUTE, static_cast<cudaStream_t>(stream));
  return cuda_status(launch_permute(a, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_permute(const ra_tensor* x, ra_tensor* y, int32_t layout, int32_t n_shards, int32_t seq_dim,
                            void* stream) {
  return permute_common(x, y, layout, n_shards, seq_dim, 0, nullptr, 0, stream);
}

ra_status ring_attn_unpermute(const ra_tensor* y, ra_tensor* x, int32_t layout, int32_t n_shards, int32_t seq_dim,
                              void* stream) {
  return permute_common(y, x, layout, n_shards, seq_dim, 1, nullptr, 0, stream);
}

static ra_status varlen_permute_common(const ra_tensor* src, ra_tensor* dst, const int32_t* cu_dev,
                                       const int32_t* cu_host, int32_t n_seqs, int32_t layout, int32_t n_shards,
                                       int32_t seq_dim, int inverse, void* stream) {
  long long total = 0;
  RA_TRY(check_cu(cu_dev, cu_host, n_seqs, INT32_MAX, &total));
  RA_TRY(check_varlen_layout(layout, n_shards, cu_host, n_seqs));
  if (!src || seq_dim < 0 || seq_dim >= src->ndim || src->shape[seq_dim] != total) return RA_ERR_INVALID_ARG;
  return permute_common(src, dst, layout, n_shards, seq_dim, inverse, cu_dev, n_seqs, stream);
}

ra_status ring_attn_varlen_permute(const ra_tensor* x, ra_tensor* y, const int32_t* cu_seqlens_dev,
                                   const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t layout, int32_t n_shards,
                                   int32_t seq_dim, void* stream) {
  return varlen_permute_common(x, y, cu_seqlens_dev, cu_seqlens_host, n_seqs, layout, n_shards, seq_dim, 0, stream);
}

ra_status ring_attn_varlen_unpermute(const ra_tensor* y, ra_tensor* x, const int32_t* cu_seqlens_dev,
                                     const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t layout, int32_t n_shards,
                                     int32_t seq_dim, void* stream) {
  return varlen_permute_common(y, x, cu_seqlens_dev, cu_seqlens_host, n_seqs, layout, n_shards, seq_dim, 1, stream);
}

size_t ring_attn_varlen_workspace_size(int32_t op, int64_t total, int64_t h, int64_t d, int32_t layout,
                                       int32_t n_shards) {
  if (total < 1 || h < 1 || (d != 64 && d != 128) || n_shards < 1 || total % n_shards) return 0;
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG) return 0;
  if (op == RA_OP_FWD) return layout == RA_LAYOUT_ZIGZAG ? zz_fwd_bytes(total, h, d) : 0;
  if (op != RA_OP_BWD) return 0;
  return layout == RA_LAYOUT_ZIGZAG ? zz_bwd_bytes(total, h, d, n_shards) : bwd_ws_bytes(1, h, total, n_shards);
}

size_t ring_attn_workspace_size(int32_t op, int64_t b, int64_t h, int64_t s, int64_t d, int32_t n_shards) {
  if (b < 1 || h < 1 || s < 1 || d < 1 || n_shards < 1 || s % n_shards) return 0;
  if (op == RA_OP_BWD) return bwd_ws_bytes(b, h, s, n_shards);
  return 0;
}

ra_status ring_attn_check_device_error(void* stream, int32_t* info) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return RA_ERR_CUDA;
  DevCtl c;
  RA_TRY(dev_ctl(&c));
  int host[2] = {0, 0};
  if (cudaMemcpy(host, c.err_word, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return RA_ERR_CUDA;
  if (host[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(c.err_word, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return RA_ERR_CUDA;
  }
  if (info) *info = host[1];
  if (host[0] == 0) return RA_OK;
  return host[0] == DEV_TIMEOUT ? RA_ERR_TIMEOUT : RA_ERR_DEVICE;
}

ra_status ring_attn_set_knob(int32_t knob, int64_t value) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (knob == RA_KNOB_WAIT_LIMIT_NS) {
    if (value < 1000) return RA_ERR_INVALID_ARG;
    g_wait_limit_ns = (unsigned long long)value;
    return RA_OK;
  }
  if (knob == RA_KNOB_DEBUG_FLAGS) {
    if (value < 0 || value > 7) return RA_ERR_INVALID_ARG;  // bits 0, 1 and 2
    g_debug_flags = (int)value;
    return RA_OK;
  }
  if (knob == RA_KNOB_DKDV_PAIR) {
    if (value < 0 || value > 1) return RA_ERR_INVALID_ARG;
    __atomic_store_n(&g_dkdv_pair, (int)value, __ATOMIC_RELAXED);
    return RA_OK;
  }
  return RA_ERR_INVALID_ARG;
}

ra_status ring_attn_timing_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing_on = on != 0;
  for (auto& t : g_timing) t.used = 0;
  return RA_OK;
}

ra_status ring_attn_timing_read(int32_t kernel, double* total_ms, int64_t* launches) {
  if (kernel < 0 || kernel >= RA_KERNEL_COUNT || !total_ms || !launches) return RA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  TimingSlot& t = g_timing[kernel];
  double sum = 0.0;
  for (size_t i = 0; i < t.used; ++i) {
    if (cudaEventSynchronize(t.pool[i].second) != cudaSuccess) return RA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.pool[i].first, t.pool[i].second) != cudaSuccess) return RA_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *launches = (int64_t)t.used;
  t.used = 0;
  return RA_OK;
}

const char* ra_status_string(int32_t status) {
  switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_INVALID_ARG: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported configuration";
    case RA_ERR_ALIGNMENT: return "stride or pointer alignment unusable for TMA tiles";
    case RA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case RA_ERR_CUDA: return "CUDA runtime error";
    case RA_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case RA_ERR_DEVICE: return "device-side error";
    case RA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the library's static array holds";
    default: return "unknown status";
  }
}

int32_t ring_attn_version(void) { return 200; }

int32_t ring_attn_debug_bounds(void) {
#ifdef RA_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"
