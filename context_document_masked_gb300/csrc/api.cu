// C ABI of libfcp (see include/fcp.h): argument validation, TMA descriptor
// encoding and kernel launches. Every check runs on the host before any
// launch; nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "plan.h"

namespace {

using fcp::Plan;

int64_t g_wait_ns = 2000000000LL;  // bounded device waits give up after 2 s

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

// Token-major [rows][heads][d] 16-bit tensor, boxes of 64 x 1 x 128 with the
// 128-byte swizzle (one swizzle panel of a 128-row tile).
bool make_map(CUtensorMap* m, const void* ptr, int d, int heads, int64_t rows, bool f16 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows][heads][d] tensor, boxes of 32 x 1 x 128 with the 128-byte
// swizzle: the target of the backward's dQ reduce-adds.
bool make_map_f32(CUtensorMap* m, void* ptr, int d, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)heads * d * 4};
  cuuint32_t box[3] = {32, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 [rows][heads][d] tensor (one byte per element), boxes of d x 1 x 128
// (d = 128: one 128-byte swizzled row per key or query).
bool make_map_u8(CUtensorMap* m, void* ptr, int d, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)heads * d};
  cuuint32_t box[3] = {(cuuint32_t)d, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

const int32_t* table(const fcp_dev_plan* dp, int tb) { return dp->base + dp->tables[tb]; }

// Host copy of a table entry (the serialized tables live in the plan).
int32_t host_at(const Plan* p, int tb, int64_t i) { return p->dev[p->tab_off[tb] + i]; }

int check_dims(const fcp_dims& d, const Plan* p) {
  if (d.T <= 0 || d.hq <= 0 || d.hkv <= 0) return FCP_ERR_INVALID_ARG;
  if (d.d != 64 && d.d != 128) return FCP_ERR_UNSUPPORTED;
  if (d.hq % d.hkv != 0) return FCP_ERR_UNSUPPORTED;
  if (p && d.T != p->T) return FCP_ERR_INVALID_ARG;
  return FCP_OK;
}

float softmax_scale(const fcp_dims& d) { return d.scale > 0.f ? d.scale : 1.0f / std::sqrt((float)d.d); }

int64_t remote_rows_of(const Plan* p, int32_t shard) {
  return shard < 0 ? p->total_remote : p->shards[shard].remote_rows;
}

}  // namespace

namespace fcp {
int64_t wait_limit_ns() { return g_wait_ns; }

// A device-plan handle must describe its host plan exactly: the kernels index
// the device tables with these offsets and counts, so a handle that was
// corrupted, hand-edited or bound to another plan is rejected before anything
// is launched.
int check_dev_plan(const fcp_dev_plan* dp, int32_t shard) {
  if (!dp || !dp->host || !dp->base) return FCP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dp->base) & 15) != 0) return FCP_ERR_INVALID_ARG;
  const Plan* p = dp->host;
  if (dp->n_shards != p->N || (int64_t)dp->T != p->T || dp->total_remote_rows != p->total_remote ||
      dp->bytes != (int64_t)p->dev.size() * 4)
    return FCP_ERR_INVALID_ARG;
  for (int t = 0; t < fcp::TB_COUNT; ++t)
    if (dp->tables[t] != p->tab_off[t] || dp->counts[t] != p->tab_cnt[t]) return FCP_ERR_INVALID_ARG;
  for (int t = fcp::TB_COUNT; t < 16; ++t)
    if (dp->tables[t] != 0 || dp->counts[t] != 0) return FCP_ERR_INVALID_ARG;
  if (shard < -1 || shard >= dp->n_shards) return FCP_ERR_INVALID_ARG;
  return FCP_OK;
}
}  // namespace fcp

using fcp::check_dev_plan;

extern "C" {

const char* fcp_strerror(int s) {
  switch (s) {
    case FCP_OK: return "ok";
    case FCP_ERR_INVALID_ARG: return "invalid argument";
    case FCP_ERR_UNSUPPORTED: return "unsupported shape";
    case FCP_ERR_CUDA: return "CUDA error";
    case FCP_ERR_TIMEOUT: return "bounded device wait expired";
    case FCP_ERR_INFEASIBLE: return "policy infeasible for this input";
    case FCP_ERR_CAPACITY: return "buffer too small";
    case FCP_ERR_MISSING_PART: return "partial result missing or duplicated";
    default: return "unknown status";
  }
}

int fcp_plan(const int32_t* doclens, int32_t n_docs, int32_t cp, int32_t policy,
             double target_imbalance, fcp_plan_t** out) {
  if (!out) return FCP_ERR_INVALID_ARG;
  *out = nullptr;
  return fcp::make_plan(doclens, n_docs, cp, policy, target_imbalance, out);
}

void fcp_plan_free(fcp_plan_t* plan) { delete plan; }

int fcp_plan_shard(const fcp_plan_t* plan, int32_t shard, fcp_shard_view* out) {
  if (!plan || !out || shard < 0 || shard >= plan->N) return FCP_ERR_INVALID_ARG;
  const fcp::Shard& s = plan->shards[shard];
  static_assert(sizeof(fcp::Piece) == sizeof(fcp_range), "piece layout");
  out->n_pieces = (int32_t)s.pieces.size();
  out->pieces = reinterpret_cast<const fcp_range*>(s.pieces.data());
  out->n_need = (int32_t)s.kv_need.size();
  out->kv_need = s.kv_need.data();
  out->n_remote = (int32_t)s.kv_remote.size();
  out->kv_remote = s.kv_remote.data();
  out->tokens = s.tokens;
  out->useful_pairs = s.W;
  out->remote_rows = s.remote_rows;
  out->kbuf_base = s.kbuf_base;
  out->fwd_tiles = s.fwd_tiles;
  out->fwd_qtiles = s.fwd_qtiles;
  out->fwd_masked = s.fwd_masked;
  out->bwd_tiles = s.bwd_tiles;
  out->bwd_ktiles = s.bwd_ktiles;
  return FCP_OK;
}

int fcp_plan_query_indices(const fcp_plan_t* plan, int32_t shard, int32_t* idx, int64_t cap,
                           int64_t* n) {
  if (!plan || !n || shard < 0 || shard >= plan->N || cap < 0) return FCP_ERR_INVALID_ARG;
  const fcp::Shard& s = plan->shards[shard];
  *n = s.tokens;
  if (cap < s.tokens) return FCP_ERR_CAPACITY;
  if (!idx && s.tokens > 0) return FCP_ERR_INVALID_ARG;
  int64_t k = 0;
  for (const fcp::Piece& p : s.pieces)
    for (int32_t t = p.start; t < p.end; ++t) idx[k++] = t;
  return FCP_OK;
}

int fcp_plan_stats(const fcp_plan_t* plan, fcp_plan_stats_t* out) {
  if (!plan || !out) return FCP_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->cp = plan->N;
  out->n_docs = (int32_t)plan->D.size();
  out->T = plan->T;
  out->imbalance = plan->imbalance;
  for (const fcp::Shard& s : plan->shards) {
    out->max_pairs = std::max(out->max_pairs, s.W);
    out->total_pairs += s.W;
    out->remote_rows_total += s.remote_rows;
    out->remote_rows_max = std::max(out->remote_rows_max, s.remote_rows);
  }
  out->eq4_tokens = plan->eq4;
  out->eq5_tokens = plan->eq5;
  out->eq2_max_dev = plan->eq2dev;
  out->iterations = plan->iterations;
  for (uint8_t f : plan->per_doc) out->n_per_doc += f;
  return FCP_OK;
}

int fcp_plan_per_doc_flags(const fcp_plan_t* plan, int32_t* out, int32_t n_docs) {
  if (!plan || !out || n_docs != (int32_t)plan->D.size()) return FCP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_docs; ++i) out[i] = plan->per_doc[i];
  return FCP_OK;
}

int64_t fcp_plan_device_bytes(const fcp_plan_t* plan) {
  return plan ? (int64_t)plan->dev.size() * 4 : 0;
}

int fcp_plan_device_image(const fcp_plan_t* plan, void* dst, int64_t bytes) {
  if (!plan || !dst) return FCP_ERR_INVALID_ARG;
  const int64_t need = fcp_plan_device_bytes(plan);
  if (bytes < need) return FCP_ERR_CAPACITY;
  std::memcpy(dst, plan->dev.data(), (size_t)need);
  return FCP_OK;
}

int fcp_plan_bind(const fcp_plan_t* plan, const void* dev_buf, int64_t bytes, fcp_dev_plan* out) {
  if (!plan || !dev_buf || !out) return FCP_ERR_INVALID_ARG;
  if (!aligned16(dev_buf)) return FCP_ERR_INVALID_ARG;
  const int64_t need = fcp_plan_device_bytes(plan);
  if (bytes < need) return FCP_ERR_CAPACITY;
  std::memset(out, 0, sizeof(*out));
  out->host = plan;
  out->base = static_cast<const int32_t*>(dev_buf);
  out->bytes = need;
  out->n_shards = plan->N;
  out->T = (int32_t)plan->T;
  out->total_remote_rows = plan->total_remote;
  for (int t = 0; t < fcp::TB_COUNT; ++t) {
    out->tables[t] = plan->tab_off[t];
    out->counts[t] = plan->tab_cnt[t];
  }
  return FCP_OK;
}

int fcp_plan_upload(const fcp_plan_t* plan, void* dev_buf, int64_t bytes, void* stream,
                    fcp_dev_plan* out) {
  const int st = fcp_plan_bind(plan, dev_buf, bytes, out);
  if (st != FCP_OK) return st;
  if (cudaMemcpyAsync(dev_buf, plan->dev.data(), (size_t)out->bytes, cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCP_ERR_CUDA;
  return FCP_OK;
}

// Workspace layout (each region 256-byte aligned): [0, 256) error word (byte
// 0) and the persistent kernels' work counter (byte kWorkCounterOff); D_i
// (fp32 [Hq][T]); fp16 copies of Q and dO ([T][Hq][d] each, backward); fp16
// copies of V ([T][Hkv][d]) and of the received V rows ([R][Hkv][d], R = all
// shards' remote rows of the plan), the forward's P*V operands.
constexpr int64_t kWorkCounterOff = 64;

struct WsLayout {
  int64_t delta, q16, do16, v16, vb16, q8, k8, kb8, total;
};

// Header words of the e4m3 Q K^T forward: amax bits of Q and K, then their
// scales 2^kq and 2^kk.
constexpr int64_t kQkAmaxOff = 128;
constexpr int64_t kQkScaleOff = 136;
// Diagnostic counter of the forward: online-softmax rescales of O after a
// query tile's first key tile (one count per warp and event).
constexpr int64_t kRescaleCountOff = 192;

static int64_t ws_align(int64_t x) { return (x + 255) / 256 * 256; }

static WsLayout ws_layout(const fcp_dims& d, int64_t remote_rows) {
  const int64_t T = std::max(d.T, 0), hq = std::max(d.hq, 0), hkv = std::max(d.hkv, 0),
                dd = std::max(d.d, 0);
  WsLayout w;
  w.delta = 256;
  w.q16 = w.delta + ws_align(hq * T * 4);
  w.do16 = w.q16 + ws_align(T * hq * dd * 2);
  w.v16 = w.do16 + ws_align(T * hq * dd * 2);
  w.vb16 = w.v16 + ws_align(T * hkv * dd * 2);
  const int64_t R = std::max<int64_t>(remote_rows, 0);
  w.q8 = w.vb16 + ws_align(R * hkv * dd * 2);
  w.k8 = w.q8 + ws_align(T * hq * dd);
  w.kb8 = w.k8 + ws_align(T * hkv * dd);
  w.total = w.kb8 + ws_align(R * hkv * dd);
  return w;
}

int64_t fcp_workspace_bytes(fcp_dims dims, const fcp_plan_t* plan) {
  return ws_layout(dims, plan ? plan->total_remote : 0).total;
}

int fcp_gather_kv(const void* k, const void* v, const fcp_dev_plan* plan, int32_t shard,
                  int32_t hkv, int32_t d, void* kbuf, void* vbuf, void* stream) {
  int st = check_dev_plan(plan, shard);
  if (st) return st;
  if (hkv <= 0 || (d != 64 && d != 128)) return FCP_ERR_UNSUPPORTED;
  const Plan* p = plan->host;
  const int64_t rows = remote_rows_of(p, shard);
  if (rows == 0) return FCP_OK;
  if (!k || !v || !kbuf || !vbuf) return FCP_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kbuf) || !aligned16(vbuf)) return FCP_ERR_INVALID_ARG;
  int32_t t0 = 0, t1 = plan->counts[fcp::TB_COPY], shift = 0;
  if (shard >= 0) {
    t0 = host_at(p, fcp::TB_CSHARD, shard);
    t1 = host_at(p, fcp::TB_CSHARD, shard + 1);
    shift = (int32_t)p->shards[shard].kbuf_base;
  }
  return fcp::launch_gather(k, v, table(plan, fcp::TB_COPY) + 4 * t0, t1 - t0, shift,
                            (int64_t)hkv * d * 2, kbuf, vbuf, plan->T, (int32_t)rows, num_sms(),
                            static_cast<cudaStream_t>(stream));
}

// Forward over the plan's gathered key layout (ring < -1: own rows from K/V,
// received rows from kbuf/vbuf) or in ring order (ring >= -1: every needed key
// from its owner's rows of K/V, owners visited by ring distance; ring = -1 all
// of them in one pass, ring = s only the keys of owner (shard - s) mod N).
static int attn_fwd_impl(const void* q, const void* k, const void* v, const void* kbuf, const void* vbuf,
                         const fcp_dev_plan* plan, int32_t shard, int32_t kv_lo, int32_t kv_hi,
                         fcp_dims dims, int32_t out_dtype, void* out, float* lse, void* ws,
                         int64_t ws_bytes, void* stream, int32_t ring, bool qk8 = false) {
  const bool ring_order = ring >= -1;
  int st = check_dev_plan(plan, shard);
  if (st) return st;
  const Plan* p = plan->host;
  if ((st = check_dims(dims, p))) return st;
  if (!q || !k || !v || !out || !lse || !ws) return FCP_ERR_INVALID_ARG;
  if (out_dtype != FCP_OUT_BF16 && out_dtype != FCP_OUT_F32) return FCP_ERR_INVALID_ARG;
  if (kv_lo < 0 || kv_hi > dims.T || kv_lo > kv_hi) return FCP_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(dims, p->total_remote);
  if (ws_bytes < wl.total) return FCP_ERR_CAPACITY;
  if (ring_order && ring >= plan->n_shards) return FCP_ERR_INVALID_ARG;
  const int64_t rrows = ring_order ? 0 : remote_rows_of(p, shard);
  if (rrows > 0 && (!kbuf || !vbuf)) return FCP_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)out, (const void*)lse, (const void*)ws})
    if (!aligned16(ptr)) return FCP_ERR_INVALID_ARG;
  if (rrows > 0 && (!aligned16(kbuf) || !aligned16(vbuf))) return FCP_ERR_INVALID_ARG;

  // fp16 copies of V and of the received V rows: the P*V operands.
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* wsb = static_cast<char*>(ws);
  void* v16 = wsb + wl.v16;
  void* vb16 = wsb + wl.vb16;
  int* counter = reinterpret_cast<int*>(wsb + kWorkCounterOff);
  if (qk8) {
    // e4m3 copies of Q, K and the received K rows (with K's scale: they are
    // copies of K rows), each tensor with its own power-of-two scale.
    if (dims.d != 128) return FCP_ERR_UNSUPPORTED;
    unsigned* amax = reinterpret_cast<unsigned*>(wsb + kQkAmaxOff);
    float* scales = reinterpret_cast<float*>(wsb + kQkScaleOff);
    if (cudaMemsetAsync(amax, 0, 2 * sizeof(unsigned), cs) != cudaSuccess) return FCP_ERR_CUDA;
    int sq = fcp::launch_quant_e4m3(q, wsb + wl.q8, (int64_t)dims.T * dims.hq * dims.d, amax, scales,
                                    num_sms(), cs);
    if (sq == FCP_OK)
      sq = fcp::launch_quant_e4m3(k, wsb + wl.k8, (int64_t)dims.T * dims.hkv * dims.d, amax + 1, scales + 1,
                                  num_sms(), cs);
    if (sq == FCP_OK && rrows > 0)
      sq = fcp::launch_quant_e4m3_with(kbuf, wsb + wl.kb8, rrows * dims.hkv * dims.d, amax + 1, num_sms(), cs);
    if (sq) return sq;
  }
  int st2 = fcp::launch_convert_f16(v, v16, (int64_t)dims.T * dims.hkv * dims.d, static_cast<int*>(ws),
                                    counter, num_sms(), cs);
  if (st2 == FCP_OK && rrows > 0)
    st2 = fcp::launch_convert_f16(vbuf, vb16, rrows * dims.hkv * dims.d, static_cast<int*>(ws), nullptr,
                                  num_sms(), cs);
  if (st2) return st2;

  fcp::FwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  bool ok = make_map(&a.tm_v, v16, dims.d, dims.hkv, dims.T, true);
  if (qk8) {
    ok = ok && make_map_u8(&a.tm_q, wsb + wl.q8, dims.d, dims.hq, dims.T) &&
         make_map_u8(&a.tm_k, wsb + wl.k8, dims.d, dims.hkv, dims.T) &&
         make_map_u8(&a.tm_kb, rrows > 0 ? wsb + wl.kb8 : wsb + wl.k8, dims.d, dims.hkv, rrows > 0 ? rrows : dims.T);
  } else {
    ok = ok && make_map(&a.tm_q, q, dims.d, dims.hq, dims.T) && make_map(&a.tm_k, k, dims.d, dims.hkv, dims.T) &&
         make_map(&a.tm_kb, rrows > 0 ? kbuf : k, dims.d, dims.hkv, rrows > 0 ? rrows : dims.T);
  }
  ok = ok && make_map(&a.tm_vb, rrows > 0 ? vb16 : v16, dims.d, dims.hkv, rrows > 0 ? rrows : dims.T, true);
  if (!ok) return FCP_ERR_CUDA;
  a.qk8 = qk8;
  fcp::FwdParams& fp = a.p;
  fp.pieces = table(plan, ring_order ? fcp::TB_RPIECES : fcp::TB_PIECES);
  fp.segs = table(plan, ring_order ? fcp::TB_RSEGS : fcp::TB_SEGS);
  fp.seg_filter = ring_order ? ring : -1;
  fp.tiles = table(plan, fcp::TB_FTILES);
  if (shard < 0) {
    fp.order = table(plan, fcp::TB_FORDER);
    fp.n_items = plan->counts[fcp::TB_FTILES];
    fp.kbuf_shift = 0;
  } else {
    const int32_t t0 = host_at(p, fcp::TB_FSHARD, shard), t1 = host_at(p, fcp::TB_FSHARD, shard + 1);
    fp.order = table(plan, fcp::TB_IDENT) + t0;
    fp.n_items = t1 - t0;
    fp.kbuf_shift = ring_order ? 0 : (int32_t)p->shards[shard].kbuf_base;
  }
  fp.kv_lo = kv_lo;
  fp.kv_hi = kv_hi;
  fp.T = dims.T;
  fp.hq = dims.hq;
  fp.hkv = dims.hkv;
  fp.scale_log2 = softmax_scale(dims) * 1.4426950408889634f;
  fp.out_f32 = out_dtype == FCP_OUT_F32;
  fp.out = out;
  fp.lse = lse;
  fp.err = static_cast<int*>(ws);
  fp.work_counter = counter;
  fp.qk_scale = qk8 ? reinterpret_cast<const float*>(wsb + kQkScaleOff) : nullptr;
  fp.rescale_count = reinterpret_cast<int*>(wsb + kRescaleCountOff);
  fp.n_tiles = plan->counts[fcp::TB_FTILES];
  fp.n_pieces = plan->counts[ring_order ? fcp::TB_RPIECES : fcp::TB_PIECES];
  fp.n_segs = plan->counts[ring_order ? fcp::TB_RSEGS : fcp::TB_SEGS];
  fp.kb_rows = rrows > 0 ? (int32_t)rrows : dims.T;
  fp.wait_ns = g_wait_ns;
  a.d = dims.d;
  a.num_sms = num_sms();
  return fcp::launch_attn_fwd(a, cs);
}

int fcp_attn_fwd(const void* q, const void* k, const void* v, const void* kbuf, const void* vbuf,
                 const fcp_dev_plan* plan, int32_t shard, int32_t kv_lo, int32_t kv_hi,
                 fcp_dims dims, int32_t out_dtype, void* out, float* lse, void* ws,
                 int64_t ws_bytes, void* stream) {
  return attn_fwd_impl(q, k, v, kbuf, vbuf, plan, shard, kv_lo, kv_hi, dims, out_dtype, out, lse, ws,
                       ws_bytes, stream, -2);
}

int fcp_attn_fwd_qk8(const void* q, const void* k, const void* v, const void* kbuf, const void* vbuf,
                     const fcp_dev_plan* plan, int32_t shard, int32_t kv_lo, int32_t kv_hi, fcp_dims dims,
                     int32_t out_dtype, void* out, float* lse, void* ws, int64_t ws_bytes, void* stream) {
  return attn_fwd_impl(q, k, v, kbuf, vbuf, plan, shard, kv_lo, kv_hi, dims, out_dtype, out, lse, ws,
                       ws_bytes, stream, -2, true);
}

int fcp_quant_e4m3(const void* x, int64_t n, void* out, float* scale_out, void* scratch, void* stream) {
  if (n < 0 || n % 8 != 0) return FCP_ERR_INVALID_ARG;
  if (n == 0) return FCP_OK;
  if (!x || !out || !scale_out || !scratch) return FCP_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(out) & 7) || (reinterpret_cast<uintptr_t>(scratch) & 3))
    return FCP_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned), cs) != cudaSuccess) return FCP_ERR_CUDA;
  return fcp::launch_quant_e4m3(x, out, n, static_cast<unsigned*>(scratch), scale_out, num_sms(), cs);
}

int fcp_round_bf16(const float* x, int64_t n, void* out, void* stream) {
  if (n < 0 || n % 8 != 0) return FCP_ERR_INVALID_ARG;
  if (n == 0) return FCP_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return FCP_ERR_INVALID_ARG;
  return fcp::launch_round_bf16(x, out, n, num_sms(), static_cast<cudaStream_t>(stream));
}

int fcp_attn_fwd_ring(const void* q, const void* k, const void* v, const fcp_dev_plan* plan,
                      int32_t shard, int32_t ring_step, fcp_dims dims, int32_t out_dtype, void* out,
                      float* lse, void* ws, int64_t ws_bytes, void* stream) {
  if (ring_step < -1) return FCP_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, nullptr, nullptr, plan, shard, 0, dims.T, dims, out_dtype, out, lse, ws,
                       ws_bytes, stream, ring_step);
}

int fcp_merge(const float* o_parts, const float* lse_parts, int32_t B, int64_t rows, int32_t hq,
              int32_t d, void* out, float* lse_out, void* stream) {
  if (B < 1 || rows < 0 || hq < 1) return FCP_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FCP_ERR_UNSUPPORTED;
  if (B > d / 4 || rows * hq >= (int64_t(1) << 30)) return FCP_ERR_UNSUPPORTED;
  if (rows == 0) return FCP_OK;
  if (!o_parts || !lse_parts || !out || !lse_out) return FCP_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(out)) return FCP_ERR_INVALID_ARG;
  return fcp::launch_merge(o_parts, lse_parts, B, rows, hq, d, out, lse_out, num_sms(),
                           static_cast<cudaStream_t>(stream));
}

int fcp_merge_ring(const fcp_dev_plan* plan, const float* o_parts, const float* lse_parts,
                   const int32_t* part_step, int32_t B, int32_t hq, int32_t d, void* out, float* lse_out,
                   void* stream) {
  int st = check_dev_plan(plan, -1);
  if (st) return st;
  if (!part_step && B > 0) return FCP_ERR_INVALID_ARG;
  const int32_t N = plan->n_shards;
  if (B != N) return FCP_ERR_MISSING_PART;
  std::vector<uint8_t> seen(N, 0);
  for (int32_t b = 0; b < B; ++b) {
    const int32_t s = part_step[b];
    if (s < 0 || s >= N || seen[s]) return FCP_ERR_MISSING_PART;
    seen[s] = 1;
  }
  return fcp_merge(o_parts, lse_parts, B, plan->T, hq, d, out, lse_out, stream);
}

int fcp_attn_bwd(const void* q, const void* k, const void* v, const void* kbuf, const void* vbuf,
                 const void* out, int32_t out_dtype, const float* lse, const void* dout,
                 const fcp_dev_plan* plan, int32_t shard, fcp_dims dims, float* dq, float* dk,
                 float* dv, void* ws, int64_t ws_bytes, void* stream) {
  int st = check_dev_plan(plan, shard);
  if (st) return st;
  const Plan* p = plan->host;
  if ((st = check_dims(dims, p))) return st;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !ws) return FCP_ERR_INVALID_ARG;
  if (out_dtype != FCP_OUT_BF16 && out_dtype != FCP_OUT_F32) return FCP_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(dims, p->total_remote);
  if (ws_bytes < wl.total) return FCP_ERR_CAPACITY;
  const int64_t rrows = remote_rows_of(p, shard);
  if (rrows > 0 && (!kbuf || !vbuf)) return FCP_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, out, (const void*)lse, dout, (const void*)dq, (const void*)dk,
                          (const void*)dv, (const void*)ws})
    if (!aligned16(ptr)) return FCP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* wsb = static_cast<char*>(ws);
  float* delta = reinterpret_cast<float*>(wsb + wl.delta);
  void* q16 = wsb + wl.q16;
  void* do16 = wsb + wl.do16;

  // Row statistics D_i and dQ = 0 for the shard's query rows.
  int32_t r0 = 0, r1 = plan->counts[fcp::TB_ROWS];
  if (shard >= 0) {
    r0 = host_at(p, fcp::TB_RSHARD, shard);
    r1 = host_at(p, fcp::TB_RSHARD, shard + 1);
  }
  st = fcp::launch_bwd_preprocess(out, out_dtype == FCP_OUT_F32, dout, q, table(plan, fcp::TB_ROWS),
                                  table(plan, fcp::TB_IDENT) + r0, r1 - r0, plan->counts[fcp::TB_ROWS], dims.T,
                                  dims.hq, dims.d,
                                  delta, dq, q16, do16, static_cast<int*>(ws),
                                  reinterpret_cast<int*>(wsb + kWorkCounterOff), s);
  if (st) return st;

  fcp::BwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  bool ok = make_map(&a.tm_q, q16, dims.d, dims.hq, dims.T, true) &&
            make_map(&a.tm_do, do16, dims.d, dims.hq, dims.T, true) &&
            make_map(&a.tm_k, k, dims.d, dims.hkv, dims.T) && make_map(&a.tm_v, v, dims.d, dims.hkv, dims.T) &&
            make_map_f32(&a.tm_dq, dq, dims.d, dims.hq, dims.T) &&
            make_map_f32(&a.tm_dk, dk, dims.d, dims.hkv, dims.T) &&
            make_map_f32(&a.tm_dv, dv, dims.d, dims.hkv, dims.T);
  if (rrows > 0)
    ok = ok && make_map(&a.tm_kb, kbuf, dims.d, dims.hkv, rrows) &&
         make_map(&a.tm_vb, vbuf, dims.d, dims.hkv, rrows);
  else
    ok = ok && make_map(&a.tm_kb, k, dims.d, dims.hkv, dims.T) && make_map(&a.tm_vb, v, dims.d, dims.hkv, dims.T);
  if (!ok) return FCP_ERR_CUDA;
  fcp::BwdParams& bp = a.p;
  bp.pieces = table(plan, fcp::TB_PIECES);
  bp.tiles = table(plan, fcp::TB_BTILES);
  if (shard < 0) {
    bp.order = table(plan, fcp::TB_BORDER);
    bp.n_items = plan->counts[fcp::TB_BTILES];
    bp.kbuf_shift = 0;
  } else {
    const int32_t t0 = host_at(p, fcp::TB_BSHARD, shard), t1 = host_at(p, fcp::TB_BSHARD, shard + 1);
    bp.order = table(plan, fcp::TB_IDENT) + t0;
    bp.n_items = t1 - t0;
    bp.kbuf_shift = (int32_t)p->shards[shard].kbuf_base;
  }
  bp.T = dims.T;
  bp.hq = dims.hq;
  bp.hkv = dims.hkv;
  bp.scale = softmax_scale(dims);
  bp.scale_log2 = bp.scale * 1.4426950408889634f;
  bp.lse = lse;
  bp.delta = delta;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  bp.err = static_cast<int*>(ws);
  bp.work_counter = reinterpret_cast<int*>(wsb + kWorkCounterOff);
  bp.n_tiles = plan->counts[fcp::TB_BTILES];
  bp.kb_rows = rrows > 0 ? (int32_t)rrows : dims.T;
  bp.wait_ns = g_wait_ns;
  a.d = dims.d;
  a.num_sms = num_sms();
  return fcp::launch_attn_bwd(a, s);
}

int fcp_get_device_status(void* ws, void* stream) {
  if (!ws) return FCP_ERR_INVALID_ARG;
  int word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FCP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FCP_ERR_CUDA;
  if (word == 0) return FCP_OK;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return FCP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FCP_ERR_CUDA;
  if (word & 1) return FCP_ERR_TIMEOUT;
  if (word & 4) return FCP_ERR_UNSUPPORTED;  // an input exceeds the fp16 operand range
  if (word & fcp::kErrBadTable) return FCP_ERR_INVALID_ARG;  // checked build: a table index out of range
  return FCP_ERR_CUDA;
}

void fcp_debug_set_wait_limit(int64_t ns) { g_wait_ns = ns == 0 ? 2000000000LL : ns; }

int fcp_debug_rescale_events(void* ws, void* stream, int64_t* count) {
  if (!ws || !count) return FCP_ERR_INVALID_ARG;
  int word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* counter = static_cast<char*>(ws) + kRescaleCountOff;
  if (cudaMemcpyAsync(&word, counter, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FCP_ERR_CUDA;
  if (cudaMemsetAsync(counter, 0, sizeof(int), s) != cudaSuccess) return FCP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FCP_ERR_CUDA;
  *count = word;
  return FCP_OK;
}

}  // extern "C"
