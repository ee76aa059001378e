// fcp_attn_fwd_noalloc: the attention forward for callers that must not
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving or training
// process that reserves all device memory up front (or hands it to another
// allocator) and forbids any allocation on its request path, where a
// cudaMalloc would synchronise the device and may fail once memory is
// fragmented. For them this entry point keeps its scratch (the error word and
// the fp16 copies of V and of the received V rows that the P*V product reads)
// in one file-scope device array, sized once when the library is loaded.
//
// The array lives on every GPU that loads the library until the process
// exits. Every call shares it: the error word is cleared at the start of each
// call and the fp16 copies are fully rewritten before they are read, but two
// calls whose work overlaps on the GPU (different streams, no ordering between
// them) race on the array and must not be issued.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "plan.h"

namespace {

// Scratch of the allocation-free forward (FCP_NOALLOC_SCRATCH_BYTES bytes).
static __device__ __align__(256) unsigned char g_fwd_scratch[FCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (host code only sees a host-side stand-in under the array's name).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FCP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return FCP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FCP_OK;
}

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

bool make_map(CUtensorMap* m, const void* ptr, int d, int heads, int64_t rows, bool f16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

extern "C" int fcp_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* kbuf,
                                    const void* vbuf, const fcp_dev_plan* plan, int32_t shard,
                                    int32_t kv_lo, int32_t kv_hi, fcp_dims dims, int32_t out_dtype,
                                    void* out, float* lse, void* stream) {
  if (int st0 = fcp::check_dev_plan(plan, shard)) return st0;
  const fcp::Plan* p = plan->host;
  if (dims.T <= 0 || dims.hq <= 0 || dims.hkv <= 0 || dims.T != p->T) return FCP_ERR_INVALID_ARG;
  if (dims.d != 64 && dims.d != 128) return FCP_ERR_UNSUPPORTED;
  if (dims.hq % dims.hkv != 0) return FCP_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out || !lse) return FCP_ERR_INVALID_ARG;
  if (out_dtype != FCP_OUT_BF16 && out_dtype != FCP_OUT_F32) return FCP_ERR_INVALID_ARG;
  if (kv_lo < 0 || kv_hi > dims.T || kv_lo > kv_hi) return FCP_ERR_INVALID_ARG;
  const int64_t rrows = shard < 0 ? p->total_remote : p->shards[shard].remote_rows;
  if (rrows > 0 && (!kbuf || !vbuf)) return FCP_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, (const void*)out, (const void*)lse})
    if (!aligned16(ptr)) return FCP_ERR_INVALID_ARG;
  if (rrows > 0 && (!aligned16(kbuf) || !aligned16(vbuf))) return FCP_ERR_INVALID_ARG;

  // Scratch layout: error word (byte 0) and the forward kernel's work counter
  // (byte 64) in the first 256 bytes, fp16 V [T][Hkv][d], fp16 received V
  // [rrows][Hkv][d].
  const int64_t v16_off = 256;
  const int64_t vb16_off = v16_off + align256((int64_t)dims.T * dims.hkv * dims.d * 2);
  const int64_t need = vb16_off + align256(rrows * dims.hkv * dims.d * 2);
  if (need > (int64_t)FCP_NOALLOC_SCRATCH_BYTES) return FCP_ERR_CAPACITY;

  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st) return st;
  char* base = static_cast<char*>(scratch);
  int* err = reinterpret_cast<int*>(base);
  void* v16 = base + v16_off;
  void* vb16 = base + vb16_off;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(err, 0, sizeof(int), cs) != cudaSuccess) return FCP_ERR_CUDA;
  int* counter = reinterpret_cast<int*>(base + 64);  // the forward kernel's work counter
  st = fcp::launch_convert_f16(v, v16, (int64_t)dims.T * dims.hkv * dims.d, err, counter, num_sms(), cs);
  if (st == FCP_OK && rrows > 0)
    st = fcp::launch_convert_f16(vbuf, vb16, rrows * dims.hkv * dims.d, err, nullptr, num_sms(), cs);
  if (st) return st;

  fcp::FwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  bool ok = make_map(&a.tm_q, q, dims.d, dims.hq, dims.T, false) &&
            make_map(&a.tm_k, k, dims.d, dims.hkv, dims.T, false) &&
            make_map(&a.tm_v, v16, dims.d, dims.hkv, dims.T, true);
  if (rrows > 0)
    ok = ok && make_map(&a.tm_kb, kbuf, dims.d, dims.hkv, rrows, false) &&
         make_map(&a.tm_vb, vb16, dims.d, dims.hkv, rrows, true);
  else
    ok = ok && make_map(&a.tm_kb, k, dims.d, dims.hkv, dims.T, false) &&
         make_map(&a.tm_vb, v16, dims.d, dims.hkv, dims.T, true);
  if (!ok) return FCP_ERR_CUDA;
  const int32_t* tb = plan->base;
  fcp::FwdParams& fp = a.p;
  fp.pieces = tb + plan->tables[fcp::TB_PIECES];
  fp.segs = tb + plan->tables[fcp::TB_SEGS];
  fp.tiles = tb + plan->tables[fcp::TB_FTILES];
  if (shard < 0) {
    fp.order = tb + plan->tables[fcp::TB_FORDER];
    fp.n_items = plan->counts[fcp::TB_FTILES];
    fp.kbuf_shift = 0;
  } else {
    const int32_t t0 = p->dev[p->tab_off[fcp::TB_FSHARD] + shard];
    const int32_t t1 = p->dev[p->tab_off[fcp::TB_FSHARD] + shard + 1];
    fp.order = tb + plan->tables[fcp::TB_IDENT] + t0;
    fp.n_items = t1 - t0;
    fp.kbuf_shift = (int32_t)p->shards[shard].kbuf_base;
  }
  fp.kv_lo = kv_lo;
  fp.kv_hi = kv_hi;
  fp.seg_filter = -1;
  fp.T = dims.T;
  fp.hq = dims.hq;
  fp.hkv = dims.hkv;
  const float scale = dims.scale > 0.f ? dims.scale : 1.0f / std::sqrt((float)dims.d);
  fp.scale_log2 = scale * 1.4426950408889634f;
  fp.out_f32 = out_dtype == FCP_OUT_F32;
  fp.out = out;
  fp.lse = lse;
  fp.err = err;
  fp.work_counter = counter;
  fp.rescale_count = nullptr;
  fp.n_tiles = plan->counts[fcp::TB_FTILES];
  fp.n_pieces = plan->counts[fcp::TB_PIECES];
  fp.n_segs = plan->counts[fcp::TB_SEGS];
  fp.kb_rows = rrows > 0 ? (int32_t)rrows : dims.T;
  fp.wait_ns = fcp::wait_limit_ns();
  a.d = dims.d;
  a.num_sms = num_sms();
  return fcp::launch_attn_fwd(a, cs);
}
