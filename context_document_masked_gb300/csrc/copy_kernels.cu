// Bandwidth-bound kernels of libfcp: the sharding-aware KV gather, the
// (O, LSE) merge of partial results, and the backward row statistics.
//
// All three move contiguous rows with 128-bit loads and stores, several
// independent loads in flight per thread, and grids sized in multiples of the
// SM count.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace fcp {

namespace {

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ gather
// "FlashCP" §3.2: each shard receives only the prefix keys of its documents
// held by other shards, compacted into one contiguous buffer. A task copies
// `nrows` consecutive rows (contiguous in source and destination) of K and V.
constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                  const int32_t* __restrict__ tasks, int32_t n_tasks, int32_t dst_shift,
                  int64_t row_vecs, uint4* __restrict__ kbuf, uint4* __restrict__ vbuf, int32_t src_rows,
                  int32_t dst_rows) {
  for (int t = blockIdx.x; t < n_tasks; t += gridDim.x) {
    const int src = __ldg(tasks + 4 * t + 0);
    const int dst = __ldg(tasks + 4 * t + 1) - dst_shift;
    const int nrows = __ldg(tasks + 4 * t + 2);
    // Checked build: a run outside K/V or outside the destination buffer is
    // skipped (the call has no error word; the attention kernels that read
    // the same plan report such tables).
    if (kDeviceChecks && (nrows < 0 || src < 0 || src > src_rows - nrows || dst < 0 || dst > dst_rows - nrows))
      continue;
    const int64_t n = (int64_t)nrows * row_vecs;
    const uint4* ks = k + (int64_t)src * row_vecs;
    const uint4* vs = v + (int64_t)src * row_vecs;
    uint4* kd = kbuf + (int64_t)dst * row_vecs;
    uint4* vd = vbuf + (int64_t)dst * row_vecs;
    const int64_t step = (int64_t)kGatherThreads * kGatherUnroll;
    for (int64_t base = threadIdx.x; base < n; base += step) {
      uint4 a[kGatherUnroll], b[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kGatherThreads;
        if (i < n) {
          a[u] = __ldg(ks + i);
          b[u] = __ldg(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kGatherThreads;
        if (i < n) {
          kd[i] = a[u];
          vd[i] = b[u];
        }
      }
    }
  }
}

// ------------------------------------------------------------------- merge
// "LLM Context Parallel in Production", "Core Principle" / "Ring Attention":
// LSE = ln sum_b exp(LSE_b), O = sum_b exp(LSE_b - LSE) O_b.
//
// A warp takes G = 32 / BP consecutive rows of one head (BP = B rounded up to
// a power of two). Weight phase: lane (u, b) reads part b's LSE of row u, the
// max and the sum reduce over BP lanes (log2 BP shuffles), and each lane keeps
// its normalised weight exp(LSE_b - LSE); lane (u, 0) writes LSE. Data phase:
// row by row, D/4 lanes stream one float4 each of every non-empty part (four
// parts' loads in flight at a time) with the weight shuffled from lane (u, b).
// Parts whose LSE is -inf (no key of that block visible) are not read.
constexpr int kMergeThreads = 256;

template <int D, int BP>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const float4* __restrict__ o_parts, const float* __restrict__ lse_parts, int B,
                 int rows, int hq, uint2* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int V = D / 4;               // lanes (float4) per (row, head): 32 or 16
  constexpr int kRowsPerPass = 32 / V;   // rows one data pass covers
  constexpr int G = 32 / BP;             // rows per weight phase
  static_assert(G >= kRowsPerPass, "B too large for this head dimension");
  const float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const int wu = lane / BP, wb = lane % BP;   // weight phase: row in the group, part
  const int vec = lane % V, sub = lane / V;   // data phase: float4 of the row, row in the pass
  const int h = blockIdx.y;                   // one query head per grid row
  const int64_t lstride = (int64_t)hq * rows;
  const int64_t part_stride = (int64_t)rows * hq * V;  // float4 between consecutive parts
  const float* lse_h = lse_parts + (int64_t)h * rows;
  float* lse_o = lse_out + (int64_t)h * rows;
  const int rstep = gridDim.x * (kMergeThreads / 32) * G;
  int r0 = (blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5)) * G;
  // Neighbouring warps read neighbouring rows of the same LSE lines; the next
  // group's LSEs are fetched while this group's O parts stream.
  auto lse_at = [&](int base) {
    const int r = base + wu;
    return (r < rows && wb < B) ? __ldg(lse_h + wb * lstride + r) : -INFINITY;
  };
  float l_next = lse_at(r0);
  for (; r0 < rows; r0 += rstep) {
    const float l = l_next;
    l_next = lse_at(r0 + rstep);
    float m = l;
#pragma unroll
    for (int o = 1; o < BP; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float w = (l == -INFINITY) ? 0.f : ex2f((l - m) * kLog2e);
    float tw = w;
#pragma unroll
    for (int o = 1; o < BP; o <<= 1) tw += __shfl_xor_sync(0xffffffffu, tw, o);
    // A row with no visible key anywhere (all parts empty) has m = -inf:
    // zero output and LSE -inf.
    w = (m == -INFINITY) ? 0.f : w * (1.f / tw);
    if (wb == 0 && r0 + wu < rows) lse_o[r0 + wu] = (m == -INFINITY) ? -INFINITY : m + logf(tw);
    // Bit u * BP + b: part b of row u has a nonzero weight.
    const uint32_t nz = __ballot_sync(0xffffffffu, w != 0.f);
#pragma unroll 2
    for (int u0 = 0; u0 < G; u0 += kRowsPerPass) {
      const int u = u0 + sub;
      const int row = r0 + u;
      const float4* op = o_parts + ((int64_t)row * hq + h) * V + vec;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (kRowsPerPass == 1) {
        // One row per pass (d = 128): the row's nonzero parts are the same in
        // every lane, so empty parts cost neither a shuffle nor a load, and
        // an empty group of four costs nothing.
        const uint32_t rb = (nz >> (u * BP)) & (BP == 32 ? 0xffffffffu : ((1u << BP) - 1u));
        for (int b0 = 0; b0 < B; b0 += 4) {
          const uint32_t g = (rb >> b0) & 0xFu;
          if (g == 0) continue;
          float wk[4];
          float4 o[4];
          const float4* opb = op + b0 * part_stride;
#pragma unroll
          for (int k = 0; k < 4; ++k) wk[k] = (g >> k) & 1u ? __shfl_sync(0xffffffffu, w, u * BP + b0 + k) : 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o[k] = (g >> k) & 1u ? __ldg(opb + k * part_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc.x = fmaf(wk[k], o[k].x, acc.x);
            acc.y = fmaf(wk[k], o[k].y, acc.y);
            acc.z = fmaf(wk[k], o[k].z, acc.z);
            acc.w = fmaf(wk[k], o[k].w, acc.w);
          }
        }
        if (row < rows) out[((int64_t)row * hq + h) * V + vec] = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
        continue;
      }
      for (int b0 = 0; b0 < B; b0 += 4) {
        float wk[4];
        float4 o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = __shfl_sync(0xffffffffu, w, u * BP + ((b0 + k) % BP));
          wk[k] = b0 + k < B ? x : 0.f;
        }
        // With more than one group of four parts, a group empty for every row
        // of the pass is skipped by the whole warp (a vote: with d = 64 a pass
        // covers two rows). Causal key blocks leave most rows' later groups
        // empty.
        if constexpr (BP > 4) {
          if (__all_sync(0xffffffffu, wk[0] == 0.f && wk[1] == 0.f && wk[2] == 0.f && wk[3] == 0.f)) continue;
        }
        // wk != 0 implies row < rows and part b0 + k non-empty.
        const float4* opb = op + b0 * part_stride;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          o[k] = wk[k] != 0.f ? __ldg(opb + k * part_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc.x = fmaf(wk[k], o[k].x, acc.x);
          acc.y = fmaf(wk[k], o[k].y, acc.y);
          acc.z = fmaf(wk[k], o[k].z, acc.z);
          acc.w = fmaf(wk[k], o[k].w, acc.w);
        }
      }
      if (row < rows) out[((int64_t)row * hq + h) * V + vec] = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
    }
  }
}

// ------------------------------------------------------- bwd preprocess
// D_i = <dO_i, O_i> (the row term of dS = P (dP - D)), dQ rows zeroed so the
// backward kernel can accumulate into them, and fp16 copies of Q and dO (the
// backward's tensor-core operands; exact for bf16 values inside the fp16
// range, error bit 4 otherwise).
constexpr int kPreThreads = 256;

__device__ __forceinline__ uint32_t cvt_pair(uint32_t x, bool& ovf) {
  const float lo = __uint_as_float(x << 16), hi = __uint_as_float(x & 0xFFFF0000u);
  ovf |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D, bool OF32>
__global__ void __launch_bounds__(kPreThreads)
    preprocess_kernel(const void* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                      const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ rows,
                      const int32_t* __restrict__ order, int n_chunks, int n_rows_table, int T, int hq,
                      float* __restrict__ delta, float* __restrict__ dq, __half* __restrict__ q16,
                      __half* __restrict__ do16, int* __restrict__ err, int* __restrict__ zero_word) {
  if (zero_word && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *zero_word = 0;
  // A chunk's rows, all heads, are one contiguous [rows][hq][D] block. Each
  // thread takes 8 consecutive elements (16-byte loads of dO and Q, 16 or 32
  // bytes of O); L = D / 8 lanes hold one (row, head) and reduce its D_i.
  constexpr int L = D / 8;
  const int lane = threadIdx.x & 31;
  const int stride = kPreThreads * gridDim.y;
  bool ovf = false;
  for (int c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const int chunk = __ldg(order + c);
    if constexpr (kDeviceChecks) {
      if (chunk < 0 || chunk >= n_rows_table) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadTable);
        continue;
      }
    }
    const int r0 = __ldg(rows + 2 * chunk), nr = __ldg(rows + 2 * chunk + 1);
    if constexpr (kDeviceChecks) {
      if (nr < 0 || r0 < 0 || r0 > T - nr) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadTable);
        continue;
      }
    }
    const int total = nr * hq * L;  // 16-byte groups of the chunk
    const int64_t e0 = (int64_t)r0 * hq * D;
    // Warp-uniform trip count: every lane of a warp takes part in the
    // shuffles; lanes past the end hold s = 0 and store nothing.
    for (int g = threadIdx.x + kPreThreads * blockIdx.y; g - lane < total; g += stride) {
      const bool live = g < total;
      const int64_t base = e0 + (int64_t)g * 8;
      uint4 b = make_uint4(0, 0, 0, 0), x = b;
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (live) {
        b = __ldg(reinterpret_cast<const uint4*>(dout + base));
        x = __ldg(reinterpret_cast<const uint4*>(q + base));
        if constexpr (OF32) {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(out) + base);
          const float4 a0 = __ldg(p), a1 = __ldg(p + 1);
          o[0] = a0.x; o[1] = a0.y; o[2] = a0.z; o[3] = a0.w;
          o[4] = a1.x; o[5] = a1.y; o[6] = a1.z; o[7] = a1.w;
        } else {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(out) + base));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(ws[i] << 16);
            o[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
          }
        }
      }
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w}, xw[4] = {x.x, x.y, x.z, x.w};
      uint32_t oq[4], od[4];
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s = fmaf(o[2 * i], __uint_as_float(bw[i] << 16), s);
        s = fmaf(o[2 * i + 1], __uint_as_float(bw[i] & 0xFFFF0000u), s);
        oq[i] = cvt_pair(xw[i], ovf);
        od[i] = cvt_pair(bw[i], ovf);
      }
      if (live) {
        *reinterpret_cast<uint4*>(q16 + base) = make_uint4(oq[0], oq[1], oq[2], oq[3]);
        *reinterpret_cast<uint4*>(do16 + base) = make_uint4(od[0], od[1], od[2], od[3]);
        float4* z = reinterpret_cast<float4*>(dq + base);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int m = L / 2; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
      if (live && (g % L) == 0) {
        const int u = g / L;  // (row, head) within the chunk
        delta[(int64_t)(u % hq) * T + r0 + u / hq] = s;
      }
    }
  }
  if (ovf) atomicOr(err, 4);
}

// ------------------------------------------------------- bf16 -> fp16
// fp16 copy of a bf16 tensor (exact inside the fp16 range; error bit 4 when a
// value exceeds it). The forward's P*V product runs on fp16 operands.
constexpr int kCvtThreads = 256;

__global__ void __launch_bounds__(kCvtThreads)
    convert_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n, int* err,
                   int* zero_word) {
  if (zero_word && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0;
  bool ovf = false;
  for (int64_t i = (int64_t)blockIdx.x * kCvtThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kCvtThreads) {
    uint4 x = __ldg(src + i);
    x.x = cvt_pair(x.x, ovf);
    x.y = cvt_pair(x.y, ovf);
    x.z = cvt_pair(x.z, ovf);
    x.w = cvt_pair(x.w, ovf);
    dst[i] = x;
  }
  if (ovf) atomicOr(err, 4);
}

// ------------------------------------------------------- fp32 -> bf16
// The final-output form of an fp32 O: each element rounded to the nearest
// bf16 (ties to even). Eight elements per thread: two 16-byte loads, one
// 16-byte store.
__global__ void __launch_bounds__(kCvtThreads)
    round_bf16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kCvtThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kCvtThreads) {
    const float4 a = __ldg(src + 2 * i), b = __ldg(src + 2 * i + 1);
    dst[i] = make_uint4(pack2(a.x, a.y), pack2(a.z, a.w), pack2(b.x, b.y), pack2(b.z, b.w));
  }
}

// ------------------------------------------------------- e4m3 quantisation
// Per-tensor power-of-two scale 2^k, the largest with max|x| * 2^k <= 448
// (the largest finite e4m3 value), so scaling and dequantising are exact;
// rounding to nearest, ties to even, saturating (cvt .rn.satfinite).
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
    amax_kernel(const uint4* __restrict__ x, int64_t n, unsigned* __restrict__ amax_bits) {
  float m = 0.f;
  for (int64_t i = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kQuantThreads) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // m >= 0: bits order as values
}

// 2^k from the bits of amax = (1 + f) 2^e: k = (f <= 0.75 ? 8 : 7) - e.
__device__ __forceinline__ float e4m3_scale(unsigned amax_bits) {
  if (amax_bits == 0) return 1.f;
  const int e = (int)((amax_bits >> 23) & 0xFFu) - 127;
  int k = ((amax_bits & 0x7FFFFFu) <= 0x600000u ? 8 : 7) - e;
  k = max(-126, min(127, k));
  return __uint_as_float((uint32_t)(k + 127) << 23);
}

// Four floats to four e4m3 bytes, a at the lowest address.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void __launch_bounds__(kQuantThreads)
    quant_kernel(const uint4* __restrict__ x, uint2* __restrict__ y, int64_t n,
                 const unsigned* __restrict__ amax_bits, float* __restrict__ scale_out) {
  const float s = e4m3_scale(*amax_bits);
  if (scale_out && blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
  for (int64_t i = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kQuantThreads) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16) * s;
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * s;
    }
    y[i] = make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
  }
}

}  // namespace

int launch_quant_e4m3(const void* src, void* dst, int64_t n_elems, unsigned* amax_bits, float* scale_out,
                      int num_sms, cudaStream_t st) {
  const int64_t n = n_elems / 8;
  int64_t grid = (n + kQuantThreads - 1) / kQuantThreads;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  if (grid < 1) grid = 1;
  amax_kernel<<<(int)grid, kQuantThreads, 0, st>>>(static_cast<const uint4*>(src), n, amax_bits);
  quant_kernel<<<(int)grid, kQuantThreads, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint2*>(dst), n,
                                                    amax_bits, scale_out);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_quant_e4m3_with(const void* src, void* dst, int64_t n_elems, const unsigned* amax_bits,
                           int num_sms, cudaStream_t st) {
  const int64_t n = n_elems / 8;
  if (n == 0) return FCP_OK;
  int64_t grid = (n + kQuantThreads - 1) / kQuantThreads;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  quant_kernel<<<(int)grid, kQuantThreads, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint2*>(dst), n,
                                                    amax_bits, nullptr);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_convert_f16(const void* src, void* dst, int64_t n_elems, int* err, int* zero_word,
                       int num_sms, cudaStream_t st) {
  const int64_t n = n_elems / 8;
  if (n == 0 && !zero_word) return FCP_OK;
  int64_t grid = (n + kCvtThreads - 1) / kCvtThreads;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  if (grid < 1) grid = 1;
  convert_kernel<<<(int)grid, kCvtThreads, 0, st>>>(static_cast<const uint4*>(src),
                                                    static_cast<uint4*>(dst), n, err, zero_word);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_round_bf16(const float* src, void* dst, int64_t n_elems, int num_sms, cudaStream_t st) {
  const int64_t n = n_elems / 8;
  if (n == 0) return FCP_OK;
  int64_t grid = (n + kCvtThreads - 1) / kCvtThreads;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  round_bf16_kernel<<<(int)grid, kCvtThreads, 0, st>>>(reinterpret_cast<const float4*>(src),
                                                       static_cast<uint4*>(dst), n);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_gather(const void* k, const void* v, const int32_t* tasks, int32_t n_tasks,
                  int32_t dst_shift, int64_t row_bytes, void* kbuf, void* vbuf, int32_t src_rows,
                  int32_t dst_rows, int num_sms, cudaStream_t st) {
  if (n_tasks == 0) return FCP_OK;
  const int grid = n_tasks < num_sms * 8 ? n_tasks : num_sms * 8;
  gather_kernel<<<grid, kGatherThreads, 0, st>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), tasks, n_tasks, dst_shift,
      row_bytes / 16, static_cast<uint4*>(kbuf), static_cast<uint4*>(vbuf), src_rows, dst_rows);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_merge(const float* o_parts, const float* lse_parts, int32_t B, int64_t rows, int32_t hq,
                 int32_t d, void* out, float* lse_out, int num_sms, cudaStream_t st) {
  if (rows == 0) return FCP_OK;
  if (B > d / 4 || rows * hq >= (int64_t(1) << 30)) return FCP_ERR_UNSUPPORTED;
  int bp = 1;
  while (bp < B) bp *= 2;
  const int64_t rows_per_block = (kMergeThreads / 32) * (32 / bp);
  int64_t gx = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = std::max<int64_t>(1, (int64_t)num_sms * 32 / hq);
  if (gx > cap) gx = cap;
  const dim3 grid((unsigned)gx, (unsigned)hq);
  const float4* op = reinterpret_cast<const float4*>(o_parts);
  uint2* o = static_cast<uint2*>(out);
  auto go = [&](auto kernel) { kernel<<<grid, kMergeThreads, 0, st>>>(op, lse_parts, B, (int)rows, hq, o, lse_out); };
  if (d == 128) {
    switch (bp) {
      case 1: go(merge_kernel<128, 1>); break;
      case 2: go(merge_kernel<128, 2>); break;
      case 4: go(merge_kernel<128, 4>); break;
      case 8: go(merge_kernel<128, 8>); break;
      case 16: go(merge_kernel<128, 16>); break;
      default: go(merge_kernel<128, 32>); break;
    }
  } else {
    switch (bp) {
      case 1: go(merge_kernel<64, 1>); break;
      case 2: go(merge_kernel<64, 2>); break;
      case 4: go(merge_kernel<64, 4>); break;
      case 8: go(merge_kernel<64, 8>); break;
      default: go(merge_kernel<64, 16>); break;
    }
  }
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_bwd_preprocess(const void* out, bool out_f32, const void* dout, const void* q,
                          const int32_t* rows, const int32_t* order, int32_t n_chunks, int32_t n_rows_table,
                          int32_t T,
                          int32_t hq, int32_t d, float* delta, float* dq, void* q16, void* do16,
                          int* err, int* zero_word, cudaStream_t st) {
  if (n_chunks == 0 && !zero_word) return FCP_OK;
  const dim3 grid(n_chunks > 0 ? n_chunks : 1, 8);  // a chunk's (row, head) pairs over 8 blocks
  using B = __nv_bfloat16;
  auto go = [&](auto kernel) {
    kernel<<<grid, kPreThreads, 0, st>>>(out, static_cast<const B*>(dout), static_cast<const B*>(q),
                                         rows, order, n_chunks, n_rows_table, T, hq, delta, dq,
                                         static_cast<__half*>(q16), static_cast<__half*>(do16), err,
                                         zero_word);
  };
  if (d == 128)
    out_f32 ? go(preprocess_kernel<128, true>) : go(preprocess_kernel<128, false>);
  else
    out_f32 ? go(preprocess_kernel<64, true>) : go(preprocess_kernel<64, false>);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

}  // namespace fcp
