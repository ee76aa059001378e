// Document-masked attention backward on sm_103a (tcgen05 + TMA + TMEM).
//
// The exact gradient of the forward in attn_fwd.cu, for an upstream dO:
//   P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>,
//   dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q.
// "FlashCP" Fig. 6 names this "Attention BWD" and pairs it with a
// ReduceScatter of the KV gradients; on one GPU that reduction is the
// scatter-add of every key tile's dK/dV into the keys' global rows.
//
// Work unit: one key tile (<= 128 keys of one key segment of one piece) for
// one KV head. The CTA loops over the query heads of that GQA group and the
// piece's query tiles that can see the keys, so dK and dV accumulate in TMEM
// over the whole group and reach global memory once per unit.
//
// Per step (one query head, one 128-row query tile), with keys as rows:
//   S^T = K Q^T, dP^T = V dO^T                (TMEM)
//   P^T = exp2(S^T scale log2e - LSE log2e)   (masked; bf16, back into TMEM)
//   dS^T = P^T (dP^T - D)                     (bf16, shared memory)
//   dV += P^T dO  (A operand from TMEM),  dK += dS^T Q,  dQ = dS K
// and dQ is added to global memory with fp32 vector atomics.
//
// Tensor-core operands are fp16 (11 significant bits against bf16's 8): Q and
// dO arrive as fp16 copies made by the preprocess pass, K and V tiles are
// converted from bf16 in shared memory once per work unit, and P and dS are
// rounded to fp16. Every bf16 input inside the fp16 range converts exactly;
// P <= 1 and |dS| stay far inside it.
//
// CTA roles (384 threads, persistent): warp 0 loads (TMA for K, V, Q, dO;
// plain loads for LSE and D), warp 1 issues MMAs, warps 2-3 convert the K/V
// tiles, warps 4-7 compute P and dS (one key row per thread) and write dK/dV,
// warps 8-11 drain dQ (one query row per thread).
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "sm103.cuh"

namespace fcp {

using namespace dev;

namespace {

constexpr int kThreads = 384;

template <int D>
struct BwdCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;           // 2 stages
  static constexpr int kDO = 4 * kTile;          // 2 stages
  static constexpr int kDS = 6 * kTile;          // 128 x 128 bf16
  static constexpr int kStat = kDS + 128 * 128 * 2;  // [stage][lse2 | delta][128] fp32
  static constexpr int kSmem = kStat + 2 * 2 * 128 * 4;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;           // S^T, then P^T (bf16) in its first 64 columns
  static constexpr uint32_t kColDP = 128;        // dP^T, then dQ
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

struct BwdItem {
  int piece_start, piece_end, key0, n, src, src_row, qt_first, n_qt, g;
};

__device__ __forceinline__ BwdItem decode(const BwdParams& p, int w) {
  const int item = __ldg(p.order + w / p.hkv);
  const int* t = p.tiles + 8 * item;
  const int piece = __ldg(t + 0);
  BwdItem it;
  it.piece_start = __ldg(p.pieces + 8 * piece + 2);
  it.piece_end = __ldg(p.pieces + 8 * piece + 3);
  it.key0 = __ldg(t + 2);
  it.n = __ldg(t + 3);
  it.src = __ldg(t + 4);
  it.src_row = __ldg(t + 5) - (it.src ? p.kbuf_shift : 0);
  it.qt_first = __ldg(t + 6);
  it.n_qt = __ldg(t + 7);
  it.g = w % p.hkv;
  return it;
}

// MMA with the A operand in TMEM (kind::f16, bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  tmem_st32(taddr, f);
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vb,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_kv_full, bar_kv_conv, bar_kv_empty, bar_drain;
  __shared__ __align__(8) uint64_t bar_qdo_full[2], bar_qdo_empty[2];
  __shared__ __align__(8) uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready, bar_ds_free;
  __shared__ __align__(8) uint64_t bar_dq_full, bar_dq_free, bar_dkdv_full, bar_dkdv_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    if (tid == 0) atomicOr(p.err, 2);
    return;
  }
  if (tid == 0) {
    mbar_init(&bar_kv_full, 1);
    mbar_init(&bar_kv_conv, 64);
    mbar_init(&bar_kv_empty, 1);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_qdo_full[s], 2);
      mbar_init(&bar_qdo_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_ready, 128);
    mbar_init(&bar_ds_ready, 128);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_free, 128);
    mbar_init(&bar_dkdv_full, 1);
    mbar_init(&bar_dkdv_free, 128);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_kb);
    prefetch_tmap(&tm_vb);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const WaitCtl wc{&abort_sh, p.err, p.wait_ns};
  const int n_work = p.n_items * p.hkv;
  const int G = p.hq / p.hkv;
  float* stat = reinterpret_cast<float*>(smem + C::kStat);

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    uint32_t kv_items = 0, qdo_cnt = 0;
    uint32_t issued_q[2] = {0, 0};
    bool ok = true;
    const float kLog2e = 1.4426950408889634f;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const BwdItem it = decode(p, w);
      if (kv_items > 0) {
        ok = mbar_wait(&bar_kv_empty, (kv_items - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_kv_full, 2 * C::kTile);
        const CUtensorMap* tk = it.src ? &tm_kb : &tm_k;
        const CUtensorMap* tv = it.src ? &tm_vb : &tm_v;
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_3d(smem + C::kK + pn * 16384, tk, &bar_kv_full, pn * 64, it.g, it.src_row);
          tma_load_3d(smem + C::kV + pn * 16384, tv, &bar_kv_full, pn * 64, it.g, it.src_row);
        }
      }
      ++kv_items;
      const int nsteps = G * it.n_qt;
      for (int j = 0; j < nsteps; ++j) {
        const int h = it.g * G + j / it.n_qt;
        const int q0 = it.piece_start + (it.qt_first + j % it.n_qt) * 128;
        const int q_rows = min(128, it.piece_end - q0);
        const int s = qdo_cnt & 1;
        if (qdo_cnt >= 2) {
          ok = mbar_wait(&bar_qdo_empty[s], ((qdo_cnt >> 1) - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_qdo_full[s], 2 * C::kTile);
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_3d(smem + C::kQ + s * C::kTile + pn * 16384, &tm_q, &bar_qdo_full[s], pn * 64, h, q0);
            tma_load_3d(smem + C::kDO + s * C::kTile + pn * 16384, &tm_do, &bar_qdo_full[s], pn * 64, h, q0);
          }
          ++issued_q[s];
        }
        float* st = stat + s * 256;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = lane + 32 * u;
          const bool valid = r < q_rows;
          st[r] = valid ? __ldg(p.lse + (size_t)h * p.T + q0 + r) * kLog2e : INFINITY;
          st[128 + r] = valid ? __ldg(p.delta + (size_t)h * p.T + q0 + r) : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_qdo_full[s]);
        ++qdo_cnt;
      }
    }
    if (lane == 0) {  // every copy this warp started has landed before the CTA exits
      if (kv_items) mbar_drain(&bar_kv_full, (kv_items - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (issued_q[s]) mbar_drain(&bar_qdo_full[s], (issued_q[s] - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f16kind(128, 128, false, false, false);  // S^T, dP^T
      constexpr uint32_t id_kd = idesc_f16kind(128, D, false, true, false);     // dV, dK
      constexpr uint32_t id_dq = idesc_f16kind(128, D, true, true, false);      // dQ = dS K
      const uint32_t sK = smem_u32(smem + C::kK), sV = smem_u32(smem + C::kV);
      const uint32_t sDS = smem_u32(smem + C::kDS);
      uint32_t kv_items = 0, qdo_cnt = 0, gstep = 0, items = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
        const BwdItem it = decode(p, w);
        const int nsteps = G * it.n_qt;
        if (!(ok = mbar_wait(&bar_kv_conv, kv_items & 1, wc))) break;
        for (int j = 0; j < nsteps; ++j, ++gstep) {
          const uint32_t c = qdo_cnt + j, s = c & 1;
          const uint32_t sQ = smem_u32(smem + C::kQ + s * C::kTile);
          const uint32_t sDO = smem_u32(smem + C::kDO + s * C::kTile);
          if (!(ok = mbar_wait(&bar_qdo_full[s], (c >> 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColS, smem_desc_sw128(sK + off, 0, 1024),
                        smem_desc_sw128(sQ + off, 0, 1024), id_sq, kk > 0);
          }
          mma_commit(&bar_s_full);
          if (gstep > 0 && !(ok = mbar_wait(&bar_dq_free, (gstep - 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColDP, smem_desc_sw128(sV + off, 0, 1024),
                        smem_desc_sw128(sDO + off, 0, 1024), id_sq, kk > 0);
          }
          mma_commit(&bar_dp_full);
          if (!(ok = mbar_wait(&bar_p_ready, gstep & 1, wc))) break;
          if (j == 0 && items > 0 && !(ok = mbar_wait(&bar_dkdv_free, (items - 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + C::kColDV, tmem + C::kColS + kk * 8,
                        smem_desc_sw128(sDO + kk * 2048, 16384, 1024), id_kd, (j > 0 || kk > 0));
          if (!(ok = mbar_wait(&bar_ds_ready, gstep & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColDK, smem_desc_sw128(sDS + aoff, 0, 1024),
                        smem_desc_sw128(sQ + kk * 2048, 16384, 1024), id_kd, (j > 0 || kk > 0));
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + C::kColDP, smem_desc_sw128(sDS + kk * 2048, 16384, 1024),
                        smem_desc_sw128(sK + kk * 2048, 16384, 1024), id_dq, kk > 0);
          mma_commit(&bar_dq_full);
          mma_commit(&bar_ds_free);
          mma_commit(&bar_qdo_empty[s]);
        }
        if (!ok) break;
        mma_commit(&bar_dkdv_full);
        mma_commit(&bar_kv_empty);
        qdo_cnt += nsteps;
        ++kv_items;
        ++items;
      }
      // Every MMA this thread issued has finished before TMEM is released.
      mma_commit(&bar_drain);
      mbar_drain(&bar_drain, 0);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ K/V to fp16
    const int t = tid - 64;
    uint32_t items = 0;
    bool ok = true, ovf = false;
    uint4* kv = reinterpret_cast<uint4*>(smem + C::kK);  // K and V tiles are contiguous
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      ok = mbar_wait(&bar_kv_full, items & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll 4
      for (int i = t; i < 2 * C::kTile / 16; i += 64) {
        uint4 x = kv[i];
        x.x = bf16x2_to_f16x2(x.x, ovf);
        x.y = bf16x2_to_f16x2(x.y, ovf);
        x.z = bf16x2_to_f16x2(x.z, ovf);
        x.w = bf16x2_to_f16x2(x.w, ovf);
        kv[i] = x;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar_kv_conv);
      ++items;
    }
    if (ovf) atomicOr(p.err, 4);
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ P and dS
    const int kr = tid - 128;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t ds_row = smem_u32(smem + C::kDS);
    uint32_t qdo_cnt = 0, gstep = 0, items = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const BwdItem it = decode(p, w);
      const int nsteps = G * it.n_qt;
      const bool key_valid = kr < it.n;
      const int key = it.key0 + kr;
      for (int j = 0; j < nsteps; ++j, ++gstep) {
        const uint32_t c = qdo_cnt + j, s = c & 1;
        const int q0 = it.piece_start + (it.qt_first + j % it.n_qt) * 128;
        const int lim = key - q0;  // query columns below lim cannot see this key
        ok = mbar_wait(&bar_s_full, gstep & 1, wc) && mbar_wait(&bar_qdo_full[s], (c >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float* st = stat + s * 256;
        uint32_t pk[64];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float v[32];
          tmem_ld32(lane_base + C::kColS + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = cc * 32 + e;
            float p0 = ex2(fmaf(v[e], p.scale_log2, -st[col]));
            float p1 = ex2(fmaf(v[e + 1], p.scale_log2, -st[col + 1]));
            if (!key_valid || col < lim) p0 = 0.f;
            if (!key_valid || col + 1 < lim) p1 = 0.f;
            pk[col >> 1] = pack_f16(p0, p1);
          }
        }
        {
          uint32_t a[32], b[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            a[e] = pk[e];
            b[e] = pk[32 + e];
          }
          tmem_st32u(lane_base + C::kColS, a);
          tmem_st32u(lane_base + C::kColS + 32, b);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar_p_ready);
        ok = mbar_wait(&bar_dp_full, gstep & 1, wc);
        if (ok && gstep > 0) ok = mbar_wait(&bar_ds_free, (gstep - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float v[32];
          tmem_ld32(lane_base + C::kColDP + cc * 32, v);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = cc * 32 + e;
            const uint32_t pp = pk[col >> 1];
            const float d0 = f16_lo(pp) * (v[e] - st[128 + col]);
            const float d1 = f16_hi(pp) * (v[e + 1] - st[128 + col + 1]);
            o[e >> 1] = pack_f16(d0, d1);
          }
          // 32 query columns = 4 swizzle chunks of 8 in panel cc/2.
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = (cc & 1) * 4 + q4;
            st_shared_v4(ds_row + (cc >> 1) * 16384 + sw128_offset(kr, chunk), o[4 * q4],
                         o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_ds_ready);
      }
      if (!ok) break;
      qdo_cnt += nsteps;
      // dK, dV of this key tile -> global rows (scatter-add over shards and pieces).
      ok = mbar_wait(&bar_dkdv_full, items & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const size_t gbase = ((size_t)key * p.hkv + it.g) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float v[32], k2[32];
        tmem_ld32(lane_base + C::kColDV + cc * 32, v);
        tmem_ld32(lane_base + C::kColDK + cc * 32, k2);
        tmem_ld_wait();
        if (key_valid) {
          float4* dvp = reinterpret_cast<float4*>(p.dv + gbase + cc * 32);
          float4* dkp = reinterpret_cast<float4*>(p.dk + gbase + cc * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            atomicAdd(dvp + e, make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]));
            atomicAdd(dkp + e, make_float4(k2[4 * e] * p.scale, k2[4 * e + 1] * p.scale,
                                           k2[4 * e + 2] * p.scale, k2[4 * e + 3] * p.scale));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_dkdv_free);
      ++items;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain
    const int r = tid - 256;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t gstep = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const BwdItem it = decode(p, w);
      const int nsteps = G * it.n_qt;
      for (int j = 0; j < nsteps; ++j, ++gstep) {
        const int h = it.g * G + j / it.n_qt;
        const int q0 = it.piece_start + (it.qt_first + j % it.n_qt) * 128;
        const bool row_valid = r < min(128, it.piece_end - q0);
        ok = mbar_wait(&bar_dq_full, gstep & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        float4* dst = reinterpret_cast<float4*>(p.dq + ((size_t)(q0 + r) * p.hq + h) * D);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          float v[32];
          tmem_ld32(lane_base + C::kColDP + cc * 32, v);
          tmem_ld_wait();
          if (row_valid) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              atomicAdd(dst + cc * 8 + e, make_float4(v[4 * e] * p.scale, v[4 * e + 1] * p.scale,
                                                      v[4 * e + 2] * p.scale, v[4 * e + 3] * p.scale));
          }
        }
        tc_fence_before();
        mbar_arrive(&bar_dq_free);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

template <int D>
static int launch_bwd_impl(const BwdLaunch& a, cudaStream_t st) {
  using C = BwdCfg<D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmem) != cudaSuccess)
      return FCP_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int n_work = a.p.n_items * a.p.hkv;
  if (n_work == 0) return FCP_OK;
  const int grid = n_work < a.num_sms ? n_work : a.num_sms;
  attn_bwd_kernel<D><<<grid, kThreads, C::kSmem, st>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.tm_kb,
                                                      a.tm_vb, a.p);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_attn_bwd(const BwdLaunch& a, cudaStream_t st) {
  if (a.d == 128) return launch_bwd_impl<128>(a, st);
  if (a.d == 64) return launch_bwd_impl<64>(a, st);
  return FCP_ERR_UNSUPPORTED;
}

}  // namespace fcp
