// Document-masked attention backward on sm_103a (tcgen05 + TMA + TMEM).
//
// The exact gradient of the forward in attn_fwd.cu, for an upstream dO:
//   P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>,
//   dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q.
// "FlashCP" Fig. 6 names this "Attention BWD" and pairs it with a
// ReduceScatter of the KV gradients; on one GPU that reduction is the
// scatter-add of every key tile's dK/dV into the keys' global rows.
//
// Work unit: one key tile (<= 128 keys of one key segment) for one KV head.
// The CTA loops over the query heads of that GQA group and the query tiles
// that can see the keys -- those of the piece, and of the shard's earlier
// piece of the same document when the tile lies before that piece's end -- so
// dK and dV accumulate in TMEM over the whole group and reach global memory
// once per unit.
//
// Per step (one query head, one 128-row query tile), with keys as rows:
//   S^T = K Q^T, dP^T = V dO^T                (TMEM)
//   P^T = exp2(S^T scale log2e - LSE log2e)   (masked; fp16, back into TMEM)
//   dS^T = P^T (dP^T - D)                     (fp16, shared memory)
//   dV += P^T dO  (A operand from TMEM),  dK += dS^T Q,  dQ = dS K
// and dQ leaves TMEM through shared memory with TMA bulk reduce-adds
// (32-column chunks), one instruction per 16 KB.
//
// Tensor-core operands are fp16 (11 significant bits against bf16's 8): Q and
// dO arrive as fp16 copies made by the preprocess pass, K and V tiles are
// converted from bf16 in shared memory once per work unit, and P and dS are
// rounded to fp16. Every bf16 input inside the fp16 range converts exactly;
// P <= 1 and |dS| stay far inside it.
//
// CTA roles (512 threads, persistent):
//   warp 0       loads (TMA for K, V, Q, dO; plain loads for LSE and D)
//   warp 1       issues MMAs and owns TMEM
//   warps 2-3    convert each unit's K/V tiles to fp16
//   warps 4-7    P and dS for query columns 0-63 (one key row per thread);
//                dV to global at the end of a unit
//   warps 8-11   P and dS for query columns 64-127; dK to global
//   warps 12-15  dQ: TMEM -> shared memory -> TMA reduce-add into global
// MMA order per step j, so that the exp work of step j+1 overlaps the dK/dQ
// products of step j:  dV_j, S_{j+1}, dQ_j, dK_j, dP_{j+1}. Q tiles are
// double-buffered; the dO tile is single-buffered (its last reader, dV_j,
// runs first in the step).
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "sm103.cuh"

namespace fcp {

using namespace dev;

namespace {

constexpr int kThreads = 512;

template <int D>
struct BwdCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;           // 2 stages
  static constexpr int kDO = 4 * kTile;          // 1 stage
  static constexpr int kStage = 5 * kTile;       // 2 x [128 rows][32 fp32] dQ chunks
  static constexpr int kDS = kStage + 2 * 16384; // 128 x 128 fp16 (two 64-column panels)
  static constexpr int kStat = kDS + 128 * 128 * 2;  // [stage][lse2 | delta][128] fp32
  static constexpr int kSmem = kStat + 2 * 2 * 128 * 4;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;           // S^T; P^T (fp16) in cols [0,32) and [64,96)
  static constexpr uint32_t kColDP = 128;        // dP^T, then dQ
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

struct BwdItem {
  int key0, n, src, src_row, qa0, qa_end, na, qb0, qb_end, nb, nq, g;
  bool bad;  // checked build: the unit's table entries are out of range (skip it)
};

// Query tiles q0, q0 + 128, ... (n of them) lie inside [0, q_end] and q_end <= T.
__device__ __forceinline__ bool qrange_ok(int q0, int q_end, int n, int T) {
  return n == 0 || (n > 0 && q0 >= 0 && q_end <= T && (int64_t)q0 + (int64_t)(n - 1) * 128 < q_end);
}

__device__ __forceinline__ BwdItem decode(const BwdParams& p, int w) {
  const WorkSlot ws = work_slot(w, p.n_items, p.hkv, p.order_block);
  const int item = __ldg(p.order + ws.pos);
  BwdItem it;
  it.bad = false;
  if constexpr (kDeviceChecks) {
    if (item < 0 || item >= p.n_tiles) {
      it = BwdItem{0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, true};
      return it;
    }
  }
  const int* t = p.tiles + kBwdTileInts * item;
  it.key0 = __ldg(t + 0);
  it.n = __ldg(t + 1);
  it.src = __ldg(t + 2);
  it.src_row = __ldg(t + 3) - (it.src ? p.kbuf_shift : 0);
  it.qa0 = __ldg(t + 4);
  it.qa_end = __ldg(t + 5);
  it.na = __ldg(t + 6);
  it.qb0 = __ldg(t + 7);
  it.qb_end = __ldg(t + 8);
  it.nb = __ldg(t + 9);
  it.nq = it.na + it.nb;
  it.g = ws.head;
  if constexpr (kDeviceChecks) {
    const int rows = it.src ? p.kb_rows : p.T;
    it.bad = it.n < 1 || it.n > 128 || it.key0 < 0 || it.key0 > p.T - it.n || (it.src != 0 && it.src != 1) ||
             it.src_row < 0 || it.src_row > rows - it.n || !qrange_ok(it.qa0, it.qa_end, it.na, p.T) ||
             !qrange_ok(it.qb0, it.qb_end, it.nb, p.T);
  }
  return it;
}

// Query tile of step j of a unit: head index within the group j / nq, then
// the first range's tiles and the second range's.
struct StepRows {
  int h, q0, q_end;
};
__device__ __forceinline__ StepRows step_rows(const BwdItem& it, int G, int j) {
  StepRows r;
  const int jh = j / it.nq, jj = j - jh * it.nq;
  r.h = it.g * G + jh;
  if (jj < it.na) {
    r.q0 = it.qa0 + jj * 128;
    r.q_end = it.qa_end;
  } else {
    r.q0 = it.qb0 + (jj - it.na) * 128;
    r.q_end = it.qb_end;
  }
  return r;
}

// TMA bulk reduce-add of a shared-memory tile into global memory.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, const void* src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void drain_group_sync() {  // the 128 threads of the dQ warpgroup
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// AND of `ok` over the 128 threads of the dQ warpgroup, so that its four warps
// leave (or stay in) the loop together and never strand one at bar.sync.
__device__ __forceinline__ bool drain_group_all(bool ok) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)ok)
      : "memory");
  return out != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vb,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_kv_full, bar_kv_conv, bar_kv_empty, bar_drain;
  __shared__ __align__(8) uint64_t bar_q_full[2], bar_q_empty[2], bar_do_full, bar_do_empty;
  __shared__ __align__(8) uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready, bar_ds_free;
  __shared__ __align__(8) uint64_t bar_dq_full, bar_dq_free, bar_dkdv_full, bar_dkdv_free;
  __shared__ __align__(8) uint64_t bar_stg_full[2], bar_stg_free[2];  // dV / dK staging, per half
  __shared__ WorkRing<4> ring;
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
      mbar_init(&bar_q_full[s], 2);
      mbar_init(&bar_q_empty[s], 1);
    }
    mbar_init(&bar_do_full, 1);
    mbar_init(&bar_do_empty, 1);
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_ready, 256);
    mbar_init(&bar_ds_ready, 256);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_free, 128);
    mbar_init(&bar_dkdv_full, 1);
    mbar_init(&bar_dkdv_free, 256);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bar_stg_full[h], 128);
      mbar_init(&bar_stg_free[h], 1);
    }
    ring.init(1 + 2 + 8 + 4);  // MMA thread, conversion, compute and dQ warps
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
    prefetch_tmap(&tm_dq);
    prefetch_tmap(&tm_dk);
    prefetch_tmap(&tm_dv);
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
    uint32_t kv_items = 0, qc = 0, dc = 0;
    uint32_t issued_q[2] = {0, 0};
    bool ok = true;
    const float kLog2e = 1.4426950408889634f;
    uint32_t k = 0;
    for (int w = blockIdx.x; ok;) {
      if (lane == 0) ok = ring.put(k, w, wc);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
      ++k;
      if (!ok || w >= n_work) break;
      // The next unit is claimed now (measured a little ahead of claiming it
      // after this unit's loads).
      int w_next = 0;
      if (lane == 0) w_next = next_work(p.work_counter);
      w_next = __shfl_sync(0xffffffffu, w_next, 0);
      const BwdItem it = decode(p, w);
      if (it.bad) {  // checked build: skipped by every role
        if (lane == 0) atomicOr(p.err, kErrBadTable);
        w = w_next;
        continue;
      }
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
      const int nsteps = G * it.nq;
      // No L2 prefetches: issued through the tensor-memory accelerator, which
      // also carries this CTA's loads and dQ reduce-adds, they cost more in its
      // queue than they saved.
      for (int j = 0; j < nsteps; ++j) {
        const StepRows sr = step_rows(it, G, j);
        const int h = sr.h, q0 = sr.q0;
        const int q_rows = min(128, sr.q_end - q0);
        // Q tile and the rows' LSE / D into Q stage s.
        const int s = qc & 1;
        if (qc >= 2) {
          ok = mbar_wait(&bar_q_empty[s], ((qc >> 1) - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_q_full[s], C::kTile);
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kQ + s * C::kTile + pn * 16384, &tm_q, &bar_q_full[s], pn * 64, h, q0);
          ++issued_q[s];
        }
        float* st = stat + s * 256;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = lane + 32 * u;
          const bool valid = r < q_rows;
          // Stored negated (-LSE log2 e, -D): the compute warps add them with
          // packed f32x2 arithmetic. Rows past the piece get P = 0.
          st[r] = valid ? -__ldg(p.lse + (size_t)h * p.T + q0 + r) * kLog2e : -INFINITY;
          st[128 + r] = valid ? -__ldg(p.delta + (size_t)h * p.T + q0 + r) : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_q_full[s]);
        ++qc;
        // dO tile into the single dO buffer once dV of the previous step is done.
        if (dc >= 1) {
          ok = mbar_wait(&bar_do_empty, (dc - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_do_full, C::kTile);
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kDO + pn * 16384, &tm_do, &bar_do_full, pn * 64, h, q0);
        }
        ++dc;
      }
      w = w_next;
    }
    if (lane == 0) {  // every copy this warp started has landed before the CTA exits
      if (kv_items) mbar_drain(&bar_kv_full, (kv_items - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (issued_q[s]) mbar_drain(&bar_q_full[s], (issued_q[s] - 1) & 1);
      if (dc) mbar_drain(&bar_do_full, (dc - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_sq = idesc_f16kind(128, 128, false, false, false);  // S^T, dP^T
      constexpr uint32_t id_kd = idesc_f16kind(128, D, false, true, false);     // dV, dK
      constexpr uint32_t id_dq = idesc_f16kind(128, D, true, true, false);      // dQ = dS K
      const uint32_t sK = smem_u32(smem + C::kK), sV = smem_u32(smem + C::kV);
      const uint32_t sDO = smem_u32(smem + C::kDO), sDS = smem_u32(smem + C::kDS);
      uint32_t kv_items = 0, qc = 0, dc = 0, gstep = 0, items = 0;
      bool ok = true;
      auto qaddr = [&](uint32_t c) { return smem_u32(smem + C::kQ + (c & 1) * C::kTile); };
      auto issue_s = [&](uint32_t c) {
        const uint32_t sQ = qaddr(c);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + C::kColS, smem_desc_sw128(sK + off, 0, 1024),
                      smem_desc_sw128(sQ + off, 0, 1024), id_sq, kk > 0);
        }
        mma_commit(&bar_s_full);
      };
      auto issue_dp = [&]() {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ss(tmem + C::kColDP, smem_desc_sw128(sV + off, 0, 1024),
                      smem_desc_sw128(sDO + off, 0, 1024), id_sq, kk > 0);
        }
        mma_commit(&bar_dp_full);
      };
      for (uint32_t k = 0; ok; ++k) {
        int w;
        if (!(ok = ring.get(k, w, wc))) break;
        ring.release(k);
        if (w >= n_work) break;
        const BwdItem it = decode(p, w);
        if (it.bad) continue;
        const int nsteps = G * it.nq;
        if (!(ok = mbar_wait(&bar_kv_conv, kv_items & 1, wc))) break;
        tc_fence_after();
        // Prologue of the unit: S_0 and dP_0.
        if (!(ok = mbar_wait(&bar_q_full[qc & 1], (qc >> 1) & 1, wc))) break;
        tc_fence_after();
        issue_s(qc);
        if (gstep > 0 && !(ok = mbar_wait(&bar_dq_free, (gstep - 1) & 1, wc))) break;
        if (!(ok = mbar_wait(&bar_do_full, dc & 1, wc))) break;
        tc_fence_after();
        issue_dp();
        for (int j = 0; j < nsteps; ++j, ++gstep) {
          const uint32_t c = qc + j;
          const uint32_t sQ = qaddr(c);
          if (!(ok = mbar_wait(&bar_p_ready, gstep & 1, wc))) break;
          if (j == 0 && items > 0 && !(ok = mbar_wait(&bar_dkdv_free, (items - 1) & 1, wc))) break;
          tc_fence_after();
          // dV += P^T dO, P^T from TMEM: q columns 0-63 in cols [0,32), 64-127 in [64,96).
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ts(tmem + C::kColDV, tmem + C::kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                       smem_desc_sw128(sDO + kk * 2048, 16384, 1024), id_kd, (j > 0 || kk > 0));
          mma_commit(&bar_do_empty);
          if (j + 1 < nsteps) {  // S region is free once dV (issued above) has read P^T
            if (!(ok = mbar_wait(&bar_q_full[(c + 1) & 1], ((c + 1) >> 1) & 1, wc))) break;
            tc_fence_after();
            issue_s(c + 1);
          }
          if (!(ok = mbar_wait(&bar_ds_ready, gstep & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + C::kColDP, smem_desc_sw128(sDS + kk * 2048, 16384, 1024),
                        smem_desc_sw128(sK + kk * 2048, 16384, 1024), id_dq, kk > 0);
          mma_commit(&bar_dq_full);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColDK, smem_desc_sw128(sDS + aoff, 0, 1024),
                        smem_desc_sw128(sQ + kk * 2048, 16384, 1024), id_kd, (j > 0 || kk > 0));
          }
          mma_commit(&bar_ds_free);
          mma_commit(&bar_q_empty[c & 1]);
          if (j + 1 < nsteps) {  // DP region is free once dQ_j has been read out
            if (!(ok = mbar_wait(&bar_dq_free, gstep & 1, wc))) break;
            if (!(ok = mbar_wait(&bar_do_full, (dc + j + 1) & 1, wc))) break;
            tc_fence_after();
            issue_dp();
          }
        }
        if (!ok) break;
        mma_commit(&bar_dkdv_full);
        mma_commit(&bar_kv_empty);
        qc += nsteps;
        dc += nsteps;
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
    for (uint32_t k = 0; ok; ++k) {
      int w = 0;
      ok = ring.get(k, w, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) ring.release(k);
      if (w >= n_work) break;
      if constexpr (kDeviceChecks) {
        if (decode(p, w).bad) continue;
      }
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
  } else if (warp < 12) {
    // ------------------------------------------------------------ P and dS
    const int half = (warp - 4) >> 2;       // query columns [64*half, 64*half + 64)
    const int kr = (warp & 3) * 32 + lane;  // key row == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_cols = lane_base + C::kColS + 64 * half;
    const uint32_t dp_cols = lane_base + C::kColDP + 64 * half;
    const uint32_t ds_panel = smem_u32(smem + C::kDS) + half * 16384;
    uint32_t qc = 0, gstep = 0, items = 0, stg = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      int w = 0;
      ok = ring.get(k, w, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) ring.release(k);
      if (w >= n_work) break;
      const BwdItem it = decode(p, w);
      if (it.bad) continue;
      const int nsteps = G * it.nq;
      const bool key_valid = kr < it.n;
      const int key = it.key0 + kr;
      for (int j = 0; j < nsteps; ++j, ++gstep) {
        const uint32_t c = qc + j, s = c & 1;
        const int q0 = step_rows(it, G, j).q0;
        const int lim = key - q0 - 64 * half;  // local columns below lim cannot see this key
        // Whole tile below the diagonal with 128 keys: no element needs a mask
        // (query rows past the piece end have LSE = +inf, hence P = 0).
        const bool unmasked = it.n == 128 && it.key0 + 127 <= q0;
        ok = mbar_wait(&bar_s_full, gstep & 1, wc) && mbar_wait(&bar_q_full[s], (c >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float4* st4 = reinterpret_cast<const float4*>(stat + s * 256 + 64 * half);
        uint32_t pk[32];
        {
          // Both 32-column halves of this group's S^T in flight together.
          float va[32], vb[32];
          tmem_ld32(s_cols, va);
          tmem_ld32(s_cols + 32, vb);
          tmem_ld_wait();
          const uint64_t c2 = f2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const float* v = e < 32 ? va + e : vb + (e - 32);
            const float4 l4 = st4[e >> 2];  // -LSE log2 e of the four query columns
            float p0, p1, p2, p3;
            f2_split(f2_fma(f2(v[0], v[1]), c2, f2(l4.x, l4.y)), p0, p1);
            f2_split(f2_fma(f2(v[2], v[3]), c2, f2(l4.z, l4.w)), p2, p3);
            p0 = ex2(p0);
            p1 = ex2(p1);
            p2 = ex2(p2);
            p3 = ex2(p3);
            if (!unmasked) {
              if (!key_valid || e < lim) p0 = 0.f;
              if (!key_valid || e + 1 < lim) p1 = 0.f;
              if (!key_valid || e + 2 < lim) p2 = 0.f;
              if (!key_valid || e + 3 < lim) p3 = 0.f;
            }
            pk[e >> 1] = pack_f16(p0, p1);
            pk[(e >> 1) + 1] = pack_f16(p2, p3);
          }
        }
        {
          float f[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(pk[e]);
          tmem_st32(s_cols, f);  // P^T over the S values just read (same rows, own columns)
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar_p_ready);
        ok = mbar_wait(&bar_dp_full, gstep & 1, wc);
        if (ok && gstep > 0) ok = mbar_wait(&bar_ds_free, (gstep - 1) & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // dS = P (dP - D) in packed fp16: (dP - D) and the product are each
        // rounded to fp16, the operand type of the dK and dQ products.
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float v[32];
          tmem_ld32(dp_cols + cc * 32, v);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int col = cc * 32 + e;
            const float4 d4 = st4[32 + (col >> 2)];  // -D of the four query columns
            float a0, a1, a2, a3;
            f2_split(f2_add(f2(v[e], v[e + 1]), f2(d4.x, d4.y)), a0, a1);
            f2_split(f2_add(f2(v[e + 2], v[e + 3]), f2(d4.z, d4.w)), a2, a3);
            const __half2 x01 = __floats2half2_rn(a0, a1);
            const __half2 x23 = __floats2half2_rn(a2, a3);
            const uint32_t p01 = pk[col >> 1], p23 = pk[(col >> 1) + 1];
            const __half2 r01 = __hmul2(*reinterpret_cast<const __half2*>(&p01), x01);
            const __half2 r23 = __hmul2(*reinterpret_cast<const __half2*>(&p23), x23);
            o[e >> 1] = *reinterpret_cast<const uint32_t*>(&r01);
            o[(e >> 1) + 1] = *reinterpret_cast<const uint32_t*>(&r23);
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(ds_panel + sw128_offset(kr, cc * 4 + q4), o[4 * q4], o[4 * q4 + 1],
                         o[4 * q4 + 2], o[4 * q4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_ds_ready);
      }
      if (!ok) break;
      qc += nsteps;
      // dV (columns-0 group) or dK (columns-64 group) of this key tile ->
      // global rows: 32-column chunks staged in this group's half of the dS
      // buffer (free once the unit's MMAs are done; the 128-byte swizzled
      // layout of a [128 rows][32 fp32] TMA box) and reduce-added by one
      // thread with TMA. Rows of keys past the tile hold zeros.
      ok = mbar_wait(&bar_dkdv_full, items & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t src_col = lane_base + (half == 0 ? C::kColDV : C::kColDK);
      const float mul = half == 0 ? 1.f : p.scale;
      const CUtensorMap* tm_out = half == 0 ? &tm_dv : &tm_dk;
      // Two chunks in registers: the TMEM read of chunk cc + 2 is issued once
      // chunk cc is staged and waited for two chunks later, so its latency
      // (a TMEM read waits behind the MMAs' own TMEM traffic) overlaps the
      // reduce-adds of the chunks between.
      constexpr int kChunks = D / 32;
      float vv[2][32];
      tmem_ld32(src_col, vv[0]);
      tmem_ld32(src_col + 32, vv[1]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < kChunks; ++cc, ++stg) {
        if (!ok) break;
        float* v = vv[cc & 1];
        if (stg > 0) {  // the previous chunk's reduce has read the staging tile
          ok = mbar_wait(&bar_stg_free[half], (stg - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        if (cc >= 2) tmem_ld_wait();  // this chunk was read after chunk cc - 2 was staged
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float a0 = key_valid ? v[4 * q4] * mul : 0.f, a1 = key_valid ? v[4 * q4 + 1] * mul : 0.f;
          const float a2 = key_valid ? v[4 * q4 + 2] * mul : 0.f, a3 = key_valid ? v[4 * q4 + 3] * mul : 0.f;
          st_shared_v4(ds_panel + sw128_offset(kr, q4), __float_as_uint(a0), __float_as_uint(a1),
                       __float_as_uint(a2), __float_as_uint(a3));
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar_stg_full[half]);
        if (cc + 2 < kChunks) tmem_ld32(src_col + (cc + 2) * 32, vv[cc & 1]);
        if (kr == 0) {
          ok = mbar_wait(&bar_stg_full[half], stg & 1, wc);
          if (ok) {
            tma_reduce_add_3d(tm_out, smem + C::kDS + half * 16384, cc * 32, it.g, it.key0);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bar_stg_free[half]);
        }
        ok = __all_sync(0xffffffffu, ok);  // the issuing lane's outcome, warp-wide
      }
      tmem_ld_wait();  // no TMEM read left in flight, also when the loop gave up early
      // The last chunk's tile is read before dS of the next unit lands there.
      if (ok) ok = mbar_wait(&bar_stg_free[half], (stg - 1) & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_before();
      mbar_arrive(&bar_dkdv_free);
      ++items;
    }
    if (kr == 0) bulk_wait_all();  // this thread's reduces are complete before the CTA exits
  } else {
    // ------------------------------------------------------------ dQ drain
    // Thread r holds query row q0 + r. Each 32-column chunk goes to one of two
    // shared-memory staging tiles (the 128-byte swizzled layout of a
    // [128 rows][32 fp32] TMA box) and one thread reduce-adds it into dQ.
    // Rows past the piece end hold exact zeros (their P and dS are zero).
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t* stage = smem + C::kStage;
    uint32_t gstep = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      int w = 0;
      ok = drain_group_all(ring.get(k, w, wc));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) ring.release(k);
      if (w >= n_work) break;
      const BwdItem it = decode(p, w);
      if (it.bad) continue;
      const int nsteps = G * it.nq;
      for (int j = 0; j < nsteps; ++j, ++gstep) {
        const StepRows sr = step_rows(it, G, j);
        const int h = sr.h, q0 = sr.q0;
        ok = drain_group_all(mbar_wait(&bar_dq_full, gstep & 1, wc));
        if (!ok) break;
        tc_fence_after();
        // Two 32-column chunks at a time: both loads in flight together, the
        // TMEM columns released as soon as every chunk has been read.
        constexpr int kPairs = D / 64;
        float a[32], b[32];
        tmem_ld32(lane_base + C::kColDP, a);
        tmem_ld32(lane_base + C::kColDP + 32, b);
        tmem_ld_wait();
        if (kPairs == 1) {
          tc_fence_before();
          mbar_arrive(&bar_dq_free);  // every dQ column of this step has been read
        }
#pragma unroll 1
        for (int pr = 0; pr < kPairs; ++pr) {
          if (r == 0) bulk_wait_read_all();  // earlier reduces are done reading the tiles
          drain_group_sync();
          const uint32_t b0 = smem_u32(stage), b1 = smem_u32(stage + 16384);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            st_shared_v4(b0 + sw128_offset(r, q4), __float_as_uint(a[4 * q4] * p.scale),
                         __float_as_uint(a[4 * q4 + 1] * p.scale), __float_as_uint(a[4 * q4 + 2] * p.scale),
                         __float_as_uint(a[4 * q4 + 3] * p.scale));
            st_shared_v4(b1 + sw128_offset(r, q4), __float_as_uint(b[4 * q4] * p.scale),
                         __float_as_uint(b[4 * q4 + 1] * p.scale), __float_as_uint(b[4 * q4 + 2] * p.scale),
                         __float_as_uint(b[4 * q4 + 3] * p.scale));
          }
          if (pr + 1 < kPairs) {
            tmem_ld32(lane_base + C::kColDP + 64 * (pr + 1), a);
            tmem_ld32(lane_base + C::kColDP + 64 * (pr + 1) + 32, b);
            tmem_ld_wait();
            if (pr + 2 == kPairs) {
              tc_fence_before();
              mbar_arrive(&bar_dq_free);  // every dQ column of this step has been read
            }
          }
          fence_proxy_async_smem();
          drain_group_sync();
          if (r == 0) {
            tma_reduce_add_3d(&tm_dq, stage, 64 * pr, h, q0);
            tma_reduce_add_3d(&tm_dq, stage + 16384, 64 * pr + 32, h, q0);
            bulk_commit();
          }
        }
      }
    }
    if (r == 0) bulk_wait_all();
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
  // Blocks of key tiles that fill the grid with one KV head: the CTAs running
  // together stream the same query rows (Q, dO, dQ) of that head group.
  BwdParams p = a.p;
  p.order_block = grid;
  attn_bwd_kernel<D><<<grid, kThreads, C::kSmem, st>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.tm_kb,
                                                      a.tm_vb, a.tm_dq, a.tm_dk, a.tm_dv, p);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

int launch_attn_bwd(const BwdLaunch& a, cudaStream_t st) {
  if (a.d == 128) return launch_bwd_impl<128>(a, st);
  if (a.d == 64) return launch_bwd_impl<64>(a, st);
  return FCP_ERR_UNSUPPORTED;
}

}  // namespace fcp
