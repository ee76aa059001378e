// Document-masked attention forward on sm_103a (tcgen05 + TMA + TMEM).
//
// Computes, for every query row i of the selected shard(s) and query head h,
//   s_ij = scale <q_ih, k_jg>   over keys j of doc(i) with j <= i,
//   LSE_ih = ln sum_j exp(s_ij),  O_ih = sum_j exp(s_ij - LSE_ih) v_jg
// ("FlashCP: Load-Balanced Communication-Efficient Context Parallelism for
// LLM Training", §2.1 and Fig. 1(a): the intra-document causal mask), with
// the keys a shard needs read from its own rows of K/V and from the
// compacted buffer of received prefix keys (§3.2). The softmax is evaluated
// online, keeping a running row maximum and exponential sum ("LLM Context
// Parallel in Production", "Core Principle: Split Q, Circulate KV").
//
// Work unit: one 128-row query tile of one piece (a shard's query range inside
// one document) for TWO query heads of the same GQA group, which read the
// same K/V tiles (a group of odd size, MHA included, pairs its last head with
// a repeat of itself whose results are not stored; that form of the kernel is
// a separate instantiation). Key tiles are 128 keys of one key segment (a run
// of keys held by the shard or received from others), so only tiles that contain
// useful (q, k) pairs are visited; tiles on the diagonal or at a segment end
// are masked element by element.
//
// CTA roles (320 threads, persistent over the work list):
//   warp 0      TMA producer: Q tiles of both heads, then K/V tiles into a
//               ring of shared-memory stages.
//   warp 1      MMA issuer (one thread): S_i = Q_i K^T and O_i += P_i V with
//               tcgen05.mma, accumulators in TMEM; allocates TMEM.
//   warps 2-5   softmax for head 0 of the pair, warps 6-9 for head 1: read
//               S from TMEM (one row per thread), mask, update the running
//               max / sum, write P (fp16) back into TMEM over S, rescale O in
//               TMEM when the max grows by more than 2^8, and finish the rows.
// P V takes P straight from TMEM (the A operand) and V from shared memory.
// Q K^T runs on the bf16 inputs; P V runs on fp16 operands (P <= 2^8 after
// the lazy rescale, V from an fp16 copy), whose 11 significant bits keep the
// rounding of P four times below bf16's. The MMAs of one thread run in issue
// order, so S_i(t+1), issued after P_i(t) V, lands only after that product
// has read P_i(t) and updated O_i: its completion also tells the softmax
// group that O_i may be rescaled.
// The two heads ping-pong: while one softmax group works on its S, the
// tensor core runs the other head's P*V and next S.
#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "sm103.cuh"

namespace fcp {

using namespace dev;

namespace {

constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

template <int D>
struct FwdCfg {
  static constexpr int kStages = D == 128 ? 5 : 8;
  static constexpr int kPanels = D / 64;                 // 64-column swizzle panels per row
  static constexpr int kTileBytes = 128 * D * 2;         // one Q/K/V tile
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kSmem = kKVOff + kStages * kTileBytes;
  static constexpr int kSmemAlloc = kSmem + 1024;        // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;                   // S_i at i*128; P_i (fp16) over its first 64
  static constexpr uint32_t kColO = 256;                 // O_i at 256 + i*D
};

// Key tiles of one query tile: every segment of the piece (those whose first
// field equals `filter`, if filter >= 0), clipped to the key block [lo, hi)
// and to keys <= q_last, cut into tiles of 128 keys. Segments may come in any
// key order (the ring order lists them by owner).
struct Walker {
  const int32_t* seg;
  int s, s_end, q_last, lo, hi, shift, filter;
  int pos, end, ks, src, srow;

  __device__ void init(const int32_t* segs, int seg_begin, int seg_count, int q_last_, int lo_,
                       int hi_, int shift_, int filter_) {
    seg = segs;
    s = seg_begin - 1;
    s_end = seg_begin + seg_count;
    q_last = q_last_;
    lo = lo_;
    hi = hi_;
    shift = shift_;
    filter = filter_;
    pos = end = 0;
  }
  __device__ bool next(int& src_o, int& row_o, int& key_o, int& n_o) {
    while (pos >= end) {
      if (++s >= s_end) return false;
      const int* g = seg + 4 * s;
      ks = __ldg(g + 2);
      src = __ldg(g + 0);
      if (ks > q_last || (filter >= 0 && src != filter)) continue;  // pos >= end still holds
      const int len = __ldg(g + 3);
      srow = __ldg(g + 1) - (src ? shift : 0);
      pos = max(ks, lo);
      end = min(min(ks + len, hi), q_last + 1);
    }
    src_o = src;
    row_o = srow + (pos - ks);
    key_o = pos;
    n_o = min(128, end - pos);
    pos += 128;
    return true;
  }
};

// A key segment's keys and source rows lie inside the sequence and inside
// the tensor its source names (own K/V rows, or the received rows behind
// tm_kb, `shift` rows into them). Checked build only.
__device__ __forceinline__ bool segment_ok(const FwdParams& p, const int* g) {
  const int src = __ldg(g + 0), row = __ldg(g + 1) - (__ldg(g + 0) ? p.kbuf_shift : 0);
  const int ks = __ldg(g + 2), len = __ldg(g + 3);
  const int rows = src ? p.kb_rows : p.T;
  return len >= 0 && ks >= 0 && ks <= p.T - len && row >= 0 && row <= rows - len;
}

// Key tiles a query tile visits; -1 (checked build) if one of its segments
// fails segment_ok.
__device__ __forceinline__ int count_key_tiles(const FwdParams& p, const int32_t* segs, int seg_begin,
                                               int seg_count, int q_last, int lo, int hi, int filter) {
  int n = 0;
  for (int s = seg_begin; s < seg_begin + seg_count; ++s) {
    const int* g = segs + 4 * s;
    if constexpr (kDeviceChecks) {
      if (!segment_ok(p, g)) return -1;
    }
    const int ks = __ldg(g + 2);
    if (ks > q_last || (filter >= 0 && __ldg(g) != filter)) continue;
    const int a = max(ks, lo);
    const int e = min(min(ks + __ldg(g + 3), hi), q_last + 1);
    if (e > a) n += (e - a + 127) / 128;
  }
  return n;
}

struct WorkItem {
  int q_start, q_rows, seg_begin, seg_count, h0, h1, g;
  bool bad;  // checked build: the unit's table entries are out of range (skip it)
};

// Head pairs per query tile: each GQA group's heads two at a time; an odd
// group's last pair holds one head (its second slot repeats the first and
// stores nothing).
__host__ __device__ __forceinline__ int head_pairs(int hq, int hkv) { return hkv * ((hq / hkv + 1) / 2); }

template <bool ODD>
__device__ __forceinline__ WorkItem decode(const FwdParams& p, int w) {
  const int hp_count = ODD ? head_pairs(p.hq, p.hkv) : p.hq / 2;
  const WorkSlot ws = work_slot(w, p.n_items, hp_count, p.order_block);
  const int item = __ldg(p.order + ws.pos);
  const int hp = ws.head;
  WorkItem it;
  it.bad = false;
  if constexpr (kDeviceChecks) {
    if (item < 0 || item >= p.n_tiles) {
      it = WorkItem{0, 0, 0, 0, 0, 0, 0, true};
      return it;
    }
  }
  const int* t = p.tiles + 4 * item;
  const int piece = __ldg(t + 0);
  if constexpr (kDeviceChecks) {
    if (piece < 0 || piece >= p.n_pieces) {
      it = WorkItem{0, 0, 0, 0, 0, 0, 0, true};
      return it;
    }
  }
  it.q_start = __ldg(t + 1);
  it.q_rows = __ldg(t + 2);
  it.seg_begin = __ldg(p.pieces + 8 * piece + 5);
  it.seg_count = __ldg(p.pieces + 8 * piece + 6);
  if constexpr (kDeviceChecks) {
    it.bad = it.q_rows < 1 || it.q_rows > 128 || it.q_start < 0 || it.q_start > p.T - it.q_rows ||
             it.seg_begin < 0 || it.seg_count < 0 || it.seg_begin > p.n_segs - it.seg_count;
  }
  if constexpr (ODD) {
    const int G = p.hq / p.hkv, per_group = (G + 1) / 2;
    it.g = hp / per_group;
    it.h0 = it.g * G + 2 * (hp % per_group);
    it.h1 = it.h0 + 1 < (it.g + 1) * G ? it.h0 + 1 : it.h0;
  } else {
    it.h0 = 2 * hp;
    it.h1 = it.h0 + 1;
    it.g = it.h0 / (p.hq / p.hkv);
  }
  return it;
}

template <int D, bool QK8, bool ODD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
                    const __grid_constant__ CUtensorMap tm_vb, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty, bar_drain;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kStages], bar_kv_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_p_ready[2], bar_o_done[2], bar_o_free[2];
  __shared__ WorkRing<4> ring;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_drain, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_ready[i], 128);
      mbar_init(&bar_o_done[i], 1);
      mbar_init(&bar_o_free[i], 128);
    }
    ring.init(1 + 8);  // the MMA thread and the eight softmax warps
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
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
  const int n_work = p.n_items * (ODD ? head_pairs(p.hq, p.hkv) : p.hq / 2);

  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sKV = smem + C::kKVOff;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kv_cnt = 0, q_iter = 0;
      uint32_t issued[C::kStages];
      for (int s = 0; s < C::kStages; ++s) issued[s] = 0;
      bool ok = true;
      uint32_t k = 0;
      for (int w = blockIdx.x; ok; w = next_work(p.work_counter)) {
        if (!(ok = ring.put<true>(k++, w, wc)) || w >= n_work) break;
        const WorkItem it = decode<ODD>(p, w);
        const int q_last = it.q_start + it.q_rows - 1;
        const int nt = it.bad ? -1 : count_key_tiles(p, p.segs, it.seg_begin, it.seg_count, q_last, p.kv_lo, p.kv_hi, p.seg_filter);
        if (nt < 0) atomicOr(p.err, kErrBadTable);
        if (nt <= 0) continue;
        if (q_iter > 0 && !(ok = mbar_wait_inline(&bar_q_empty, (q_iter - 1) & 1, wc))) break;
        if constexpr (QK8) {  // e4m3 rows of D bytes: one box per head
          mbar_arrive_expect_tx(&bar_q_full, 2 * 128 * D);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sQ + h * C::kTileBytes, &tm_q, &bar_q_full, 0, h ? it.h1 : it.h0, it.q_start);
        } else {
          mbar_arrive_expect_tx(&bar_q_full, 2 * C::kTileBytes);
          for (int h = 0; h < 2; ++h)
            for (int pn = 0; pn < C::kPanels; ++pn)
              tma_load_3d(sQ + h * C::kTileBytes + pn * 16384, &tm_q, &bar_q_full, pn * 64, h ? it.h1 : it.h0,
                          it.q_start);
        }
        ++q_iter;
        Walker wk;
        wk.init(p.segs, it.seg_begin, it.seg_count, q_last, p.kv_lo, p.kv_hi, p.kbuf_shift, p.seg_filter);
        int src, row, key, n;
        while (ok && wk.next(src, row, key, n)) {
          for (int kv = 0; kv < 2; ++kv) {
            const int s = kv_cnt % C::kStages;
            if (kv_cnt >= (uint32_t)C::kStages &&
                !(ok = mbar_wait_inline(&bar_kv_empty[s], ((kv_cnt / C::kStages) - 1) & 1, wc)))
              break;
            const CUtensorMap* tm = kv == 0 ? (src ? &tm_kb : &tm_k) : (src ? &tm_vb : &tm_v);
            if (QK8 && kv == 0) {  // e4m3 K tile: one box of D-byte rows
              mbar_arrive_expect_tx(&bar_kv_full[s], 128 * D);
              tma_load_3d(sKV + s * C::kTileBytes, tm, &bar_kv_full[s], 0, it.g, row);
            } else {
              mbar_arrive_expect_tx(&bar_kv_full[s], C::kTileBytes);
              for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(sKV + s * C::kTileBytes + pn * 16384, tm, &bar_kv_full[s], pn * 64, it.g,
                            row);
            }
            ++issued[s];
            ++kv_cnt;
          }
        }
      }
      // Every copy this thread started has landed before the CTA exits.
      for (int s = 0; s < C::kStages; ++s)
        if (issued[s]) mbar_drain(&bar_kv_full[s], (issued[s] - 1) & 1);
      if (q_iter) mbar_drain(&bar_q_full, (q_iter - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = QK8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_f16kind(128, D, false, true, false);  // fp16 P, V
      uint32_t kv_cnt = 0, q_iter = 0, items = 0;
      uint32_t p_cnt[2] = {0, 0};
      bool ok = true;
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      auto issue_s = [&](int i, uint32_t kstage) {
        const uint32_t qa = q_base + i * C::kTileBytes;
        const uint32_t ka = kv_base + kstage * C::kTileBytes;
        if constexpr (QK8) {  // K steps of 32 e4m3 values (32 bytes) along one 128-byte row
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_f8_ss(tmem + C::kColS + i * 128, smem_desc_sw128(qa + kk * 32, 0, 1024),
                      smem_desc_sw128(ka + kk * 32, 0, 1024), idesc_s, kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColS + i * 128, smem_desc_sw128(qa + off, 0, 1024),
                        smem_desc_sw128(ka + off, 0, 1024), idesc_s, kk > 0);
          }
        }
      };
      auto issue_o = [&](int i, uint32_t vstage, bool acc) {
        const uint32_t va = kv_base + vstage * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(tmem + C::kColO + i * D, tmem + C::kColS + i * 128 + kk * 8,
                     smem_desc_sw128(va + kk * 2048, 16384, 1024), idesc_o, (acc || kk > 0));
      };
      for (uint32_t k = 0; ok; ++k) {
        int w;
        if (!(ok = ring.get<true>(k, w, wc))) break;
        ring.release(k);
        if (w >= n_work) break;
        const WorkItem it = decode<ODD>(p, w);
        const int q_last = it.q_start + it.q_rows - 1;
        const int nt = it.bad ? -1 : count_key_tiles(p, p.segs, it.seg_begin, it.seg_count, q_last, p.kv_lo, p.kv_hi, p.seg_filter);
        if (nt <= 0) continue;
        if (!(ok = mbar_wait_inline(&bar_q_full, q_iter & 1, wc))) break;
        tc_fence_after();
        // S_0, S_1 of the first key tile.
        {
          const uint32_t c = kv_cnt, s = c % C::kStages;
          if (!(ok = mbar_wait_inline(&bar_kv_full[s], (c / C::kStages) & 1, wc))) break;
          tc_fence_after();
          issue_s(0, s);
          mma_commit(&bar_s_full[0]);
          issue_s(1, s);
          mma_commit(&bar_s_full[1]);
          mma_commit(&bar_kv_empty[s]);
          if (nt == 1) mma_commit(&bar_q_empty);  // no S left to issue: Q may be replaced
        }
        for (int t = 0; t < nt && ok; ++t) {
          const uint32_t cv = kv_cnt + 2 * t + 1, sv = cv % C::kStages;
          if (!(ok = mbar_wait_inline(&bar_kv_full[sv], (cv / C::kStages) & 1, wc))) break;
          for (int i = 0; i < 2; ++i) {
            if (!(ok = mbar_wait_inline(&bar_p_ready[i], p_cnt[i] & 1, wc))) break;
            ++p_cnt[i];
            if (t == 0 && items > 0 && !(ok = mbar_wait_inline(&bar_o_free[i], (items - 1) & 1, wc))) break;
            tc_fence_after();
            issue_o(i, sv, t > 0);
            if (t + 1 == nt) mma_commit(&bar_o_done[i]);  // O_i final: the epilogue may read it
            if (i == 1) mma_commit(&bar_kv_empty[sv]);
            if (t + 1 < nt) {
              const uint32_t ck = kv_cnt + 2 * (t + 1), sk = ck % C::kStages;
              if (!(ok = mbar_wait_inline(&bar_kv_full[sk], (ck / C::kStages) & 1, wc))) break;
              tc_fence_after();
              issue_s(i, sk);
              mma_commit(&bar_s_full[i]);
              if (i == 1) mma_commit(&bar_kv_empty[sk]);
              // After the last tile's S of both heads, Q is not read again:
              // the next unit's Q tiles may load while this unit finishes.
              if (i == 1 && t + 2 == nt) mma_commit(&bar_q_empty);
            }
          }
        }
        if (!ok) break;
        kv_cnt += 2 * nt;
        ++q_iter;
        ++items;
      }
      // Every MMA this thread issued has finished before TMEM is released.
      mma_commit(&bar_drain);
      mbar_drain(&bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // A warp reaches TMEM lanes 32 * (warp % 4) and up: warps 2-5 (and 6-9)
    // cover the four lane quarters of one head's tile.
    const int i = (warp - 2) >> 2;          // which head of the pair
    const int r = 32 * (warp & 3) + lane;   // tile row == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + C::kColS + i * 128;
    const uint32_t o_col = lane_base + C::kColO + i * D;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    const bool out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
    // e4m3 Q K^T: S comes out scaled by 2^kq 2^kk (powers of two, exact).
    const float scale_log2 = QK8 ? p.scale_log2 / (p.qk_scale[0] * p.qk_scale[1]) : p.scale_log2;
    for (uint32_t k = 0; ok; ++k) {
      int w = 0;
      ok = ring.get<true>(k, w, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) ring.release(k);
      if (w >= n_work) break;
      const WorkItem it = decode<ODD>(p, w);
      const int q_last = it.q_start + it.q_rows - 1;
      const int nt = it.bad ? -1 : count_key_tiles(p, p.segs, it.seg_begin, it.seg_count, q_last, p.kv_lo, p.kv_hi, p.seg_filter);
      if (nt < 0) continue;  // checked build: a unit with out-of-range table entries stores nothing
      const int q = it.q_start + r;
      bool row_valid = r < it.q_rows;
      int head = it.h0 + i;
      float m_run = -INFINITY, l = 0.f;
      if (nt > 0) {
        Walker wk;
        wk.init(p.segs, it.seg_begin, it.seg_count, q_last, p.kv_lo, p.kv_hi, p.kbuf_shift, p.seg_filter);
        int src, row, key, n;
        for (int t = 0; t < nt; ++t) {
          wk.next(src, row, key, n);
          ok = mbar_wait_inline(&bar_s_full[i], s_cnt & 1, wc);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          ++s_cnt;
          tc_fence_after();
          float s[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(s_col + c * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) s[c * 32 + j] = v[j];
          }
          tmem_ld_wait();
          if (key + 127 > it.q_start || n < 128) {
            const int lim = min(n, q - key + 1);  // keys [key, key+lim) are visible to row q
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) s[c] = -INFINITY;
          }
          // Row max: eight independent chains of three-input maxima (one warp
          // per scheduler: keep the dependent-latency chains short).
          float mx8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float m = fmaxf(s[j], s[j + 8]);
#pragma unroll
            for (int c = j + 16; c < 128; c += 16) m = fmax3(m, s[c], s[c + 8]);
            mx8[j] = m;
          }
          const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], fmax3(mx8[5], mx8[6], mx8[7]))) *
                           scale_log2;
          const float m_new = fmaxf(m_run, mx);
          const bool rescale = m_new > m_run + kRescaleThreshold;
          float alpha = 1.f;
          if (rescale) {
            alpha = ex2(m_run - m_new);
            m_run = m_new;
          }
          const float m_use = m_run == -INFINITY ? 0.f : m_run;
          // P = exp2(s * scale * log2e - m): fp16 pairs straight into TMEM columns
          // [0, 64) of S_i, 64 score columns at a time. The scaling and the row
          // sum run on packed pairs; sums of column c go to accumulator c mod 8.
          const uint64_t c2 = f2(scale_log2, scale_log2), nm2 = f2(-m_use, -m_use);
          uint64_t rs2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // 32 score columns -> 16 TMEM columns of P
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int c = 32 * q4 + 2 * j;
              float x0, x1;
              f2_split(f2_fma(f2(s[c], s[c + 1]), c2, nm2), x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              rs2[j & 3] = f2_add(rs2[j & 3], f2(p0, p1));
              pk[j] = pack_f16(p0, p1);
            }
            tmem_st16(s_col + 16 * q4, pk);
          }
          float rs[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) f2_split(rs2[j], rs[2 * j], rs[2 * j + 1]);
          const float rowsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
          // P_i(t-1) V has completed (see above), so O_i can be rescaled now.
          if (t > 0 && __any_sync(0xffffffffu, rescale)) {
            if (lane == 0 && p.rescale_count) atomicAdd(p.rescale_count, 1);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float v[32];
              tmem_ld32(o_col + c * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] *= alpha;
              tmem_st32(o_col + c * 32, v);
            }
          }
          l = l * alpha + rowsum;
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bar_p_ready[i]);
        }
        if (!ok) break;
        ok = mbar_wait_inline(&bar_o_done[i], o_cnt & 1, wc);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        ++o_cnt;
        tc_fence_after();
      }
      // Epilogue: O / l and LSE for this row. The second slot of an odd
      // group's last pair repeats the first head: it runs but stores nothing.
      if constexpr (ODD) {
        head = i ? it.h1 : it.h0;
        row_valid = row_valid && (i == 0 || it.h1 != it.h0);
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t obase = ((size_t)q * p.hq + head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        if (nt > 0) {
          tmem_ld32(o_col + c * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        // A thread writes its own row: 32-byte stores where `out` allows
        // them (each row segment is then whole sectors), else 16-byte ones.
        if (row_valid) {
          if (p.out_f32) {
            float* dst = static_cast<float*>(p.out) + obase + c * 32;
            if (out_v8) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_global_v8(dst + 8 * j, __float_as_uint(v[8 * j] * inv), __float_as_uint(v[8 * j + 1] * inv),
                             __float_as_uint(v[8 * j + 2] * inv), __float_as_uint(v[8 * j + 3] * inv),
                             __float_as_uint(v[8 * j + 4] * inv), __float_as_uint(v[8 * j + 5] * inv),
                             __float_as_uint(v[8 * j + 6] * inv), __float_as_uint(v[8 * j + 7] * inv));
            } else {
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv);
            }
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + obase + c * 32;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16(v[2 * j] * inv, v[2 * j + 1] * inv);
            if (out_v8) {
              st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int j = 0; j < 4; ++j) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            }
          }
        }
      }
      if (row_valid)
        p.lse[(size_t)head * p.T + q] = l > 0.f ? (m_run + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (nt > 0) {
        tc_fence_before();
        mbar_arrive(&bar_o_free[i]);
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

template <int D, bool QK8, bool ODD>
static int launch_fwd_impl(const FwdLaunch& a, cudaStream_t st) {
  using C = FwdCfg<D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_fwd_kernel<D, QK8, ODD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemAlloc) != cudaSuccess)
      return FCP_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int n_work = a.p.n_items * head_pairs(a.p.hq, a.p.hkv);
  if (n_work == 0) return FCP_OK;
  const int grid = n_work < a.num_sms ? n_work : a.num_sms;
  // Blocks of query tiles such that one block's head pairs of one KV head
  // fill the grid: the CTAs running together stream the same K/V rows.
  FwdParams p = a.p;
  const int pairs_per_kv = head_pairs(p.hq, p.hkv) / p.hkv;
  p.order_block = grid / pairs_per_kv > 0 ? grid / pairs_per_kv : 1;
  attn_fwd_kernel<D, QK8, ODD><<<grid, kThreads, C::kSmemAlloc, st>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_kb, a.tm_vb,
                                                                p);
  return cudaGetLastError() == cudaSuccess ? FCP_OK : FCP_ERR_CUDA;
}

template <bool ODD>
static int launch_fwd_any(const FwdLaunch& a, cudaStream_t st) {
  if (a.qk8) return a.d == 128 ? launch_fwd_impl<128, true, ODD>(a, st) : FCP_ERR_UNSUPPORTED;
  if (a.d == 128) return launch_fwd_impl<128, false, ODD>(a, st);
  if (a.d == 64) return launch_fwd_impl<64, false, ODD>(a, st);
  return FCP_ERR_UNSUPPORTED;
}

int launch_attn_fwd(const FwdLaunch& a, cudaStream_t st) {
  return (a.p.hq / a.p.hkv) % 2 ? launch_fwd_any<true>(a, st) : launch_fwd_any<false>(a, st);
}

}  // namespace fcp
