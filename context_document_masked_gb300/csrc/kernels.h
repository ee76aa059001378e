// Launch interfaces of the libfcp device kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/fcp.h"

// FCP_DEVICE_CHECKS=1 builds the checked library: every index the kernels
// read from the plan's device tables is checked against the table sizes and
// the tensors' rows before use; a failed check sets bit kErrBadTable of the
// error word (fcp_get_device_status: FCP_ERR_INVALID_ARG) and the kernel
// skips that work unit. It never traps.
#ifndef FCP_DEVICE_CHECKS
#define FCP_DEVICE_CHECKS 0
#endif

namespace fcp {

constexpr bool kDeviceChecks = FCP_DEVICE_CHECKS != 0;
constexpr int kErrBadTable = 8;

// Ints per backward unit in the plan's TB_BTILES table.
constexpr int kBwdTileInts = 12;

struct FwdParams {
  const int32_t* pieces;   // plan piece table
  const int32_t* segs;     // key segments
  const int32_t* tiles;    // query tiles (piece, q_start, q_rows, cost)
  const int32_t* order;    // tile indices to run, longest first
  int32_t n_items;
  int32_t kbuf_shift;      // subtracted from received-key rows (one-shard launches)
  int32_t kv_lo, kv_hi;    // key block
  int32_t seg_filter;      // -1: every key segment; else only segments whose first field equals it
  int32_t T, hq, hkv;
  float scale_log2;        // softmax scale * log2(e)
  int32_t out_f32;
  void* out;
  float* lse;
  int* err;
  int* work_counter;       // zero at launch (set by the preceding kernel of the call)
  const float* qk_scale;   // e4m3 Q K^T variant: the scales 2^kq, 2^kk of Q and K (else unused)
  int* rescale_count;      // if not null: +1 per warp each time O is rescaled after a later key tile
  int32_t order_block;     // work decode: items per block (set by the launch, see work_slot)
  int32_t n_tiles, n_pieces, n_segs, kb_rows;  // table sizes, rows behind tm_kb (checked build)
  int64_t wait_ns;
};

struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_kb, tm_vb;
  FwdParams p;
  int d;
  int num_sms;
  bool qk8;                // Q, K, received K as e4m3 (boxes of 128 bytes x 1 x 128)
};

struct BwdParams {
  const int32_t* pieces;
  const int32_t* tiles;    // backward units, kBwdTileInts ints each (plan.h, TB_BTILES)
  const int32_t* order;
  int32_t n_items;
  int32_t kbuf_shift;
  int32_t T, hq, hkv;
  float scale;             // softmax scale
  float scale_log2;
  const float* lse;        // [Hq][T]
  const float* delta;      // [Hq][T] rowsum(dO * O)
  float* dq;               // [T][Hq][d] fp32, accumulated
  float* dk;               // [T][Hkv][d] fp32, accumulated
  float* dv;
  int* err;
  int* work_counter;       // zero at launch (set by the preprocess)
  int32_t order_block;     // work decode: items per block (set by the launch, see work_slot)
  int32_t n_tiles, kb_rows;  // TB_BTILES size, rows behind tm_kb/tm_vb (checked build)
  int64_t wait_ns;
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_kb, tm_vb;
  CUtensorMap tm_dq;  // dQ fp32 [T][Hq][d], boxes of 32 x 1 x 128 (reduce-add target)
  CUtensorMap tm_dk, tm_dv;  // dK, dV fp32 [T][Hkv][d], same boxes (reduce-add targets)
  BwdParams p;
  int d;
  int num_sms;
};

int launch_attn_fwd(const FwdLaunch& a, cudaStream_t st);
int launch_attn_bwd(const BwdLaunch& a, cudaStream_t st);

// Limit of every bounded device wait (fcp_debug_set_wait_limit), in ns.
int64_t wait_limit_ns();

// Row statistics D_i = <dO_i, O_i> for the rows of the given row chunks, dQ
// rows set to zero, and fp16 copies of Q and dO for the backward's MMAs.
// *zero_word (if not null) is set to 0: the work counter of the kernel that
// follows in the same stream.
// n_rows_table: entries of `rows` (the checked build bounds the chunk indices).
int launch_bwd_preprocess(const void* out, bool out_f32, const void* dout, const void* q,
                          const int32_t* rows,
                          const int32_t* order, int32_t n_chunks, int32_t n_rows_table, int32_t T, int32_t hq,
                          int32_t d,
                          float* delta, float* dq, void* q16, void* do16, int* err, int* zero_word,
                          cudaStream_t st);

// fp16 copy of a bf16 array of n_elems (a multiple of 8) elements; *zero_word
// (if not null) is set to 0, as above.
int launch_convert_f16(const void* src, void* dst, int64_t n_elems, int* err, int* zero_word,
                       int num_sms, cudaStream_t st);

// bf16 copy (round to nearest even) of an fp32 array of n_elems (a multiple
// of 8) elements.
int launch_round_bf16(const float* src, void* dst, int64_t n_elems, int num_sms, cudaStream_t st);

// e4m3 copy of a bf16 array of n_elems (a multiple of 8) elements, scaled by
// the power of two 2^k, the largest with max|x| * 2^k <= 448 (exact to undo).
// *amax_bits must be zero on entry (it receives the bits of max|x|); the
// scale goes to *scale_out.
int launch_quant_e4m3(const void* src, void* dst, int64_t n_elems, unsigned* amax_bits,
                      float* scale_out, int num_sms, cudaStream_t st);
// The same with a scale computed before (from *amax_bits of another tensor):
// rows copied from that tensor share its scale.
int launch_quant_e4m3_with(const void* src, void* dst, int64_t n_elems, const unsigned* amax_bits,
                           int num_sms, cudaStream_t st);

// Gather of received KV rows: tasks (src_row, dst_row, nrows, shard); K/V
// hold src_rows rows, kbuf/vbuf dst_rows (bounds of the checked build).
int launch_gather(const void* k, const void* v, const int32_t* tasks, int32_t n_tasks,
                  int32_t dst_shift, int64_t row_bytes, void* kbuf, void* vbuf, int32_t src_rows,
                  int32_t dst_rows, int num_sms, cudaStream_t st);

int launch_merge(const float* o_parts, const float* lse_parts, int32_t B, int64_t rows, int32_t hq,
                 int32_t d, void* out, float* lse_out, int num_sms, cudaStream_t st);

}  // namespace fcp
