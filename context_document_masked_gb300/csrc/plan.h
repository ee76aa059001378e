// Host plan object of libfcp and the device work tables derived from it.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/fcp.h"

namespace fcp {

constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // keys per tile
constexpr int kCopyRows = 32; // rows per gather task
constexpr int kRowChunk = 128;

struct Piece {
  int32_t doc, start, end;
};

struct Shard {
  std::vector<Piece> pieces;
  std::vector<fcp_range> kv_need;
  std::vector<fcp_range> kv_remote;
  int64_t tokens = 0, W = 0, remote_rows = 0, kbuf_base = 0;
  // Tiles the kernels visit (per query head): forward query x key tiles,
  // forward query tiles, forward tiles needing a per-element mask; backward
  // key x query tiles and backward key tiles.
  int64_t fwd_tiles = 0, fwd_qtiles = 0, fwd_masked = 0, bwd_tiles = 0, bwd_ktiles = 0;
};

// Device table ids (index into fcp_dev_plan::tables / counts).
enum Table {
  TB_PIECES = 0,   // 8 ints: shard, doc, start, end, doc_start, seg_begin, seg_count, pad
  TB_SEGS,         // 4 ints: src (0 own K/V, 1 kbuf/vbuf), src_row, key_start, len
  TB_FTILES,       // 4 ints: piece, q_start, q_rows, cost   (grouped by shard)
  TB_FORDER,       // all-shards longest-first order of TB_FTILES
  TB_FSHARD,       // N+1 offsets into TB_FTILES
  TB_BTILES,       // kBwdTileInts ints: key_start, key_rows, src, src_row, then two query
                   // ranges (first tile start, piece end, tile count; the first may be
                   // empty), piece, seg
  TB_BORDER,
  TB_BSHARD,
  TB_COPY,         // 4 ints: src_row, dst_row, nrows, shard (grouped by shard)
  TB_CSHARD,
  TB_ROWS,         // 2 ints: start, nrows (grouped by shard)
  TB_RSHARD,
  TB_IDENT,        // 0, 1, 2, ... (indirection for one-shard launches)
  TB_KBASE,        // N+1 kbuf row offsets
  TB_RPIECES,      // TB_PIECES with seg_begin / seg_count into TB_RSEGS
  TB_RSEGS,        // 4 ints: ring distance, src_row (= key_start), key_start, len
  TB_COUNT
};

struct Plan {
  int32_t N = 0;
  int64_t T = 0;
  std::vector<int32_t> D, off;
  std::vector<Shard> shards;
  std::vector<uint8_t> per_doc;
  std::vector<int32_t> pd_order;
  double imbalance = 1.0;
  int64_t eq4 = 0, eq5 = 0, eq2dev = 0, total_remote = 0;
  int32_t iterations = 1;
  std::vector<int32_t> dev;          // serialized device tables
  int32_t tab_off[TB_COUNT] = {0};
  int32_t tab_cnt[TB_COUNT] = {0};

  int build_llama3();
  int build_perdoc();
  int build_algorithm1(double R, bool tiles);
  void finish(std::vector<std::vector<Piece>>& wp);
  void build_work_tables();
};

}  // namespace fcp

struct fcp_plan : fcp::Plan {};

namespace fcp {
int make_plan(const int32_t* doclens, int32_t n_docs, int32_t cp, int32_t policy, double R,
              fcp_plan_t** out);

// FCP_OK if `dp` describes its host plan exactly (table offsets, counts, sizes,
// a 16-byte aligned base) and -1 <= shard < the plan's shard count;
// FCP_ERR_INVALID_ARG otherwise. Host only, no CUDA call.
int check_dev_plan(const fcp_dev_plan* dp, int32_t shard);
}  // namespace fcp
