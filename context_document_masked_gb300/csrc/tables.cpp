// Device work tables of a plan.
//
// From each shard's pieces (query ranges) and key needs the planner derives
// what the kernels iterate over:
//   - key segments: the keys a piece needs, [doc start, piece end), cut into
//     runs that the shard holds itself (read from K/V at their global rows)
//     and runs received from other shards (read from the compacted
//     kbuf/vbuf, in the order of the shard's kv_remote list);
//   - forward query tiles of <= 128 rows, each inside one piece;
//   - backward units: key tiles of <= 128 keys, each inside one segment,
//     with the query tiles that see them. Where a shard holds two pieces of
//     one document, every key tile of the earlier piece is also a key tile of
//     the later one (both walks cut [doc start, earlier end) at the same
//     points), so that tile is one unit whose steps run over both pieces'
//     query tiles: dK/dV of the tile leave the kernel once, not twice;
//   - gather runs (<= kCopyRows rows) and preprocess row chunks.
// Tiles are listed piece by piece (pieces ordered by their longest tile) and,
// inside a piece, longest first (by the number of tile pairs they cover): the
// CTAs running at the same time then share one piece's query rows and keys
// in L2, and the long rows start early.
#include <algorithm>
#include <array>
#include <numeric>

#include "kernels.h"
#include "plan.h"

namespace fcp {

namespace {

struct Seg { int32_t src, src_row, key_start, len; };

int64_t count_key_tiles(const std::vector<Seg>& segs, int32_t seg_begin, int32_t seg_count,
                        int32_t q_last) {
  int64_t n = 0;
  for (int32_t s = seg_begin; s < seg_begin + seg_count; ++s) {
    const Seg& g = segs[s];
    if (g.key_start > q_last) break;
    int64_t len = std::min<int64_t>(g.len, (int64_t)q_last - g.key_start + 1);
    n += (len + kTileN - 1) / kTileN;
  }
  return n;
}

// Key tiles of query tile [q0, q_last] that need a per-element mask: those
// reaching past q0 (the diagonal) or shorter than a full tile (a segment end).
int64_t count_masked_tiles(const std::vector<Seg>& segs, int32_t seg_begin, int32_t seg_count,
                           int32_t q0, int32_t q_last) {
  int64_t n = 0;
  for (int32_t s = seg_begin; s < seg_begin + seg_count; ++s) {
    const Seg& g = segs[s];
    if (g.key_start > q_last) break;
    const int32_t end = std::min<int64_t>((int64_t)g.key_start + g.len, (int64_t)q_last + 1);
    for (int32_t k = g.key_start; k < end; k += kTileN) {
      const int32_t nk = std::min(kTileN, end - k);
      if (k + kTileN - 1 > q0 || nk < kTileN) ++n;
    }
  }
  return n;
}

void append(std::vector<int32_t>& dev, int32_t* off, int32_t* cnt, int tb,
            const std::vector<int32_t>& data, int32_t n_entries) {
  while (dev.size() % 4) dev.push_back(0);  // 16-byte alignment of every table
  off[tb] = (int32_t)dev.size();
  cnt[tb] = n_entries;
  dev.insert(dev.end(), data.begin(), data.end());
}

}  // namespace

void Plan::build_work_tables() {
  std::vector<int32_t> pieces, segs_flat, ftiles, btiles, copy, rows;
  std::vector<Seg> segs;
  std::vector<int32_t> fshard(N + 1, 0), bshard(N + 1, 0), cshard(N + 1, 0), rshard(N + 1, 0);
  std::vector<int64_t> fcost, bcost;
  std::vector<int32_t> fpiece, bpiece;
  struct PieceInfo { int32_t id, doc, start, end, seg_begin, seg_count; };
  int32_t piece_id = 0;
  for (int32_t j = 0; j < N; ++j) {
    const Shard& sh = shards[j];
    fshard[j] = (int32_t)(ftiles.size() / 4);
    bshard[j] = (int32_t)(btiles.size() / kBwdTileInts);
    cshard[j] = (int32_t)(copy.size() / 4);
    rshard[j] = (int32_t)(rows.size() / 2);
    // Position of each remote range inside this shard's kbuf.
    std::vector<int64_t> rpos(sh.kv_remote.size());
    int64_t acc = sh.kbuf_base;
    for (size_t r = 0; r < sh.kv_remote.size(); ++r) {
      rpos[r] = acc;
      const fcp_range& rr = sh.kv_remote[r];
      for (int32_t a = rr.start; a < rr.end; a += kCopyRows) {
        int32_t nr = std::min(kCopyRows, rr.end - a);
        copy.insert(copy.end(), {a, (int32_t)(acc + (a - rr.start)), nr, j});
      }
      acc += rr.end - rr.start;
    }
    std::vector<PieceInfo> pinfo;
    for (const Piece& p : sh.pieces) {
      const int32_t ds = off[p.doc];
      const int32_t seg_begin = (int32_t)segs.size();
      // Walk [ds, p.end): own pieces of this doc and remote ranges of this doc
      // are disjoint and together cover the needed range.
      int32_t t = ds;
      while (t < p.end) {
        bool found = false;
        for (const Piece& o : sh.pieces) {
          if (o.doc == p.doc && o.start <= t && t < o.end) {
            int32_t e = std::min(o.end, p.end);
            segs.push_back(Seg{0, t, t, e - t});
            t = e;
            found = true;
            break;
          }
        }
        if (found) continue;
        for (size_t r = 0; r < sh.kv_remote.size(); ++r) {
          const fcp_range& rr = sh.kv_remote[r];
          if (rr.doc == p.doc && rr.start <= t && t < rr.end) {
            int32_t e = std::min(rr.end, p.end);
            segs.push_back(Seg{1, (int32_t)(rpos[r] + (t - rr.start)), t, e - t});
            t = e;
            found = true;
            break;
          }
        }
        if (!found) break;  // unreachable for a consistent plan
      }
      const int32_t seg_count = (int32_t)segs.size() - seg_begin;
      pieces.insert(pieces.end(), {j, p.doc, p.start, p.end, ds, seg_begin, seg_count, 0});
      // Forward query tiles.
      for (int32_t q0 = p.start; q0 < p.end; q0 += kTileM) {
        int32_t qr = std::min(kTileM, p.end - q0);
        int64_t c = count_key_tiles(segs, seg_begin, seg_count, q0 + qr - 1);
        ftiles.insert(ftiles.end(), {piece_id, q0, qr, (int32_t)std::min<int64_t>(c, 1 << 30)});
        fcost.push_back(c);
        fpiece.push_back(piece_id);
        shards[j].fwd_tiles += c;
        shards[j].fwd_qtiles += 1;
        shards[j].fwd_masked += count_masked_tiles(segs, seg_begin, seg_count, q0, q0 + qr - 1);
      }
      pinfo.push_back(PieceInfo{piece_id, p.doc, p.start, p.end, seg_begin, seg_count});
      for (int32_t a = p.start; a < p.end; a += kRowChunk)
        rows.insert(rows.end(), {a, std::min(kRowChunk, p.end - a)});
      ++piece_id;
    }
    // Backward units: every key tile of every segment of a piece; the queries
    // that see it are the piece's rows at or after the tile start. A document
    // with exactly two pieces in this shard gives one unit per key tile of the
    // later piece, the earlier piece's query tiles attached to the tiles that
    // lie before its end.
    auto q_tiles = [](const PieceInfo& pc, int32_t key, int32_t* q0, int32_t* n) {
      const int32_t qt_first = (std::max(key, pc.start) - pc.start) / kTileM;
      *q0 = pc.start + qt_first * kTileM;
      *n = (pc.end - pc.start + kTileM - 1) / kTileM - qt_first;
    };
    for (size_t i = 0; i < pinfo.size(); ++i) {
      const PieceInfo& pc = pinfo[i];
      int n_same = 0, partner = -1;
      for (size_t o = 0; o < pinfo.size(); ++o)
        if (pinfo[o].doc == pc.doc) {
          ++n_same;
          if (o != i) partner = (int)o;
        }
      if (n_same != 2) partner = -1;
      if (partner >= 0 && pinfo[partner].start > pc.start) continue;  // emitted with the later piece
      for (int32_t s = pc.seg_begin; s < pc.seg_begin + pc.seg_count; ++s) {
        const Seg& g = segs[s];
        for (int32_t k0 = 0; k0 < g.len; k0 += kTileN) {
          const int32_t kr = std::min(kTileN, g.len - k0);
          const int32_t key = g.key_start + k0;
          int32_t qa0 = 0, qa_end = 0, na = 0, qb0, nb;
          if (partner >= 0 && key < pinfo[partner].end) {
            q_tiles(pinfo[partner], key, &qa0, &na);
            qa_end = pinfo[partner].end;
          }
          q_tiles(pc, key, &qb0, &nb);
          btiles.insert(btiles.end(), {key, kr, g.src, g.src_row + k0, qa0, qa_end, na, qb0, pc.end, nb, pc.id, s});
          bcost.push_back(na + nb);
          bpiece.push_back(pc.id);
          shards[j].bwd_tiles += na + nb;
          shards[j].bwd_ktiles += 1;
        }
      }
    }
  }
  fshard[N] = (int32_t)(ftiles.size() / 4);
  bshard[N] = (int32_t)(btiles.size() / kBwdTileInts);
  cshard[N] = (int32_t)(copy.size() / 4);
  rshard[N] = (int32_t)(rows.size() / 2);
  // Piece-major, longest-first orders. A piece's rank is the position of its
  // longest tile among all pieces' longest tiles.
  auto ranks = [&](const std::vector<int64_t>& cost, const std::vector<int32_t>& piece) {
    const int32_t np = piece_id;
    std::vector<int64_t> pmax(np, -1);
    for (size_t i = 0; i < cost.size(); ++i) pmax[piece[i]] = std::max(pmax[piece[i]], cost[i]);
    std::vector<int32_t> idx(np), rank(np);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return pmax[a] > pmax[b]; });
    for (int32_t r = 0; r < np; ++r) rank[idx[r]] = r;
    return rank;
  };
  const std::vector<int32_t> frank = ranks(fcost, fpiece), brank = ranks(bcost, bpiece);
  auto sort_group = [](std::vector<int32_t>& tab, int width, std::vector<int64_t>& cost,
                       std::vector<int32_t>& piece, const std::vector<int32_t>& rank,
                       const std::vector<int32_t>& shard_off, int N) {
    std::vector<int32_t> out(tab.size()), pout(piece.size());
    std::vector<int64_t> cout(cost.size());
    for (int j = 0; j < N; ++j) {
      std::vector<int32_t> idx(shard_off[j + 1] - shard_off[j]);
      std::iota(idx.begin(), idx.end(), shard_off[j]);
      std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
        if (rank[piece[a]] != rank[piece[b]]) return rank[piece[a]] < rank[piece[b]];
        return cost[a] > cost[b];
      });
      for (size_t i = 0; i < idx.size(); ++i) {
        std::copy(tab.begin() + (size_t)idx[i] * width, tab.begin() + (size_t)(idx[i] + 1) * width,
                  out.begin() + (size_t)(shard_off[j] + i) * width);
        cout[shard_off[j] + i] = cost[idx[i]];
        pout[shard_off[j] + i] = piece[idx[i]];
      }
    }
    tab.swap(out);
    cost.swap(cout);
    piece.swap(pout);
  };
  sort_group(ftiles, 4, fcost, fpiece, frank, fshard, N);
  sort_group(btiles, kBwdTileInts, bcost, bpiece, brank, bshard, N);
  std::vector<int32_t> forder(fcost.size()), border(bcost.size());
  std::iota(forder.begin(), forder.end(), 0);
  std::iota(border.begin(), border.end(), 0);
  std::stable_sort(forder.begin(), forder.end(), [&](int32_t a, int32_t b) {
    if (frank[fpiece[a]] != frank[fpiece[b]]) return frank[fpiece[a]] < frank[fpiece[b]];
    return fcost[a] > fcost[b];
  });
  std::stable_sort(border.begin(), border.end(), [&](int32_t a, int32_t b) {
    if (brank[bpiece[a]] != brank[bpiece[b]]) return brank[bpiece[a]] < brank[bpiece[b]];
    return bcost[a] > bcost[b];
  });
  size_t nid = std::max({forder.size(), border.size(), copy.size() / 4, rows.size() / 2, (size_t)1});
  std::vector<int32_t> ident(nid);
  std::iota(ident.begin(), ident.end(), 0);
  std::vector<int32_t> kbase(N + 1);
  for (int32_t j = 0; j < N; ++j) kbase[j] = (int32_t)shards[j].kbuf_base;
  kbase[N] = (int32_t)total_remote;

  // Ring order ("LLM Context Parallel in Production", "Ring Attention": at
  // step s shard j holds the KV block of shard (j - s) mod N). A piece's
  // needed keys [doc start, piece end) are cut into runs by the shard that
  // owns them and listed by ring distance (j - owner) mod N, own keys first,
  // each run read from K/V at its global rows.
  std::vector<std::vector<std::array<int32_t, 3>>> doc_runs(D.size());  // (start, end, owner)
  for (int32_t j = 0; j < N; ++j)
    for (const Piece& p : shards[j].pieces) doc_runs[p.doc].push_back({p.start, p.end, j});
  for (auto& v : doc_runs) std::sort(v.begin(), v.end());
  std::vector<int32_t> rpieces, rsegs;
  for (int32_t j = 0; j < N; ++j) {
    for (const Piece& p : shards[j].pieces) {
      std::vector<std::array<int32_t, 3>> runs;  // (distance, start, len)
      for (const auto& r : doc_runs[p.doc]) {
        if (r[0] >= p.end) break;
        const int32_t e = std::min(r[1], p.end);
        const int32_t dist = ((j - r[2]) % N + N) % N;
        if (!runs.empty() && runs.back()[0] == dist && runs.back()[1] + runs.back()[2] == r[0])
          runs.back()[2] += e - r[0];
        else
          runs.push_back({dist, r[0], e - r[0]});
      }
      std::stable_sort(runs.begin(), runs.end(),
                       [](const std::array<int32_t, 3>& a, const std::array<int32_t, 3>& b) { return a[0] < b[0]; });
      const int32_t begin = (int32_t)(rsegs.size() / 4);
      for (const auto& r : runs) rsegs.insert(rsegs.end(), {r[0], r[1], r[1], r[2]});
      rpieces.insert(rpieces.end(), {j, p.doc, p.start, p.end, off[p.doc], begin, (int32_t)runs.size(), 0});
    }
  }

  for (const Seg& g : segs) segs_flat.insert(segs_flat.end(), {g.src, g.src_row, g.key_start, g.len});
  dev.clear();
  append(dev, tab_off, tab_cnt, TB_PIECES, pieces, (int32_t)(pieces.size() / 8));
  append(dev, tab_off, tab_cnt, TB_SEGS, segs_flat, (int32_t)segs.size());
  append(dev, tab_off, tab_cnt, TB_FTILES, ftiles, (int32_t)(ftiles.size() / 4));
  append(dev, tab_off, tab_cnt, TB_FORDER, forder, (int32_t)forder.size());
  append(dev, tab_off, tab_cnt, TB_FSHARD, fshard, N + 1);
  append(dev, tab_off, tab_cnt, TB_BTILES, btiles, (int32_t)(btiles.size() / kBwdTileInts));
  append(dev, tab_off, tab_cnt, TB_BORDER, border, (int32_t)border.size());
  append(dev, tab_off, tab_cnt, TB_BSHARD, bshard, N + 1);
  append(dev, tab_off, tab_cnt, TB_COPY, copy, (int32_t)(copy.size() / 4));
  append(dev, tab_off, tab_cnt, TB_CSHARD, cshard, N + 1);
  append(dev, tab_off, tab_cnt, TB_ROWS, rows, (int32_t)(rows.size() / 2));
  append(dev, tab_off, tab_cnt, TB_RSHARD, rshard, N + 1);
  append(dev, tab_off, tab_cnt, TB_IDENT, ident, (int32_t)ident.size());
  append(dev, tab_off, tab_cnt, TB_KBASE, kbase, N + 1);
  append(dev, tab_off, tab_cnt, TB_RPIECES, rpieces, (int32_t)(rpieces.size() / 8));
  append(dev, tab_off, tab_cnt, TB_RSEGS, rsegs, (int32_t)(rsegs.size() / 4));
  while ((dev.size() * 4) % 256) dev.push_back(0);
}

}  // namespace fcp
