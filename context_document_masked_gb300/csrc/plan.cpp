// Host sharding planner of libfcp.
//
// Builds, from the document lengths of one packed sequence, the CP sharding
// plans described in "FlashCP: Load-Balanced Communication-Efficient Context
// Parallelism for LLM Training":
//   - Llama3 CP (§2.2): the sequence in 2N equal chunks, worker i holds
//     chunks i and 2N-1-i (the pairing rule of §2.3);
//   - Per-Doc (§2.3): every document in 2N chunks with floor(cL/2N)
//     boundaries, worker i holds chunks i and 2N-1-i;
//   - Whole-Doc and hybrid (§3.3, §3.4, Algorithm 1): greedy whole-document
//     placement by workload, an equal-token repair that moves or splits the
//     most recent piece of the worker with the largest token excess (its head
//     goes to the worker with the largest deficit), and, while the imbalance
//     exceeds R, the longest remaining document moves to Per-Doc sharding.
// and derives the per-shard key needs of §3.2 (a piece [a,b) of a document
// starting at o needs keys [o,b); keys held by other shards are "remote").
// Workload of a piece: W = (2p + s + 1) s / 2 (§3.1).
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <limits>

namespace fcp {

static inline int64_t piece_work(int64_t p, int64_t s) { return (2 * p + s + 1) * s / 2; }

// The 2N Per-Doc chunks of one document, as pieces per worker.
static void perdoc_pieces(int32_t doc, int64_t L, int64_t o, int32_t N,
                          std::vector<std::vector<Piece>>& out) {
  for (int32_t i = 0; i < N; ++i) {
    const int32_t cs[2] = {i, 2 * N - 1 - i};
    for (int32_t c : cs) {
      int64_t a = o + (int64_t)c * L / (2 * N);
      int64_t b = o + (int64_t)(c + 1) * L / (2 * N);
      if (b > a) out[i].push_back(Piece{doc, (int32_t)a, (int32_t)b});
    }
  }
}

static int64_t sum_work(const std::vector<Piece>& ps, const std::vector<int32_t>& off) {
  int64_t w = 0;
  for (const Piece& p : ps) w += piece_work(p.start - off[p.doc], p.end - p.start);
  return w;
}

// Kernel-unit cost of a shard (the hybrid_tiles policy): for each of its
// ceil(s/128) query tiles, the ceil((p + e)/128) key tiles of the document's
// causal prefix up to the tile's local end e, plus one per query tile -- the
// tiles the attention kernels visit when the keys form one run from the
// document start. Measured per-shard time on GB300 (forward + backward)
// fits visited tiles and query tiles with equal weights.
static int64_t tile_cost(int64_t p, int64_t s) {
  const int64_t nq = (s + kTileM - 1) / kTileM;
  int64_t c = nq;
  for (int64_t t = 0; t < nq; ++t) c += (p + std::min<int64_t>(kTileM * (t + 1), s) + kTileN - 1) / kTileN;
  return c;
}

static int64_t sum_cost(const std::vector<Piece>& ps, const std::vector<int32_t>& off, bool tiles) {
  if (!tiles) return sum_work(ps, off);
  int64_t w = 0;
  for (const Piece& p : ps) w += tile_cost(p.start - off[p.doc], p.end - p.start);
  return w;
}

static int64_t sum_tokens(const std::vector<Piece>& ps) {
  int64_t t = 0;
  for (const Piece& p : ps) t += p.end - p.start;
  return t;
}

void Plan::finish(std::vector<std::vector<Piece>>& wp) {
  const int32_t n = (int32_t)D.size();
  shards.assign(N, Shard{});
  for (int32_t j = 0; j < N; ++j) {
    std::vector<Piece> ps = wp[j];
    std::stable_sort(ps.begin(), ps.end(),
                     [](const Piece& a, const Piece& b) { return a.start < b.start; });
    Shard& sh = shards[j];
    for (const Piece& p : ps) {  // adjacent pieces of one document form one shard
      if (!sh.pieces.empty() && sh.pieces.back().doc == p.doc && sh.pieces.back().end == p.start)
        sh.pieces.back().end = p.end;
      else
        sh.pieces.push_back(p);
    }
    // kv_need: per document touched, [doc start, max piece end).
    for (size_t a = 0; a < sh.pieces.size();) {
      int32_t doc = sh.pieces[a].doc;
      int32_t e = sh.pieces[a].end;
      size_t b = a + 1;
      while (b < sh.pieces.size() && sh.pieces[b].doc == doc) e = std::max(e, sh.pieces[b++].end);
      sh.kv_need.push_back(fcp_range{doc, off[doc], e});
      // kv_remote: the needed range minus this shard's own pieces of the doc.
      int32_t t = off[doc];
      for (size_t c = a; c < b; ++c) {
        if (sh.pieces[c].start > t) sh.kv_remote.push_back(fcp_range{doc, t, sh.pieces[c].start});
        t = std::max(t, sh.pieces[c].end);
      }
      if (t < e) sh.kv_remote.push_back(fcp_range{doc, t, e});
      a = b;
    }
    sh.tokens = sum_tokens(sh.pieces);
    sh.W = sum_work(sh.pieces, off);
    sh.remote_rows = 0;
    for (const fcp_range& r : sh.kv_remote) sh.remote_rows += r.end - r.start;
  }
  int64_t sumW = 0, maxW = 0;
  for (const Shard& s : shards) { sumW += s.W; maxW = std::max(maxW, s.W); }
  imbalance = sumW > 0 ? (double)maxW / ((double)sumW / (double)N) : 1.0;
  // S^: all pieces of a split document except its last one (§3.2, Eq. 5).
  std::vector<int32_t> last_start(n, -1), npieces(n, 0);
  for (const Shard& s : shards)
    for (const Piece& p : s.pieces) {
      last_start[p.doc] = std::max(last_start[p.doc], p.start);
      npieces[p.doc]++;
    }
  int64_t max_nonlast = 0;
  for (const Shard& s : shards) {
    int64_t nl = 0;
    for (const Piece& p : s.pieces)
      if (npieces[p.doc] >= 2 && p.start != last_start[p.doc]) nl += p.end - p.start;
    max_nonlast = std::max(max_nonlast, nl);
  }
  eq4 = (T % N == 0) ? 4 * (T / N) * (N - 1) : 4 * T * (N - 1) / N;
  eq5 = 4 * max_nonlast * (N - 1);
  eq2dev = 0;
  for (const Shard& s : shards) eq2dev = std::max<int64_t>(eq2dev, std::llabs(s.tokens * N - T) / N);
  int64_t base = 0;
  for (Shard& s : shards) { s.kbuf_base = base; base += s.remote_rows; }
  total_remote = base;
}

int Plan::build_llama3() {
  if (T % (2 * N) != 0) return FCP_ERR_INFEASIBLE;
  const int64_t c = T / (2 * N);
  std::vector<std::vector<Piece>> wp(N);
  for (int32_t i = 0; i < N; ++i) {
    const int32_t cs[2] = {i, 2 * N - 1 - i};
    for (int32_t ch : cs) {
      int64_t t = ch * c, b = (ch + 1) * c;
      while (t < b) {  // cut the chunk at document boundaries
        int32_t doc = (int32_t)(std::upper_bound(off.begin(), off.end(), (int32_t)t) - off.begin()) - 1;
        int64_t e = std::min<int64_t>(b, (int64_t)off[doc] + D[doc]);
        wp[i].push_back(Piece{doc, (int32_t)t, (int32_t)e});
        t = e;
      }
    }
  }
  per_doc.assign(D.size(), 0);
  iterations = 1;
  finish(wp);
  return FCP_OK;
}

int Plan::build_perdoc() {
  std::vector<std::vector<Piece>> wp(N);
  for (int32_t doc = 0; doc < (int32_t)D.size(); ++doc) perdoc_pieces(doc, D[doc], off[doc], N, wp);
  per_doc.assign(D.size(), 1);
  iterations = 1;
  finish(wp);
  return FCP_OK;
}

// Algorithm 1 of FlashCP (§3.4). `tiles`: a piece's workload is its kernel
// tile cost instead of W (placement and imbalance alike).
int Plan::build_algorithm1(double R, bool tiles) {
  if (T % N != 0) return FCP_ERR_INFEASIBLE;
  const int32_t n = (int32_t)D.size();
  const int64_t target_total = T / N;
  // Line 1: documents by length, descending; ties keep document order.
  std::vector<int32_t> order(n);
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return D[a] > D[b]; });
  std::vector<uint8_t> is_pd(n, 0);
  std::vector<std::vector<Piece>> base(N), tmp(N);
  iterations = 0;
  for (;;) {
    ++iterations;
    // Per-doc shards of the documents popped so far are each worker's base
    // (popped in `order` sequence, so iterate the pop list).
    for (auto& v : base) v.clear();
    for (int32_t doc : pd_order) perdoc_pieces(doc, D[doc], off[doc], N, base);
    std::vector<int64_t> load(N), target(N), tokens(N, 0);
    for (int32_t j = 0; j < N; ++j) {
      load[j] = sum_cost(base[j], off, tiles);
      target[j] = target_total - sum_tokens(base[j]);
    }
    std::vector<int64_t> base_w = load;
    // Lines 5-9: every remaining document, whole, to the least-loaded worker.
    for (auto& v : tmp) v.clear();
    for (int32_t doc : order) {
      if (is_pd[doc]) continue;
      int32_t j = 0;
      for (int32_t w = 1; w < N; ++w)
        if (load[w] < load[j]) j = w;
      tmp[j].push_back(Piece{doc, off[doc], off[doc] + D[doc]});
      load[j] += tiles ? tile_cost(0, D[doc]) : piece_work(0, D[doc]);
      tokens[j] += D[doc];
    }
    // Lines 11-16: equal-token repair with Whole-Doc sharding.
    for (;;) {
      bool equal = true;
      for (int32_t j = 0; j < N; ++j) equal &= (tokens[j] == target[j]);
      if (equal) break;
      int32_t A = 0, B = 0;
      for (int32_t w = 1; w < N; ++w) {
        if (tokens[w] - target[w] > tokens[A] - target[A]) A = w;
        if (tokens[w] - target[w] < tokens[B] - target[B]) B = w;
      }
      int64_t ea = tokens[A] - target[A], eb = tokens[B] - target[B];
      if (ea <= 0 || eb >= 0 || tmp[A].empty()) break;
      int64_t delta = std::min(ea, -eb);
      Piece& last = tmp[A].back();
      int64_t moved;
      if (last.end - last.start <= delta) {
        Piece p = last;
        tmp[A].pop_back();
        tmp[B].push_back(p);
        moved = p.end - p.start;
      } else {
        Piece head{last.doc, last.start, (int32_t)(last.start + delta)};
        last.start += (int32_t)delta;
        tmp[B].push_back(head);
        moved = delta;
      }
      tokens[A] -= moved;
      tokens[B] += moved;
    }
    // Line 18: imbalance of the complete plan.
    int64_t sumW = 0, maxW = 0;
    for (int32_t j = 0; j < N; ++j) {
      int64_t w = base_w[j] + sum_cost(tmp[j], off, tiles);
      sumW += w;
      maxW = std::max(maxW, w);
    }
    double cur_r = sumW > 0 ? (double)maxW / ((double)sumW / (double)N) : 1.0;
    int32_t longest = -1;
    for (int32_t doc : order)
      if (!is_pd[doc]) { longest = doc; break; }
    // Lines 19-23: move the longest remaining document to Per-Doc.
    if (cur_r > R && longest >= 0) {
      is_pd[longest] = 1;
      pd_order.push_back(longest);
      continue;
    }
    break;
  }
  std::vector<std::vector<Piece>> wp(N);
  for (int32_t j = 0; j < N; ++j) {
    wp[j] = base[j];
    wp[j].insert(wp[j].end(), tmp[j].begin(), tmp[j].end());
  }
  per_doc = is_pd;
  finish(wp);
  return FCP_OK;
}

int make_plan(const int32_t* doclens, int32_t n_docs, int32_t cp, int32_t policy, double R,
              fcp_plan_t** out) {
  if (!doclens || !out || n_docs < 1 || cp < 1) return FCP_ERR_INVALID_ARG;
  if (policy < FCP_POLICY_LLAMA3 || policy > FCP_POLICY_HYBRID_TILES) return FCP_ERR_INVALID_ARG;
  if ((policy == FCP_POLICY_HYBRID || policy == FCP_POLICY_HYBRID_TILES) && !(R > 0)) return FCP_ERR_INVALID_ARG;
  fcp_plan_t* p = new fcp_plan_t();
  p->N = cp;
  p->D.assign(doclens, doclens + n_docs);
  p->off.resize(n_docs);
  int64_t acc = 0;
  for (int32_t i = 0; i < n_docs; ++i) {
    if (doclens[i] < 1) { delete p; return FCP_ERR_INVALID_ARG; }
    p->off[i] = (int32_t)acc;
    acc += doclens[i];
    if (acc >= (int64_t(1) << 31)) { delete p; return FCP_ERR_INVALID_ARG; }
  }
  p->T = acc;
  int st;
  switch (policy) {
    case FCP_POLICY_LLAMA3: st = p->build_llama3(); break;
    case FCP_POLICY_PER_DOC: st = p->build_perdoc(); break;
    case FCP_POLICY_WHOLE_DOC: st = p->build_algorithm1(std::numeric_limits<double>::infinity(), false); break;
    case FCP_POLICY_HYBRID_TILES: st = p->build_algorithm1(R, true); break;
    default: st = p->build_algorithm1(R, false); break;
  }
  if (st != FCP_OK) { delete p; return st; }
  p->build_work_tables();
  *out = p;
  return FCP_OK;
}

}  // namespace fcp
