"""Oracle of the FlashCP sharding policies and their cost model.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU baseline, never by the library. The C++ planner of the
library is a separate implementation of the same rules and must reproduce
every index list here bit for bit.

Notation follows the FlashCP paper ("FlashCP: Load-Balanced
Communication-Efficient Context Parallelism for LLM Training", §3.1): CP size
N, context window C (= T tokens), documents D = [d_1..d_n], document shards
s_i with prefix length p_i (tokens of the same document before the shard),
and the workload of a shard W_i = (2 p_i + s_i + 1) s_i / 2 (§3.1, after
Eq. 3). A whole document of length L therefore has W = L(L+1)/2.

Policies:
  llama3   §2.2 / Fig. 1(b): the whole sequence is cut into 2N equal chunks;
           worker i takes chunks i and 2N-1-i (the pairing rule §2.3 states
           for Per-Doc and zigzag sharding; Fig. 1(b) is not legible).
  perdoc   §2.3: every document is cut into 2N chunks; worker i takes chunks
           i and 2N-1-i. Chunk boundaries are floor(c L / 2N).
  wholedoc Algorithm 1 (§3.4) with the Per-Doc branch never taken (R = inf).
  hybrid   Algorithm 1 with target imbalance R.
  hybrid_tiles  Algorithm 1 with target imbalance R, a piece's workload
           measured in the attention kernels' own units instead of W: the
           128 x 128 tiles its query rows touch in the document's causal
           prefix (keys taken as one run from the document start) plus one
           per query tile. The weights are those of a least-squares fit of
           measured per-shard forward + backward time on GB300 against visited
           tiles and query tiles, which came out equal. FlashCP §2.2 ("Reduced
           Kernel Efficiency", Fig. 3) is the motivation: short shards cost
           more per useful pair. The greedy placement and Cur_R both use it.

Readings of Algorithm 1 where the text is open:
  * "least-loaded worker" (Min_Worker_Add) is by workload W, ties to the
    lowest worker index; the per-doc shards of earlier-popped documents count
    toward a worker's load.
  * Max_Token_Worker_Pop / Whole_Doc_Shard_and_Add (the equal-token loop,
    §3.3 and Fig. 4(2)): take the worker A with the largest token excess over
    its target and the worker B with the largest deficit (ties: lowest index),
    Delta = min(excess, deficit). A's most recently added whole-doc piece moves
    to B whole if it is no longer than Delta; otherwise its first Delta tokens
    (its head) move to B and the tail stays. Only the head, a non-last shard,
    then has to be communicated, so the exchanged volume is bounded by the
    largest Delta (§3.3).
  * Targets: worker j must hold C/N tokens in total, per-doc shards included.
    If a worker with excess has no whole-doc piece left (only possible when
    per-doc rounding already overfills it) the loop stops and the deviation
    from Eq. 2 is reported.
  * Cur_R = max_j W_j / mean_j W_j over the complete plan (§3.4 text); the
    outer loop pops the longest remaining document into Per-Doc while
    Cur_R > R and documents remain.
Communication:
  * A shard's needed keys for a piece [a, b) of a document starting at o are
    [o, b) (§3.2: a query attends only to its document's prefix).
  * kv_remote = needed keys not held by the shard itself (receiver side).
  * Eq. 4 (full KV exchange) and Eq. 5 (sharding-aware) volumes are reported
    as token counts: 4 * (C/N) * (N-1) and 4 * max_j sum_{i in S^} x_ij s_i *
    (N-1), where S^ holds every shard of a split document except its last
    one; multiply by heads x head dim x bytes for a byte count.
"""
from __future__ import annotations

import dataclasses
import math

POLICIES = ("llama3", "perdoc", "wholedoc", "hybrid", "hybrid_tiles")
DEFAULT_R = 1.05


class Infeasible(ValueError):
    pass


@dataclasses.dataclass
class Piece:
    doc: int
    start: int   # global token index
    end: int     # exclusive

    @property
    def s(self) -> int:
        return self.end - self.start


@dataclasses.dataclass
class Shard:
    pieces: list            # Piece, ascending by start
    kv_need: list           # (doc, start, end) per document touched, ascending
    kv_remote: list         # (doc, start, end), ascending, disjoint
    tokens: int
    W: int
    remote_rows: int


@dataclasses.dataclass
class Plan:
    N: int
    T: int
    lengths: list
    offsets: list
    shards: list
    per_doc: list           # per document: 1 if sharded Per-Doc, else 0
    imbalance: float
    eq4_tokens: int
    eq5_tokens: int
    eq2_max_dev: int        # max_j |tokens_j - T/N|
    iterations: int         # outer-loop passes of Algorithm 1 (1 for others)

    def query_indices(self, j: int) -> list:
        out = []
        for p in self.shards[j].pieces:
            out.extend(range(p.start, p.end))
        return out


def workload(p: int, s: int) -> int:
    """W_i = (2 p_i + s_i + 1) s_i / 2, exact in integers."""
    return (2 * p + s + 1) * s // 2


TILE = 128


def tile_cost(p: int, s: int) -> int:
    """Kernel-unit cost of a shard of s tokens whose document prefix is p
    tokens: for each of its ceil(s/128) query tiles, the ceil((p + e)/128) key
    tiles of the causal prefix up to the tile's local end e, plus one per
    query tile."""
    nq = -(-s // TILE)
    return sum(-(-(p + min(TILE * (t + 1), s)) // TILE) for t in range(nq)) + nq


def _offsets(D):
    o, acc = [], 0
    for L in D:
        o.append(acc)
        acc += L
    return o, acc


def _perdoc_chunks(L: int, o: int, N: int):
    """The 2N chunks of a document at offset o: [o + floor(cL/2N), o + floor((c+1)L/2N))."""
    return [(o + (c * L) // (2 * N), o + ((c + 1) * L) // (2 * N)) for c in range(2 * N)]


def _perdoc_pieces(doc: int, L: int, o: int, N: int):
    """Pieces of one Per-Doc sharded document, per worker."""
    ch = _perdoc_chunks(L, o, N)
    out = [[] for _ in range(N)]
    for i in range(N):
        for c in (i, 2 * N - 1 - i):
            a, b = ch[c]
            if b > a:
                out[i].append(Piece(doc, a, b))
    return out




def _split_by_docs(a: int, b: int, offsets, lengths):
    """Cut the token range [a, b) at document boundaries."""
    out = []
    t = a
    import bisect
    while t < b:
        i = bisect.bisect_right(offsets, t) - 1
        e = min(b, offsets[i] + lengths[i])
        out.append(Piece(i, t, e))
        t = e
    return out


def _finish(N, T, lengths, offsets, worker_pieces, per_doc, iterations) -> Plan:
    shards = []
    for j in range(N):
        ps = []
        # Adjacent pieces of one document on one worker form one shard.
        for p in sorted(worker_pieces[j], key=lambda p: p.start):
            if ps and ps[-1].doc == p.doc and ps[-1].end == p.start:
                ps[-1] = Piece(p.doc, ps[-1].start, p.end)
            else:
                ps.append(Piece(p.doc, p.start, p.end))
        need = {}
        for p in ps:
            need[p.doc] = max(need.get(p.doc, 0), p.end)
        kv_need = [(doc, offsets[doc], e) for doc, e in sorted(need.items())]
        kv_remote = []
        for doc, a, b in kv_need:
            own = sorted((p.start, p.end) for p in ps if p.doc == doc)
            t = a
            for s, e in own:
                if s > t:
                    kv_remote.append((doc, t, s))
                t = max(t, e)
            if t < b:
                kv_remote.append((doc, t, b))
        tokens = sum(p.s for p in ps)
        W = sum(workload(p.start - offsets[p.doc], p.s) for p in ps)
        shards.append(Shard(ps, kv_need, kv_remote, tokens, W,
                            sum(e - s for _, s, e in kv_remote)))
    Ws = [s.W for s in shards]
    sumW = sum(Ws)
    imb = (max(Ws) / (sumW / N)) if sumW > 0 else 1.0
    # S^: every piece of a split document except its last one.
    by_doc = {}
    for j, s in enumerate(shards):
        for p in s.pieces:
            by_doc.setdefault(p.doc, []).append((p.start, p.end, j))
    nonlast = [0] * N
    for doc, lst in by_doc.items():
        if len(lst) < 2:
            continue
        lst.sort()
        for a, b, j in lst[:-1]:
            nonlast[j] += b - a
    eq4 = 4 * (T // N) * (N - 1) if T % N == 0 else 4 * T * (N - 1) // N
    eq5 = 4 * max(nonlast) * (N - 1)
    dev = max(abs(s.tokens * N - T) for s in shards) // N if N else 0
    return Plan(N, T, list(lengths), offsets, shards, per_doc, imb, eq4, eq5, dev, iterations)


def plan_llama3(D, N: int) -> Plan:
    offsets, T = _offsets(D)
    if T % (2 * N) != 0:
        raise Infeasible("Llama3 2xCP sharding needs T divisible by 2N")
    c = T // (2 * N)
    wp = [[] for _ in range(N)]
    for i in range(N):
        for ch in (i, 2 * N - 1 - i):
            wp[i].extend(_split_by_docs(ch * c, (ch + 1) * c, offsets, D))
    return _finish(N, T, D, offsets, wp, [0] * len(D), 1)


def plan_perdoc(D, N: int) -> Plan:
    offsets, T = _offsets(D)
    wp = [[] for _ in range(N)]
    for doc, L in enumerate(D):
        for j, ps in enumerate(_perdoc_pieces(doc, L, offsets[doc], N)):
            wp[j].extend(ps)
    return _finish(N, T, D, offsets, wp, [1] * len(D), 1)


def plan_algorithm1(D, N: int, R: float, cost=None) -> Plan:
    """Algorithm 1 of FlashCP (§3.4): Whole-Doc placement with Per-Doc for the
    documents that keep the imbalance above R. `cost(p, s)` measures a
    piece's workload (default W)."""
    cost = workload if cost is None else cost
    offsets, T = _offsets(D)
    n = len(D)
    if T % N != 0:
        raise Infeasible("equal-token sharding needs T divisible by N")
    target_total = T // N
    # Line 1: sort D descending by length (stable: ties keep document order).
    order = sorted(range(n), key=lambda i: (-D[i], i))
    per_doc_P = []            # lines 2, 21-22: documents given Per-Doc sharding
    cur_r = math.inf          # line 3
    iterations = 0
    while True:
        iterations += 1
        # Per-doc shards of the popped documents are each worker's base.
        base = [[] for _ in range(N)]
        for doc in per_doc_P:
            for j, ps in enumerate(_perdoc_pieces(doc, D[doc], offsets[doc], N)):
                base[j].extend(ps)
        base_W = [sum(cost(p.start - offsets[p.doc], p.s) for p in ps) for ps in base]
        base_tok = [sum(p.s for p in ps) for ps in base]
        target = [target_total - base_tok[j] for j in range(N)]
        # Lines 5-9: each remaining document goes whole to the least-loaded worker.
        load = list(base_W)
        tmp_P = [[] for _ in range(N)]     # per worker, in the order pieces arrive
        for doc in order:
            if doc in per_doc_P:
                continue
            j = min(range(N), key=lambda w: (load[w], w))
            tmp_P[j].append(Piece(doc, offsets[doc], offsets[doc] + D[doc]))
            load[j] += cost(0, D[doc])
        # Lines 11-16: restore equal token counts (Eq. 2) with Whole-Doc sharding.
        tokens = [sum(p.s for p in ps) for ps in tmp_P]
        while True:
            excess = [tokens[j] - target[j] for j in range(N)]
            if all(e == 0 for e in excess):
                break
            A = max(range(N), key=lambda w: (excess[w], -w))
            B = max(range(N), key=lambda w: (-excess[w], -w))
            if excess[A] <= 0 or excess[B] >= 0 or not tmp_P[A]:
                break
            delta = min(excess[A], -excess[B])
            last = tmp_P[A][-1]
            if last.s <= delta:
                tmp_P[A].pop()
                tmp_P[B].append(last)
                moved = last.s
            else:
                head = Piece(last.doc, last.start, last.start + delta)
                last.start += delta
                tmp_P[B].append(head)
                moved = delta
            tokens[A] -= moved
            tokens[B] += moved
        # Line 18: imbalance of the complete plan.
        Wj = [base_W[j] + sum(cost(p.start - offsets[p.doc], p.s) for p in tmp_P[j])
              for j in range(N)]
        sumW = sum(Wj)
        cur_r = (max(Wj) / (sumW / N)) if sumW > 0 else 1.0
        remaining = [doc for doc in order if doc not in per_doc_P]
        # Lines 19-23: pop the longest remaining document into Per-Doc.
        if cur_r > R and remaining:
            per_doc_P.append(remaining[0])
            continue
        break
    wp = [base[j] + tmp_P[j] for j in range(N)]
    flags = [1 if i in per_doc_P else 0 for i in range(n)]
    return _finish(N, T, D, offsets, wp, flags, iterations)


def make_plan(D, N: int, policy: str, R: float = DEFAULT_R) -> Plan:
    D = [int(x) for x in D]
    if N < 1 or any(L < 1 for L in D) or not D:
        raise ValueError("bad plan input")
    if policy == "llama3":
        return plan_llama3(D, N)
    if policy == "perdoc":
        return plan_perdoc(D, N)
    if policy == "wholedoc":
        return plan_algorithm1(D, N, math.inf)
    if policy == "hybrid":
        return plan_algorithm1(D, N, R)
    if policy == "hybrid_tiles":
        return plan_algorithm1(D, N, R, cost=tile_cost)
    raise ValueError(policy)
