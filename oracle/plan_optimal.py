"""Exhaustive optimal sharding for tiny inputs: a stand-in for the ILP that
FlashCP compares its heuristic against (§3.4 "ILP-based Sharding", §4 Table 2).

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.

The ILP of §3.1 / §3.4 assigns document shards of "a given sharding
granularity" to workers: every shard to one worker (Eq. 1), the same token
count on every worker (Eq. 2), minimising the largest worker workload (Eq. 3)
with the communication of Eq. 5 in the objective. The pages give neither the
granularity nor the weight of the two terms. Reading taken here: documents are
cut into chunks of g tokens (a document's last chunk may be shorter); a plan
assigns every chunk to a worker; adjacent chunks of a document on the same
worker form one shard; the objective is lexicographic -- first the largest
workload max_j W_j, then the Eq. 5 volume max_j (tokens of worker j's non-last
shards). The search is a depth-first enumeration over chunks with the workers
labelled in order of first use (a plan and its relabellings are one plan) and
branches cut when they cannot beat the best plan found.
"""
from __future__ import annotations

import dataclasses

from .plan import workload


@dataclasses.dataclass
class OptimalPlan:
    assign: list        # worker of each chunk, in document order
    chunks: list        # (doc, start, end) global token ranges
    max_w: int          # largest worker workload (W summed over its shards)
    comm: int           # max over workers of its non-last shard tokens (Eq. 5 without constants)
    sum_w: int
    N: int

    @property
    def imbalance(self) -> float:
        return self.max_w / (self.sum_w / self.N) if self.sum_w else 1.0


def chunks_of(D, g: int) -> list:
    """Documents cut into chunks of g tokens: (doc, start, end), global."""
    out, o = [], 0
    for i, L in enumerate(D):
        for a in range(0, L, g):
            out.append((i, o + a, o + min(a + g, L)))
        o += L
    return out


def evaluate(D, chunks, assign, N: int):
    """(max_w, comm, sum_w) of a chunk assignment: W per worker (W is a sum
    over tokens, so per chunk: the chunk's W at its prefix) and, per worker,
    the tokens of its shards that are not a document's last shard."""
    offsets = []
    o = 0
    for L in D:
        offsets.append(o)
        o += L
    W = [0] * N
    nonlast = [0] * N
    # Shards: maximal runs of a document's consecutive chunks on one worker.
    i = 0
    while i < len(chunks):
        doc, a, _ = chunks[i]
        j = i
        while j + 1 < len(chunks) and chunks[j + 1][0] == doc and assign[j + 1] == assign[i]:
            j += 1
        b = chunks[j][2]
        w = assign[i]
        W[w] += workload(a - offsets[doc], b - a)
        if b != offsets[doc] + D[doc]:
            nonlast[w] += b - a
        i = j + 1
    return max(W), max(nonlast), sum(W)


def optimal_plan(D, N: int, g: int) -> OptimalPlan:
    """Best g-granular plan under the lexicographic objective (max W, then
    Eq. 5), by depth-first enumeration. Tiny inputs only (a few dozen chunks
    at most, fewer for larger N)."""
    D = [int(x) for x in D]
    T = sum(D)
    if T % N:
        raise ValueError("equal-token sharding needs T divisible by N")
    target = T // N
    chunks = chunks_of(D, g)
    offsets = []
    o = 0
    for L in D:
        offsets.append(o)
        o += L
    cw = [workload(a - offsets[doc], b - a) for doc, a, b in chunks]
    cs = [b - a for _, a, b in chunks]
    rest_w = [0] * (len(chunks) + 1)
    for k in range(len(chunks) - 1, -1, -1):
        rest_w[k] = rest_w[k + 1] + cw[k]
    best = {"key": None, "assign": None}
    assign = [0] * len(chunks)
    W = [0] * N
    tok = [0] * N

    def dfs(k: int, used: int):
        if k == len(chunks):
            if any(t != target for t in tok):
                return
            mw, comm, _ = evaluate(D, chunks, assign, N)
            key = (mw, comm)
            if best["key"] is None or key < best["key"]:
                best["key"], best["assign"] = key, list(assign)
            return
        # Bound: the largest workload can only grow, and the rest must fit.
        if best["key"] is not None and max(W) > best["key"][0]:
            return
        for w in range(min(used + 1, N)):
            if tok[w] + cs[k] > target:
                continue
            assign[k] = w
            W[w] += cw[k]
            tok[w] += cs[k]
            if best["key"] is None or W[w] <= best["key"][0]:
                dfs(k + 1, max(used, w + 1))
            W[w] -= cw[k]
            tok[w] -= cs[k]

    dfs(0, 0)
    if best["key"] is None:
        raise ValueError("no g-granular plan with equal token counts")
    mw, comm, sw = evaluate(D, chunks, best["assign"], N)
    return OptimalPlan(best["assign"], chunks, mw, comm, sw, N)
