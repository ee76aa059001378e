"""Pins of the sharding-plan oracle.

Checks against what the FlashCP paper fixes: Eq. 1 (each shard on exactly one
worker), Eq. 2 (C/N tokens per worker), the workload W_i = (2p_i+s_i+1)s_i/2
counted by brute force, the Fig. 4(1) ideal case, the S^ rule of §3.2 (whole
documents and last shards are never communicated), and hand-derived cases
stored in tests/golden/plan_hand_cases.json.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import plan as P
from oracle.attention import useful_pairs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_hand_cases.json")


def _pieces(plan):
    return [[[p.doc, p.start, p.end] for p in s.pieces] for s in plan.shards]


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_cases(case):
    plan = P.make_plan(case["D"], case["N"], case["policy"], case.get("R", P.DEFAULT_R))
    assert _pieces(plan) == case["shards"]
    assert [s.W for s in plan.shards] == case["W"]
    assert [s.remote_rows for s in plan.shards] == case["remote_rows"]
    assert plan.imbalance == pytest.approx(case["imbalance"], rel=1e-12)
    if "eq5_tokens" in case:
        assert plan.eq5_tokens == case["eq5_tokens"]
    if "eq4_tokens" in case:
        assert plan.eq4_tokens == case["eq4_tokens"]
    if "iterations" in case:
        assert plan.iterations == case["iterations"]


def _brute_pairs(piece, offset):
    """Count (query, key) pairs of a piece by enumeration: keys of the same
    document at or before the query."""
    return sum(q - offset + 1 for q in range(piece.start, piece.end))


def _all_cases():
    out = []
    for cfg in (1, 2, 3, 4):
        D = synth.doc_lengths(cfg)
        N = synth.WORKLOADS[cfg].cp
        for pol in P.POLICIES:
            out.append((f"cfg{cfg}-{pol}", D, N, pol))
    for seed in range(6):
        T = 2 * 4 * 64
        D = synth.random_doc_lengths(T, seed=100 + seed)
        for pol in P.POLICIES:
            out.append((f"rand{seed}-{pol}", D, 4, pol))
    return out


CASES = _all_cases()


@pytest.mark.parametrize("name,D,N,pol", CASES, ids=[c[0] for c in CASES])
def test_plan_invariants(name, D, N, pol):
    plan = P.make_plan(D, N, pol)
    T = sum(D)
    offsets = plan.offsets
    # Eq. 1: every token is in exactly one shard.
    owner = np.full(T, -1)
    for j, s in enumerate(plan.shards):
        for p in s.pieces:
            assert 0 <= p.start < p.end <= T
            assert offsets[p.doc] <= p.start and p.end <= offsets[p.doc] + D[p.doc]
            assert (owner[p.start:p.end] == -1).all()
            owner[p.start:p.end] = j
        qi = plan.query_indices(j)
        assert qi == sorted(qi)
    assert (owner >= 0).all()
    # Eq. 2: C/N tokens per worker (Per-Doc up to floor rounding).
    if pol in ("llama3", "wholedoc"):
        assert all(s.tokens == T // N for s in plan.shards)
        assert plan.eq2_max_dev == 0
    else:
        # Per-Doc chunk rounding moves at most one token per document and
        # worker; Whole-Doc pieces absorb it unless a worker's Per-Doc share
        # alone already exceeds C/N.
        assert plan.eq2_max_dev <= sum(plan.per_doc)
        assert all(abs(s.tokens - T / N) <= sum(plan.per_doc) for s in plan.shards)
    # Workload: W per piece equals the enumerated pair count; totals equal
    # sum L(L+1)/2.
    for s in plan.shards:
        assert s.W == sum(_brute_pairs(p, offsets[p.doc]) for p in s.pieces)
    assert sum(s.W for s in plan.shards) == useful_pairs(D)
    Ws = [s.W for s in plan.shards]
    assert plan.imbalance == pytest.approx(max(Ws) / np.mean(Ws))
    # S^ rule: remote keys are prefixes held by other workers and never lie in a
    # whole document or in the last shard of a document.
    last_start = {}
    for s in plan.shards:
        for p in s.pieces:
            last_start[p.doc] = max(last_start.get(p.doc, -1), p.start)
    for j, s in enumerate(plan.shards):
        for doc, a, b in s.kv_remote:
            assert (owner[a:b] != j).all()
            assert b <= last_start[doc]
        need = set()
        for p in s.pieces:
            need.update(range(offsets[p.doc], p.end))
        have = set(plan.query_indices(j))
        remote = set()
        for doc, a, b in s.kv_remote:
            remote.update(range(a, b))
        assert remote == need - have
        assert s.remote_rows == len(remote)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_perdoc_is_balanced_and_llama3_is_not(cfg):
    D = synth.doc_lengths(cfg)
    N = synth.WORKLOADS[cfg].cp
    pd = P.make_plan(D, N, "perdoc")
    assert pd.imbalance < 1.05
    if cfg >= 2:
        assert P.make_plan(D, N, "llama3").imbalance > 1.1


def test_hybrid_meets_target_or_exhausts_documents():
    for cfg in (2, 3, 4):
        D = synth.doc_lengths(cfg)
        N = synth.WORKLOADS[cfg].cp
        plan = P.make_plan(D, N, "hybrid", 1.05)
        assert plan.imbalance <= 1.05 or all(plan.per_doc)


@pytest.mark.parametrize("p,s", [(0, 1), (0, 128), (0, 129), (5, 1), (5, 300), (127, 2), (128, 128),
                                 (200, 257), (1000, 31), (0, 700), (333, 513)])
def test_tile_cost_counts_touched_tiles(p, s):
    """hybrid_tiles cost of a shard: the (query tile, key tile) cells holding
    at least one causal pair -- query tiles from the shard start, key tiles
    from the document start -- enumerated pair by pair, plus its query tiles."""
    cells = {((q - p) // 128, k // 128) for q in range(p, p + s) for k in range(q + 1)}
    assert P.tile_cost(p, s) == len(cells) + -(-s // 128)


def test_tile_cost_whole_document_closed_form():
    for L in (1, 127, 128, 129, 4096, 8833):
        n = -(-L // 128)
        assert P.tile_cost(0, L) == n * (n + 1) // 2 + n


def test_hybrid_tiles_meets_target_in_its_cost():
    """Algorithm 1 with the tile cost stops once the cost imbalance is within
    R, or after every document went Per-Doc."""
    for cfg in (2, 3, 4):
        D = synth.doc_lengths(cfg)
        N = synth.WORKLOADS[cfg].cp
        plan = P.make_plan(D, N, "hybrid_tiles", 1.05)
        costs = [sum(P.tile_cost(pc.start - plan.offsets[pc.doc], pc.s) for pc in sh.pieces) for sh in plan.shards]
        assert max(costs) / (sum(costs) / N) <= 1.05 or all(plan.per_doc)


def test_wholedoc_cuts_communication():
    """Whole-Doc exchanges no more than Per-Doc on the skewed workloads (§3.2,
    Eq. 4 vs Eq. 5)."""
    for cfg in (2, 4):
        D = synth.doc_lengths(cfg)
        N = synth.WORKLOADS[cfg].cp
        wd = P.make_plan(D, N, "wholedoc")
        pd = P.make_plan(D, N, "perdoc")
        assert wd.eq5_tokens <= pd.eq5_tokens
        assert sum(s.remote_rows for s in wd.shards) < sum(s.remote_rows for s in pd.shards)


def test_llama3_needs_T_divisible_by_2N():
    with pytest.raises(P.Infeasible):
        P.make_plan([5, 4], 2, "llama3")


def test_workload_closed_form():
    # A whole document of length L: L(L+1)/2 (CP variance article's pair count).
    for L in (1, 2, 7, 128, 1000):
        assert P.workload(0, L) == L * (L + 1) // 2
    # Splitting a document anywhere conserves the total.
    for L in (9, 100):
        for c in range(1, L):
            assert P.workload(0, c) + P.workload(c, L - c) == P.workload(0, L)
    assert math.isinf(float("inf"))
