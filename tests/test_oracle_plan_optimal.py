"""Pins of the exhaustive optimal planner (the stand-in for FlashCP's ILP,
§3.4 and §4 Table 2) and its comparison with Algorithm 1 on tiny inputs."""
import itertools
import math

import numpy as np
import pytest

from oracle import plan as P
from oracle import plan_optimal as O


def _enumerate_all(D, N, g):
    """Every balanced chunk assignment, no pruning, no symmetry breaking."""
    chunks = O.chunks_of(D, g)
    target = sum(D) // N
    best = None
    for assign in itertools.product(range(N), repeat=len(chunks)):
        tok = [0] * N
        for (doc, a, b), w in zip(chunks, assign):
            tok[w] += b - a
        if any(t != target for t in tok):
            continue
        mw, comm, _ = O.evaluate(D, chunks, list(assign), N)
        if best is None or (mw, comm) < best:
            best = (mw, comm)
    return best


@pytest.mark.parametrize("D,N,g", [
    ([8, 8], 2, 4), ([12, 4], 2, 4), ([5, 9, 2], 2, 4), ([10, 6, 8], 3, 4),
    ([16, 3, 5], 2, 3), ([7, 7, 4], 3, 3), ([20, 4], 2, 4),
])
def test_search_equals_plain_enumeration(D, N, g):
    opt = O.optimal_plan(D, N, g)
    assert (opt.max_w, opt.comm) == _enumerate_all(D, N, g)


def test_fig4_ideal_case_two_equal_documents():
    """FlashCP Fig. 4(1): two documents of equal length on two workers are
    kept whole, one per worker: balanced and nothing to communicate."""
    opt = O.optimal_plan([64, 64], 2, 16)
    assert opt.imbalance == 1.0 and opt.comm == 0


@pytest.mark.parametrize("seed", range(6))
def test_optimum_respects_lower_bound_and_beats_per_chunk_heuristics(seed):
    rng = np.random.default_rng(seed)
    N = 2
    D = [int(x) for x in rng.integers(4, 40, size=4)]
    D[-1] += (-sum(D)) % (N * 8)
    opt = O.optimal_plan(D, N, 8)
    total_w = sum(L * (L + 1) // 2 for L in D)
    assert opt.sum_w == total_w
    assert opt.max_w >= math.ceil(total_w / N)
    # Any other balanced 8-granular assignment is no better: spot-check random ones.
    chunks = O.chunks_of(D, 8)
    target = sum(D) // N
    for _ in range(200):
        assign = list(rng.integers(0, N, size=len(chunks)))
        tok = [0] * N
        for (_, a, b), w in zip(chunks, assign):
            tok[w] += b - a
        if all(t == target for t in tok):
            mw, comm, _ = O.evaluate(D, chunks, assign, N)
            assert (opt.max_w, opt.comm) <= (mw, comm)


def table2_style(mixes, N, g, R=1.05):
    """Imbalance and communication saving (1 - Eq.5 / Eq.4) of Algorithm 1
    (hybrid) and of the g-granular optimum, averaged over the mixes."""
    rows = []
    for D in mixes:
        h = P.make_plan(D, N, "hybrid", R)
        opt = O.optimal_plan(D, N, g)
        T = sum(D)
        rows.append((h.imbalance, 1 - h.eq5_tokens / h.eq4_tokens, opt.imbalance, 1 - opt.comm / (T // N)))
    return np.array(rows).mean(axis=0)


def test_table2_style_comparison_on_tiny_mixes():
    """The §4 Table 2 comparison on seeded tiny mixes (the Pile dataset is not
    used): the optimum's imbalance is near 1 and the heuristic stays close."""
    rng = np.random.default_rng(11)
    N, g = 2, 8
    mixes = []
    while len(mixes) < 8:
        D = [int(x) for x in rng.integers(8, 48, size=int(rng.integers(3, 5)))]
        D[-1] += (-sum(D)) % (N * g)
        if sum(D) <= 120:
            mixes.append(D)
    h_imb, h_save, o_imb, o_save = table2_style(mixes, N, g)
    print(f"[table2] heuristic imbalance {h_imb:.3f} saving {h_save:.2f}; optimum imbalance {o_imb:.3f} saving {o_save:.2f}")
    assert o_imb < 1.1
    assert 0.0 <= o_save <= 1.0 and 0.0 <= h_save <= 1.0
