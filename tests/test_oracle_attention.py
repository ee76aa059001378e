"""Pins of the fp64 attention oracle against facts fixed outside it.

Each check ties the oracle to something it does not compute itself: a library
routine (torch SDPA / autograd in fp64), a closed form, brute force, or an
invariant of the document mask (FlashCP §2.1, Fig. 1(a)) and of the
online-softmax merge (production CP guide, "Core Principle: Split Q,
Circulate KV").
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as A


def _inputs(lengths, Hq=4, Hkv=2, d=16, seed=0):
    T = sum(lengths)
    q, k, v = synth.make_qkv(T, Hq, Hkv, d, seed)
    return synth.cu_from_lengths(lengths), q, k, v


MIXES = [
    [1, 7, 1, 40, 3, 1, 19],
    [64],
    [5, 5, 5, 5],
    synth.random_doc_lengths(180, seed=3),
]


@pytest.mark.parametrize("lengths", MIXES)
def test_per_doc_equals_bruteforce(lengths):
    cu, q, k, v = _inputs(lengths)
    ob, lb = A.attention_bruteforce(q, k, v, cu)
    op, lp = A.attention_per_doc(q, k, v, cu)
    np.testing.assert_allclose(op, ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lp, lb, atol=1e-12, rtol=0)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (4, 1), (6, 3)])
def test_single_doc_is_causal_sdpa(Hq, Hkv):
    """A single document is plain causal attention: compare with torch SDPA."""
    T, d = 97, 32
    q, k, v = synth.make_qkv(T, Hq, Hkv, d, seed=11)
    cu = np.array([0, T])
    o, lse = A.attention_per_doc(q, k, v, cu)
    G = Hq // Hkv
    qt = q.double().permute(1, 0, 2)                        # [Hq,T,d]
    kt = k.double().permute(1, 0, 2).repeat_interleave(G, 0)
    vt = v.double().permute(1, 0, 2).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
    s = (qt @ kt.transpose(1, 2)) / math.sqrt(d)
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12, rtol=0)


def test_first_token_returns_its_v_row():
    lengths = [3, 1, 50, 2, 9]
    cu, q, k, v = _inputs(lengths, Hq=4, Hkv=2, d=16)
    o, lse = A.attention_per_doc(q, k, v, cu)
    qd, kd, vd = A.to_f64(q), A.to_f64(k), A.to_f64(v)
    for s in cu[:-1]:
        for h in range(4):
            g = h // 2
            assert np.array_equal(o[s, h], vd[s, g])
            assert lse[h, s] == pytest.approx(float(qd[s, h] @ kd[s, g]) / 4.0, abs=1e-12)


def test_doc_permutation_equivariance():
    lengths = [10, 3, 25, 1, 7]
    cu, q, k, v = _inputs(lengths, seed=5)
    o, lse = A.attention_per_doc(q, k, v, cu)
    perm = [3, 0, 4, 2, 1]
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in perm])
    cu2 = synth.cu_from_lengths([lengths[i] for i in perm])
    o2, lse2 = A.attention_bruteforce(q[idx], k[idx], v[idx], cu2)
    np.testing.assert_allclose(o2, o[idx], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse2, lse[:, idx], atol=1e-12, rtol=0)


def test_mask_keeps_L_times_L_plus_1_over_2_pairs():
    """The document mask keeps exactly sum L(L+1)/2 pairs (the pair count the
    CP variance article states for causal attention)."""
    lengths = [1, 2, 9, 30, 4]
    doc = A.doc_ids(synth.cu_from_lengths(lengths))
    T = len(doc)
    brute = sum(1 for i in range(T) for j in range(T) if doc[i] == doc[j] and j <= i)
    assert brute == A.useful_pairs(lengths) == sum(L * (L + 1) // 2 for L in lengths)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_over_contiguous_key_blocks(seed):
    rng = np.random.default_rng(seed)
    lengths = synth.random_doc_lengths(150, seed=seed + 20)
    cu, q, k, v = _inputs(lengths, seed=seed)
    T = int(cu[-1])
    o, lse = A.attention_per_doc(q, k, v, cu)
    B = int(rng.integers(2, 6))
    cuts = np.sort(rng.integers(0, T + 1, size=B - 1))
    bounds = [0, *cuts.tolist(), T]                 # empty blocks allowed
    parts = [A.attention_per_doc(q, k, v, cu, key_range=(bounds[b], bounds[b + 1]))
             for b in range(B)]
    om, lm = A.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(om, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lm, lse, atol=1e-12, rtol=0)


def test_merge_over_arbitrary_key_partition():
    """Merge over a random (non-contiguous) partition of the keys, partials
    from the brute-force form with explicit key masks."""
    rng = np.random.default_rng(9)
    lengths = [12, 1, 30, 8]
    cu, q, k, v = _inputs(lengths, seed=9)
    T = int(cu[-1])
    o, lse = A.attention_bruteforce(q, k, v, cu)
    owner = rng.integers(0, 4, size=T)
    parts = [A.attention_bruteforce(q, k, v, cu, key_allowed=(owner == b)) for b in range(4)]
    assert any(np.isneginf(p[1]).any() for p in parts)  # some rows empty in some block
    om, lm = A.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(om, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lm, lse, atol=1e-12, rtol=0)


@pytest.mark.parametrize("lengths", MIXES)
def test_per_doc_key_mask_equals_bruteforce(lengths):
    """The per-document form with a key mask (the keys one CP owner holds)
    against the full T x T mask of the brute-force form; rows left without a
    key get O = 0, LSE = -inf in both."""
    cu, q, k, v = _inputs(lengths)
    T = int(cu[-1])
    mask = np.random.default_rng(T).random(T) < 0.4
    ob, lb = A.attention_bruteforce(q, k, v, cu, key_allowed=mask)
    op, lp = A.attention_per_doc(q, k, v, cu, key_allowed=mask)
    np.testing.assert_allclose(op, ob, atol=1e-12, rtol=0)
    assert np.array_equal(np.isneginf(lp), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lp[fin], lb[fin], atol=1e-12, rtol=0)


@pytest.mark.parametrize("policy", ["llama3", "perdoc", "hybrid"])
def test_merge_over_ring_owner_blocks(policy):
    """Ring order ("LLM Context Parallel in Production", "Ring Attention"): at
    step s shard j holds shard (j - s) mod N's KV block. For every shard's
    rows, merging the N step partials (each over one owner's keys) gives the
    unsplit result."""
    from oracle import plan as P
    lengths = [40, 7, 1, 60, 19, 33]
    cu, q, k, v = _inputs(lengths)
    N = 4
    T = int(cu[-1])
    pad = (-T) % (2 * N)
    if pad:  # the Llama3 split needs T % 2N == 0
        lengths = lengths[:-1] + [lengths[-1] + pad]
        cu, q, k, v = _inputs(lengths)
        T = int(cu[-1])
    plan = P.make_plan(lengths, N, policy)
    owner = np.full(T, -1)
    for j, sh in enumerate(plan.shards):
        for pc in sh.pieces:
            owner[pc.start:pc.end] = j
    assert (owner >= 0).all()
    o_full, l_full = A.attention_per_doc(q, k, v, cu)
    for j in range(N):
        rows = np.array(plan.query_indices(j), dtype=np.int64)
        parts = [A.attention_per_doc(q, k, v, cu, key_allowed=owner == (j - s) % N) for s in range(N)]
        o_parts = np.stack([p_[0][rows] for p_ in parts])
        l_parts = np.stack([p_[1][:, rows] for p_ in parts])
        om, lm = A.merge(o_parts, l_parts)
        np.testing.assert_allclose(om, o_full[rows], atol=1e-12, rtol=0)
        np.testing.assert_allclose(lm, l_full[:, rows], atol=1e-12, rtol=0)


def test_merge_all_empty_rows():
    o_parts = np.zeros((3, 2, 1, 4))
    lse_parts = np.full((3, 1, 2), -np.inf)
    lse_parts[1, 0, 1] = 0.5
    o_parts[1, 1, 0] = [1, 2, 3, 4]
    o, lse = A.merge(o_parts, lse_parts)
    assert np.array_equal(o[0, 0], np.zeros(4)) and lse[0, 0] == -np.inf
    assert np.array_equal(o[1, 0], [1, 2, 3, 4]) and lse[0, 1] == 0.5
    assert not np.isnan(o).any()


def _torch_ref_forward(q, k, v, cu, Hq, Hkv):
    """fp64 autograd-able brute-force document-masked attention in torch."""
    T, _, d = q.shape
    G = Hq // Hkv
    doc = torch.as_tensor(A.doc_ids(cu))
    idx = torch.arange(T)
    allowed = (doc[:, None] == doc[None, :]) & (idx[None, :] <= idx[:, None])
    kk = k.repeat_interleave(G, 1)
    vv = v.repeat_interleave(G, 1)
    s = torch.einsum("thd,shd->hts", q, kk) / math.sqrt(d)
    s = s.masked_fill(~allowed, float("-inf"))
    p = torch.softmax(s, dim=-1)
    return torch.einsum("hts,shd->thd", p, vv)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (2, 2), (3, 1)])
def test_backward_matches_autograd(Hq, Hkv):
    lengths = [1, 14, 3, 27, 2]
    T, d = sum(lengths), 8
    cu, q, k, v = _inputs(lengths, Hq=Hq, Hkv=Hkv, d=d, seed=4)
    do = synth.make_dout(T, Hq, d, seed=4)
    qt, kt, vt = (x.double().requires_grad_(True) for x in (q, k, v))
    out = _torch_ref_forward(qt, kt, vt, cu, Hq, Hkv)
    out.backward(do.double())
    o, lse = A.attention_per_doc(q, k, v, cu)
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12, rtol=0)
    dq, dk, dv = A.attention_bwd_per_doc(q, k, v, o, lse, do, cu, row_chunk=5)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11, rtol=0)


def test_backward_central_finite_differences():
    lengths = [4, 6]
    T, Hq, Hkv, d = 10, 2, 1, 4
    cu, q, k, v = _inputs(lengths, Hq=Hq, Hkv=Hkv, d=d, seed=8)
    do = A.to_f64(synth.make_dout(T, Hq, d, seed=8))
    qd, kd, vd = A.to_f64(q), A.to_f64(k), A.to_f64(v)
    o, lse = A.attention_per_doc(qd, kd, vd, cu)
    dq, dk, dv = A.attention_bwd_per_doc(qd, kd, vd, o, lse, do, cu)

    def loss(q, k, v):
        oo, _ = A.attention_per_doc(q, k, v, cu)
        return float(np.sum(oo * do))

    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, x, g in (("q", qd, dq), ("k", kd, dk), ("v", vd, dv)):
        for _ in range(6):
            i = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            args_p = {"q": qd, "k": kd, "v": vd}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**args_p) - loss(**args_m)) / (2 * eps)
            assert abs(fd - g[i]) <= 1e-6 * max(1.0, abs(g[i])), (name, i, fd, g[i])


def test_rows_sampler_matches_per_doc():
    lengths = [40, 1, 77, 13]
    cu, q, k, v = _inputs(lengths, Hq=4, Hkv=2, d=16, seed=2)
    o, lse = A.attention_per_doc(q, k, v, cu)
    rows = [0, 39, 40, 41, 100, 130]
    heads = [0, 3]
    os_, ls = A.attention_rows(q, k, v, cu, rows, heads)
    np.testing.assert_allclose(os_, o[rows][:, heads], atol=1e-12, rtol=0)
    np.testing.assert_allclose(ls, lse[heads][:, rows], atol=1e-12, rtol=0)
    os2, ls2 = A.attention_rows(q[rows], k, v, cu, rows, heads, q_holds_rows=True)
    np.testing.assert_array_equal(os2, os_)
    np.testing.assert_array_equal(ls2, ls)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 1), (2, 2)])
def test_sampled_row_gradients_match_autograd(Hq, Hkv):
    """The row-by-row gradient functions used for full-size spot checks
    (dQ at sampled query rows, dK/dV at sampled key rows) equal torch
    autograd of the brute-force document-masked attention at those rows,
    including first and last rows of documents and 1-token documents."""
    lengths = [1, 14, 3, 27, 2, 9]
    T, d = sum(lengths), 8
    cu, q, k, v = _inputs(lengths, Hq=Hq, Hkv=Hkv, d=d, seed=12)
    do = synth.make_dout(T, Hq, d, seed=12)
    qt, kt, vt = (x.double().requires_grad_(True) for x in (q, k, v))
    _torch_ref_forward(qt, kt, vt, cu, Hq, Hkv).backward(do.double())
    rows = [0, 1, 5, 14, 15, 17, 18, 30, 44, 45, 46, 47, T - 1]
    dq = A.attention_bwd_query_rows(q, k, v, do, cu, rows, list(range(Hq)))
    np.testing.assert_allclose(dq, qt.grad.numpy()[rows], atol=1e-11, rtol=0)
    key_rows = [0, 1, 7, 14, 16, 17, 40, 44, 45, 46, T - 2, T - 1]
    dk, dv = A.attention_bwd_key_rows(q, k, v, do, cu, key_rows)
    np.testing.assert_allclose(dk, kt.grad.numpy()[key_rows], atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy()[key_rows], atol=1e-11, rtol=0)


def test_sampled_row_gradients_with_a_scale():
    """The same with a non-default softmax scale (central differences of the
    per-row functions' loss would need the full forward; here the scale enters
    autograd through scaled queries: attention(q * c / (1/sqrt(d))) at the
    default scale equals attention(q) at scale c)."""
    lengths = [5, 11]
    T, Hq, Hkv, d = 16, 2, 1, 8
    cu, q, k, v = _inputs(lengths, Hq=Hq, Hkv=Hkv, d=d, seed=13)
    do = synth.make_dout(T, Hq, d, seed=13)
    c = 0.3
    factor = c * math.sqrt(d)
    qt = (A.to_f64(q) * 1.0)
    qs = torch.tensor(qt * factor, requires_grad=True)
    kt, vt = (x.double().requires_grad_(True) for x in (k, v))
    _torch_ref_forward(qs, kt, vt, cu, Hq, Hkv).backward(do.double())
    rows = list(range(T))
    dq = A.attention_bwd_query_rows(q, k, v, do, cu, rows, list(range(Hq)), scale=c)
    np.testing.assert_allclose(dq, qs.grad.numpy() * factor, atol=1e-11, rtol=0)
    dk, dv = A.attention_bwd_key_rows(q, k, v, do, cu, rows, scale=c)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11, rtol=0)
