"""GPU parity of the ring-order forward (fcp_attn_fwd_ring) against the fp64
oracle, through the C ABI.

"LLM Context Parallel in Production", "Ring Attention": at step s of the ring
shard j holds the KV block of shard (j - s) mod N and folds its partial
result into the online softmax. The fused mode (ring_step = -1) visits every
owner's keys in that order in one pass, reading them from the owners' rows of
K/V (no gathered buffer); ring_step = s gives the partial (O, LSE) of step s
alone, which fcp_merge combines. Tolerances as in test_gpu_attention.py.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import plan as P

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3

CASES = [
    # name, doc lengths, Hq, Hkv, d, cp, policy
    ("cfg1_llama3", synth.doc_lengths(1), 4, 2, 64, 2, "llama3"),
    ("ragged_d128_perdoc", synth.random_doc_lengths(1024, seed=7), 4, 2, 128, 4, "perdoc"),
    ("ragged_d128_hybrid", synth.random_doc_lengths(2048, seed=9), 8, 2, 128, 4, "hybrid"),
    ("gqa3_d128_perdoc", synth.random_doc_lengths(1536, seed=13), 6, 2, 128, 3, "perdoc"),
    ("tiles_edges_perdoc", [1, 127, 128, 129, 255, 256, 1, 1, 600, 2], 4, 2, 128, 3, "perdoc"),
    ("long_doc_wholedoc", [3000, 40, 1, 55, 900], 8, 2, 128, 4, "wholedoc"),
]


def _setup(name, D, hq, hkv, d, cp, pol, seed=0):
    from context_document_masked_gb300.session import CPAttention
    T = sum(D)
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=seed)
    s = CPAttention(D, cp, pol, hq, hkv, d)
    return s, synth.cu_from_lengths(D), q, k, v


def _owners(D, cp, pol):
    plan = P.make_plan(D, cp, pol)
    owner = np.full(sum(D), -1)
    for j, sh in enumerate(plan.shards):
        for pc in sh.pieces:
            owner[pc.start:pc.end] = j
    assert (owner >= 0).all()
    return plan, owner


def _err(a, b):
    a = np.asarray(a, dtype=np.float64)
    assert np.isfinite(a).all()
    return float(np.max(np.abs(a - b))) if a.size else 0.0


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ring_fused_matches_oracle_and_gathered_forward(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v = _setup(*case)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = s.forward_ring(qd, kd, vd, ring_step=-1, out_dtype=torch.float32)
    s.gather(kd, vd)
    out_g, lse_g = s.forward(qd, kd, vd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    e_o, e_l = _err(out.cpu(), o_ref), _err(lse.cpu(), lse_ref)
    print(f"[err] ring fused O {e_o:.3e} LSE {e_l:.3e}")
    assert e_o <= TOL_O and e_l <= TOL_LSE
    # The same function as the gathered forward; only the key order differs.
    assert float((out - out_g).abs().max()) <= 2e-3
    assert float((lse - lse_g).abs().max()) <= 1e-4


@pytest.mark.parametrize("case", CASES[1:3], ids=[c[0] for c in CASES[1:3]])
def test_ring_fused_one_shard_at_a_time(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v = _setup(*case)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.full((s.T, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((hq, s.T), float("nan"), dtype=torch.float32, device="cuda")
    for j in range(cp):
        s.forward_ring(qd, kd, vd, ring_step=-1, shard=j, out=out, lse=lse, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    assert _err(out.cpu(), o_ref) <= TOL_O
    assert _err(lse.cpu(), lse_ref) <= TOL_LSE


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ring_steps_match_owner_blocks_and_merge(cuda, case):
    """Ring step s of every shard at once: shard j's rows against the oracle
    restricted to owner (j - s) mod N's keys (rows with none: O = 0,
    LSE = -inf); the N step partials merged by fcp_merge give the full result."""
    from context_document_masked_gb300 import fcp
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v = _setup(*case)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    plan, owner = _owners(D, cp, pol)
    o_parts = torch.empty(cp, s.T, hq, d, dtype=torch.float32, device="cuda")
    l_parts = torch.empty(cp, hq, s.T, dtype=torch.float32, device="cuda")
    for st in range(cp):
        s.forward_ring(qd, kd, vd, ring_step=st, out=o_parts[st], lse=l_parts[st], out_dtype=torch.float32)
    out = torch.empty(s.T, hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(hq, s.T, dtype=torch.float32, device="cuda")
    fcp.merge(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    e_o = e_l = 0.0
    for j in range(cp):
        rows = np.array(plan.query_indices(j), dtype=np.int64)
        for st in range(cp):
            o_r, l_r = A.attention_per_doc(q, k, v, cu, key_allowed=owner == (j - st) % cp)
            lp = l_parts[st][:, rows].cpu().numpy()
            assert np.array_equal(np.isneginf(lp), np.isneginf(l_r[:, rows]))
            fin = np.isfinite(l_r[:, rows])
            e_l = max(e_l, float(np.abs(lp[fin] - l_r[:, rows][fin]).max()) if fin.any() else 0.0)
            e_o = max(e_o, _err(o_parts[st][rows].cpu(), o_r[rows]))
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    e_m = float((np.abs(out.float().cpu().numpy() - o_ref) - half_ulp).max())
    e_ml = _err(lse.cpu(), lse_ref)
    print(f"[err] ring steps O {e_o:.3e} LSE {e_l:.3e}; merged O beyond half-ulp {e_m:.3e}, LSE {e_ml:.3e}")
    assert e_o <= TOL_O and e_l <= TOL_LSE
    assert e_m <= TOL_O and e_ml <= TOL_LSE


def test_ring_rejects_bad_step(cuda):
    from context_document_masked_gb300 import fcp
    name, D, hq, hkv, d, cp, pol = CASES[1]
    s, cu, q, k, v = _setup(*CASES[1])
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for bad in (-2, cp):
        with pytest.raises(fcp.FcpError):
            s.forward_ring(qd, kd, vd, ring_step=bad)


def test_merge_ring_checks_the_partials_and_matches_merge(cuda):
    """fcp_merge_ring: with every ring step's partial present (tags in any
    order) it equals fcp_merge of the same partials bit for bit and the
    oracle; with one step's partial lost it reports FCP_ERR_MISSING_PART and
    leaves the outputs untouched."""
    from context_document_masked_gb300 import fcp
    name, D, hq, hkv, d, cp, pol = CASES[1]
    s, cu, q, k, v = _setup(*CASES[1])
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    order = [2, 0, 3, 1]                      # the order the partials "arrived" in
    o_parts = torch.empty(cp, s.T, hq, d, dtype=torch.float32, device="cuda")
    l_parts = torch.empty(cp, hq, s.T, dtype=torch.float32, device="cuda")
    for b, st in enumerate(order):
        s.forward_ring(qd, kd, vd, ring_step=st, out=o_parts[b], lse=l_parts[b], out_dtype=torch.float32)
    out = torch.full((s.T, hq, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((hq, s.T), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(fcp.FcpError) as e:          # the partial of step 1 never arrived
        fcp.merge_ring(s.dplan, o_parts[:3], l_parts[:3], order[:3], out, lse)
    assert e.value.status == fcp.ERR_MISSING_PART
    with pytest.raises(fcp.FcpError) as e:          # step 0 twice, step 1 lost
        fcp.merge_ring(s.dplan, o_parts, l_parts, [2, 0, 3, 0], out, lse)
    assert e.value.status == fcp.ERR_MISSING_PART
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    fcp.merge_ring(s.dplan, o_parts, l_parts, order, out, lse)
    ref_o = torch.empty_like(out)
    ref_l = torch.empty_like(lse)
    fcp.merge(o_parts, l_parts, ref_o, ref_l)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    assert float((np.abs(out.float().cpu().numpy() - o_ref) - half_ulp).max()) <= TOL_O
    assert _err(lse.cpu(), lse_ref) <= TOL_LSE
