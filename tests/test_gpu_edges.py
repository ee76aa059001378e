"""Degenerate cases of the CUDA path, checked against closed forms that do not
go through the oracle.

With Q = 0 every score is 0, so under the document mask each query row
attends uniformly to its visible keys: O_i = mean of v_j over j in doc(i),
j <= i, and LSE_i = ln(i - start(i) + 1) ("FlashCP", §2.1 and Fig. 1(a): the
intra-document causal mask; the softmax of equal scores is uniform). The
gradient then has closed forms too (P_ij = 1/n_i with n_i the row's visible
key count): dV_j = sum over rows i that see j of dO_i / n_i; dK = 0 because
every dS_ij multiplies q_i = 0; dQ_i = scale/n_i * sum_j (dO_i.v_j - D_i) k_j
with D_i = dO_i.O_i. An empty key block leaves every row with no visible key:
O = 0 and LSE = -inf exactly.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _session(D, hq, hkv, d, cp, pol):
    from context_document_masked_gb300.session import CPAttention
    return CPAttention(D, cp, pol, hq, hkv, d)


def _prefix_forms(D, k, v, do, hq, hkv, d):
    """Closed forms for Q = 0 (float64, per document, running sums)."""
    k = k.double().numpy()
    v = v.double().numpy()
    do = do.double().numpy()
    T = sum(D)
    G = hq // hkv
    scale = 1.0 / np.sqrt(d)
    O = np.zeros((T, hq, d))
    L = np.zeros((hq, T))
    dQ = np.zeros((T, hq, d))
    dV = np.zeros((T, hkv, d))
    s0 = 0
    for n_doc in D:
        idx = np.arange(s0, s0 + n_doc)
        cnt = np.arange(1, n_doc + 1, dtype=np.float64)
        for h in range(hq):
            g = h // G
            vs, ks, dos = v[idx, g], k[idx, g], do[idx, h]
            o = np.cumsum(vs, axis=0) / cnt[:, None]
            O[idx, h] = o
            L[h, idx] = np.log(cnt)
            Dr = np.sum(dos * o, axis=1)                       # D_i = dO_i . O_i
            # sum_{j<=i} (dO_i . v_j) k_j = dO_i^T (sum_{j<=i} v_j k_j^T), kept as a running d x d sum.
            M = np.zeros((d, d))
            ksum = np.zeros(d)
            for t in range(n_doc):
                M += np.outer(vs[t], ks[t])
                ksum += ks[t]
                dQ[idx[t], h] = scale / cnt[t] * (dos[t] @ M - Dr[t] * ksum)
            # dV_j = sum_{i>=j} dO_i / n_i: a suffix sum.
            w = dos / cnt[:, None]
            dV[idx, g] += np.cumsum(w[::-1], axis=0)[::-1]
        s0 += n_doc
    return O, L, dQ, dV


CASES = [
    ("ragged_d128_perdoc", synth.random_doc_lengths(1024, seed=41), 4, 2, 128, 4, "perdoc"),
    ("edges_d64_llama3", [1, 127, 128, 129, 63, 64], 4, 2, 64, 2, "llama3"),
    ("gqa4_d128_hybrid", synth.random_doc_lengths(768, seed=42), 8, 2, 128, 3, "hybrid"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_zero_queries_give_prefix_means_and_closed_form_gradients(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    T = sum(D)
    _, k, v = synth.make_qkv(T, hq, hkv, d, seed=5)
    do = synth.make_dout(T, hq, d, seed=5)
    q = torch.zeros(T, hq, d, dtype=torch.bfloat16)
    s = _session(D, hq, hkv, d, cp, pol)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd, out_dtype=torch.float32)
    dq, dk, dv = s.backward(qd, kd, vd, out, lse, dod)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    O, L, dQ, dV = _prefix_forms(D, k, v, do, hq, hkv, d)
    e = {"O": np.abs(out.cpu().double().numpy() - O).max(),
         "LSE": np.abs(lse.cpu().double().numpy() - L).max(),
         "dQ": np.abs(dq.cpu().double().numpy() - dQ).max(),
         "dV": np.abs(dv.cpu().double().numpy() - dV).max()}
    print(f"[err] {name} q=0: " + ", ".join(f"{a} {b:.2e}" for a, b in e.items()))
    assert e["O"] <= 1e-3 and e["LSE"] <= 1e-5
    assert e["dQ"] <= 1e-2 and e["dV"] <= 1e-2
    assert torch.count_nonzero(dk).item() == 0          # dS_ij q_i with q = 0


def test_zero_queries_e4m3_path(cuda):
    """The e4m3 Q K^T forward on Q = 0: the quantiser's zero-amax scale (2^0),
    all-zero codes, uniform attention."""
    D = synth.random_doc_lengths(1024, seed=43)
    T, hq, hkv, d = sum(D), 4, 2, 128
    _, k, v = synth.make_qkv(T, hq, hkv, d, seed=6)
    do = synth.make_dout(T, hq, d, seed=6)
    q = torch.zeros(T, hq, d, dtype=torch.bfloat16)
    s = _session(D, hq, hkv, d, 4, "perdoc")
    s.gather(k.cuda(), v.cuda())
    out, lse = s.forward_qk8(q.cuda(), k.cuda(), v.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    O, L, _, _ = _prefix_forms(D, k, v, do, hq, hkv, d)
    assert np.abs(out.cpu().double().numpy() - O).max() <= 1e-3
    assert np.abs(lse.cpu().double().numpy() - L).max() <= 1e-5


@pytest.mark.parametrize("where", ["start", "middle", "end"])
def test_empty_key_block_gives_zero_and_minus_inf(cuda, where):
    D = synth.random_doc_lengths(1024, seed=44)
    T, hq, hkv, d = sum(D), 4, 2, 128
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=7)
    s = _session(D, hq, hkv, d, 4, "perdoc")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s.gather(kd, vd)
    lo = {"start": 0, "middle": T // 2, "end": T}[where]
    for dt in (torch.float32, torch.bfloat16):
        out = torch.full((T, hq, d), 7.0, dtype=dt, device="cuda")
        lse = torch.full((hq, T), 7.0, device="cuda")
        s.forward(qd, kd, vd, out=out, lse=lse, kv_block=(lo, lo), out_dtype=dt)
        torch.cuda.synchronize()
        assert s.device_status() == 0
        assert torch.count_nonzero(out).item() == 0
        assert bool(torch.all(torch.isneginf(lse)))


def test_merge_of_zero_rows_is_a_no_op(cuda):
    from context_document_masked_gb300 import fcp
    o_parts = torch.empty(2, 0, 4, 128, device="cuda")
    l_parts = torch.empty(2, 4, 0, device="cuda")
    out = torch.empty(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, 0, device="cuda")
    fcp.merge(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
