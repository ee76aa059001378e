"""Parity at the full workload sizes, in the launch configuration the
benchmark times (every shard in one launch; forward output in fp32 for the
backward).

The fp64 oracle cannot recompute these sizes whole, so it checks samples it
can compute one by one: random query rows of every document (all heads) for
O and LSE; dQ at sampled query rows and dK, dV at the last key rows of every
document, long ones included (the gradient's definition row by row); and
complete documents short enough for the exact per-document gradient.
Documents are independent under the document mask, so a document's slice of
the inputs determines its slice of every output. Tolerances as in
test_gpu_attention.py.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 1e-2


def _run(cfg, policy=None, merge_blocks=0, bwd=True, rows_per_doc=6, max_bwd_doc=2100, seed=0,
         key_rows_per_doc=3):
    from context_document_masked_gb300 import fcp
    from context_document_masked_gb300.session import CPAttention
    w = synth.WORKLOADS[cfg]
    D = synth.doc_lengths(cfg)
    T, hq, hkv, d = w.T, w.Hq, w.Hkv, w.d
    dev = torch.device("cuda:0")
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=1000 + cfg, device=dev)
    s = CPAttention(D, w.cp, policy or w.policy, hq, hkv, d, device=dev)
    s.gather(k, v)
    out, lse = s.forward(q, k, v, out_dtype=torch.float32)
    out_bf, lse_bf = s.forward(q, k, v)
    merged = None
    if merge_blocks:
        B = merge_blocks
        bounds = [T * b // B for b in range(B + 1)]
        o_parts = torch.empty(B, T, hq, d, dtype=torch.float32, device=dev)
        l_parts = torch.empty(B, hq, T, dtype=torch.float32, device=dev)
        for b in range(B):
            s.forward(q, k, v, out=o_parts[b], lse=l_parts[b], kv_block=(bounds[b], bounds[b + 1]),
                      out_dtype=torch.float32)
        mo = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
        ml = torch.empty(hq, T, dtype=torch.float32, device=dev)
        fcp.merge(o_parts, l_parts, mo, ml)
        merged = (mo, ml)
        del o_parts, l_parts
    grads = None
    if bwd:
        do = synth.make_dout(T, hq, d, seed=1000 + cfg, device=dev)
        grads = s.backward(q, k, v, out, lse, do)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    cu = synth.cu_from_lengths(D)
    rng = np.random.default_rng(seed + cfg)
    errs = {"O": 0.0, "LSE": 0.0, "O_bf16_excess": 0.0, "merge": 0.0, "dQ": 0.0, "dK": 0.0, "dV": 0.0,
            "dQ_rows": 0.0, "dK_rows": 0.0, "dV_rows": 0.0}
    heads = list(range(hq))
    for i, L in enumerate(D):
        s0, s1 = int(cu[i]), int(cu[i + 1])
        local = sorted(set([0, L - 1] + rng.integers(0, L, size=rows_per_doc).tolist()))
        ks, vs = A.to_f64(k[s0:s1]), A.to_f64(v[s0:s1])      # upcast once per document
        cu_l = np.array([0, L])
        o_r, l_r = A.attention_rows(q[[s0 + r for r in local]].cpu(), ks, vs, cu_l, local, heads,
                                    q_holds_rows=True)
        rows = [s0 + r for r in local]
        g_o = out[rows].cpu().double().numpy()
        g_l = lse[:, rows].cpu().double().numpy()
        errs["O"] = max(errs["O"], float(np.abs(g_o - o_r).max()))
        errs["LSE"] = max(errs["LSE"], float(np.abs(g_l - l_r).max()))
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_r), 1e-30))) - 8)
        g_bf = out_bf[rows].cpu().double().numpy()
        errs["O_bf16_excess"] = max(errs["O_bf16_excess"], float((np.abs(g_bf - o_r) - half_ulp).max()))
        assert torch.equal(lse_bf[:, rows], lse[:, rows])
        if merged is not None:
            g_m = merged[0][rows].cpu().double().numpy()
            errs["merge"] = max(errs["merge"], float((np.abs(g_m - o_r) - half_ulp).max()))
            errs["LSE"] = max(errs["LSE"], float(np.abs(merged[1][:, rows].cpu().double().numpy() - l_r).max()))
        if grads is not None:
            # dQ at two sampled rows and the last row; dK, dV at the last key rows.
            for r in sorted(set([L - 1] + rng.integers(0, L, size=2).tolist())):
                dq_r = A.attention_bwd_query_rows(q[s0 + r:s0 + r + 1].cpu(), ks, vs, do[s0 + r:s0 + r + 1].cpu(),
                                                  cu_l, [r], heads, q_offset=r)
                g = grads[0][s0 + r:s0 + r + 1].cpu().double().numpy()
                errs["dQ_rows"] = max(errs["dQ_rows"], float(np.abs(g - dq_r).max()))
            kr0 = max(0, L - key_rows_per_doc)
            dk_r, dv_r = A.attention_bwd_key_rows(q[s0 + kr0:s1].cpu(), ks, vs, do[s0 + kr0:s1].cpu(), cu_l,
                                                  list(range(kr0, L)), q_offset=kr0)
            errs["dK_rows"] = max(errs["dK_rows"], float(np.abs(grads[1][s0 + kr0:s1].cpu().double().numpy()
                                                                - dk_r).max()))
            errs["dV_rows"] = max(errs["dV_rows"], float(np.abs(grads[2][s0 + kr0:s1].cpu().double().numpy()
                                                                - dv_r).max()))
        if grads is not None and L <= max_bwd_doc:
            qs, dos = q[s0:s1].cpu(), do[s0:s1].cpu()
            o_d, l_d = A.attention_per_doc(qs, ks, vs, cu_l)
            dq_r, dk_r, dv_r = A.attention_bwd_per_doc(qs, ks, vs, o_d, l_d, dos, cu_l)
            for name, g, ref in (("dQ", grads[0], dq_r), ("dK", grads[1], dk_r), ("dV", grads[2], dv_r)):
                errs[name] = max(errs[name], float(np.abs(g[s0:s1].cpu().double().numpy() - ref).max()))
    print(f"[err] cfg{cfg} {policy or w.policy}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["O"] <= TOL_O and errs["LSE"] <= TOL_LSE and errs["O_bf16_excess"] <= TOL_O
    assert errs["merge"] <= TOL_O
    assert errs["dQ"] <= TOL_GRAD and errs["dK"] <= TOL_GRAD and errs["dV"] <= TOL_GRAD
    assert errs["dQ_rows"] <= TOL_GRAD and errs["dK_rows"] <= TOL_GRAD and errs["dV_rows"] <= TOL_GRAD
    return errs


def test_packed32k_perdoc_fwd_bwd(cuda):
    _run(2)


def test_packed128k_hybrid_fwd_bwd_and_merge_over_8_blocks(cuda):
    _run(3, merge_blocks=8, rows_per_doc=4)


@pytest.mark.parametrize("policy", ["wholedoc", "perdoc", "llama3"])
def test_packed64k_shortdocs(cuda, policy):
    _run(4, policy=policy, rows_per_doc=3)


def test_packed512k_hybrid_fwd_bwd(cuda):
    _run(5, rows_per_doc=2, max_bwd_doc=1500)
