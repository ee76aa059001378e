"""GPU parity on inputs that drive the forward's online-softmax rescale, with a
non-default softmax scale, and the fp16-range guard of the tensor-core
operands, through the C ABI.

The online softmax ("LLM Context Parallel in Production", "Core Principle:
Split Q, Circulate KV" and "Ring Attention") keeps a running row maximum m and
exponential sum; the kernels rescale the accumulated O only when a later key
tile raises m by more than 2^8 (5.545 nats). With Q, K ~ N(0, 1) and the
1/sqrt(d) scale a row's maximum grows by ~3 nats at most after its first key
tile, so those inputs never take that branch. Here Q is scaled by 2 and each
document's K rows by a ramp that grows (or shrinks) along the document, so
the keys a query tile visits last (first) carry scores ~20 nats above the
others. Each case asserts, from the inputs alone, that some row's maximum
grows by more than 5.545 nats after the keys its first tile can hold, and
reads the kernels' rescale counter to show the branch ran.

Tolerances as in test_gpu_attention.py: max-abs 1e-2 on O and the gradients,
1e-3 on LSE, against the fp64 oracle on the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import fp8 as F

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 1e-2
RESCALE_NATS = 8.0 * np.log(2.0)   # the kernels' threshold, 2^8, in nats

# name, doc lengths, Hq, Hkv, d, cp, policy, softmax scale (None = 1/sqrt(d))
CASES = [
    ("perdoc_d128", [1200, 700, 2, 900, 129, 1165], 8, 2, 128, 4, "perdoc", None),
    ("hybrid_d128_scale", [1500, 1, 640, 300, 1655], 4, 2, 128, 4, "hybrid", 0.07),
    ("llama3_d64_gqa3", [1000, 536, 1, 511], 6, 2, 64, 2, "llama3", 0.1),
]


def _ramp_inputs(D, hq, hkv, d, seed, up=True, q_gain=2.0, span=1.5):
    """Seeded N(0,1) bf16 inputs with Q scaled by q_gain and the K rows of each
    document scaled by 1 + span * x, x running 0 -> 1 (up) or 1 -> 0 along the
    document; rounded back to bf16 (both sides read the same values)."""
    T = sum(D)
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=seed)
    pos = np.concatenate([np.arange(L) / max(L - 1, 1) for L in D])
    r = 1.0 + span * (pos if up else 1.0 - pos)
    k = (k.double() * torch.from_numpy(r)[:, None, None]).to(torch.bfloat16)
    q = (q.double() * q_gain).to(torch.bfloat16)
    return q, k, v


def _growth_after_first_tile(q, k, D, hq, hkv, scale):
    """Largest growth, over rows and heads, of a row's score maximum beyond the
    maximum over the first 128 keys of its document (a query tile's first key
    tile, in key order, lies inside them). Above RESCALE_NATS the kernels must
    rescale O at least once."""
    cu = synth.cu_from_lengths(D)
    G = hq // hkv
    qf, kf = A.to_f64(q), A.to_f64(k)
    best = 0.0
    for i in range(len(D)):
        a, b = int(cu[i]), int(cu[i + 1])
        if b - a <= 128:
            continue
        vis = np.tril(np.ones((b - a, b - a), dtype=bool))
        for h in range(hq):
            s = np.where(vis, scale * (qf[a:b, h] @ kf[a:b, h // G].T), -np.inf)
            best = max(best, float((s.max(axis=1) - s[:, :128].max(axis=1)).max()))
    return best


def _err(a, b, what):
    a = np.asarray(a, dtype=np.float64)
    assert np.isfinite(a).all(), what
    e = float(np.max(np.abs(a - b))) if a.size else 0.0
    print(f"[err] {what} max-abs {e:.3e}")
    return e


def _session(D, cp, pol, hq, hkv, d, scale):
    from context_document_masked_gb300.session import CPAttention
    return CPAttention(D, cp, pol, hq, hkv, d, scale=scale or 0.0)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rescale_forward_variants_and_backward(cuda, lib, case):
    fcp = lib
    name, D, hq, hkv, d, cp, pol, scale = case
    sc = A.default_scale(d) if scale is None else scale
    q, k, v = _ramp_inputs(D, hq, hkv, d, seed=41)
    g = _growth_after_first_tile(q, k, D, hq, hkv, sc)
    print(f"[rescale] {name}: row maximum grows by {g:.2f} nats after the first key tile")
    assert g > RESCALE_NATS + 2.0
    cu = synth.cu_from_lengths(D)
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu, scale=sc)
    s = _session(D, cp, pol, hq, hkv, d, scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert fcp.debug_rescale_events(s.ws) == 0

    # Gathered keys, fp32 and bf16 output, all shards in one launch.
    s.gather(kd, vd)
    out32, lse32 = s.forward(qd, kd, vd, out_dtype=torch.float32)
    out16, lse16 = s.forward(qd, kd, vd)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    n_ev = fcp.debug_rescale_events(s.ws)
    print(f"[rescale] {name}: gathered forward rescale events {n_ev}")
    assert n_ev > 0
    assert _err(out32.cpu(), o_ref, "O(fp32)") <= TOL_O
    assert _err(lse32.cpu(), lse_ref, "LSE") <= TOL_LSE
    assert torch.equal(out16, out32.to(torch.bfloat16)) and torch.equal(lse16, lse32)

    # One shard at a time, each with only its own received rows.
    o1 = torch.full_like(out32, float("nan"))
    l1 = torch.full_like(lse32, float("nan"))
    for j in range(cp):
        s.gather(kd, vd, shard=j)
        s.forward(qd, kd, vd, shard=j, out=o1, lse=l1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fcp.debug_rescale_events(s.ws) > 0
    assert _err(o1.cpu(), o_ref, "O(fp32, one shard per launch)") <= TOL_O
    assert _err(l1.cpu(), lse_ref, "LSE(one shard per launch)") <= TOL_LSE

    # Backward from the fp32 output.
    do = synth.make_dout(s.T, hq, d, seed=42)
    s.gather(kd, vd)
    dq, dk, dv = s.backward(qd, kd, vd, out32, lse32, do.cuda())
    torch.cuda.synchronize()
    assert s.device_status() == 0
    dq_ref, dk_ref, dv_ref = A.attention_bwd_per_doc(q, k, v, o_ref, lse_ref, do, cu, scale=sc)
    assert _err(dv.cpu(), dv_ref, "dV") <= TOL_GRAD
    assert _err(dk.cpu(), dk_ref, "dK") <= TOL_GRAD
    assert _err(dq.cpu(), dq_ref, "dQ") <= TOL_GRAD

    # The allocation-free forward runs the same kernel on the same inputs: its
    # rows equal the workspace forward's bit for bit.
    on = torch.full_like(out32, float("nan"))
    ln = torch.full_like(lse32, float("nan"))
    fcp.attn_fwd_noalloc(qd, kd, vd, s.kbuf, s.vbuf, s.dplan, -1, on, ln, scale=scale or 0.0)
    torch.cuda.synchronize()
    assert torch.equal(on, out32) and torch.equal(ln, lse32)


@pytest.mark.parametrize("case", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_rescale_ring_fused(cuda, lib, case):
    """The fused ring visits a shard's own keys first, then the other owners'
    by ring distance; with K shrinking along each document the earlier keys,
    visited later, carry the largest scores."""
    fcp = lib
    name, D, hq, hkv, d, cp, pol, scale = case
    sc = A.default_scale(d) if scale is None else scale
    q, k, v = _ramp_inputs(D, hq, hkv, d, seed=43, up=False)
    cu = synth.cu_from_lengths(D)
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu, scale=sc)
    s = _session(D, cp, pol, hq, hkv, d, scale)
    out, lse = s.forward_ring(q.cuda(), k.cuda(), v.cuda(), ring_step=-1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    n_ev = fcp.debug_rescale_events(s.ws)
    print(f"[rescale] {name}: fused ring rescale events {n_ev}")
    assert n_ev > 0
    assert _err(out.cpu(), o_ref, "O(ring fused)") <= TOL_O
    assert _err(lse.cpu(), lse_ref, "LSE(ring fused)") <= TOL_LSE


def test_rescale_e4m3_qk(cuda, lib):
    """The e4m3 Q K^T forward on the ramp inputs, against the oracle on the
    dequantised Q and K (the scales are powers of two)."""
    fcp = lib
    name, D, hq, hkv, d, cp, pol, scale = CASES[0]
    sc = A.default_scale(d)
    q, k, v = _ramp_inputs(D, hq, hkv, d, seed=44)
    qdq = torch.from_numpy(F.dequantized_tensor(A.to_f64(q)))
    kdq = torch.from_numpy(F.dequantized_tensor(A.to_f64(k)))
    cu = synth.cu_from_lengths(D)
    o_ref, lse_ref = A.attention_per_doc(qdq, kdq, v, cu, scale=sc)
    assert _growth_after_first_tile(qdq, kdq, D, hq, hkv, sc) > RESCALE_NATS + 2.0
    s = _session(D, cp, pol, hq, hkv, d, scale)
    kd, vd = k.cuda(), v.cuda()
    s.gather(kd, vd)
    out, lse = s.forward_qk8(q.cuda(), kd, vd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    n_ev = fcp.debug_rescale_events(s.ws)
    print(f"[rescale] e4m3 Q K^T forward rescale events {n_ev}")
    assert n_ev > 0
    assert _err(out.cpu(), o_ref, "O(e4m3 QK)") <= TOL_O
    assert _err(lse.cpu(), lse_ref, "LSE(e4m3 QK)") <= TOL_LSE


def test_standard_inputs_do_not_rescale(cuda, lib):
    """The converse: on N(0,1) inputs with the default scale no row grows by
    2^8 after its first key tile, and the counter stays at zero."""
    fcp = lib
    D = [1200, 700, 2, 900, 129, 1165]
    hq, hkv, d = 8, 2, 128
    q, k, v = synth.make_qkv(sum(D), hq, hkv, d, seed=45)
    assert _growth_after_first_tile(q, k, D, hq, hkv, A.default_scale(d)) < RESCALE_NATS
    s = _session(D, 4, "perdoc", hq, hkv, d, None)
    kd, vd = k.cuda(), v.cuda()
    s.gather(kd, vd)
    s.forward(q.cuda(), kd, vd)
    torch.cuda.synchronize()
    assert fcp.debug_rescale_events(s.ws) == 0


F16_MAX_PAST = 7.0e4   # > 65504, the largest finite fp16 value; a bf16 value


@pytest.mark.parametrize("where", ["q", "dout", "v"])
def test_fp16_range_guard_reports_and_recovers(cuda, lib, where):
    """One input element beyond the fp16 range of the tensor-core operands:
    V is converted by the forward, Q and dO by the backward's preprocess. The
    call completes (its results for that input are not meaningful) and
    fcp_get_device_status reports FCP_ERR_UNSUPPORTED; the next call on clean
    inputs, same workspace, is correct and reports nothing."""
    fcp = lib
    D = [300, 1, 500, 223]
    hq, hkv, d, cp = 4, 2, 128, 2
    T = sum(D)
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=46)
    do = synth.make_dout(T, hq, d, seed=46)
    bad = {"q": q.clone(), "dout": do.clone(), "v": v.clone()}[where]
    bad.view(-1)[12345 % bad.numel()] = F16_MAX_PAST
    assert float(bad.float().abs().max()) > 65504.0
    inputs = {"q": q, "dout": do, "v": v}
    inputs[where] = bad
    s = _session(D, cp, "perdoc", hq, hkv, d, None)
    kd = k.cuda()
    qd, vd, dod = inputs["q"].cuda(), inputs["v"].cuda(), inputs["dout"].cuda()
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd, out_dtype=torch.float32)
    if where != "v":
        s.backward(qd, kd, vd, out, lse, dod)
    torch.cuda.synchronize()
    assert s.device_status() == fcp.ERR_UNSUPPORTED
    assert s.device_status() == fcp.OK          # reading the status cleared it

    qd, vd, dod = q.cuda(), v.cuda(), do.cuda()
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd, out_dtype=torch.float32)
    dq, dk, dv = s.backward(qd, kd, vd, out, lse, dod)
    torch.cuda.synchronize()
    assert s.device_status() == fcp.OK
    cu = synth.cu_from_lengths(D)
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    dq_ref, dk_ref, dv_ref = A.attention_bwd_per_doc(q, k, v, o_ref, lse_ref, do, cu)
    assert _err(out.cpu(), o_ref, "O after recovery") <= TOL_O
    assert _err(lse.cpu(), lse_ref, "LSE after recovery") <= TOL_LSE
    assert _err(dq.cpu(), dq_ref, "dQ after recovery") <= TOL_GRAD
    assert _err(dk.cpu(), dk_ref, "dK after recovery") <= TOL_GRAD
    assert _err(dv.cpu(), dv_ref, "dV after recovery") <= TOL_GRAD
