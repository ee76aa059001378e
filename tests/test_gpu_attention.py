"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Tolerances: max-abs 1e-2 on O, dQ, dK, dV and 1e-3 on LSE (bf16 inputs, fp32
accumulation); bit-exact for the gather. Inputs are the seeded synthetic
tensors of `synth`, the same for both sides.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import plan as P

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_GRAD = 1e-2, 1e-3, 1e-2

SMALL = [
    # name, doc lengths, Hq, Hkv, d, cp, policy
    ("cfg1", synth.doc_lengths(1), 4, 2, 64, 2, "llama3"),
    ("ragged_d128_perdoc", synth.random_doc_lengths(1024, seed=7), 4, 2, 128, 4, "perdoc"),
    ("ragged_d128_wholedoc", synth.random_doc_lengths(1024, seed=8), 4, 2, 128, 4, "wholedoc"),
    ("ragged_d128_hybrid", synth.random_doc_lengths(2048, seed=9), 8, 2, 128, 4, "hybrid"),
    ("ragged_d64_llama3", synth.random_doc_lengths(1536, seed=10), 4, 2, 64, 3, "llama3"),
    ("tiles_edges", [1, 127, 128, 129, 255, 256, 1, 1, 600, 2], 4, 2, 128, 3, "perdoc"),
    ("long_doc_gqa4", [3000, 40, 1, 55], 8, 2, 128, 2, "perdoc"),
    ("single_doc", [1536], 4, 2, 128, 2, "llama3"),
    ("mha_d128_perdoc", synth.random_doc_lengths(1024, seed=11), 4, 4, 128, 4, "perdoc"),
    ("gqa3_d64_hybrid", synth.random_doc_lengths(1536, seed=12), 6, 2, 64, 3, "hybrid"),
]


def _setup(name, D, hq, hkv, d, cp, pol, seed=0):
    from context_document_masked_gb300.session import CPAttention
    T = sum(D)
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=seed)
    cu = synth.cu_from_lengths(D)
    s = CPAttention(D, cp, pol, hq, hkv, d)
    dev = s.device
    return s, cu, q, k, v, q.to(dev), k.to(dev), v.to(dev)


def _maxabs(a, b, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape
    assert np.isfinite(a).all()
    e = float(np.max(np.abs(a - b))) if a.size else 0.0
    print(f"[err] {what} max-abs {e:.3e}")
    return e


def _bf16_excess(out_bf16, ref):
    """Error of a bf16-stored output beyond the half-ulp the bf16 format itself
    adds when it stores the exact value (round to nearest even)."""
    a = out_bf16.float().cpu().numpy().astype(np.float64)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 8)
    e = float(np.max(np.abs(a - ref) - half_ulp))
    print(f"[err] O(bf16) max-abs beyond half-ulp {e:.3e}")
    return e


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_forward_all_shards(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    s.gather(kd, vd)
    out32, lse32 = s.forward(qd, kd, vd, out_dtype=torch.float32)
    out, lse = s.forward(qd, kd, vd)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    assert _maxabs(out32.cpu(), o_ref, "O(fp32)") <= TOL_O
    assert _maxabs(lse32.cpu(), lse_ref, "LSE") <= TOL_LSE
    assert torch.equal(lse, lse32)
    assert torch.equal(out, out32.to(torch.bfloat16))
    assert _bf16_excess(out, o_ref) <= TOL_O


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_forward_output_only_16_byte_aligned(cuda, dtype):
    """The API asks for 16-byte alignment of `out`; the kernel stores 32 bytes
    at a time only when the pointer allows it. Output written at a 16-byte
    offset (the narrower stores) equals the aligned output bit for bit."""
    case = SMALL[3]
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    s.gather(kd, vd)
    ref, lse_ref = s.forward(qd, kd, vd, out_dtype=dtype)
    shift = 16 // torch.tensor([], dtype=dtype).element_size()
    flat = torch.full((s.T * hq * d + shift,), float("nan"), dtype=dtype, device=s.device)
    out = flat[shift:].view(s.T, hq, d)
    assert out.data_ptr() % 32 == 16
    lse = torch.empty_like(lse_ref)
    s.forward(qd, kd, vd, out=out, lse=lse, out_dtype=dtype)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    assert torch.equal(out, ref) and torch.equal(lse, lse_ref)
    assert torch.isnan(flat[:shift].float()).all()  # nothing written before `out`


@pytest.mark.parametrize("case", SMALL[:6], ids=[c[0] for c in SMALL[:6]])
def test_forward_one_shard_at_a_time(cuda, case):
    """Each shard alone, with only its own received keys gathered: assembling
    the shards' rows by their query index lists gives the unsharded result."""
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    out = torch.full((s.T, hq, d), float("nan"), dtype=torch.bfloat16, device=s.device)
    lse = torch.full((hq, s.T), float("nan"), dtype=torch.float32, device=s.device)
    ref_plan = P.make_plan(D, cp, pol)
    for j in range(cp):
        s.kbuf.fill_(float("nan"))          # only this shard's gathered rows may be read
        s.vbuf.fill_(float("nan"))
        s.gather(kd, vd, shard=j)
        s.forward(qd, kd, vd, shard=j, out=out, lse=lse)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    covered = np.concatenate([ref_plan.query_indices(j) for j in range(cp)])
    assert np.array_equal(np.sort(covered), np.arange(s.T))
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    assert _bf16_excess(out, o_ref) <= TOL_O
    assert _maxabs(lse.cpu(), lse_ref, "LSE") <= TOL_LSE


def test_first_token_row_is_exact(cuda):
    D = [1, 9, 130, 1, 300]
    s, cu, q, k, v, qd, kd, vd = _setup("first", D, 4, 2, 128, 2, "perdoc")
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd)
    torch.cuda.synchronize()
    for st in cu[:-1]:
        for h in range(4):
            assert torch.equal(out[st, h].cpu(), v[st, h // 2])


def test_round_bf16_is_the_forward_bf16_output(cuda):
    """fcp_round_bf16 of the fp32 output equals the forward's own bf16 output,
    and, on random values with exact ties, subnormals, infinities and values
    near the bf16 maximum, equals round-to-nearest-even (PyTorch's CPU cast)."""
    from context_document_masked_gb300 import fcp
    case = SMALL[3]
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    s.gather(kd, vd)
    out32, _ = s.forward(qd, kd, vd, out_dtype=torch.float32)
    out16, _ = s.forward(qd, kd, vd)
    r = torch.empty_like(out16)
    fcp.round_bf16(out32, r)
    torch.cuda.synchronize()
    assert torch.equal(r, out16)
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1 << 16, generator=g) * torch.exp2(torch.randint(-140, 128, (1 << 16,), generator=g).float())
    bits = torch.randint(0, 1 << 16, (4096,), generator=g, dtype=torch.int32)
    x[:4096] = ((bits << 16) | 0x8000).view(torch.float32)     # exactly halfway between two bf16
    x[4096:4100] = torch.tensor([float("inf"), -float("inf"), 3.3895e38, -0.0])
    x = x[torch.isfinite(x) | torch.isinf(x)]
    x = x[: x.numel() // 8 * 8]
    y = torch.empty(x.numel(), dtype=torch.bfloat16, device="cuda")
    fcp.round_bf16(x.cuda(), y)
    torch.cuda.synchronize()
    ref = x.to(torch.bfloat16)
    assert torch.equal(y.cpu().view(torch.int16), ref.view(torch.int16))


def test_gather_is_byte_exact(cuda):
    D = synth.doc_lengths(2)[:5]
    T = sum(D) - sum(D) % 8
    D[-1] -= sum(D) - T
    s, cu, q, k, v, qd, kd, vd = _setup("g", D, 8, 2, 128, 4, "perdoc")
    s.gather(kd, vd)
    torch.cuda.synchronize()
    ref = P.make_plan(D, 4, "perdoc")
    rows = [t for sh in ref.shards for (_, a, b) in sh.kv_remote for t in range(a, b)]
    assert s.dplan.total_remote_rows == len(rows)
    assert torch.equal(s.kbuf[: len(rows)].cpu(), k[rows])
    assert torch.equal(s.vbuf[: len(rows)].cpu(), v[rows])


@pytest.mark.parametrize("case", [SMALL[0], SMALL[3], SMALL[5]], ids=["cfg1", "hybrid", "edges"])
def test_partial_blocks_and_merge(cuda, case):
    """Ring-style: the forward over B key blocks gives partial (O, LSE) equal to
    the oracle's per block, and the merge kernel recombines them."""
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    s.gather(kd, vd)
    B = 4
    bounds = np.linspace(0, s.T, B + 1).astype(int)
    bounds[1] = max(1, bounds[1] - 37)  # ragged blocks
    o_parts = torch.empty(B, s.T, hq, d, dtype=torch.float32, device=s.device)
    l_parts = torch.empty(B, hq, s.T, dtype=torch.float32, device=s.device)
    for b in range(B):
        s.forward(qd, kd, vd, out=o_parts[b], lse=l_parts[b], kv_block=(int(bounds[b]), int(bounds[b + 1])),
                  out_dtype=torch.float32)
    out = torch.empty(s.T, hq, d, dtype=torch.bfloat16, device=s.device)
    lse = torch.empty(hq, s.T, dtype=torch.float32, device=s.device)
    from context_document_masked_gb300 import fcp
    fcp.merge(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
    for b in range(B):
        o_b, l_b = A.attention_per_doc(q, k, v, cu, key_range=(int(bounds[b]), int(bounds[b + 1])))
        assert _maxabs(o_parts[b].cpu(), o_b, "O(fp32 part)") <= TOL_O
        lp = l_parts[b].cpu().numpy()
        assert np.array_equal(np.isneginf(lp), np.isneginf(l_b))
        fin = np.isfinite(l_b)
        assert np.max(np.abs(lp[fin] - l_b[fin])) <= TOL_LSE
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    assert _bf16_excess(out, o_ref) <= TOL_O
    assert _maxabs(lse.cpu(), lse_ref, "LSE") <= TOL_LSE


MERGE_CASES = [(1, 128), (2, 128), (3, 128), (4, 128), (5, 128), (8, 128), (13, 128), (32, 128),
               (1, 64), (2, 64), (4, 64), (7, 64), (16, 64)]


@pytest.mark.parametrize("B,d", MERGE_CASES, ids=[f"B{b}-d{d}" for b, d in MERGE_CASES])
def test_merge_kernel_against_oracle(cuda, B, d):
    """Every part count the kernel specialises on (B rounded up to a power of
    two, up to d/4), with a row count that leaves a ragged last row group."""
    from context_document_masked_gb300 import fcp
    g = torch.Generator().manual_seed(3 + B)
    rows, hq = 777, 4
    o_parts = torch.randn(B, rows, hq, d, generator=g)
    l_parts = torch.randn(B, hq, rows, generator=g) * 3
    mask = torch.rand(B, hq, rows, generator=g) < 0.3
    l_parts[mask] = float("-inf")
    o_parts[mask.permute(0, 2, 1)] = 0.0
    l_parts[:, :, 5] = float("-inf")       # a row empty in every block
    o_parts[:, 5] = 0.0
    out = torch.empty(rows, hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(hq, rows, dtype=torch.float32, device="cuda")
    fcp.merge(o_parts.cuda(), l_parts.cuda(), out, lse)
    torch.cuda.synchronize()
    o_ref, l_ref = A.merge(o_parts.numpy(), l_parts.numpy())
    assert _bf16_excess(out, o_ref) <= TOL_O
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.max(np.abs(lg[fin] - l_ref[fin])) <= TOL_LSE


def _merge_patterns(B, rows, hq, g):
    """Emptiness patterns of B parts x rows (True = part has no visible key)."""
    r = torch.arange(rows)
    causal = torch.stack([r < b * rows // B for b in range(B)])           # contiguous key blocks
    one = torch.ones(B, rows, dtype=torch.bool)                          # a single non-empty part per row
    pick = torch.randint(0, B, (rows,), generator=g)
    one[pick, r] = False
    ends = torch.ones(B, rows, dtype=torch.bool)                         # first part (even rows) or last (odd)
    ends[0, r % 2 == 0] = False
    ends[B - 1, r % 2 == 1] = False
    return {"causal": causal, "one": one, "ends": ends}


@pytest.mark.parametrize("d,B", [(128, 5), (128, 8), (128, 13), (128, 16), (128, 32), (64, 8), (64, 11), (64, 16)])
def test_merge_kernel_empty_part_patterns(cuda, d, B):
    """Structured emptiness: whole groups of four parts empty for a row (or
    for every row of a pass), the case the kernel skips without touching the
    parts, beside rows where any single part is the only non-empty one."""
    from context_document_masked_gb300 import fcp
    g = torch.Generator().manual_seed(100 + B + d)
    rows, hq = 389, 3
    for name, empty in _merge_patterns(B, rows, hq, g).items():
        o_parts = torch.randn(B, rows, hq, d, generator=g)
        l_parts = torch.randn(B, hq, rows, generator=g) * 3
        m = empty[:, None, :].expand(B, hq, rows)
        l_parts[m] = float("-inf")
        o_parts[m.permute(0, 2, 1)] = 0.0
        out = torch.empty(rows, hq, d, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(hq, rows, dtype=torch.float32, device="cuda")
        fcp.merge(o_parts.cuda(), l_parts.cuda(), out, lse)
        torch.cuda.synchronize()
        o_ref, l_ref = A.merge(o_parts.numpy(), l_parts.numpy())
        assert _bf16_excess(out, o_ref) <= TOL_O, name
        lg = lse.cpu().numpy()
        assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref)), name
        fin = np.isfinite(l_ref)
        assert np.max(np.abs(lg[fin] - l_ref[fin])) <= TOL_LSE, name


BWD = [SMALL[0], SMALL[1], SMALL[3], SMALL[5], SMALL[6], SMALL[8], SMALL[9]]


@pytest.mark.parametrize("case", BWD, ids=[c[0] for c in BWD])
def test_backward_all_shards(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    do = synth.make_dout(s.T, hq, d, seed=1)
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd, out_dtype=torch.float32)
    dq, dk, dv = s.backward(qd, kd, vd, out, lse, do.to(s.device))
    torch.cuda.synchronize()
    assert s.device_status() == 0
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    dq_ref, dk_ref, dv_ref = A.attention_bwd_per_doc(q, k, v, o_ref, lse_ref, do, cu)
    assert _maxabs(dv.cpu(), dv_ref, "dV") <= TOL_GRAD
    assert _maxabs(dk.cpu(), dk_ref, "dK") <= TOL_GRAD
    assert _maxabs(dq.cpu(), dq_ref, "dQ") <= TOL_GRAD


@pytest.mark.parametrize("case", [SMALL[1], SMALL[3]], ids=["perdoc", "hybrid"])
def test_backward_one_shard_at_a_time(cuda, case):
    """Summing every shard's dK/dV contributions (the simulated ReduceScatter)
    gives the global gradient; dQ rows come from their owner shard."""
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    do = synth.make_dout(s.T, hq, d, seed=2).to(s.device)
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd, out_dtype=torch.float32)
    dq = torch.full((s.T, hq, d), float("nan"), device=s.device)
    dk = torch.zeros(s.T, hkv, d, device=s.device)
    dv = torch.zeros(s.T, hkv, d, device=s.device)
    for j in range(cp):
        s.gather(kd, vd, shard=j)
        s.backward(qd, kd, vd, out, lse, do, shard=j, dq=dq, dk=dk, dv=dv, zero_kv_grads=False)
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    dq_ref, dk_ref, dv_ref = A.attention_bwd_per_doc(q, k, v, o_ref, lse_ref, do.cpu(), cu)
    assert _maxabs(dv.cpu(), dv_ref, "dV") <= TOL_GRAD
    assert _maxabs(dk.cpu(), dk_ref, "dK") <= TOL_GRAD
    assert _maxabs(dq.cpu(), dq_ref, "dQ") <= TOL_GRAD


def test_backward_from_bf16_output(cuda):
    """The backward may also be given the bf16-stored output. D_i = <dO_i, O_i>
    then carries O's storage rounding (up to 2^-9 |O| per element), which a
    dS term passes to dK and dQ: the bound here adds that term's worst case
    over this input, scale * max|q| * sum_d |dO_d| |O_d| 2^-9."""
    case = SMALL[1]
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    do = synth.make_dout(s.T, hq, d, seed=1)
    s.gather(kd, vd)
    out, lse = s.forward(qd, kd, vd)
    assert out.dtype == torch.bfloat16
    dq, dk, dv = s.backward(qd, kd, vd, out, lse, do.to(s.device))
    torch.cuda.synchronize()
    o_ref, lse_ref = A.attention_per_doc(q, k, v, cu)
    dq_ref, dk_ref, dv_ref = A.attention_bwd_per_doc(q, k, v, o_ref, lse_ref, do, cu)
    dD = np.max(np.sum(np.abs(A.to_f64(do)) * np.abs(o_ref), axis=-1)) * 2.0 ** -9
    extra = dD * np.max(np.abs(A.to_f64(q))) / np.sqrt(d)
    assert _maxabs(dv.cpu(), dv_ref, "dV") <= TOL_GRAD
    assert _maxabs(dk.cpu(), dk_ref, "dK(bf16 O)") <= TOL_GRAD + extra
    assert _maxabs(dq.cpu(), dq_ref, "dQ(bf16 O)") <= TOL_GRAD + extra


def test_timeout_path_reports_error_and_recovers(cuda):
    """A bounded wait that gives up at once sets the error word; the context
    stays usable and the next run is correct."""
    from context_document_masked_gb300 import fcp
    case = SMALL[1]
    s, cu, q, k, v, qd, kd, vd = _setup(*case)
    s.gather(kd, vd)
    fcp.debug_set_wait_limit(-1)
    try:
        s.forward(qd, kd, vd)
        torch.cuda.synchronize()
        st = s.device_status()
    finally:
        fcp.debug_set_wait_limit(0)
    assert st == fcp.ERR_TIMEOUT
    out, lse = s.forward(qd, kd, vd)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    o_ref, _ = A.attention_per_doc(q, k, v, cu)
    assert _bf16_excess(out, o_ref) <= TOL_O
