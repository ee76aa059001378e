"""The binding's checks on GPU tensors: a wrong dtype, a wrong shape, a
non-contiguous view or received-key buffers shorter than the plan's
received rows are refused with ValueError before anything is launched (the
library would otherwise read or write past them), and a valid call after
them still gives the right result."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

T, HQ, HKV, D, CP = 2048, 4, 2, 128, 4
DOCS = [1500, 300, 248]


@pytest.fixture()
def setup(cuda):
    from context_document_masked_gb300.session import CPAttention
    s = CPAttention(DOCS, CP, "perdoc", HQ, HKV, D, device=cuda)
    q, k, v = synth.make_qkv(T, HQ, HKV, D, seed=5, device=cuda)
    do = synth.make_dout(T, HQ, D, seed=5, device=cuda)
    return s, q, k, v, do


def test_forward_argument_checks(setup):
    from context_document_masked_gb300 import fcp
    s, q, k, v, do = setup
    assert s.dplan.c.total_remote_rows > 0
    out = torch.empty(T, HQ, D, dtype=torch.float32, device="cuda")
    lse = torch.empty(HQ, T, dtype=torch.float32, device="cuda")
    bad = {
        "q fp32": dict(q=q.float()),
        "k shape": dict(k=k[:, :1].contiguous()),
        "q view": dict(q=q.transpose(0, 1).contiguous().transpose(0, 1)),
        "lse shape": dict(lse=torch.empty(T, HQ, device="cuda")),
        "out fp16": dict(out=torch.empty(T, HQ, D, dtype=torch.float16, device="cuda")),
        "kbuf short": dict(kbuf=s.kbuf[: s.dplan.c.total_remote_rows - 1].contiguous()),
        "vbuf dtype": dict(vbuf=s.vbuf.float()),
    }
    base = dict(q=q, k=k, v=v, kbuf=s.kbuf, vbuf=s.vbuf, out=out, lse=lse)
    for what, over in bad.items():
        a = {**base, **over}
        with pytest.raises(ValueError):
            fcp.attn_fwd(a["q"], a["k"], a["v"], a["kbuf"], a["vbuf"], s.dplan, -1, a["out"], a["lse"], s.ws)
        with pytest.raises(ValueError):
            fcp.attn_fwd_noalloc(a["q"], a["k"], a["v"], a["kbuf"], a["vbuf"], s.dplan, -1, a["out"], a["lse"])
    with pytest.raises(ValueError):
        fcp.gather_kv(k, v, s.dplan, -1, s.kbuf[:1].contiguous(), s.vbuf[:1].contiguous())
    # A valid call afterwards: the same as the session's.
    s.gather(k, v)
    o1, l1 = s.forward(q, k, v, out_dtype=torch.float32)
    fcp.attn_fwd(q, k, v, s.kbuf, s.vbuf, s.dplan, -1, out, lse, s.ws)
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(lse, l1)
    assert s.device_status() == 0


def test_backward_and_merge_argument_checks(setup):
    from context_document_masked_gb300 import fcp
    s, q, k, v, do = setup
    s.gather(k, v)
    o, lse = s.forward(q, k, v, out_dtype=torch.float32)
    dq = torch.empty(T, HQ, D, dtype=torch.float32, device="cuda")
    dk = torch.zeros(T, HKV, D, dtype=torch.float32, device="cuda")
    dv = torch.zeros(T, HKV, D, dtype=torch.float32, device="cuda")
    args = [q, k, v, s.kbuf, s.vbuf, o, lse, do, s.dplan, -1, dq, dk, dv, s.ws]
    for i, bad in ((7, do.float()), (10, dq.to(torch.bfloat16)), (11, dk[:, :1].contiguous()),
                   (12, torch.zeros(T, HKV, D, dtype=torch.float32))):   # dv on the host
        a = list(args)
        a[i] = bad
        with pytest.raises(ValueError):
            fcp.attn_bwd(*a)
    parts = torch.zeros(2, T, HQ, D, device="cuda")
    lparts = torch.full((2, HQ, T), float("-inf"), device="cuda")
    mo = torch.empty(T, HQ, D, dtype=torch.bfloat16, device="cuda")
    ml = torch.empty(HQ, T, device="cuda")
    for a in ((parts, lparts[:, :, :-1].contiguous(), mo, ml), (parts, lparts, mo.float(), ml),
              (parts.to(torch.bfloat16), lparts, mo, ml)):
        with pytest.raises(ValueError):
            fcp.merge(*a)
    with pytest.raises(ValueError):
        fcp.round_bf16(o, torch.empty(T, HQ, D - 8, dtype=torch.bfloat16, device="cuda"))
    fcp.attn_bwd(*args)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    dq2, dk2, dv2 = s.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert torch.allclose(dq, dq2, rtol=1e-5, atol=1e-6)
    assert torch.allclose(dk, dk2, rtol=1e-5, atol=1e-6) and torch.allclose(dv, dv2, rtol=1e-5, atol=1e-6)


def test_one_shard_buffers_sized_for_that_shard(setup):
    """For one shard the received-key buffers need only that shard's received
    rows (its row 0 is the shard's first); one row fewer is refused."""
    from context_document_masked_gb300 import fcp
    s, q, k, v, do = setup
    s.gather(k, v)
    o_all, l_all = s.forward(q, k, v, out_dtype=torch.float32)
    for j in range(CP):
        rows = s.dplan.remote_rows(j)
        kb = torch.empty(max(1, rows), HKV, D, dtype=torch.bfloat16, device="cuda")
        vb = torch.empty_like(kb)
        fcp.gather_kv(k, v, s.dplan, j, kb, vb)
        out = torch.zeros(T, HQ, D, dtype=torch.float32, device="cuda")
        lse = torch.full((HQ, T), float("nan"), device="cuda")
        fcp.attn_fwd(q, k, v, kb, vb, s.dplan, j, out, lse, s.ws)
        torch.cuda.synchronize()
        for _, a, b in s.plan.shard(j)["pieces"]:
            assert torch.equal(out[a:b], o_all[a:b]) and torch.equal(lse[:, a:b], l_all[:, a:b])
        if rows > 1:
            with pytest.raises(ValueError):
                fcp.attn_fwd(q, k, v, kb[:-1].contiguous(), vb[:-1].contiguous(), s.dplan, j, out, lse, s.ws)
    assert s.device_status() == 0
