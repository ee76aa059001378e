"""The allocation-free forward entry point (fcp_attn_fwd_noalloc).

It serves callers that cannot allocate device memory when they call the
library (all device memory reserved up front, no allocation allowed on the
request path); its scratch is a fixed device array inside the library. This
file is collected last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def test_noalloc_forward_matches_workspace_forward(cuda, lib):
    """Both entry points run the same kernel on the same inputs, and every
    output row's arithmetic is independent of which CTA computes it, so the
    results agree bit for bit (two calls in a row share the scratch)."""
    from context_document_masked_gb300 import fcp
    from context_document_masked_gb300.session import CPAttention
    D = synth.random_doc_lengths(1536, seed=31)
    T, hq, hkv, d = sum(D), 8, 2, 128
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=31, device=cuda)
    s = CPAttention(D, 4, "perdoc", hq, hkv, d, device=cuda)
    s.gather(k, v)
    ref_out, ref_lse = s.forward(q, k, v)            # the workspace entry point
    torch.cuda.synchronize()
    for _ in range(2):                               # two calls in a row share the scratch
        out = torch.full((T, hq, d), float("nan"), dtype=torch.bfloat16, device=cuda)
        lse = torch.full((hq, T), float("nan"), dtype=torch.float32, device=cuda)
        fcp.attn_fwd_noalloc(q, k, v, s.kbuf, s.vbuf, s.dplan, -1, out, lse)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)


def test_noalloc_one_shard_at_a_time(cuda, lib):
    """Per-shard calls (the shard's own received rows at the head of the key
    buffer): each shard's rows equal the workspace forward's for that shard."""
    from context_document_masked_gb300 import fcp
    from context_document_masked_gb300.session import CPAttention
    D = synth.random_doc_lengths(2048, seed=32)
    T, hq, hkv, d, cp = sum(D), 4, 2, 128, 4
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=32, device=cuda)
    s = CPAttention(D, cp, "perdoc", hq, hkv, d, device=cuda)
    for j in range(cp):
        rows = torch.from_numpy(s.plan.query_indices(j).astype(np.int64)).to(cuda)
        s.gather(k, v, shard=j)
        ref_out, ref_lse = s.forward(q, k, v, shard=j, out_dtype=torch.float32)
        out = torch.full((T, hq, d), float("nan"), dtype=torch.float32, device=cuda)
        lse = torch.full((hq, T), float("nan"), dtype=torch.float32, device=cuda)
        fcp.attn_fwd_noalloc(q, k, v, s.kbuf, s.vbuf, s.dplan, j, out, lse)
        torch.cuda.synchronize()
        assert rows.numel() > 0
        assert torch.equal(out[rows], ref_out[rows])
        assert torch.equal(lse[:, rows], ref_lse[:, rows])


def test_noalloc_rejects_inputs_beyond_its_scratch(cuda, lib):
    from context_document_masked_gb300 import fcp
    from context_document_masked_gb300.session import CPAttention
    # V alone needs T * Hkv * d * 2 bytes: 262144 * 2 * 128 * 2 = 128 MiB > 64 MiB.
    T, hq, hkv, d = 262144, 4, 2, 128
    D = [T // 2, T // 2]
    s = CPAttention(D, 2, "wholedoc", hq, hkv, d, device=cuda)
    q = torch.zeros(T, hq, d, dtype=torch.bfloat16, device=cuda)
    kv = torch.zeros(T, hkv, d, dtype=torch.bfloat16, device=cuda)
    out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(hq, T, dtype=torch.float32, device=cuda)
    with pytest.raises(fcp.FcpError) as e:
        fcp.attn_fwd_noalloc(q, kv, kv, s.kbuf, s.vbuf, s.dplan, -1, out, lse)
    assert e.value.status == fcp.ERR_CAPACITY
