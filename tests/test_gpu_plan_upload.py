"""Both ways of putting a plan's work tables on the device -- the C call that
copies from the plan's own host memory, and the binding's copy staged through
pinned memory -- leave the same bytes, equal to the plan's device image."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg,pol", [(1, "llama3"), (2, "perdoc"), (4, "hybrid")])
def test_upload_paths_agree(cuda, cfg, pol):
    from context_document_masked_gb300 import fcp
    D = synth.doc_lengths(cfg)
    p = fcp.Plan(D, synth.WORKLOADS[cfg].cp, pol)
    n = p.device_bytes() // 4
    a = torch.full((n,), -7, dtype=torch.int32, device=cuda)
    b = torch.full((n,), -9, dtype=torch.int32, device=cuda)
    s = torch.cuda.Stream()
    dp = fcp.DevPlan()
    st = fcp.raw_call("fcp_plan_upload", p._ptr, ctypes.c_void_p(a.data_ptr()), n * 4,
                      ctypes.c_void_p(s.cuda_stream), ctypes.byref(dp))
    assert st == fcp.OK
    h = p.upload(b, stream=s)
    s.synchronize()
    img = p.device_image()
    assert np.array_equal(a.cpu().numpy(), img)
    assert np.array_equal(b.cpu().numpy(), img)
    assert h.c.bytes == dp.bytes and list(h.c.tables) == list(dp.tables) and list(h.c.counts) == list(dp.counts)
