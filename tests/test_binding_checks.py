"""The binding checks every tensor before its raw pointer reaches the
library (which sees neither dtypes, strides nor devices): tensors that are
not on the GPU are refused with ValueError before anything is called. The
dtype, shape, layout and buffer-size checks run on the GPU
(tests/test_gpu_binding_checks.py)."""
import ctypes

import pytest

import synth

torch = pytest.importorskip("torch")

FAKE = ctypes.c_void_p(1 << 24)


@pytest.fixture()
def dplan(lib):
    D = synth.doc_lengths(1)
    p = lib.Plan(D, 2, "hybrid")
    dp = lib.DevPlan()
    assert lib.raw_call("fcp_plan_bind", p._ptr, FAKE, p.device_bytes(), ctypes.byref(dp)) == lib.OK
    return lib.DevicePlan(dp, p, None), sum(D)


def _calls(lib, dp, T):
    hq, hkv, d = 4, 2, 64
    q = torch.zeros(T, hq, d, dtype=torch.bfloat16)
    k = torch.zeros(T, hkv, d, dtype=torch.bfloat16)
    kb = torch.zeros(max(1, dp.c.total_remote_rows), hkv, d, dtype=torch.bfloat16)
    out = torch.zeros(T, hq, d, dtype=torch.float32)
    lse = torch.zeros(hq, T, dtype=torch.float32)
    g = torch.zeros(T, hkv, d, dtype=torch.float32)
    ws = torch.zeros(1024, dtype=torch.int32)
    parts = torch.zeros(2, T, hq, d)
    lparts = torch.zeros(2, hq, T)
    ob = torch.zeros(T, hq, d, dtype=torch.bfloat16)
    return {
        "gather_kv": lambda: lib.gather_kv(k, k, dp, -1, kb, kb),
        "attn_fwd": lambda: lib.attn_fwd(q, k, k, kb, kb, dp, -1, out, lse, ws),
        "attn_fwd_qk8": lambda: lib.attn_fwd_qk8(q, k, k, kb, kb, dp, -1, out, lse, ws),
        "attn_fwd_ring": lambda: lib.attn_fwd_ring(q, k, k, dp, -1, -1, out, lse, ws),
        "attn_fwd_noalloc": lambda: lib.attn_fwd_noalloc(q, k, k, kb, kb, dp, -1, out, lse),
        "attn_bwd": lambda: lib.attn_bwd(q, k, k, kb, kb, out, lse, q, dp, -1, out, g, g, ws),
        "merge": lambda: lib.merge(parts, lparts, ob, lse),
        "round_bf16": lambda: lib.round_bf16(out, ob),
        "quant_e4m3": lambda: lib.quant_e4m3(q, torch.zeros(q.numel(), dtype=torch.uint8),
                                             torch.zeros(1), torch.zeros(1, dtype=torch.int32)),
        "device_status": lambda: lib.device_status(ws),
        "debug_rescale_events": lambda: lib.debug_rescale_events(ws),
    }


@pytest.mark.parametrize("name", ["gather_kv", "attn_fwd", "attn_fwd_qk8", "attn_fwd_ring", "attn_fwd_noalloc",
                                  "attn_bwd", "merge", "round_bf16", "quant_e4m3", "device_status",
                                  "debug_rescale_events"])
def test_host_tensors_are_refused(lib, dplan, name):
    dp, T = dplan
    with pytest.raises(ValueError, match="CUDA tensor"):
        _calls(lib, dp, T)[name]()
