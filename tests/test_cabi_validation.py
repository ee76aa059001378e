"""Host-side fault injection at the C ABI, on CPU: corrupted device-plan
handles, shape and shard mismatches, and a lost or duplicated ring-step
partial at the merge. Every case must be rejected by the host checks with an
error status before anything is launched (no GPU is needed or touched: the
device pointers below are never dereferenced).

"LLM Context Parallel in Production", "Go-Live Checklist": a faulty or lost
rank is to be reported, not absorbed; here the equivalents are a plan handle
that no longer describes its plan and a missing partial result.
"""
import ctypes

import pytest

import synth

FAKE = ctypes.c_void_p(1 << 24)          # 16-byte aligned, never dereferenced


@pytest.fixture()
def bound(lib):
    D = synth.doc_lengths(2)
    p = lib.Plan(D, 4, "perdoc")
    dp = lib.DevPlan()
    assert lib.raw_call("fcp_plan_bind", p._ptr, FAKE, p.device_bytes(), ctypes.byref(dp)) == lib.OK
    return p, dp, lib.dims(sum(D), 8, 2, 128)


def _calls(lib, dp, dm):
    """Every entry point that takes a device plan, with otherwise valid arguments."""
    ws_bytes = 1 << 40
    steps = (ctypes.c_int32 * dp.n_shards)(*range(dp.n_shards))
    return {
        "fcp_gather_kv": lambda: lib.raw_call("fcp_gather_kv", FAKE, FAKE, ctypes.byref(dp), -1, dm.hkv, dm.d,
                                              FAKE, FAKE, None),
        "fcp_attn_fwd": lambda: lib.raw_call("fcp_attn_fwd", FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(dp), -1, 0,
                                             dm.T, dm, 0, FAKE, FAKE, FAKE, ws_bytes, None),
        "fcp_attn_fwd_qk8": lambda: lib.raw_call("fcp_attn_fwd_qk8", FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(dp),
                                                 -1, 0, dm.T, dm, 0, FAKE, FAKE, FAKE, ws_bytes, None),
        "fcp_attn_fwd_ring": lambda: lib.raw_call("fcp_attn_fwd_ring", FAKE, FAKE, FAKE, ctypes.byref(dp), -1, -1,
                                                  dm, 0, FAKE, FAKE, FAKE, ws_bytes, None),
        "fcp_attn_fwd_noalloc": lambda: lib.raw_call("fcp_attn_fwd_noalloc", FAKE, FAKE, FAKE, FAKE, FAKE,
                                                     ctypes.byref(dp), -1, 0, dm.T, dm, 0, FAKE, FAKE, None),
        "fcp_attn_bwd": lambda: lib.raw_call("fcp_attn_bwd", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE,
                                             ctypes.byref(dp), -1, dm, FAKE, FAKE, FAKE, FAKE, ws_bytes, None),
        "fcp_merge_ring": lambda: lib.raw_call("fcp_merge_ring", ctypes.byref(dp), FAKE, FAKE, steps, dp.n_shards,
                                               dm.hq, dm.d, FAKE, FAKE, None),
    }


CORRUPTIONS = {
    "table_offset": lambda dp: setattr_item(dp.tables, 1, dp.tables[1] + 4),
    "table_count": lambda dp: setattr_item(dp.counts, 2, dp.counts[2] + 1),
    "unused_slot": lambda dp: setattr_item(dp.counts, 15, 3),
    "shard_count": lambda dp: setattr(dp, "n_shards", dp.n_shards + 1),
    "tokens": lambda dp: setattr(dp, "T", dp.T - 128),
    "remote_rows": lambda dp: setattr(dp, "total_remote_rows", dp.total_remote_rows + 1),
    "bytes": lambda dp: setattr(dp, "bytes", dp.bytes - 256),
    "base_misaligned": lambda dp: setattr(dp, "base", (1 << 24) + 8),
    "no_host_plan": lambda dp: setattr(dp, "host", None),
}


def setattr_item(arr, i, v):
    arr[i] = v


@pytest.mark.parametrize("what", sorted(CORRUPTIONS))
def test_corrupted_plan_handle_is_rejected_before_launch(lib, bound, what):
    p, dp, dm = bound
    CORRUPTIONS[what](dp)
    for name, call in _calls(lib, dp, dm).items():
        assert call() == lib.ERR_INVALID_ARG, name


def test_shard_index_and_token_count_are_checked(lib, bound):
    p, dp, dm = bound
    for shard in (-2, dp.n_shards):
        assert lib.raw_call("fcp_attn_fwd", FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(dp), shard, 0, dm.T, dm, 0,
                            FAKE, FAKE, FAKE, 1 << 40, None) == lib.ERR_INVALID_ARG
        assert lib.raw_call("fcp_gather_kv", FAKE, FAKE, ctypes.byref(dp), shard, dm.hkv, dm.d, FAKE, FAKE,
                            None) == lib.ERR_INVALID_ARG
    other = lib.dims(dm.T + 8, dm.hq, dm.hkv, dm.d)          # dims of another sequence
    assert lib.raw_call("fcp_attn_bwd", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, ctypes.byref(dp), -1,
                        other, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == lib.ERR_INVALID_ARG
    # A key block outside the sequence.
    assert lib.raw_call("fcp_attn_fwd", FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(dp), -1, 0, dm.T + 1, dm, 0,
                        FAKE, FAKE, FAKE, 1 << 40, None) == lib.ERR_INVALID_ARG


@pytest.mark.parametrize("steps", [[0, 1, 3], [0, 1, 1, 3], [0, 1, 2, 4], [3, 2, 1, 0, 0], [], [-1, 0, 1, 2]],
                         ids=["lost", "duplicated", "outside_ring", "extra", "none", "negative"])
def test_merge_reports_a_missing_ring_partial(lib, bound, steps):
    """A ring-step partial that never arrived (a lost shard's message), arrived
    twice, or carries a tag outside the ring: the merge refuses before any
    launch with FCP_ERR_MISSING_PART."""
    p, dp, dm = bound
    arr = (ctypes.c_int32 * max(1, len(steps)))(*steps) if steps else None
    st = lib.raw_call("fcp_merge_ring", ctypes.byref(dp), FAKE, FAKE, arr, len(steps), dm.hq, dm.d, FAKE, FAKE,
                      None)
    assert st == lib.ERR_MISSING_PART
    assert lib.strerror(lib.ERR_MISSING_PART) == "partial result missing or duplicated"


def test_merge_ring_binding_checks_shapes(lib, bound):
    """The Python binding refuses partial tensors whose count or rows differ
    from the step list and the plan (the library would read past them)."""
    torch = pytest.importorskip("torch")
    p, dp, dm = bound
    dplan = lib.DevicePlan(dp, p, None)
    o = torch.zeros(3, dm.T, dm.hq, dm.d)
    lse = torch.zeros(3, dm.hq, dm.T)
    with pytest.raises(ValueError):
        lib.merge_ring(dplan, o, lse, [0, 1, 2, 3], o[0], lse[0])
    o2 = torch.zeros(4, dm.T - 8, dm.hq, dm.d)
    lse2 = torch.zeros(4, dm.hq, dm.T - 8)
    with pytest.raises(ValueError):
        lib.merge_ring(dplan, o2, lse2, [0, 1, 2, 3], o2[0], lse2[0])
