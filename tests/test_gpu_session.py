"""The session API used the way a training loop uses it: a session re-planned
for the next packed sequence (set_plan) and steps pipelined over two buffer
sets on three streams, ordered by events. Results must equal a fresh session
and a serial run: the forward bit for bit (each row's arithmetic does not
depend on scheduling), the gradients up to the order of their fp32
reduce-adds (dK/dV rows receive one reduce-add per key tile and query head;
dQ rows one per key tile)."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

T, HQ, HKV, D, CP = 4096, 8, 2, 128, 4
MIXES = ([3000, 40, 1, 55, 1000], [512, 2048, 1536], [4096], [1] * 96 + [4000])


def _inputs(seed, dev):
    q, k, v = synth.make_qkv(T, HQ, HKV, D, seed=seed, device=dev)
    do = synth.make_dout(T, HQ, D, seed=seed, device=dev)
    return q, k, v, do


def _step(s, q, k, v, do, stream=None):
    s.gather(k, v, stream=stream)
    o32 = torch.empty(T, HQ, D, dtype=torch.float32, device=q.device)
    lse = torch.empty(HQ, T, dtype=torch.float32, device=q.device)
    s.forward(q, k, v, out=o32, lse=lse, out_dtype=torch.float32, stream=stream)
    dq = torch.empty(T, HQ, D, dtype=torch.float32, device=q.device)
    dk = torch.zeros(T, HKV, D, dtype=torch.float32, device=q.device)
    dv = torch.zeros(T, HKV, D, dtype=torch.float32, device=q.device)
    s.backward(q, k, v, o32, lse, do, dq=dq, dk=dk, dv=dv, stream=stream)
    return o32, lse, dq, dk, dv


def _same(a, b, what):
    o, l, dq, dk, dv = a
    o2, l2, dq2, dk2, dv2 = b
    assert torch.equal(o, o2), what + ": O"
    assert torch.equal(l, l2), what + ": LSE"
    for x, y, n in ((dq, dq2, "dQ"), (dk, dk2, "dK"), (dv, dv2, "dV")):
        assert torch.allclose(x, y, rtol=1e-5, atol=1e-6), f"{what}: {n} {float((x - y).abs().max())}"


def test_set_plan_matches_a_fresh_session(cuda):
    from context_document_masked_gb300.session import CPAttention
    s = CPAttention(MIXES[0], CP, "hybrid", HQ, HKV, D, device=cuda)
    for i, mix in enumerate(MIXES):
        if i:
            s.set_plan(mix)
        fresh = CPAttention(mix, CP, "hybrid", HQ, HKV, D, device=cuda)
        q, k, v, do = _inputs(40 + i, cuda)
        a = _step(s, q, k, v, do)
        b = _step(fresh, q, k, v, do)
        torch.cuda.synchronize()
        assert s.device_status() == 0 and fresh.device_status() == 0
        _same(a, b, f"mix {i}")
    with pytest.raises(ValueError):
        s.set_plan([T - 1])


def test_pipelined_steps_match_serial_steps(cuda):
    """Step i's plan and inputs go up on one stream while step i-1 computes on
    another; its results come back on a third. Two sessions (buffer sets)
    alternate; each step uses its own document mix."""
    from context_document_masked_gb300.session import CPAttention
    n = len(MIXES)
    data = [_inputs(60 + i, cuda) for i in range(n)]
    serial = []
    for i, mix in enumerate(MIXES):
        s = CPAttention(mix, CP, "hybrid", HQ, HKV, D, device=cuda)
        serial.append([x.cpu() for x in _step(s, *data[i])])
    torch.cuda.synchronize()

    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sessions = [CPAttention(MIXES[0], CP, "hybrid", HQ, HKV, D, device=cuda) for _ in range(2)]
    torch.cuda.synchronize()  # their zeroed workspaces and first plans, written on the default stream
    ready = [torch.cuda.Event() for _ in range(n)]
    done = [torch.cuda.Event() for _ in range(n)]
    host = [None] * n
    for i in range(n):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done[i - 2])     # the step two back is done with this session
            sessions[b].set_plan(MIXES[i], stream=s_in)
            ins = [x.clone() for x in data[i]]   # this step's inputs, written on the input stream
            ready[i].record(s_in)
        for x in ins:
            x.record_stream(s_comp)              # read there after Python lets go of them
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ready[i])
            outs = _step(sessions[b], *ins, stream=s_comp)
            done[i].record(s_comp)
        for x in outs:
            x.record_stream(s_out)
        host[i] = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[i])
            for h, x in zip(host[i], outs):
                h.copy_(x, non_blocking=True)
    torch.cuda.synchronize()
    for s in sessions:
        assert s.device_status() == 0
    for i in range(n):
        _same(host[i], serial[i], f"step {i}")
