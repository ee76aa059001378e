"""One packed sequence, one CP plan, all shards on one GPU.

Holds the device copies of a plan's work tables and the buffers the C-ABI
calls need (received-key buffers, workspace), allocated once through PyTorch.
Every step of the path runs in libfcp; this class only orders the calls.
"""
from __future__ import annotations

import torch

from . import fcp


class CPAttention:
    def __init__(self, doclens, cp: int, policy: str, hq: int, hkv: int, d: int,
                 device="cuda", target_imbalance: float = 1.05, scale: float = 0.0):
        self.device = torch.device(device)
        self.plan = fcp.Plan(doclens, cp, policy, target_imbalance)
        self.T = int(sum(int(x) for x in doclens))
        self.hq, self.hkv, self.d, self.cp = hq, hkv, d, cp
        self.scale = scale
        nbytes = self.plan.device_bytes()
        self.plan_buf = torch.empty(nbytes // 4, dtype=torch.int32, device=self.device)
        self.dplan = self.plan.upload(self.plan_buf)
        rows = max(1, self.dplan.total_remote_rows)
        self.kbuf = torch.empty(rows, hkv, d, dtype=torch.bfloat16, device=self.device)
        self.vbuf = torch.empty_like(self.kbuf)
        self.dims = fcp.dims(self.T, hq, hkv, d, scale)
        ws_bytes = fcp.workspace_bytes(self.dims, self.plan)
        self.ws = torch.zeros(ws_bytes // 4, dtype=torch.int32, device=self.device)

    def set_plan(self, doclens, target_imbalance: float = 1.05, stream=None):
        """A new plan for the next packed sequence (same T, CP size, policy and
        shapes), uploaded into this session's plan buffer on `stream`; the
        received-key buffers and the workspace are kept when they are large
        enough and replaced otherwise. The previous plan's tables must no longer
        be in use by queued work on other streams."""
        if int(sum(int(x) for x in doclens)) != self.T:
            raise ValueError("set_plan: the token count differs from the session's")
        plan = fcp.Plan(doclens, self.cp, self.plan.policy, target_imbalance)
        nbytes = plan.device_bytes()
        if self.plan_buf.numel() * 4 < nbytes:
            self.plan_buf = torch.empty(nbytes // 4, dtype=torch.int32, device=self.device)
        self.plan = plan
        self.dplan = plan.upload(self.plan_buf, stream=stream)
        rows = max(1, self.dplan.total_remote_rows)
        if self.kbuf.shape[0] < rows:
            self.kbuf = torch.empty(rows, self.hkv, self.d, dtype=torch.bfloat16, device=self.device)
            self.vbuf = torch.empty_like(self.kbuf)
        ws_bytes = fcp.workspace_bytes(self.dims, plan)
        if self.ws.numel() * 4 < ws_bytes:
            self.ws = torch.zeros(ws_bytes // 4, dtype=torch.int32, device=self.device)
        return self.dplan

    def stats(self) -> dict:
        return self.plan.stats()

    def gather(self, k, v, shard: int = -1, stream=None):
        fcp.gather_kv(k, v, self.dplan, shard, self.kbuf, self.vbuf, stream)

    def forward(self, q, k, v, shard: int = -1, out=None, lse=None, kv_block=None,
                out_dtype=torch.bfloat16, stream=None):
        if out is None:
            out = torch.empty(self.T, self.hq, self.d, dtype=out_dtype, device=self.device)
        if lse is None:
            lse = torch.empty(self.hq, self.T, dtype=torch.float32, device=self.device)
        lo, hi = (0, self.T) if kv_block is None else kv_block
        fcp.attn_fwd(q, k, v, self.kbuf, self.vbuf, self.dplan, shard, out, lse, self.ws,
                     kv_lo=lo, kv_hi=hi, scale=self.scale, stream=stream)
        return out, lse

    def forward_qk8(self, q, k, v, shard: int = -1, out=None, lse=None, kv_block=None,
                    out_dtype=torch.bfloat16, stream=None):
        """forward() with Q K^T on e4m3 copies of Q and K (d = 128)."""
        if out is None:
            out = torch.empty(self.T, self.hq, self.d, dtype=out_dtype, device=self.device)
        if lse is None:
            lse = torch.empty(self.hq, self.T, dtype=torch.float32, device=self.device)
        lo, hi = (0, self.T) if kv_block is None else kv_block
        fcp.attn_fwd_qk8(q, k, v, self.kbuf, self.vbuf, self.dplan, shard, out, lse, self.ws,
                         kv_lo=lo, kv_hi=hi, scale=self.scale, stream=stream)
        return out, lse

    def forward_ring(self, q, k, v, ring_step: int = -1, shard: int = -1, out=None, lse=None,
                     out_dtype=torch.bfloat16, stream=None):
        """Forward in ring order without the gathered buffer: ring_step -1 visits
        every owner's keys in one pass, s >= 0 gives ring step s's partial."""
        if out is None:
            out = torch.empty(self.T, self.hq, self.d, dtype=out_dtype, device=self.device)
        if lse is None:
            lse = torch.empty(self.hq, self.T, dtype=torch.float32, device=self.device)
        fcp.attn_fwd_ring(q, k, v, self.dplan, shard, ring_step, out, lse, self.ws, scale=self.scale,
                          stream=stream)
        return out, lse

    def backward(self, q, k, v, out, lse, dout, shard: int = -1, dq=None, dk=None, dv=None,
                 zero_kv_grads: bool = True, stream=None):
        if dq is None:
            dq = torch.empty(self.T, self.hq, self.d, dtype=torch.float32, device=self.device)
        if dk is None:
            dk = torch.zeros(self.T, self.hkv, self.d, dtype=torch.float32, device=self.device)
        elif zero_kv_grads:
            dk.zero_()
        if dv is None:
            dv = torch.zeros(self.T, self.hkv, self.d, dtype=torch.float32, device=self.device)
        elif zero_kv_grads:
            dv.zero_()
        fcp.attn_bwd(q, k, v, self.kbuf, self.vbuf, out, lse, dout, self.dplan, shard, dq, dk, dv,
                     self.ws, scale=self.scale, stream=stream)
        return dq, dk, dv

    def device_status(self) -> int:
        return fcp.device_status(self.ws)
