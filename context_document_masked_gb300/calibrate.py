"""Per-shard kernel time against the plan's workload measures.

FlashCP motivates its sharding choices with attention-kernel efficiency
falling on short shards (§2.2, "Reduced Kernel Efficiency", Fig. 3), while
Algorithm 1 balances W, the useful (q, k) pairs of a worker (§3.1, §3.4).
The kernels here visit 128 x 128 tiles, so a shard's time follows the tiles
it touches rather than its useful pairs: a short document leaves most of
each diagonal tile masked. This module times each shard's forward and
backward on its own (one shard per launch, every SM working on that shard)
and fits the times against W and against the visited tiles:
    time ~ a * pairs            (the workload model of Algorithm 1)
    time ~ a * tiles + b * q    (tiles visited, plus a cost per query tile)
"""
from __future__ import annotations

import numpy as np
import torch

from .session import CPAttention


def shard_times(doclens, cp: int, policy: str, q, k, v, dout, reps: int = 5,
                target_imbalance: float = 1.05) -> list:
    """Forward and backward time of every shard alone (ms, CUDA events), with
    the shard's W and tile counts. q, k, v, dout: device tensors of the packed
    sequence."""
    T, hq, d = q.shape
    hkv = k.shape[1]
    s = CPAttention(doclens, cp, policy, hq, hkv, d, device=q.device, target_imbalance=target_imbalance)
    out = torch.empty(T, hq, d, dtype=torch.float32, device=q.device)
    lse = torch.empty(hq, T, dtype=torch.float32, device=q.device)
    dq = torch.empty(T, hq, d, dtype=torch.float32, device=q.device)
    dk = torch.zeros(T, hkv, d, dtype=torch.float32, device=q.device)
    dv = torch.zeros_like(dk)
    rows = []
    for j in range(cp):
        sh = s.plan.shard(j)
        s.gather(k, v, shard=j)
        fwd = lambda: s.forward(q, k, v, shard=j, out=out, lse=lse, out_dtype=torch.float32)  # noqa: E731
        bwd = lambda: s.backward(q, k, v, out, lse, dout, shard=j, dq=dq, dk=dk, dv=dv,  # noqa: E731
                                 zero_kv_grads=False)
        ms = {}
        for name, fn in (("fwd", fwd), ("bwd", bwd)):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms[name] = e0.elapsed_time(e1) / reps
        # Work over all heads: pairs and tiles are per query head, backward
        # key tiles per KV head.
        rows.append({"shard": j, "tokens": sh["tokens"], "pairs": sh["useful_pairs"] * hq,
                     "fwd_tiles": sh["fwd_tiles"] * hq, "fwd_qtiles": sh["fwd_qtiles"] * hq,
                     "fwd_masked": sh["fwd_masked"] * hq, "bwd_tiles": sh["bwd_tiles"] * hq,
                     "bwd_ktiles": sh["bwd_ktiles"] * hkv, "fwd_ms": ms["fwd"], "bwd_ms": ms["bwd"]})
    if s.device_status() != 0:
        raise RuntimeError("device status reports a failed wait while timing shards")
    return rows


def fit(rows: list, xkeys: tuple, ykey: str, intercept: bool = True) -> dict:
    """Least squares ykey ~ c0 + sum_i c_i * xkeys[i] (c0 only with
    `intercept`: a fixed cost per launch); coefficients, R^2 and the largest
    relative error of the fit over the rows."""
    x = np.array([[float(r[key]) for key in xkeys] for r in rows])
    if intercept:
        x = np.hstack([x, np.ones((len(rows), 1))])
        xkeys = tuple(xkeys) + ("launch",)
    y = np.array([float(r[ykey]) for r in rows])
    c, *_ = np.linalg.lstsq(x, y, rcond=None)
    pred = x @ c
    ss_res = float(((y - pred) ** 2).sum())
    ss_tot = float(((y - y.mean()) ** 2).sum())
    return {"coef": {key: float(v) for key, v in zip(xkeys, c)},
            "r2": 1.0 - ss_res / ss_tot if ss_tot > 0 else 1.0,
            "max_rel_err": float(np.max(np.abs(pred - y) / y))}


def imbalance(values) -> float:
    """max / mean over shards."""
    v = np.asarray(values, dtype=np.float64)
    return float(v.max() / v.mean())
