"""Benchmark of the document-masked CP attention hot path on one GB300.

One step = one pass of the whole path over one packed sequence with every CP
shard in one launch: KV gather of the received prefix keys, forward, backward
(preprocess + main kernel). The headline workload (default `--workload 5`) is
the 512K packed sequence: lognormal(9, 1.8) document lengths clipped to
[256, 262144], 32 query / 8 KV heads, d = 128, CP = 32 shards under the
hybrid plan (Algorithm 1), synthetic and seeded. Every step's inputs exceed the
129 MB L2 (Q, K, V, dO: 10.7 GB at 512K), so no explicit flush is done between
steps.

The same run also measures, as extra keys of the one JSON line: the merge of
partial (O, LSE) over key blocks and the ring-order forwards on the headline
workload; the other packed workloads (2K d = 64, 32K Per-Doc, 128K with one
64K document, 64K short documents under every policy) at their own shapes; the
per-shard timing against the plan's cost measures; the end-to-end figure
through the public API with host buffers; and the fp64 CPU oracle on a bounded
sample.

Prints one JSON line. `--impl reference` times the fp64 CPU oracle instead, on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

CFG = 5
METRIC = "doc-masked attn useful TFLOPS fwd+bwd (% of GB300 BF16 peak); merge GB/s"
UNIT = "TFLOP/s"

# tcgen05 rate measured on this part: one 128x128x128 fp16/bf16 MMA (2^22
# FLOPs) every 512 SM cycles, i.e. 8192 FLOP per cycle per SM.
MMA_FLOP_PER_CLK_SM = 8192

# DRAM bytes of one backward call (preprocess + main kernel) per workload, from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum of both
# kernels; summarised under profiles/). Valid only for the code it was taken
# on: the backward's kernels and helpers, the parts of the launch code and
# parameters that set the backward up, and the plan's work tables. Reported as
# null once any of them changes.
BWD_TRAFFIC_SOURCES = [
    ("context_document_masked_gb300/csrc/attn_bwd.cu", None, None),
    ("context_document_masked_gb300/csrc/copy_kernels.cu", None, None),
    ("context_document_masked_gb300/csrc/sm103.cuh", None, None),
    ("context_document_masked_gb300/csrc/kernels.h", "struct BwdParams", "int launch_attn_fwd"),
    ("context_document_masked_gb300/csrc/api.cu", "int fcp_attn_bwd(", "int fcp_get_device_status("),
    ("context_document_masked_gb300/csrc/tables.cpp", None, None),
]
BWD_TRAFFIC = {   # workload -> {"sha256": ..., "bytes": ...}
    5: {"sha256": "47684d10ec18d7e05001afc1a3f0340eb85072d6a0f94c694dbc61e20f14d638",
        "bytes": (17.46 + 17.42 + 239.75 + 144.04) * 1e9},   # preprocess + main kernel
}


def _bwd_sources_hash():
    import hashlib
    h = hashlib.sha256()
    for f, a, b in BWD_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f)) as fh:
            text = fh.read()
        if a is not None:
            text = text[text.index(a):text.index(b)]
        h.update(text.encode())
    return h.hexdigest()


def _bwd_traffic(cfg):
    try:
        t = BWD_TRAFFIC.get(cfg)
        return t["bytes"] if t and _bwd_sources_hash() == t["sha256"] else None
    except (OSError, ValueError):
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16": m["bf16_tflops"], "bf16_sustained": m["bf16_tflops_sustained"],
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def _workload(cfg=None):
    cfg = CFG if cfg is None else cfg
    w = synth.WORKLOADS[cfg]
    D = synth.doc_lengths(cfg)
    pairs = sum(L * (L + 1) // 2 for L in D)
    return w, D, pairs


def _input_gb(w):
    return (2 * w.T * w.Hq * w.d + 2 * w.T * w.Hkv * w.d) * 2 / 1e9


def _config(w, D, extra=None):
    c = {"workload": w.name, "tokens": w.T, "docs": len(D), "max_doc": max(D), "hq": w.Hq, "hkv": w.Hkv,
         "d": w.d, "cp": w.cp, "policy": w.policy, "shards_per_launch": "all",
         "l2": f"inputs > L2 (Q,K,V,dO {_input_gb(w):.2f} GB), no flush"}
    if extra:
        c.update(extra)
    return c


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 50 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.samples = []
        self._p = None
        self._t = None

    def _read(self):
        for line in self._p.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.samples.append(parts)

    def __enter__(self):
        try:
            self._p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                        "--format=csv,noheader,nounits", "-lms", "50"],
                                       stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)   # first sample before the timed region starts
        except OSError:
            self._p = None
        return self

    def __exit__(self, *a):
        if self._p is not None:
            time.sleep(0.1)
            self._p.terminate()
            try:
                self._p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._p.kill()
            self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(s[0]) for s in self.samples) if v is not None]
        mx = [v for v in (num(s[1]) for s in self.samples) if v is not None]
        pw = [v for v in (num(s[2]) for s in self.samples) if v is not None]
        reasons = sorted({self.NAMES[i] for s in self.samples for i in range(4) if s[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(self.samples)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time: every rank contributes its own and all get the max."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_tflops(world: int, flops_per_replica: float, ms_step: float) -> float:
    """Whole-job throughput: every rank runs one replica of the workload per
    step (weak scaling), timed by the slowest rank."""
    return world * flops_per_replica / (ms_step * 1e-3) / 1e12


def _replica_seed(rank: int) -> int:
    return 1000 + CFG + rank


def _tf(flops, ms):
    return flops / (ms * 1e-3) / 1e12


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class Step:
    """One packed sequence on the device with its session and result buffers:
    run() = gather -> forward (fp32 output) -> backward, every shard per launch."""

    def __init__(self, torch, cfg, policy, seed, dev):
        from context_document_masked_gb300.session import CPAttention
        w, D, pairs = _workload(cfg)
        self.w, self.D, self.pairs = w, D, pairs
        T, hq, hkv, d = w.T, w.Hq, w.Hkv, w.d
        self.q, self.k, self.v = synth.make_qkv(T, hq, hkv, d, seed=seed, device=dev)
        self.do = synth.make_dout(T, hq, d, seed=seed, device=dev)
        self.s = CPAttention(D, w.cp, policy or w.policy, hq, hkv, d, device=dev)
        self.out = torch.empty(T, hq, d, dtype=torch.float32, device=dev)
        self.lse = torch.empty(hq, T, dtype=torch.float32, device=dev)
        self.dq = torch.empty(T, hq, d, dtype=torch.float32, device=dev)
        self.dk = torch.empty(T, hkv, d, dtype=torch.float32, device=dev)
        self.dv = torch.empty_like(self.dk)
        self.fwd_flops = 4.0 * d * hq * pairs
        self.bwd_flops = 10.0 * d * hq * pairs

    def run(self, ev=None, i=None, stream=None, backward=True):
        s = self.s
        if ev is not None:
            ev["gather"][i].record(stream)
        s.gather(self.k, self.v)
        if ev is not None:
            ev["fwd"][i].record(stream)
        s.forward(self.q, self.k, self.v, out=self.out, lse=self.lse)
        if ev is not None:
            ev["bwd"][i].record(stream)
        if backward:
            s.backward(self.q, self.k, self.v, self.out, self.lse, self.do, dq=self.dq, dk=self.dk, dv=self.dv)
        if ev is not None:
            ev["end"][i].record(stream)

    def timed(self, torch, steps, warmup, backward=True, clock=None, dist=None, world=1):
        """Total ms of `steps` steps (CUDA events on the launching stream, a
        synchronize and, with several ranks, a barrier on both sides) and the
        mean per-kernel ms; `clock` samples the timed region only."""
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.run(backward=backward)
        torch.cuda.synchronize()
        if self.s.device_status() != 0:
            raise RuntimeError("device status reports an error after warm-up")
        ev = {n: [torch.cuda.Event(enable_timing=True) for _ in range(steps)] for n in ("gather", "fwd", "bwd", "end")}
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with (clock if clock is not None else _Null()):
            t0.record(stream)
            for i in range(steps):
                self.run(ev, i, stream, backward=backward)
            t1.record(stream)
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        if self.s.device_status() != 0:
            raise RuntimeError("device status reports an error in the timed steps")
        ms_total = t0.elapsed_time(t1)
        per = {n: statistics.mean(ev[a][i].elapsed_time(ev[b][i]) for i in range(steps))
               for n, a, b in (("gather", "gather", "fwd"), ("fwd", "fwd", "bwd"), ("bwd", "bwd", "end"))}
        return ms_total, per

    def free(self):
        for n in ("q", "k", "v", "do", "s", "out", "lse", "dq", "dk", "dv"):
            setattr(self, n, None)


def _summary(st, per, pk, backward=True):
    r = {"kernels_ms": {k_: round(v_, 4) for k_, v_ in per.items() if backward or k_ != "bwd"},
         "fwd": {"tflops": round(_tf(st.fwd_flops, per["fwd"]), 2),
                 "frac": round(_tf(st.fwd_flops, per["fwd"]) / pk["bf16"], 4)}}
    if backward:
        r["bwd"] = {"tflops": round(_tf(st.bwd_flops, per["bwd"]), 2),
                    "frac": round(_tf(st.bwd_flops, per["bwd"]) / pk["bf16"], 4)}
        step_ms = per["gather"] + per["fwd"] + per["bwd"]
        r["step"] = {"ms": round(step_ms, 4), "tflops": round(_tf(st.fwd_flops + st.bwd_flops, step_ms), 2),
                     "frac": round(_tf(st.fwd_flops + st.bwd_flops, step_ms) / pk["bf16"], 4)}
    return r


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from context_document_masked_gb300 import fcp

    world, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")
    pk = _peaks()
    st = Step(torch, CFG, None, _replica_seed(rank), dev)   # independent replica per rank
    w, D, pairs = st.w, st.D, st.pairs
    T, hq, hkv, d = w.T, w.Hq, w.Hkv, w.d
    clk = ClockSampler(local)
    ms_total, per = st.timed(torch, args.steps, args.warmup, clock=clk, dist=dist, world=world)
    if world > 1:
        ms_total = _max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = _job_tflops(world, st.fwd_flops + st.bwd_flops, ms_step)
    clocks = clk.summary()
    stats = st.s.stats()
    remote_rows = stats["remote_rows_total"]
    gather_bytes = 2 * 2 * remote_rows * hkv * d * 2

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    legs = set(args.legs.split(","))
    merge = _bench_merge(st, torch, fcp, pk) if "merge" in legs else None
    ring = _bench_ring(st, torch, fcp) if "ring" in legs else None
    fwd_flops, bwd_flops = st.fwd_flops, st.bwd_flops
    st.free()
    torch.cuda.empty_cache()
    configs = _bench_configs(torch, fcp, pk, dev) if "configs" in legs else None
    torch.cuda.empty_cache()
    shards = _bench_shards(torch, dev) if "shards" in legs else None
    torch.cuda.empty_cache()
    # End to end through the public API: pinned host inputs -> device, plan,
    # gather, forward, backward, results back to pinned host buffers.
    e2e = _bench_e2e(args, D, w, _replica_seed(rank), torch, fcp) if "e2e" in legs else None
    torch.cuda.empty_cache()

    policies = {}
    for pol in ("llama3", "perdoc", "wholedoc", "hybrid", "hybrid_tiles"):
        try:
            plan = fcp.Plan(D, w.cp, pol)
            ps = plan.stats()
            policies[pol] = {"imbalance": round(ps["imbalance"], 4), "remote_rows": ps["remote_rows_total"],
                             "eq4_tokens": ps["eq4_tokens"], "eq5_tokens": ps["eq5_tokens"],
                             "fwd_tiles": _tile_counts(plan, w.cp)}
        except fcp.FcpError as e:
            policies[pol] = {"error": str(e)}
    cpu = _cpu_baseline(args.cpu_seconds) if "cpu" in legs else None
    peak = pk["bf16"]
    bwd_ach = _tf(bwd_flops, per["bwd"])
    fwd_ach = _tf(fwd_flops, per["fwd"])
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz")
    at_clock = MMA_FLOP_PER_CLK_SM * n_sm * mhz * 1e6 / 1e12 if mhz else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, f16/bf16 MMA, f32 accumulate", "data": "synthetic",
        "config": _config(w, D, {"parallelism": f"replicas{world}" if world > 1 else "single"}),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "kernel": "fcp_attn_bwd (preprocess + main)", "achieved": round(bwd_ach, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(bwd_ach / peak, 4),
                     "peak_note": f"{pk['source']} bf16 dense burst (cuBLAS); fp16 MMA has the same nominal rate",
                     "frac_of_sustained": round(bwd_ach / pk["bf16_sustained"], 4),
                     "traffic": _bwd_traffic(CFG), "traffic_unit": "bytes per call (DRAM read + write, ncu)",
                     "algorithmic": "10*d*Hq*P flops per call, P = useful (q, k) pairs per head"},
        "mma_rate": {"flop_per_clk_per_sm": MMA_FLOP_PER_CLK_SM, "sms": n_sm, "sm_mhz": mhz,
                     "tflops_at_clock": round(at_clock, 1) if at_clock else None,
                     "fwd_frac": round(fwd_ach / at_clock, 4) if at_clock else None,
                     "bwd_frac": round(bwd_ach / at_clock, 4) if at_clock else None,
                     "step_frac": round(value / world / at_clock, 4) if at_clock else None,
                     "note": "achieved / (measured tcgen05 rate x SMs x median SM clock of the timed region)"},
        "kernels_ms": {k_: round(v_, 4) for k_, v_ in per.items()},
        "fwd": {"tflops": round(fwd_ach, 2), "frac": round(fwd_ach / peak, 4)},
        "bwd": {"tflops": round(bwd_ach, 2), "frac": round(bwd_ach / peak, 4)},
        "gather": {"GB/s": round(gather_bytes / (per["gather"] * 1e-3) / 1e9, 1),
                   "frac_hbm": round(gather_bytes / (per["gather"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                   "bytes": gather_bytes, "remote_rows": remote_rows},
        "merge": merge,
        "ring": ring,
        "configs": configs,
        "shards": shards,
        "useful_pairs": pairs,
        "imbalance": policies,
        "clocks": clocks,
        "gpu_launches": 6 * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def _tile_counts(plan, cp):
    """Forward 128 x 128 tiles over all shards, per head: visited without a
    mask (full), visited with a per-element mask (partial), and skipped --
    those a plain causal kernel over the packed sequence (key tiles 0 ..
    the query tile's last row, no document mask) would add."""
    visited = masked = causal = 0
    for j in range(cp):
        sh = plan.shard(j)
        visited += sh["fwd_tiles"]
        masked += sh["fwd_masked"]
        for _, a, b in sh["pieces"]:
            for q0 in range(a, b, 128):
                causal += (min(q0 + 128, b) - 1) // 128 + 1
    return {"full": visited - masked, "partial": masked, "skipped": causal - visited}


def _bench_configs(torch, fcp, pk, dev):
    """The other packed workloads at their own shapes (seed 2000 + workload):
    gather + forward + backward per step, every shard in one launch; the 32K
    and 64K workloads under every policy; the 128K workload also as its
    8 ring-step partials over the owners' key blocks and their merge; the 2K
    workload (d = 64) forward only, as its configuration states."""
    res = {}
    for cfg in (1, 2, 3, 4):
        if cfg == CFG:
            continue
        w = synth.WORKLOADS[cfg]
        # The 32K and 64K workloads under every policy: all shards in one
        # launch, so the figures compare the plans' kernel efficiency (tile
        # shapes), not their balance across ranks (the shards leg does that).
        policies = (w.policy,) + tuple(p for p in ("wholedoc", "perdoc", "llama3", "hybrid", "hybrid_tiles")
                                       if p != w.policy) if cfg in (2, 4) else (w.policy,)
        entry = {"workload": w.name, "cp": w.cp}
        for pol in policies:
            st = Step(torch, cfg, pol, 2000 + cfg, dev)
            steps = 20 if cfg in (1, 2, 4) else 8
            _, per = st.timed(torch, steps, 3, backward=w.backward)
            r = _summary(st, per, pk, backward=w.backward)
            r["imbalance"] = round(st.s.stats()["imbalance"], 4)
            if cfg == 3:
                r["ring_steps_merge"] = _owner_merge(st, torch, fcp, pk)
            entry[pol] = r
            st.free()
            torch.cuda.empty_cache()
        res[f"cfg{cfg}"] = entry
    return res


def _owner_merge(st, torch, fcp, pk):
    """Ring step s of every shard (the keys of owner (j - s) mod N), N fp32
    partials, then fcp_merge of the N partials into bf16 O and LSE."""
    w = st.w
    T, hq, d, N = w.T, w.Hq, w.d, w.cp
    dev = st.q.device
    o_parts = torch.empty(N, T, hq, d, dtype=torch.float32, device=dev)
    l_parts = torch.empty(N, hq, T, dtype=torch.float32, device=dev)
    for s_ in range(N):
        st.s.forward_ring(st.q, st.k, st.v, ring_step=s_, out=o_parts[s_], lse=l_parts[s_])
    r = _time_merge(o_parts, l_parts, torch, fcp, pk)
    r["blocks_kind"] = "ring-step partials (the owners' key blocks)"
    del o_parts, l_parts
    return r


def _time_merge(o_parts, l_parts, torch, fcp, pk, n=10):
    B, T, hq, d = o_parts.shape
    dev = o_parts.device
    out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(hq, T, dtype=torch.float32, device=dev)
    for _ in range(3):
        fcp.merge(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fcp.merge(o_parts, l_parts, out, lse)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    nonempty = int(torch.isfinite(l_parts).sum().item())
    empty = B * hq * T - nonempty
    rd = nonempty * (4 * d + 4) + empty * 4
    wr = T * hq * (2 * d + 4)
    dense = B * T * hq * (4 * d + 4) + wr
    gbs = (rd + wr) / (ms * 1e-3) / 1e9
    return {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "frac_8TBs": round(gbs / 8000, 4),
            "ms": round(ms, 4), "bytes": rd + wr, "dense_bytes": dense, "blocks": B,
            "note": "parts with LSE=-inf are not read (no visible key in that block)"}


def _bench_merge(st, torch, fcp, pk):
    """Forward over B contiguous key blocks (fp32 partials, B = min(N, 8)),
    then the merge kernel; GB/s on the algorithmic bytes of the merge."""
    w = st.w
    T, hq, d = w.T, w.Hq, w.d
    B = min(w.cp, 8)
    dev = st.q.device
    o_parts = torch.empty(B, T, hq, d, dtype=torch.float32, device=dev)
    l_parts = torch.empty(B, hq, T, dtype=torch.float32, device=dev)
    bounds = [T * b // B for b in range(B + 1)]
    st.s.gather(st.k, st.v)
    for b in range(B):
        st.s.forward(st.q, st.k, st.v, out=o_parts[b], lse=l_parts[b], kv_block=(bounds[b], bounds[b + 1]),
                     out_dtype=torch.float32)
    r = _time_merge(o_parts, l_parts, torch, fcp, pk, n=5 if T > 200000 else 10)
    r["blocks_kind"] = "contiguous key blocks [T b / B, T (b+1) / B)"
    del o_parts, l_parts
    torch.cuda.empty_cache()
    return r


def _bench_ring(st, torch, fcp):
    """The forward several ways, same workload, fp32 output ("LLM Context
    Parallel in Production", "Ring Attention"; FlashCP §2.2 and §4 on the cost
    of blockwise ring execution): (a) gather of the received keys + one
    forward over them (the path of the timed step), (b) the fused ring (every
    owner's keys read in ring order in one pass, no gather), (c) one partial
    forward per ring step + fcp_merge of the N partials (where N fp32 partials
    fit in memory), (d) (a) with Q K^T in e4m3."""
    w = st.w
    T, hq, d, N = w.T, w.Hq, w.d, w.cp
    dev = st.q.device
    s, q, k, v = st.s, st.q, st.k, st.v
    out, lse = st.out, st.lse
    stepwise_fits = N * T * hq * d * 4 <= 40e9

    def gathered():
        s.gather(k, v)
        s.forward(q, k, v, out=out, lse=lse)

    def fused():
        s.forward_ring(q, k, v, ring_step=-1, out=out, lse=lse)

    o_parts = l_parts = mo = ml = None
    if stepwise_fits:
        o_parts = torch.empty(N, T, hq, d, dtype=torch.float32, device=dev)
        l_parts = torch.empty(N, hq, T, dtype=torch.float32, device=dev)
        mo = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
        ml = torch.empty(hq, T, dtype=torch.float32, device=dev)

    def stepwise():
        for st_ in range(N):
            s.forward_ring(q, k, v, ring_step=st_, out=o_parts[st_], lse=l_parts[st_])
        fcp.merge(o_parts, l_parts, mo, ml)

    def gathered_qk8():
        s.gather(k, v)
        s.forward_qk8(q, k, v, out=out, lse=lse)

    big = T > 200000
    res = {}
    variants = [("gather_then_forward", gathered), ("ring_fused", fused)]
    if stepwise_fits:
        variants.append(("ring_steps_then_merge", stepwise))
    variants.append(("gather_then_forward_e4m3_qk", gathered_qk8))
    for name, fn in variants:
        for _ in range(1 if big else 3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 3 if big else 10
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        res[name] = {"ms": round(ms, 4), "tflops": round(_tf(st.fwd_flops, ms), 2)}
    if s.device_status() != 0:
        raise RuntimeError("device status reports a failed wait in the ring leg")
    del o_parts, l_parts, mo, ml
    torch.cuda.empty_cache()
    res["note"] = ("useful fwd FLOPs / time; ring_steps_then_merge includes the N partial forwards and the merge "
                   "(run only where N fp32 partials fit); the e4m3 Q K^T form includes its per-call quantisation "
                   "of Q, K and the received K rows")
    return res


def _bench_shards(torch, dev):
    """Per-shard kernel time against W and against the tiles visited, one shard
    per launch (context_document_masked_gb300.calibrate): the 32K packed
    workload under Per-Doc, the 64K short-document workload under the five
    policies and the 128K workload under three."""
    from context_document_masked_gb300 import calibrate as cal
    rows, per_policy = [], {}
    for cfg, policies in ((2, ("perdoc",)), (4, ("llama3", "perdoc", "wholedoc", "hybrid", "hybrid_tiles")),
                          (3, ("perdoc", "hybrid", "hybrid_tiles"))):
        w = synth.WORKLOADS[cfg]
        D = synth.doc_lengths(cfg)
        q, k, v = synth.make_qkv(w.T, w.Hq, w.Hkv, w.d, seed=2000 + cfg, device=dev)
        do = synth.make_dout(w.T, w.Hq, w.d, seed=2000 + cfg, device=dev)
        for pol in policies:
            r = cal.shard_times(D, w.cp, pol, q, k, v, do)
            for x in r:
                x["workload"], x["policy"] = w.name, pol
            rows += r
            per_policy[f"{w.name}/{pol}"] = {
                "imbalance_pairs": round(cal.imbalance([x["pairs"] for x in r]), 4),
                "imbalance_fwd_tiles": round(cal.imbalance([x["fwd_tiles"] for x in r]), 4),
                "imbalance_time": round(cal.imbalance([x["fwd_ms"] + x["bwd_ms"] for x in r]), 4),
                "max_shard_ms": round(max(x["fwd_ms"] + x["bwd_ms"] for x in r), 4)}
        del q, k, v, do
    fits = {
        "fwd~pairs": cal.fit(rows, ("pairs",), "fwd_ms"),
        "fwd~tiles+qtiles": cal.fit(rows, ("fwd_tiles", "fwd_qtiles"), "fwd_ms"),
        "bwd~pairs": cal.fit(rows, ("pairs",), "bwd_ms"),
        "bwd~tiles+ktiles": cal.fit(rows, ("bwd_tiles", "bwd_ktiles"), "bwd_ms"),
    }
    fits["fwd+bwd~tiles+qtiles"] = cal.fit([dict(r, both=r["fwd_ms"] + r["bwd_ms"]) for r in rows],
                                           ("fwd_tiles", "fwd_qtiles"), "both")
    for f in fits.values():
        f["coef"] = {kk: float(f"{vv:.4g}") for kk, vv in f["coef"].items()}
        f["r2"], f["max_rel_err"] = round(f["r2"], 4), round(f["max_rel_err"], 4)
    return {"fits": fits, "policies": per_policy, "n_shards_timed": len(rows),
            "rows": [[r["workload"][:12], r["policy"], r["pairs"], r["fwd_tiles"], r["fwd_qtiles"],
                      r["bwd_tiles"], r["bwd_ktiles"], round(r["fwd_ms"], 4), round(r["bwd_ms"], 4)]
                     for r in rows],
            "note": "ms per shard launch (all SMs on one shard); counts over all heads; fits with a "
                    "per-launch intercept over all timed shards"}


def _bench_e2e(args, D, w, seed, torch, fcp):
    """End to end through the public API, pipelined the way a training loop
    would run it: step i's inputs go host -> device on one stream while step
    i-1 computes (Q, K, V first, then dO, which only the backward reads), and
    its results device -> host on a third stream while step i+1 computes.
    Every step copies all of its inputs in (Q, K, V, dO bf16) and
    all of its results out (O rounded to bf16 -- the forward keeps its fp32 O
    on the device for the backward's D_i -- and dQ, dK, dV fp32), builds its
    plan and allocates its session buffers; buffers alternate between two sets,
    ordered by events."""
    from context_document_masked_gb300.session import CPAttention
    T, hq, hkv, d = w.T, w.Hq, w.Hkv, w.d
    dev = torch.device("cuda", torch.cuda.current_device())
    # Inputs drawn on the device, then parked in pinned host memory (untimed).
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=seed, device=dev)
    do = synth.make_dout(T, hq, d, seed=seed, device=dev)
    h_in = []
    for x in (q, k, v, do):
        h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        h.copy_(x)
        h_in.append(h)
    del q, k, v, do
    out_specs = (((T, hq, d), torch.bfloat16), ((T, hq, d), torch.float32), ((T, hkv, d), torch.float32),
                 ((T, hkv, d), torch.float32))
    h_out = [[torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in out_specs] for _ in range(2)]
    d_in = [[torch.empty(x.shape, dtype=x.dtype, device=dev) for x in h_in] for _ in range(2)]
    d_out = [[torch.empty(sh, dtype=dt, device=dev) for sh, dt in out_specs] for _ in range(2)]
    o32 = [torch.empty(T, hq, d, dtype=torch.float32, device=dev) for _ in range(2)]
    lse = [torch.empty(hq, T, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    do_ready = [ev(), ev()]
    fwd_done = [ev(), ev()]
    pairs = sum(L * (L + 1) // 2 for L in D)
    sessions = [None, None]
    marks = []   # (start, end) events of each step's kernels on the compute stream
    cin, cout = [], []   # (start, end) events of each step's host->device / device->host copies

    def h2d(b):
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])          # the step two back is done reading these
            # The plan is one of the step's inputs: built on the host for this
            # step's document lengths, its work tables go up on the input stream
            # with Q, K, V, dO. Each buffer set keeps one session: its key
            # buffers and workspace are reused while large enough.
            if sessions[b] is None:
                sessions[b] = CPAttention(D, w.cp, w.policy, hq, hkv, d, device=dev)
            sessions[b].set_plan(D, stream=s_in)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            # Q, K, V first: the forward needs only them; dO, the backward's
            # input, follows while the forward runs.
            for h, g in zip(h_in[:3], d_in[b][:3]):
                g.copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
            d_in[b][3].copy_(h_in[3], non_blocking=True)
            e1.record(s_in)
            cin.append((e0, e1))
            do_ready[b].record(s_in)

    def step(b):
        qd, kd, vd, dod = d_in[b]
        o16, dq, dk, dv = d_out[b]
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_ready[b])
            s_comp.wait_event(out_done[b])          # results of two steps back have left
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(s_comp)
            s = sessions[b]
            s.gather(kd, vd, stream=s_comp)
            s.forward(qd, kd, vd, out=o32[b], lse=lse[b], out_dtype=torch.float32, stream=s_comp)
            fcp.round_bf16(o32[b], o16, stream=s_comp)
            fwd_done[b].record(s_comp)
            s_comp.wait_event(do_ready[b])
            s.backward(qd, kd, vd, o32[b], lse[b], dod, dq=dq, dk=dk, dv=dv, stream=s_comp)
            c1.record(s_comp)
            marks.append((c0, c1))
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            # O is final after the forward: it leaves while the backward runs.
            s_out.wait_event(fwd_done[b])
            h_out[b][0].copy_(o16, non_blocking=True)
            s_out.wait_event(comp_done[b])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_out)
            for g, h in zip(d_out[b][1:], h_out[b][1:]):
                h.copy_(g, non_blocking=True)
            e1.record(s_out)
            cout.append((e0, e1))
            out_done[b].record(s_out)

    def run(n):
        h2d(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                h2d(b ^ 1)
            step(b)
        torch.cuda.synchronize()

    big = T > 200000
    run(2 if big else 3)              # both buffer sets warmed (allocator, pinned pages)
    n = args.e2e_steps if big else max(4, args.steps // 2)
    reps = 1 if big else 3
    # Timed runs of n steps each; with several runs the median is reported (one
    # host stall in a run -- allocation, page-in, another process -- otherwise
    # moves the whole figure).
    runs, kern, bw_in, bw_out = [], [], [], []
    h2d_bytes = sum(x.numel() * x.element_size() for x in h_in)
    grad_bytes = sum(x.numel() * x.element_size() for x in h_out[0][1:])
    clk = ClockSampler(torch.cuda.current_device())
    with clk:
        for _ in range(reps):
            marks.clear()
            cin.clear()
            cout.clear()
            t0 = time.perf_counter()
            run(n)
            runs.append((time.perf_counter() - t0) / n)
            kern.append(sum(a.elapsed_time(b) for a, b in marks) / len(marks))
            bw_in.append(statistics.median(h2d_bytes / (a.elapsed_time(b) * 1e6) for a, b in cin))
            bw_out.append(statistics.median(grad_bytes / (a.elapsed_time(b) * 1e6) for a, b in cout))
    dt = sorted(runs)[len(runs) // 2]
    for s in sessions:
        if s is not None and s.device_status() != 0:
            raise RuntimeError("device status reports an error in the e2e leg")
    d2h_bytes = sum(x.numel() * x.element_size() for x in h_out[0])
    r = {"value": round((14.0 * d * hq * pairs) / dt / 1e12, 2), "unit": UNIT, "ms_per_step": round(dt * 1e3, 3),
         "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": n,
         "includes": "per step: H2D of Q,K,V then dO (the backward waits for dO only); plan build + upload "
                     "(buffers reused per buffer set); gather; fwd; "
                     "rounding of O to bf16; bwd; D2H of O (bf16, as soon as the forward ends), dQ, dK, dV "
                     "(fp32) -- copies of neighbouring steps overlap this step's kernels on separate streams",
         "runs_ms_per_step": [round(x * 1e3, 3) for x in runs],
         # The kernels of a step (gather .. backward) on the compute stream, per
         # run: the rest of ms_per_step is the first step's inputs and the last
         # step's results, which nothing overlaps, plus any gap between steps.
         "kernels_ms_per_step": [round(x, 3) for x in kern],
         # Median copy rates of the run (Q, K, V, dO in; dQ, dK, dV out).
         "h2d_GBps": [round(x, 1) for x in bw_in], "d2h_GBps": [round(x, 1) for x in bw_out],
         "clocks": clk.summary()}
    del h_in, h_out, d_in, d_out, o32, lse, sessions
    return r


def _cpu_baseline(seconds: float):
    """The fp64 oracle (per-document form) on the host cores, on a bounded
    sample of the workload: whole documents in order, one GQA group of heads,
    until `seconds` have passed. Reported as useful TFLOP/s of the sample."""
    from oracle import attention as A
    w, D, _ = _workload()
    G = w.Hq // w.Hkv
    order = sorted(range(len(D)), key=lambda i: D[i])
    t0 = time.perf_counter()
    flops, done = 0.0, []
    rng_seed = 4242
    for i in order:
        L = D[i]
        q, k, v = synth.make_qkv(L, G, 1, w.d, seed=rng_seed + i)
        do = synth.make_dout(L, G, w.d, seed=rng_seed + i)
        cu = np.array([0, L])
        o, lse = A.attention_per_doc(q, k, v, cu)
        A.attention_bwd_per_doc(q, k, v, o, lse, do, cu)
        flops += 14.0 * w.d * G * L * (L + 1) / 2
        done.append(L)
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    try:
        import threadpoolctl
        blas = threadpoolctl.threadpool_info()
        threads = max((b.get("num_threads", 0) for b in blas), default=None)
    except ImportError:
        threads = None
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": threads or os.cpu_count(),
            "host_cpus": os.cpu_count(), "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"fp64 per-document fwd+bwd, {G} query heads (one GQA group), "
                      f"{len(done)} whole documents (lengths {done}) of the workload"}


def run_reference(args):
    world, rank = _dist()
    if rank != 0:
        return
    w, D, pairs = _workload()
    vals = []
    for _ in range(args.warmup):
        _cpu_baseline(args.ref_seconds)
    for _ in range(args.steps):
        vals.append(_cpu_baseline(args.ref_seconds))
    v = statistics.mean(x["value"] for x in vals)
    step_s = statistics.mean(x["seconds"] for x in vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, D),
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "kind": "oracle", "cores": vals[0]["cores"],
                             "sample": vals[0]["sample"]},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fcp", choices=["fcp", "reference"])
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5],
                    help="headline workload (1: 2K d=64, 2: 32K, 3: 128K, 4: 64K short docs, 5: 512K)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=3.0)
    ap.add_argument("--e2e-steps", type=int, default=6,
                    help="timed end-to-end steps on workloads above 200K tokens (one run of them; smaller "
                         "workloads take the median of three runs of max(4, steps / 2))")
    ap.add_argument("--legs", default="step,merge,ring,configs,shards,e2e,cpu",
                    help="parts to run: step (always), merge, ring, configs (the other workloads), shards "
                         "(per-shard calibration), e2e, cpu; e.g. 'step' for profiling")
    args = ap.parse_args()
    global CFG
    CFG = args.workload
    if args.warmup < 3 and args.impl == "fcp":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
