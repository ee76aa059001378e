"""Seeded synthetic inputs for document-masked context-parallel attention.

This module is the one place shared by the CPU oracle and the CUDA path. It
holds no arithmetic of the method: it only draws packed-sequence document
lengths and bf16 tensors from seeded generators.

The packed-sequence recipe follows the FlashCP paper ("FlashCP:
Load-Balanced Communication-Efficient Context Parallelism for LLM Training"),
§4.1 Datasets: documents are drawn one after another and the last one is
truncated so that the sequence fills the context window exactly. The length
distributions below stand in for the paper's WLB-LLM, Pile and RedPajama
samples, none of which is used here.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "doc_lengths",
    "random_doc_lengths",
    "cu_from_lengths",
    "make_qkv",
    "make_dout",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int          # packed tokens (the context window C)
    Hq: int
    Hkv: int
    d: int
    cp: int         # CP size N
    policy: str     # "llama3" | "perdoc" | "wholedoc" | "hybrid"
    backward: bool
    merge_blocks: int   # B > 0: the forward is also run as B key blocks + merge


# The five packed-sequence workloads. The index is the seed offset: lengths are
# drawn from numpy.random.default_rng(1000 + index).
WORKLOADS = {
    1: Workload("packed2k_uniform_h4kv2_d64_cp2_llama3", 2048, 4, 2, 64, 2, "llama3", False, 0),
    2: Workload("packed32k_lognorm_h32kv8_d128_cp4_perdoc", 32768, 32, 8, 128, 4, "perdoc", True, 0),
    3: Workload("packed128k_lognorm_plus64k_h32kv8_d128_cp8_hybrid", 131072, 32, 8, 128, 8, "hybrid", True, 8),
    4: Workload("packed64k_shortdocs_h64kv8_d128_cp16", 65536, 64, 8, 128, 16, "wholedoc", True, 0),
    5: Workload("packed512k_lognorm_h32kv8_d128_cp32_hybrid", 524288, 32, 8, 128, 32, "hybrid", True, 0),
}


def _fill(draw, T: int) -> list[int]:
    """Draw lengths until they cover T tokens, then cut the last one to fit."""
    out: list[int] = []
    total = 0
    while total < T:
        L = int(draw())
        if L < 1:
            L = 1
        out.append(L)
        total += L
    out[-1] -= total - T
    if out[-1] == 0:
        out.pop()
    return out


def doc_lengths(cfg: int, repeat: int = 0) -> list[int]:
    """Document lengths of workload `cfg` (1..5); `repeat` selects seed +1, +2, ..."""
    rng = np.random.default_rng(1000 + cfg + repeat)
    T = WORKLOADS[cfg].T
    if cfg == 1:
        ls = [int(x) for x in rng.integers(64, 641, size=6)]
        out, total = [], 0
        for L in ls:
            if total + L >= T:
                out.append(T - total)
                total = T
                break
            out.append(L)
            total += L
        if total < T:
            out[-1] += T - total
        return out
    if cfg == 2:
        return _fill(lambda: np.clip(np.rint(rng.lognormal(7.5, 1.2)), 32, 32768), T)
    if cfg == 3:
        big = 65536
        rest = _fill(lambda: np.clip(np.rint(rng.lognormal(8.0, 1.5)), 32, 65536), T - big)
        pos = int(rng.integers(0, len(rest) + 1))
        return rest[:pos] + [big] + rest[pos:]
    if cfg == 4:
        def draw():
            if rng.random() < 0.1:
                return rng.integers(4096, 16385)
            return rng.integers(128, 1025)
        return _fill(draw, T)
    if cfg == 5:
        return _fill(lambda: np.clip(np.rint(rng.lognormal(9.0, 1.8)), 256, 262144), T)
    raise ValueError(f"unknown workload {cfg}")


def random_doc_lengths(T: int, seed: int, max_len: int | None = None,
                       p_tiny: float = 0.15) -> list[int]:
    """Ragged document mix for edge-case tests: 1-token docs, docs shorter and
    longer than a 128-row tile, and a long tail."""
    rng = np.random.default_rng(seed)
    max_len = max_len or T

    def draw():
        u = rng.random()
        if u < p_tiny:
            return rng.integers(1, 4)
        if u < 0.6:
            return rng.integers(4, 200)
        return min(max_len, int(rng.integers(200, max(201, T // 2))))
    return _fill(draw, T)


def cu_from_lengths(lengths) -> np.ndarray:
    """Cumulative document offsets [0, d1, d1+d2, ...] as int32."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu.astype(np.int32)


def _normal_bf16(shape, gen, device):
    import torch
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)  # round to nearest even


def _gen(seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_qkv(T: int, Hq: int, Hkv: int, d: int, seed: int, device="cpu"):
    """Q [T,Hq,d], K and V [T,Hkv,d], bf16, N(0,1) before rounding, drawn in
    that order from one torch generator on `device`."""
    g = _gen(seed, device)
    q = _normal_bf16((T, Hq, d), g, device)
    k = _normal_bf16((T, Hkv, d), g, device)
    v = _normal_bf16((T, Hkv, d), g, device)
    return q, k, v


def make_dout(T: int, Hq: int, d: int, seed: int, device="cpu"):
    """Upstream gradient dO [T,Hq,d] bf16, N(0,1) before rounding."""
    g = _gen(seed + 7919, device)
    return _normal_bf16((T, Hq, d), g, device)
