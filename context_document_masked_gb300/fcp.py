"""Python binding of libfcp (include/fcp.h), argument marshalling only.

Every computation runs in the C++ planner or the CUDA kernels of libfcp.so;
PyTorch supplies device memory and streams. Importing this module loads the
library and raises if it has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# FCP_DEVICE_CHECKS=1 selects the checked build (device-side bounds checks on
# every plan-table index; build with build.build(checked=True)).
CHECKED = os.environ.get("FCP_DEVICE_CHECKS") == "1"
LIB_PATH = os.path.join(_HERE, "_lib_checked" if CHECKED else "_lib", "libfcp.so")

(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_INFEASIBLE, ERR_CAPACITY,
 ERR_MISSING_PART) = range(8)
POLICIES = {"llama3": 0, "perdoc": 1, "wholedoc": 2, "hybrid": 3, "hybrid_tiles": 4}
OUT_BF16, OUT_F32 = 0, 1

EXPORTED = (
    "fcp_strerror", "fcp_plan", "fcp_plan_free", "fcp_plan_shard", "fcp_plan_query_indices",
    "fcp_plan_stats", "fcp_plan_per_doc_flags", "fcp_plan_device_bytes", "fcp_plan_upload",
    "fcp_workspace_bytes", "fcp_gather_kv", "fcp_attn_fwd", "fcp_merge", "fcp_attn_bwd",
    "fcp_get_device_status", "fcp_debug_set_wait_limit", "fcp_attn_fwd_noalloc", "fcp_attn_fwd_ring",
    "fcp_attn_fwd_qk8", "fcp_quant_e4m3", "fcp_plan_device_image", "fcp_plan_bind",
    "fcp_debug_rescale_events", "fcp_round_bf16", "fcp_merge_ring",
)


class FcpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.fcp_strerror(status).decode()} (status {status})")


class Range(C.Structure):
    _fields_ = [("doc", C.c_int32), ("start", C.c_int32), ("end", C.c_int32)]


class ShardView(C.Structure):
    _fields_ = [
        ("n_pieces", C.c_int32), ("pieces", C.POINTER(Range)),
        ("n_need", C.c_int32), ("kv_need", C.POINTER(Range)),
        ("n_remote", C.c_int32), ("kv_remote", C.POINTER(Range)),
        ("tokens", C.c_int64), ("useful_pairs", C.c_int64), ("remote_rows", C.c_int64),
        ("kbuf_base", C.c_int64), ("fwd_tiles", C.c_int64), ("fwd_qtiles", C.c_int64),
        ("fwd_masked", C.c_int64), ("bwd_tiles", C.c_int64), ("bwd_ktiles", C.c_int64),
    ]


class PlanStats(C.Structure):
    _fields_ = [
        ("cp", C.c_int32), ("n_docs", C.c_int32), ("T", C.c_int64), ("imbalance", C.c_double),
        ("max_pairs", C.c_int64), ("total_pairs", C.c_int64), ("eq4_tokens", C.c_int64),
        ("eq5_tokens", C.c_int64), ("remote_rows_total", C.c_int64), ("remote_rows_max", C.c_int64),
        ("eq2_max_dev", C.c_int64), ("iterations", C.c_int32), ("n_per_doc", C.c_int32),
    ]


class DevPlan(C.Structure):
    _fields_ = [
        ("host", C.c_void_p), ("base", C.c_void_p), ("bytes", C.c_int64), ("n_shards", C.c_int32),
        ("T", C.c_int32), ("total_remote_rows", C.c_int64), ("tables", C.c_int32 * 16),
        ("counts", C.c_int32 * 16),
    ]


class Dims(C.Structure):
    _fields_ = [("T", C.c_int32), ("hq", C.c_int32), ("hkv", C.c_int32), ("d", C.c_int32),
                ("scale", C.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libfcp.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, f64 = C.c_void_p, C.c_int32, C.c_int64, C.c_double
    sig = {
        "fcp_strerror": (C.c_char_p, [C.c_int]),
        "fcp_plan": (C.c_int, [C.POINTER(C.c_int32), i32, i32, i32, f64, C.POINTER(vp)]),
        "fcp_plan_free": (None, [vp]),
        "fcp_plan_shard": (C.c_int, [vp, i32, C.POINTER(ShardView)]),
        "fcp_plan_query_indices": (C.c_int, [vp, i32, C.POINTER(C.c_int32), i64, C.POINTER(i64)]),
        "fcp_plan_stats": (C.c_int, [vp, C.POINTER(PlanStats)]),
        "fcp_plan_per_doc_flags": (C.c_int, [vp, C.POINTER(C.c_int32), i32]),
        "fcp_plan_device_bytes": (i64, [vp]),
        "fcp_plan_upload": (C.c_int, [vp, vp, i64, vp, C.POINTER(DevPlan)]),
        "fcp_plan_device_image": (C.c_int, [vp, vp, i64]),
        "fcp_plan_bind": (C.c_int, [vp, vp, i64, C.POINTER(DevPlan)]),
        "fcp_workspace_bytes": (i64, [Dims, vp]),
        "fcp_gather_kv": (C.c_int, [vp, vp, C.POINTER(DevPlan), i32, i32, i32, vp, vp, vp]),
        "fcp_attn_fwd": (C.c_int, [vp, vp, vp, vp, vp, C.POINTER(DevPlan), i32, i32, i32, Dims, i32,
                                   vp, vp, vp, i64, vp]),
        "fcp_attn_fwd_ring": (C.c_int, [vp, vp, vp, C.POINTER(DevPlan), i32, i32, Dims, i32, vp, vp, vp, i64,
                                        vp]),
        "fcp_attn_fwd_qk8": (C.c_int, [vp, vp, vp, vp, vp, C.POINTER(DevPlan), i32, i32, i32, Dims, i32,
                                       vp, vp, vp, i64, vp]),
        "fcp_quant_e4m3": (C.c_int, [vp, i64, vp, vp, vp, vp]),
        "fcp_merge": (C.c_int, [vp, vp, i32, i64, i32, i32, vp, vp, vp]),
        "fcp_attn_bwd": (C.c_int, [vp, vp, vp, vp, vp, vp, i32, vp, vp, C.POINTER(DevPlan), i32,
                                   Dims, vp, vp, vp, vp, i64, vp]),
        "fcp_get_device_status": (C.c_int, [vp, vp]),
        "fcp_attn_fwd_noalloc": (C.c_int, [vp, vp, vp, vp, vp, C.POINTER(DevPlan), i32, i32, i32, Dims,
                                           i32, vp, vp, vp]),
        "fcp_debug_set_wait_limit": (None, [i64]),
        "fcp_debug_rescale_events": (C.c_int, [vp, vp, C.POINTER(i64)]),
        "fcp_round_bf16": (C.c_int, [vp, i64, vp, vp]),
        "fcp_merge_ring": (C.c_int, [C.POINTER(DevPlan), vp, vp, C.POINTER(C.c_int32), i32, i32, i32, vp, vp,
                                     vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def _check(status: int, what: str):
    if status != OK:
        raise FcpError(status, what)


def strerror(status: int) -> str:
    return _lib.fcp_strerror(status).decode()


# ---------------------------------------------------------------- plans


class Plan:
    """A host sharding plan (fcp_plan)."""

    def __init__(self, doclens, cp: int, policy: str, target_imbalance: float = 1.05):
        d = np.ascontiguousarray(np.asarray(doclens, dtype=np.int32))
        self._ptr = C.c_void_p()
        _check(_lib.fcp_plan(d.ctypes.data_as(C.POINTER(C.c_int32)), len(d), cp, POLICIES[policy],
                             target_imbalance, C.byref(self._ptr)), "fcp_plan")
        self.doclens = d
        self.cp = cp
        self.policy = policy

    def __del__(self):
        if getattr(self, "_ptr", None) and self._ptr.value:
            _lib.fcp_plan_free(self._ptr)
            self._ptr = C.c_void_p()

    @property
    def handle(self):
        return self._ptr

    def shard(self, j: int) -> dict:
        v = ShardView()
        _check(_lib.fcp_plan_shard(self._ptr, j, C.byref(v)), "fcp_plan_shard")

        def rng(ptr, n):
            return [(ptr[i].doc, ptr[i].start, ptr[i].end) for i in range(n)]
        return {
            "pieces": rng(v.pieces, v.n_pieces), "kv_need": rng(v.kv_need, v.n_need),
            "kv_remote": rng(v.kv_remote, v.n_remote), "tokens": v.tokens,
            "useful_pairs": v.useful_pairs, "remote_rows": v.remote_rows, "kbuf_base": v.kbuf_base,
            "fwd_tiles": v.fwd_tiles, "fwd_qtiles": v.fwd_qtiles, "fwd_masked": v.fwd_masked,
            "bwd_tiles": v.bwd_tiles, "bwd_ktiles": v.bwd_ktiles,
        }

    def query_indices(self, j: int) -> np.ndarray:
        n = C.c_int64()
        st = _lib.fcp_plan_query_indices(self._ptr, j, None, 0, C.byref(n))
        if st not in (OK, ERR_CAPACITY):
            _check(st, "fcp_plan_query_indices")
        out = np.empty(n.value, dtype=np.int32)
        _check(_lib.fcp_plan_query_indices(self._ptr, j, out.ctypes.data_as(C.POINTER(C.c_int32)),
                                           n.value, C.byref(n)), "fcp_plan_query_indices")
        return out

    def stats(self) -> dict:
        s = PlanStats()
        _check(_lib.fcp_plan_stats(self._ptr, C.byref(s)), "fcp_plan_stats")
        return {f: getattr(s, f) for f, _ in PlanStats._fields_}

    def per_doc_flags(self) -> list:
        out = np.zeros(len(self.doclens), dtype=np.int32)
        _check(_lib.fcp_plan_per_doc_flags(self._ptr, out.ctypes.data_as(C.POINTER(C.c_int32)),
                                           len(out)), "fcp_plan_per_doc_flags")
        return out.tolist()

    def device_bytes(self) -> int:
        return int(_lib.fcp_plan_device_bytes(self._ptr))

    def device_image(self) -> np.ndarray:
        """The work tables as fcp_plan_upload would send them (int32 words)."""
        out = np.empty(self.device_bytes() // 4, dtype=np.int32)
        _check(_lib.fcp_plan_device_image(self._ptr, out.ctypes.data_as(C.c_void_p), out.nbytes),
               "fcp_plan_device_image")
        return out

    def bind(self, buf) -> "DevicePlan":
        """Handle for a device tensor that holds (or is about to hold) the image."""
        dp = DevPlan()
        _check(_lib.fcp_plan_bind(self._ptr, C.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(),
                                  C.byref(dp)), "fcp_plan_bind")
        return DevicePlan(dp, self, buf)

    def upload(self, buf, stream=None) -> "DevicePlan":
        """Copy the work tables into `buf` (an int32 device tensor of >= device_bytes()
        bytes) on `stream`, staged through pinned host memory so that the host does
        not wait for the stream's earlier work."""
        import torch
        n = self.device_bytes() // 4
        dp = self.bind(buf)
        host = torch.empty(n, dtype=torch.int32, pin_memory=True)
        _check(_lib.fcp_plan_device_image(self._ptr, C.c_void_p(host.data_ptr()), n * 4),
               "fcp_plan_device_image")
        if stream is None:
            s = torch.cuda.current_stream()
        elif isinstance(stream, int):
            s = torch.cuda.ExternalStream(stream)
        else:
            s = stream
        with torch.cuda.stream(s):
            buf.view(torch.int32)[:n].copy_(host, non_blocking=True)
        return dp


class DevicePlan:
    """fcp_dev_plan plus references that keep the host plan and buffer alive."""

    def __init__(self, dp: DevPlan, plan: Plan, buf):
        self.c = dp
        self.plan = plan
        self.buf = buf

    @property
    def total_remote_rows(self) -> int:
        return int(self.c.total_remote_rows)

    def remote_rows(self, shard: int) -> int:
        return self.total_remote_rows if shard < 0 else int(self.plan.shard(shard)["remote_rows"])


# ---------------------------------------------------------------- device


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _ptr(t):
    return C.c_void_p(0 if t is None else t.data_ptr())


def _t(t, name, dtypes=None, shape=None):
    """Checks a tensor before its raw pointer goes to the library, which cannot
    see dtypes, strides or devices: a contiguous CUDA tensor of one of
    `dtypes`, of `shape` (None entries free). Raises ValueError."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected one of {tuple(str(x) for x in dtypes)}")
    if shape is not None and (t.dim() != len(shape) or any(e is not None and e != x for e, x in zip(shape, t.shape))):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _qkv(q, k, v):
    """Q [T][hq][d] and K, V [T][hkv][d], bf16; returns (T, hq, hkv, d)."""
    import torch
    _t(q, "q", (torch.bfloat16,), (None, None, None))
    T, hq, d = q.shape
    _t(k, "k", (torch.bfloat16,), (T, None, d))
    _t(v, "v", (torch.bfloat16,), tuple(k.shape))
    return T, hq, k.shape[1], d


def _kbuf(kbuf, vbuf, dplan, shard, hkv, d):
    """The received-key buffers hold at least the rows the plan sends to
    `shard` (all shards' for -1): the library writes and reads them by the
    plan, not by their size."""
    import torch
    rows = max(1, dplan.remote_rows(shard))
    for t, n in ((kbuf, "kbuf"), (vbuf, "vbuf")):
        _t(t, n, (torch.bfloat16,), (None, hkv, d))
        if t.shape[0] < rows:
            raise ValueError(f"{n}: {t.shape[0]} rows, the plan receives {rows}")


def _out_lse(out, lse, T, hq, d):
    import torch
    _t(out, "out", (torch.bfloat16, torch.float32), (T, hq, d))
    _t(lse, "lse", (torch.float32,), (hq, T))


def dims(T: int, hq: int, hkv: int, d: int, scale: float = 0.0) -> Dims:
    return Dims(T, hq, hkv, d, scale)


def workspace_bytes(dm: Dims, plan: "Plan | None" = None) -> int:
    return int(_lib.fcp_workspace_bytes(dm, plan.handle if plan is not None else None))


def gather_kv(k, v, dplan: DevicePlan, shard: int, kbuf, vbuf, stream=None):
    import torch
    _t(k, "k", (torch.bfloat16,), (None, None, None))
    _t(v, "v", (torch.bfloat16,), tuple(k.shape))
    _kbuf(kbuf, vbuf, dplan, shard, k.shape[1], k.shape[2])
    _check(_lib.fcp_gather_kv(_ptr(k), _ptr(v), C.byref(dplan.c), shard, k.shape[1], k.shape[2],
                              _ptr(kbuf), _ptr(vbuf), _stream(stream)), "fcp_gather_kv")


def attn_fwd(q, k, v, kbuf, vbuf, dplan: DevicePlan, shard: int, out, lse, ws, kv_lo: int = 0,
             kv_hi: int | None = None, scale: float = 0.0, stream=None):
    import torch
    T, hq, hkv, d = _qkv(q, k, v)
    _kbuf(kbuf, vbuf, dplan, shard, hkv, d)
    _out_lse(out, lse, T, hq, d)
    _t(ws, "ws")
    dm = Dims(T, hq, hkv, d, scale)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(_lib.fcp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(kbuf), _ptr(vbuf), C.byref(dplan.c),
                             shard, kv_lo, T if kv_hi is None else kv_hi, dm, out_dtype, _ptr(out),
                             _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "fcp_attn_fwd")


def attn_fwd_qk8(q, k, v, kbuf, vbuf, dplan: DevicePlan, shard: int, out, lse, ws, kv_lo: int = 0,
                 kv_hi: int | None = None, scale: float = 0.0, stream=None):
    """fcp_attn_fwd_qk8: the forward with Q K^T on e4m3 copies of Q and K."""
    import torch
    T, hq, hkv, d = _qkv(q, k, v)
    _kbuf(kbuf, vbuf, dplan, shard, hkv, d)
    _out_lse(out, lse, T, hq, d)
    _t(ws, "ws")
    dm = Dims(T, hq, hkv, d, scale)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(_lib.fcp_attn_fwd_qk8(_ptr(q), _ptr(k), _ptr(v), _ptr(kbuf), _ptr(vbuf), C.byref(dplan.c),
                                 shard, kv_lo, T if kv_hi is None else kv_hi, dm, out_dtype, _ptr(out),
                                 _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "fcp_attn_fwd_qk8")


def quant_e4m3(x, out, scale_out, scratch, stream=None):
    """fcp_quant_e4m3: out (uint8, x.numel() bytes) = e4m3(x * 2^k); scale_out[0] = 2^k."""
    import torch
    _t(x, "x", (torch.bfloat16,))
    _t(out, "out", (torch.uint8,))
    _t(scale_out, "scale_out", (torch.float32,))
    _t(scratch, "scratch", (torch.int32,))
    if out.numel() < x.numel() or scale_out.numel() < 1 or scratch.numel() < 1:
        raise ValueError("quant_e4m3: out holds x.numel() bytes, scale_out and scratch one element each")
    _check(_lib.fcp_quant_e4m3(_ptr(x), x.numel(), _ptr(out), _ptr(scale_out), _ptr(scratch), _stream(stream)),
           "fcp_quant_e4m3")


def attn_fwd_ring(q, k, v, dplan: DevicePlan, shard: int, ring_step: int, out, lse, ws, scale: float = 0.0,
                  stream=None):
    """fcp_attn_fwd_ring: every needed key read from its owner's rows of K/V,
    owners in ring order; ring_step -1 = all owners in one pass, s >= 0 = the
    partial result of ring step s."""
    import torch
    T, hq, hkv, d = _qkv(q, k, v)
    _out_lse(out, lse, T, hq, d)
    _t(ws, "ws")
    dm = Dims(T, hq, hkv, d, scale)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(_lib.fcp_attn_fwd_ring(_ptr(q), _ptr(k), _ptr(v), C.byref(dplan.c), shard, ring_step, dm, out_dtype,
                                  _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)),
           "fcp_attn_fwd_ring")


def attn_fwd_noalloc(q, k, v, kbuf, vbuf, dplan: DevicePlan, shard: int, out, lse, kv_lo: int = 0,
                     kv_hi: int | None = None, scale: float = 0.0, stream=None):
    """fcp_attn_fwd_noalloc: the forward with the library's static scratch
    instead of a caller workspace (for callers that cannot allocate)."""
    import torch
    T, hq, hkv, d = _qkv(q, k, v)
    _kbuf(kbuf, vbuf, dplan, shard, hkv, d)
    _out_lse(out, lse, T, hq, d)
    dm = Dims(T, hq, hkv, d, scale)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(_lib.fcp_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kbuf), _ptr(vbuf), C.byref(dplan.c),
                                     shard, kv_lo, T if kv_hi is None else kv_hi, dm, out_dtype,
                                     _ptr(out), _ptr(lse), _stream(stream)),
           "fcp_attn_fwd_noalloc")


def round_bf16(x, out, stream=None):
    """fcp_round_bf16: out (bf16, same element count) = x (fp32) rounded to nearest even."""
    import torch
    _t(x, "x", (torch.float32,))
    _t(out, "out", (torch.bfloat16,))
    if x.numel() != out.numel():
        raise ValueError("round_bf16: x and out differ in element count")
    _check(_lib.fcp_round_bf16(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "fcp_round_bf16")


def _merge_args(o_parts, lse_parts, out, lse_out):
    import torch
    _t(o_parts, "o_parts", (torch.float32,), (None, None, None, None))
    B, rows, hq, d = o_parts.shape
    _t(lse_parts, "lse_parts", (torch.float32,), (B, hq, rows))
    _t(out, "out", (torch.bfloat16,), (rows, hq, d))
    _t(lse_out, "lse_out", (torch.float32,), (hq, rows))
    return B, rows, hq, d


def merge(o_parts, lse_parts, out, lse_out, stream=None):
    B, rows, hq, d = _merge_args(o_parts, lse_parts, out, lse_out)
    _check(_lib.fcp_merge(_ptr(o_parts), _ptr(lse_parts), B, rows, hq, d, _ptr(out), _ptr(lse_out),
                          _stream(stream)), "fcp_merge")


def merge_ring(dplan: DevicePlan, o_parts, lse_parts, part_step, out, lse_out, stream=None):
    """fcp_merge_ring: merge of the N ring-step partials; part_step[b] is the
    ring step that produced partial b (a missing or duplicated step raises
    FcpError with status ERR_MISSING_PART before anything is launched)."""
    B, rows, hq, d = o_parts.shape
    steps = np.ascontiguousarray(np.asarray(part_step, dtype=np.int32))
    if len(steps) != B or rows != dplan.c.T or tuple(lse_parts.shape) != (B, hq, rows):
        raise ValueError("merge_ring: one step tag per partial, each partial [T][hq][d] with T the plan's")
    _merge_args(o_parts, lse_parts, out, lse_out)
    _check(_lib.fcp_merge_ring(C.byref(dplan.c), _ptr(o_parts), _ptr(lse_parts),
                               steps.ctypes.data_as(C.POINTER(C.c_int32)), len(steps), hq, d, _ptr(out),
                               _ptr(lse_out), _stream(stream)), "fcp_merge_ring")


def attn_bwd(q, k, v, kbuf, vbuf, out, lse, dout, dplan: DevicePlan, shard: int, dq, dk, dv, ws,
             scale: float = 0.0, stream=None):
    import torch
    T, hq, hkv, d = _qkv(q, k, v)
    _kbuf(kbuf, vbuf, dplan, shard, hkv, d)
    _out_lse(out, lse, T, hq, d)
    _t(dout, "dout", (torch.bfloat16,), (T, hq, d))
    _t(dq, "dq", (torch.float32,), (T, hq, d))
    _t(dk, "dk", (torch.float32,), (T, hkv, d))
    _t(dv, "dv", (torch.float32,), (T, hkv, d))
    _t(ws, "ws")
    dm = Dims(T, hq, hkv, d, scale)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(_lib.fcp_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(kbuf), _ptr(vbuf), _ptr(out), out_dtype,
                             _ptr(lse), _ptr(dout), C.byref(dplan.c), shard, dm, _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "fcp_attn_bwd")


def device_status(ws, stream=None) -> int:
    _t(ws, "ws")
    return int(_lib.fcp_get_device_status(_ptr(ws), _stream(stream)))


def debug_set_wait_limit(ns: int):
    _lib.fcp_debug_set_wait_limit(ns)


def debug_rescale_events(ws, stream=None) -> int:
    """Rescales of O after a later key tile since the last read (then cleared)."""
    _t(ws, "ws")
    n = C.c_int64()
    _check(_lib.fcp_debug_rescale_events(_ptr(ws), _stream(stream), C.byref(n)), "fcp_debug_rescale_events")
    return int(n.value)


def raw_call(name: str, *args):
    """Direct C-ABI call (for tests of argument validation)."""
    return getattr(_lib, name)(*args)
