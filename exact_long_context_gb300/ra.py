"""ctypes binding of libra.so: torch tensors in, C-ABI calls out.

Argument marshalling only - every step of the computation runs in the library's CUDA
kernels.  The library must be built (``python -m exact_long_context_gb300.build``);
if it is missing, or a tensor is not on a CUDA device, the call raises.  There is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# RA_LIBRARY=debug selects the bounds-checked debug build (build.py --debug-bounds)
LIB_PATH = os.path.join(_HERE, "libra_debug.so" if os.environ.get("RA_LIBRARY") == "debug" else "libra.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT, RA_ERR_BOUNDS = range(6)
RA_F32, RA_BF16 = 0, 1
LAYOUTS = {"contig": 0, "zigzag": 1, "striped": 2}
SEG_FIRST, SEG_FINAL = 1, 2


class RaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"ra status {status}: {msg}")
        self.status = status


class RaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run python -m exact_long_context_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            P, T = ctypes.c_void_p, ctypes.POINTER(RaTensor)
            i64, c_int, c_float = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            L.ra_attn_fwd.argtypes = [T, T, T, T, P, c_int, c_float, P]
            L.ra_lse_merge.argtypes = [T, P, T, P, P]
            L.ra_ring_sim_workspace_bytes.argtypes = [T, c_int]
            L.ra_ring_sim_workspace_bytes.restype = ctypes.c_size_t
            L.ra_ring_sim_workspace_bytes_for.argtypes = [T, T, T, T, c_int, c_int, c_int]
            L.ra_ring_sim_workspace_bytes_for.restype = ctypes.c_size_t
            L.ra_ring_sim_fwd.argtypes = [T, T, T, T, P, c_int, c_int, c_int, c_float, P, P]
            L.ra_attn_varlen_fwd.argtypes = [T, T, T, T, P, P, c_int, c_int, c_float, P]
            L.ra_attn_varlen_fwd.restype = c_int
            L.ra_attn_bwd_workspace_bytes.argtypes = [T]
            L.ra_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.ra_attn_bwd.argtypes = [T, T, T, T, P, T, T, T, T, c_int, c_float, P, P]
            L.ra_attn_bwd.restype = c_int
            L.ra_ring_sim_fwd_host_workspace_bytes.argtypes = [T, T, c_int]
            L.ra_ring_sim_fwd_host_workspace_bytes.restype = ctypes.c_size_t
            L.ra_ring_sim_fwd_host.argtypes = [T, T, T, T, P, c_int, c_int, c_int, c_float, P, ctypes.c_size_t, P]
            L.ra_ring_sim_fwd_host.restype = c_int
            L.ra_ring_sim_bwd_workspace_bytes.argtypes = [T, T, c_int]
            L.ra_ring_sim_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.ra_ring_sim_bwd.argtypes = [T, T, T, T, P, T, T, T, T, c_int, c_int, c_int, c_float, P, P]
            L.ra_ring_sim_bwd.restype = c_int
            L.ra_ulysses_all_to_all.argtypes = [T, T, c_int, c_int, P]
            L.ra_ulysses_all_to_all.restype = c_int
            L.ra_ring_sim_plan.argtypes = [i64, c_int, c_int, c_int, c_int, P, i64]
            L.ra_ring_sim_plan.restype = i64
            L.ra_ring_sim_bwd_plan.argtypes = [i64, c_int, c_int, c_int, c_int, c_int, P, i64]
            L.ra_ring_sim_bwd_plan.restype = i64
            L.ra_check_device_error.argtypes = [P]
            L.ra_debug_set_wait_limit_ns.argtypes = [i64]
            L.ra_debug_set_wait_limit_ns.restype = None
            L.ra_debug_set_producer_delay_ns.argtypes = [i64]
            L.ra_debug_set_producer_delay_ns.restype = None
            L.ra_debug_wait_selftest.argtypes = [i64, P]
            L.ra_debug_fail_next_launches.argtypes = [c_int]
            L.ra_debug_fail_next_launches.restype = None
            L.ra_debug_bounds_checked.restype = c_int
            L.ra_debug_time_launches.argtypes = [c_int]
            L.ra_debug_time_launches.restype = None
            L.ra_debug_launch_times.argtypes = [P, c_int, P, c_int]
            L.ra_debug_launch_times.restype = c_int
            L.ra_debug_bounds_selftest.argtypes = [P]
            L.ra_debug_bounds_selftest.restype = c_int
            L.ra_debug_work_counters_in_use.argtypes = [P]
            L.ra_debug_work_counters_in_use.restype = c_int
            L.ra_debug_host_group_bounds.argtypes = [ctypes.c_int64, c_int, c_int, P]
            L.ra_debug_host_group_bounds.restype = c_int
            L.ra_last_error.restype = ctypes.c_char_p
            L.ra_launch_count.argtypes = [c_int]
            L.ra_launch_count.restype = i64
            for name in ("ra_attn_fwd", "ra_lse_merge", "ra_ring_sim_fwd", "ra_check_device_error",
                         "ra_debug_wait_selftest"):
                getattr(L, name).restype = c_int
            _lib = L
        return _lib


def _check(status: int):
    if status != RA_OK:
        raise RaError(status, lib().ra_last_error().decode())


def _desc(t: torch.Tensor | None, name: str, host: bool = False) -> RaTensor:
    d = RaTensor()
    if t is None:
        return d
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, N, D]")
    if t.dtype == torch.float32:
        d.dtype = RA_F32
    elif t.dtype == torch.bfloat16:
        d.dtype = RA_BF16
    else:
        raise TypeError(f"{name}: dtype {t.dtype} (want float32 or bfloat16)")
    if t.numel() and t.is_cuda == host:
        raise ValueError(f"{name} must be a {'host' if host else 'CUDA'} tensor")
    d.data = t.data_ptr() if t.numel() else None
    for i in range(4):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    if t.shape[3] <= 1:
        d.stride[3] = 1  # the stride of a size-1 dimension carries no information
    return d


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None or t.numel() == 0 else t.data_ptr()


def _outputs(q, o, lse):
    B, Hq, N, _ = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, N):
        raise ValueError("lse must be a contiguous float32 [B, Hq, N] tensor")
    return o, lse


def attn_fwd(q, k, v, causal=False, scale=None, o=None, lse=None, stream=None):
    """Exact attention: returns (o, lse).  q [B,Hq,N,D]; k, v [B,Hkv,N,D]."""
    o, lse = _outputs(q, o, lse)
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(o, "o")
    _check(lib().ra_attn_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(do),
                             _ptr(lse), int(bool(causal)), float(scale or 0.0), _stream(stream)))
    return o, lse


def attn_varlen_fwd(q, k, v, cu_seqlens, causal=False, scale=None, o=None, lse=None, stream=None):
    """Packed variable-length attention: q [1,Hq,total,D], k/v [1,Hkv,total,D];
    ``cu_seqlens`` host offsets (sequence i = rows [cu[i], cu[i+1])).  Returns (o, lse)."""
    o, lse = _outputs(q, o, lse)
    cu = (ctypes.c_int32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(o, "o")
    _check(lib().ra_attn_varlen_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                    ctypes.byref(do), _ptr(lse), ctypes.cast(cu, ctypes.c_void_p),
                                    len(cu_seqlens) - 1, int(bool(causal)), float(scale or 0.0),
                                    _stream(stream)))
    return o, lse


def attn_bwd(q, k, v, o, lse, dout, causal=False, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for the loss sum(dout * o)."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dqd = _desc(q, "q")
    need = int(lib().ra_attn_bwd_workspace_bytes(ctypes.byref(dqd)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32")
    descs = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"))]
    dd = _desc(dout, "dout")
    gq, gk, gv = _desc(dq, "dq"), _desc(dk, "dk"), _desc(dv, "dv")
    _check(lib().ra_attn_bwd(*(ctypes.byref(x) for x in descs), _ptr(lse), ctypes.byref(dd),
                             ctypes.byref(gq), ctypes.byref(gk), ctypes.byref(gv),
                             int(bool(causal)), float(scale or 0.0), _ptr(workspace),
                             _stream(stream)))
    return dq, dk, dv


def ring_sim_bwd_workspace_bytes(q, k, ring_size: int) -> int:
    """Bytes of device workspace ring_sim_bwd needs."""
    dqd, dkd = _desc(q, "q"), _desc(k, "k")
    return int(lib().ra_ring_sim_bwd_workspace_bytes(ctypes.byref(dqd), ctypes.byref(dkd), int(ring_size)))


def ring_sim_bwd(q, k, v, o, lse, dout, ring_size: int, layout: str = "zigzag", causal=True, scale=None,
                 dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of ring_sim_fwd on the ring schedule, for the loss sum(dout * o)."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = ring_sim_bwd_workspace_bytes(q, k, ring_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    elif workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32")
    descs = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"))]
    dd = _desc(dout, "dout")
    gq, gk, gv = _desc(dq, "dq"), _desc(dk, "dk"), _desc(dv, "dv")
    _check(lib().ra_ring_sim_bwd(*(ctypes.byref(x) for x in descs), _ptr(lse), ctypes.byref(dd),
                                 ctypes.byref(gq), ctypes.byref(gk), ctypes.byref(gv), int(ring_size),
                                 LAYOUTS[layout], int(bool(causal)), float(scale or 0.0), _ptr(workspace),
                                 _stream(stream)))
    return dq, dk, dv


def ring_sim_bwd_plan(N: int, ring_size: int, layout="zigzag", causal=True, step=0, kind=0):
    """Host-only schedule of one backward step: list of dicts, kind 0 = dQ, 1 = dK/dV."""
    L = lib()
    args = (int(N), int(ring_size), LAYOUTS[layout], int(bool(causal)), int(step), int(kind))
    n = L.ra_ring_sim_bwd_plan(*args, None, 0)
    if n < 0:
        raise ValueError("bad ring plan arguments")
    buf = (ctypes.c_int64 * (10 * max(n, 1)))()
    L.ra_ring_sim_bwd_plan(*args, buf, n)
    keys = ("f0", "f1", "s0a", "s1a", "s0b", "s1b", "f_rank", "s_rank", "diag", "flags")
    return [dict(zip(keys, buf[10 * i:10 * i + 10])) for i in range(n)]


def ulysses_all_to_all(x, sp: int, to_heads: bool, out=None, stream=None):
    """Sequence shards [sp, S/sp, H, D] <-> head shards [sp, S, H/sp, D] (exact copy)."""
    if out is None:
        if to_heads:
            _, ss, H, D = x.shape
            out = torch.empty((sp, ss * sp, H // sp, D), dtype=x.dtype, device=x.device)
        else:
            _, S, hs, D = x.shape
            out = torch.empty((sp, S // sp, hs * sp, D), dtype=x.dtype, device=x.device)
    _check(lib().ra_ulysses_all_to_all(ctypes.byref(_desc(x, "in")), ctypes.byref(_desc(out, "out")),
                                       int(sp), int(bool(to_heads)), _stream(stream)))
    return out


def lse_merge(o_acc, lse_acc, o_blk, lse_blk, stream=None):
    """Fold (o_blk, lse_blk) into (o_acc, lse_acc) in place."""
    da, db = _desc(o_acc, "o_acc"), _desc(o_blk, "o_blk")
    for name, t in (("lse_acc", lse_acc), ("lse_blk", lse_blk)):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous float32")
    _check(lib().ra_lse_merge(ctypes.byref(da), _ptr(lse_acc), ctypes.byref(db), _ptr(lse_blk),
                              _stream(stream)))
    return o_acc, lse_acc


def ring_sim_workspace_bytes(q, ring_size: int, k=None, v=None, o=None, layout=None, causal=False) -> int:
    """Device workspace bytes ring_sim_fwd needs: with k, v and layout, exactly that call's
    need (0 for the single pass and the fused tensor-core ring; ``o`` defaults to a tensor
    laid out like q); with q alone, the upper bound for any call with this q."""
    if k is None:
        return int(lib().ra_ring_sim_workspace_bytes(ctypes.byref(_desc(q, "q")), int(ring_size)))
    d = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v if v is not None else k, "v"),
                                  (o if o is not None else q, "o"))]
    return int(lib().ra_ring_sim_workspace_bytes_for(*(ctypes.byref(x) for x in d), int(ring_size),
                                                     LAYOUTS[layout or "contig"], int(bool(causal))))


_ws_need: dict = {}  # the exact workspace need of recent argument layouts


def _ring_ws_need(q, k, v, o, ring_size, layout, causal) -> int:
    if ring_size == 1:
        return 0
    key = (q.shape, q.stride(), q.dtype, k.shape, k.stride(), v.stride(), o.stride(),
           q.data_ptr() % 16, k.data_ptr() % 16, v.data_ptr() % 16, o.data_ptr() % 16, ring_size, layout,
           bool(causal))
    need = _ws_need.get(key)
    if need is None:
        if len(_ws_need) > 256:
            _ws_need.clear()
        need = _ws_need[key] = ring_sim_workspace_bytes(q, ring_size, k, v, o, layout, causal)
    return need


def ring_sim_fwd(q, k, v, ring_size: int, layout="contig", causal=False, scale=None, o=None,
                 lse=None, workspace=None, stream=None):
    """Ring attention over ``ring_size`` simulated ranks on one GPU: returns (o, lse)."""
    o, lse = _outputs(q, o, lse)
    need = _ring_ws_need(q, k, v, o, ring_size, layout, causal)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace is not None and workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(o, "o")
    _check(lib().ra_ring_sim_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                 ctypes.byref(do), _ptr(lse), int(ring_size), LAYOUTS[layout],
                                 int(bool(causal)), float(scale or 0.0), _ptr(workspace),
                                 _stream(stream)))
    return o, lse


def ring_sim_fwd_host_workspace_bytes(q, k, ring_size: int) -> int:
    """Device workspace bytes ring_sim_fwd_host needs (q, k: host tensors)."""
    return int(lib().ra_ring_sim_fwd_host_workspace_bytes(ctypes.byref(_desc(q, "q", host=True)),
                                                          ctypes.byref(_desc(k, "k", host=True)),
                                                          int(ring_size)))


def ring_sim_fwd_host(q, k, v, ring_size: int = 1, layout="contig", causal=False, scale=None, o=None,
                      lse=None, workspace=None, stream=None):
    """ring_sim_fwd on contiguous HOST tensors (pinned memory for asynchronous copies):
    returns host (o, lse); the results are valid once `stream` has reached the call."""
    B, Hq, N, _ = q.shape
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32).pin_memory()
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.is_cuda:
        raise ValueError("lse must be a contiguous float32 host tensor")
    need = ring_sim_fwd_host_workspace_bytes(q, k, ring_size)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    d = [_desc(t, n, host=True) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"))]
    _check(lib().ra_ring_sim_fwd_host(*(ctypes.byref(x) for x in d), _ptr(lse), int(ring_size), LAYOUTS[layout],
                                      int(bool(causal)), float(scale or 0.0), _ptr(workspace),
                                      workspace.numel(), _stream(stream)))
    return o, lse


def ring_sim_plan(N: int, ring_size: int, layout="contig", causal=False, step=0):
    """Host-only schedule of one step: list of dicts (q0, q1, k ranges, flags, rank)."""
    L = lib()
    n = L.ra_ring_sim_plan(int(N), int(ring_size), LAYOUTS[layout], int(bool(causal)), int(step),
                           None, 0)
    if n < 0:
        raise ValueError("bad ring plan arguments")
    buf = (ctypes.c_int64 * (12 * max(n, 1)))()
    L.ra_ring_sim_plan(int(N), int(ring_size), LAYOUTS[layout], int(bool(causal)), int(step),
                       ctypes.cast(buf, ctypes.c_void_p), n)
    out = []
    for i in range(n):
        q0, q1, ka0, ka1, kb0, kb1, flags, rank, q_rank, kv_rank, diag, rs = buf[12 * i:12 * i + 12]
        ranges = [(ka0, ka1)] + ([(kb0, kb1)] if kb1 > kb0 else [])
        out.append({"q": (q0, q1), "kv": ranges, "flags": flags, "rank": rank, "q_rank": q_rank,
                    "kv_rank": kv_rank, "diag": diag, "rs": rs})
    return out


def check(stream=None):
    """Synchronise and raise if a kernel recorded a device-side error (e.g. a wait timeout)."""
    _check(lib().ra_check_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int):
    lib().ra_debug_set_wait_limit_ns(int(ns))


def set_producer_delay_ns(ns: int):
    """The tensor-core kernels' TMA producers pause ns before their first copy (0: none)."""
    lib().ra_debug_set_producer_delay_ns(int(ns))


def fail_next_launches(n: int):
    """The calling thread's next n kernel launches fail on the host (RA_ERR_CUDA)."""
    lib().ra_debug_fail_next_launches(int(n))


def time_launches(enable: bool = True):
    """Time each kernel launch of this thread on its own (two CUDA events per launch)."""
    lib().ra_debug_time_launches(1 if enable else 0)


def launch_times(cap: int = 4096) -> list[tuple[str, float]]:
    """(kernel name, ms) of the launches timed since the previous read (up to cap)."""
    L = lib()
    ms = (ctypes.c_float * cap)()
    names = ctypes.create_string_buffer(32 * cap)
    n = L.ra_debug_launch_times(ctypes.cast(ms, ctypes.c_void_p), cap, ctypes.cast(names, ctypes.c_void_p), 32)
    return [(names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode(), float(ms[i])) for i in range(min(n, cap))]


def bounds_selftest(stream=None):
    """Debug builds: a bounds check that fails on purpose (ra.check() then raises
    RA_ERR_BOUNDS)."""
    _check(lib().ra_debug_bounds_selftest(_stream(stream)))


def work_counters_in_use(stream=None) -> int:
    """Synchronise the stream, then count the forward kernels' work-counter pairs that are
    not zero (0 whenever no launch is in flight; -1 on a CUDA failure)."""
    return int(lib().ra_debug_work_counters_in_use(_stream(stream)))


def wait_selftest(limit_ns: int, stream=None):
    _check(lib().ra_debug_wait_selftest(int(limit_ns), _stream(stream)))


def launch_count(reset=False) -> int:
    return int(lib().ra_launch_count(1 if reset else 0))


def version() -> int:
    return int(lib().ra_version())


def host_group_bounds(hkv: int, ng: int, copy_bound: bool) -> list[int]:
    """Boundaries (in KV heads) of the host-buffer call's head groups (diagnostic)."""
    out = (ctypes.c_int64 * (ng + 1))()
    n = lib().ra_debug_host_group_bounds(int(hkv), int(ng), 1 if copy_bound else 0, ctypes.cast(out, ctypes.c_void_p))
    if n < 0:
        raise ValueError("host_group_bounds: arguments out of range")
    return [int(x) for x in out]
