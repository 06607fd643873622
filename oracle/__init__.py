"""The oracle: a plain, slow, obviously correct fp64 CPU statement of exact attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

Contents
- :func:`attention`     - softmax(scale * Q K^T) V and the per-row natural-log LSE,
                          row by row in C (``oracle.c``), two passes per row.
- :func:`attention_varlen` - the same per sequence of a packed batch (``cu_seqlens``).
- :mod:`oracle.merge`   - the log-sum-exp merge of two partial results.
- :mod:`oracle.ring`    - an fp64 restatement of the ring of KV-block passes
                          (contiguous / zigzag partitions), used only for invariants.

Inputs are numpy arrays laid out [B, H, N, D] (contiguous copies are taken):
float32, float64, or uint16 holding bfloat16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def library_path(plant: int = 0) -> str:
    name = "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so"
    return os.path.join(_BUILD, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile oracle.c with gcc (plain -O2, IEEE arithmetic, no fast-math)."""
    out = library_path(plant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", f"-DORACLE_PLANT={plant}",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(plant: int = 0) -> ctypes.CDLL:
    with _lock:
        lib = _libs.get(plant)
        if lib is None:
            lib = ctypes.CDLL(build(plant))
            f = lib.oracle_attention_rows
            f.restype = ctypes.c_int
            i64 = ctypes.c_int64
            f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                          i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double, i64, i64,
                          ctypes.c_void_p, i64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_plant.restype = ctypes.c_int
            _libs[plant] = lib
        return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 2
    raise TypeError(f"oracle input dtype {a.dtype} (want float32, float64 or uint16 bf16 bits)")


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def attention(q, k, v, causal: bool, scale: float | None = None, kv_lo: int = 0,
              kv_hi: int | None = None, rows=None, nthreads: int | None = None, plant: int = 0):
    """Exact attention in fp64.

    q: [B, Hq, N, D]; k, v: [B, Hkv, N, D] with Hq % Hkv == 0; query head h reads KV
    head h // (Hq // Hkv).  ``scale`` None means 1/sqrt(D).  Keys outside
    [kv_lo, kv_hi) are invisible; with ``causal`` key j is visible to row i iff j <= i.
    ``rows``: None for every row (returns o [B,Hq,N,D], lse [B,Hq,N]) or an int array
    of shape [R, 3] of (b, h, i) triples (returns o [R, D], lse [R]).
    A row with no visible key gets o = 0, lse = -inf.
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    code = _dtype_code(q)
    if _dtype_code(k) != code or _dtype_code(v) != code:
        raise TypeError("q, k, v must share one dtype")
    B, Hq, N, D = q.shape
    Bk, Hkv, Nk, Dk = k.shape
    if (Bk, Nk, Dk) != (B, N, D) or v.shape != k.shape or Hq % Hkv:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if kv_hi is None:
        kv_hi = N
    if rows is None:
        nrows = B * Hq * N
        rows_arr = None
        o = np.empty((B, Hq, N, D), np.float64)
        lse = np.empty((B, Hq, N), np.float64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        nrows = rows_arr.shape[0]
        o = np.empty((nrows, D), np.float64)
        lse = np.empty((nrows,), np.float64)
    lib = _load(plant)
    rc = lib.oracle_attention_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, code, B, Hq, Hkv, N, D, int(bool(causal)),
        float(scale), int(kv_lo), int(kv_hi),
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        o.ctypes.data, lse.ctypes.data, int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return o, lse


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, round-to-nearest-even, returned as uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(a)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def attention_varlen(q, k, v, cu_seqlens, causal: bool, scale: float | None = None,
                     nthreads: int | None = None, plant: int = 0):
    """Exact attention over a packed batch: sequence i = rows [cu[i], cu[i+1]) of the
    packed axis of q [1,Hq,T,D], k/v [1,Hkv,T,D]; a row sees only keys of its own sequence
    (and j <= i when causal).  Rows outside every sequence: o = 0, lse = -inf.

    Each sequence is the plain definition over its own rows and keys: the key window
    of :func:`attention` restricted to the sequence.
    """
    q = np.ascontiguousarray(q)
    B, Hq, T, D = q.shape
    if B != 1:
        raise ValueError("packed batches have B == 1")
    o = np.zeros((B, Hq, T, D), np.float64)
    lse = np.full((B, Hq, T), -np.inf)
    cu = [int(x) for x in cu_seqlens]
    for i in range(len(cu) - 1):
        a, b = cu[i], cu[i + 1]
        if b <= a:
            continue
        rows = np.array([(0, h, r) for h in range(Hq) for r in range(a, b)], dtype=np.int64)
        oi, li = attention(q, k, v, causal, scale, kv_lo=a, kv_hi=b, rows=rows,
                           nthreads=nthreads, plant=plant)
        o[0, rows[:, 1], rows[:, 2]] = oi
        lse[0, rows[:, 1], rows[:, 2]] = li
    return o, lse
