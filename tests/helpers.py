"""Shared test helpers: moving tensors to the oracle, sampling rows, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_long_context_gb300 import synth

# GPU-vs-oracle tolerances: bf16 inputs: max-abs on O <= 2e-2, LSE |d| <= 1e-3 max(1, |lse|);
# float32 inputs (CUDA-core path): max-abs <= 1e-5 on both.
BF16_O_TOL = 2e-2
BF16_LSE_REL = 1e-3
F32_TOL = 1e-5


def to_oracle(t: torch.Tensor) -> np.ndarray:
    """CPU numpy copy in the oracle's input encoding (bf16 -> uint16 bit patterns)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def oracle_full(q, k, v, causal, scale=None, kv_lo=0, kv_hi=None):
    return oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), causal, scale, kv_lo, kv_hi)


def sample_rows(B, Hq, N, chunk=None, n_random=16, seed=0, heads=None):
    """(b, h, i) triples: rows 0, 1, N-1, every chunk's first and last row, random rows."""
    rng = np.random.default_rng(seed)
    base = {0, min(1, N - 1), N - 1}
    if chunk:
        for c0 in range(0, N, chunk):
            base.add(c0)
            base.add(min(N, c0 + chunk) - 1)
    rows = []
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in heads:
        extra = rng.integers(0, N, size=n_random) if n_random else []
        for i in sorted(base | {int(x) for x in extra}):
            rows.append((b, h, i))
    return np.array(rows, dtype=np.int64)


def gather_rows(o: torch.Tensor, lse: torch.Tensor, rows: np.ndarray):
    idx = torch.as_tensor(rows, device=o.device)
    og = o[idx[:, 0], idx[:, 1], idx[:, 2]].float().cpu().numpy().astype(np.float64)
    lg = lse[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy().astype(np.float64)
    return og, lg


def errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o_gpu = np.asarray(o_gpu, np.float64)
    lse_gpu = np.asarray(lse_gpu, np.float64)
    assert np.all(np.isfinite(o_gpu)), "non-finite output"
    assert np.all(np.isfinite(lse_gpu)), "non-finite LSE"
    o_err = float(np.max(np.abs(o_gpu - o_ref))) if o_gpu.size else 0.0
    d = np.abs(lse_gpu - lse_ref)
    lse_rel = float(np.max(d / np.maximum(1.0, np.abs(lse_ref)))) if d.size else 0.0
    lse_abs = float(np.max(d)) if d.size else 0.0
    return o_err, lse_rel, lse_abs


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    o_err, lse_rel, lse_abs = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    if dtype == torch.bfloat16:
        assert o_err <= BF16_O_TOL, f"{what}: O max-abs {o_err:.3e} > {BF16_O_TOL}"
        assert lse_rel <= BF16_LSE_REL, f"{what}: LSE rel {lse_rel:.3e} > {BF16_LSE_REL}"
    else:
        assert o_err <= F32_TOL, f"{what}: O max-abs {o_err:.3e} > {F32_TOL}"
        assert lse_abs <= F32_TOL, f"{what}: LSE abs {lse_abs:.3e} > {F32_TOL}"
    return o_err, lse_rel


# softmax edge cases: kind -> scale (None = 1/sqrt(D))
EDGE_SCALE = {"uniform": None, "flat": 0.01, "peaked": 4.0, "ramp_up": 1.0, "ramp_down": 1.0}


def edge_inputs(kind, B, Hq, Hkv, N, D, seed, dtype=torch.bfloat16, device="cuda"):
    """Seeded Q, K, V for a softmax edge case.  "uniform": Q = 0, every score 0, each row's
    P uniform over its visible keys.  "ramp_up" / "ramp_down": key norms grow (shrink) by
    0.25 -> 3 along the sequence, so the running maximum moves on most tiles of a walk.
    "flat" / "peaked" are the plain draw under the small / large scale of EDGE_SCALE."""
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=seed, device=device)
    if kind == "uniform":
        q = torch.zeros_like(q)
    elif kind.startswith("ramp"):
        f = torch.linspace(0.25, 3.0, N, device=device)
        if kind == "ramp_down":
            f = f.flip(0)
        k = (k.float() * f.view(1, 1, N, 1)).to(dtype)
    return q, k, v


# Gradients, three bounds (tol 1e-4 float32, 2e-2 bf16):
# - over the tensor: max-abs error / max(1, max |ref|) <= tol;
# - per row: every element's error <= tol * max(1, max |ref| of its row), so a row is held to
#   its own magnitude wherever that exceeds 1 (as strict as the tensor bound for every row);
# - in bulk: the 99.9th percentile of the element-wise error relative to its row's scale
#   (max |ref| of the row + GRAD_ROW_FLOOR * max |ref| of the tensor) <= tol.
# The floor in the last bound: the rounding of P and dS (bf16, 2^-9 relative per term) adds
# up over a row's keys in proportion to the sum of the terms' sizes, and the rounding of the
# stored O inside D = rowsum(dO * O) shifts every dS of a row by the same amount (a dQ error
# ~ scale * dD * mean(K)); both follow the tensor's scale, while the row's own gradient can
# cancel far below it (uniform or nearly one-hot softmax rows; causal row 0's dQ is 0 up to
# rounding).  On the softmax edge cases (scale 4, key norms that move the running maximum)
# that rounding, times the scale, exceeds such rows' own size: there the per-row bound is
# off (per_row=False) and the tensor and percentile bounds remain; the percentile bound
# catches an error that runs through many rows.
GRAD_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
GRAD_ROW_FLOOR = 0.1


def assert_grad_close(got, ref, dtype, what="", per_row=True):
    """Checks a gradient against its fp64 reference (rows on every axis but the last);
    returns (tensor-scaled error, worst per-row scaled error, p99.9 row-relative error)."""
    if isinstance(got, torch.Tensor):
        got = got.float().cpu().numpy()
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64).reshape(-1, ref.shape[-1])
    ref = ref.reshape(got.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    tol = GRAD_TOL[dtype]
    if got.size == 0:
        return 0.0, 0.0, 0.0
    d = np.abs(got - ref)
    rmax = np.max(np.abs(ref), axis=1, keepdims=True)
    gmax = float(np.max(rmax))
    scaled = float(np.max(d)) / max(1.0, gmax)
    assert scaled <= tol, f"{what}: scaled max-abs error {scaled:.3e} > {tol}"
    row = float(np.max(d / np.maximum(1.0, rmax)))
    assert row <= tol or not per_row, f"{what}: per-row scaled error {row:.3e} > {tol}"
    scale = rmax + GRAD_ROW_FLOOR * gmax
    rel = d / np.where(scale > 0, scale, 1.0)
    p999 = float(np.quantile(rel, 0.999))
    assert p999 <= tol, f"{what}: p99.9 row-relative error {p999:.3e} > {tol} (max {float(np.max(rel)):.2e})"
    return scaled, row, p999
