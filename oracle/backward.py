"""Gradients of exact attention, fp64.  TEST INFRASTRUCTURE ONLY.

For the loss L = sum(dO * O) with O = softmax(scale Q K^T (+ mask)) V, the gradients are
written out as in the `ring_attention_backward` listing of "Ring Attention 论文解析：
在分布式环境中实现无限上下文窗口训练" (there per ring step; here for the whole key axis,
which is the sum of those per-block terms):

    D_i   = sum_t dO[i,t] O[i,t]
    P_ij  = exp(s_ij - LSE_i)                (s_ij = scale q_i . k_j, visible pairs only)
    dV_j  = sum_i P_ij dO_i
    dP_ij = dO_i . v_j
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale sum_j dS_ij k_j
    dK_j  = scale sum_i dS_ij q_i

With grouped KV heads (query head h reads KV head h // G) dK and dV of a KV head are
the sums over its G query heads.  O and LSE are computed here from the definition, so
the result is the exact gradient of the exact attention.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def attention_bwd(q, k, v, do, causal: bool, scale: float | None = None):
    """Returns (dq [B,Hq,N,D], dk [B,Hkv,N,D], dv [B,Hkv,N,D], o, lse) in fp64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    vis = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.full((B, Hq, N), -np.inf)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            s = scale * (q[b, h] @ k[b, hk].T)
            s = np.where(vis, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.where(vis, np.exp(s - m), 0.0)
            z = e.sum(axis=1, keepdims=True)
            lse_bh = (m + np.log(z))[:, 0]
            o_bh = (e / z) @ v[b, hk]
            p = np.where(vis, np.exp(s - lse_bh[:, None]), 0.0)
            d_i = np.sum(do[b, h] * o_bh, axis=1)
            dv[b, hk] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, hk].T
            ds = p * (dp - d_i[:, None])
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
            o[b, h] = o_bh
            lse[b, h] = lse_bh
    return dq, dk, dv, o, lse


def ring_backward(q, k, v, do, R: int, layout: str, causal: bool, scale: float | None = None,
                  steps: bool = False):
    """Gradients on the ring schedule of R simulated ranks.  fp64.

    The `ring_attention_backward` listing of "Ring Attention 论文解析" keeps dQ on the
    query's rank and, at step s, computes rank r's block gradients against the
    key/value block it holds, that of rank j = (r - s) mod R, with the forward's
    saved LSE and D = rowsum(dO * O); the block's dK / dV go back to rank j, which sums
    them.  The forward's causal rule on global positions applies to every block (the
    listing shows no mask; the gradient of the causal forward needs it).  O and LSE are
    the ring forward's.

    Returns (dq, dk, dv), and with ``steps=True`` also a list over steps of each step's
    (dq, dk, dv) contributions (full-size arrays, zero where the step adds nothing).
    """
    from .ring import kv_source, rank_positions, ring_forward

    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o, lse = ring_forward(q, k, v, R, layout, causal, scale)
    dvec = np.sum(do * o, axis=-1)
    positions = rank_positions(N, R, layout)
    per_step = []
    for s in range(R):
        dq_s = np.zeros_like(q)
        dk_s = np.zeros_like(k)
        dv_s = np.zeros_like(v)
        for r in range(R):
            j = kv_source(r, s, R)
            qpos, kpos = positions[r], positions[j]
            vis = (kpos[None, :] <= qpos[:, None]) if causal else np.ones((len(qpos), len(kpos)), bool)
            for b in range(B):
                for h in range(Hq):
                    hk = h // G
                    sc = scale * (q[b, h, qpos] @ k[b, hk, kpos].T)
                    p = np.where(vis, np.exp(np.where(vis, sc, 0.0) - lse[b, h, qpos][:, None]), 0.0)
                    dp = do[b, h, qpos] @ v[b, hk, kpos].T
                    ds = p * (dp - dvec[b, h, qpos][:, None])
                    dq_s[b, h, qpos] += scale * (ds @ k[b, hk, kpos])
                    dk_s[b, hk, kpos] += scale * (ds.T @ q[b, h, qpos])
                    dv_s[b, hk, kpos] += p.T @ do[b, h, qpos]
        per_step.append((dq_s, dk_s, dv_s))
    dq = sum(x[0] for x in per_step)
    dk = sum(x[1] for x in per_step)
    dv = sum(x[2] for x in per_step)
    if steps:
        return dq, dk, dv, per_step
    return dq, dk, dv


def gradient_rows(q, k, v, do, causal: bool, scale: float | None = None, q_rows=None, kv_rows=None,
                  nthreads: int | None = None):
    """Selected rows of the gradients, each from its definition, for problems too large
    for :func:`attention_bwd`.

    q_rows: (b, h, i) triples -> dq rows [n, D]; kv_rows: (b, hk, j) triples -> dk and dv
    rows [m, D].  The forward rows a gradient row needs (row i itself for dQ_i; every
    row of the G query heads that sees key j for dK_j, dV_j) come from the attention
    oracle; then, per the formulas above, with D_i = dO_i . O_i:
        dQ_i = scale sum_j P_ij (dO_i . v_j - D_i) k_j
        dK_j = scale sum_i P_ij (dO_i . v_j - D_i) q_i,   dV_j = sum_i P_ij dO_i.
    Returns (dq_rows, dk_rows, dv_rows) (None for an empty selection).
    """
    from . import attention

    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, D = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q_rows = np.zeros((0, 3), np.int64) if q_rows is None else np.asarray(q_rows, np.int64).reshape(-1, 3)
    kv_rows = np.zeros((0, 3), np.int64) if kv_rows is None else np.asarray(kv_rows, np.int64).reshape(-1, 3)
    need = set(map(tuple, q_rows.tolist()))
    for b, hk, j in kv_rows.tolist():
        lo = j if causal else 0
        for h in range(hk * G, (hk + 1) * G):
            need.update((b, h, i) for i in range(lo, N))
    need = sorted(need)
    fwd = {}
    if need:
        o_r, l_r = attention(q, k, v, causal, scale, rows=np.array(need, np.int64), nthreads=nthreads)
        for n_, key in enumerate(need):
            fwd[key] = (o_r[n_], l_r[n_])
    dq_out = None
    if len(q_rows):
        dq_out = np.zeros((len(q_rows), D))
        for n_, (b, h, i) in enumerate(q_rows.tolist()):
            hk = h // G
            o_i, lse_i = fwd[(b, h, i)]
            hi = i + 1 if causal else N
            p = np.exp(scale * (kf[b, hk, :hi] @ qf[b, h, i]) - lse_i)
            ds = p * (vf[b, hk, :hi] @ dof[b, h, i] - dof[b, h, i] @ o_i)
            dq_out[n_] = scale * (ds @ kf[b, hk, :hi])
    dk_out = dv_out = None
    if len(kv_rows):
        dk_out = np.zeros((len(kv_rows), D))
        dv_out = np.zeros((len(kv_rows), D))
        for n_, (b, hk, j) in enumerate(kv_rows.tolist()):
            lo = j if causal else 0
            for h in range(hk * G, (hk + 1) * G):
                idx = range(lo, N)
                o_i = np.array([fwd[(b, h, i)][0] for i in idx]).reshape(-1, D)
                lse_i = np.array([fwd[(b, h, i)][1] for i in idx])
                p = np.exp(scale * (qf[b, h, lo:] @ kf[b, hk, j]) - lse_i)
                ds = p * (dof[b, h, lo:] @ vf[b, hk, j] - np.sum(dof[b, h, lo:] * o_i, axis=1))
                dk_out[n_] += scale * (ds @ qf[b, h, lo:])
                dv_out[n_] += p @ dof[b, h, lo:]
    return dq_out, dk_out, dv_out
