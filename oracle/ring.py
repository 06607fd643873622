"""fp64 restatement of ring attention over R simulated ranks.  TEST INFRASTRUCTURE ONLY.

Used for invariant tests (ring result == single pass; contiguous == zigzag), never as
the parity target of the GPU path (that is :func:`oracle.attention`).  It is written
with numpy matrix products and masks and shares no code with ``oracle.c``.

Partitions
- contiguous: rank r holds rows [r*c, (r+1)*c) with c = N / R
  ("Ring Attention" glossary page (ultralytics.com), section on how ring attention
  works: the sequence is cut into one block per device).
- zigzag: the sequence is cut into 2R chunks of N / (2R) rows; rank r holds chunk r
  and chunk 2R-1-r ("序列并行与 Ring Attention：超长上下文训练技术解析",
  section "2. ZigZag Ring Attention").
- striped: rank r holds positions r, r + R, r + 2R, ... (tokens spread evenly over the
  devices: Striped Attention, named on the glossary page).

Ring schedule: at step s, rank r holds the keys/values of rank (r - s) mod R (the
worked example of the glossary page; the `ring_attention_forward` listing of
"Ring Attention 论文解析" sends to r+1 and receives from r-1).

Per step, rank r computes the unnormalised partial of its queries against the held
block, with the causal rule on global positions (the `ring_attention_causal_step`
listing of "Ring Attention 论文解析": later blocks skipped, the same block masked
above the diagonal, earlier blocks unmasked), turns it into (o, lse), and folds it
into its running result with the sigmoid-form merge of the Twinkle page.
"""
from __future__ import annotations

import numpy as np

from .merge import merge_sigmoid

CONTIG = "contig"
ZIGZAG = "zigzag"
STRIPED = "striped"


def rank_ranges(N: int, R: int, layout: str):
    """Row ranges [(start, end), ...] held by each rank, in increasing position."""
    if layout == CONTIG:
        if N % R:
            raise ValueError("contiguous layout needs N % R == 0")
        c = N // R
        return [[(r * c, (r + 1) * c)] for r in range(R)]
    if layout == ZIGZAG:
        if N % (2 * R):
            raise ValueError("zigzag layout needs N % (2R) == 0")
        h = N // (2 * R)
        return [[(r * h, (r + 1) * h), ((2 * R - 1 - r) * h, (2 * R - r) * h)] for r in range(R)]
    raise ValueError(layout)


def rank_positions(N: int, R: int, layout: str):
    """Sequence positions held by each rank (increasing)."""
    if layout == STRIPED:
        if N % R:
            raise ValueError("striped layout needs N % R == 0")
        return [np.arange(r, N, R) for r in range(R)]
    return [_positions(rr) for rr in rank_ranges(N, R, layout)]


def kv_source(r: int, s: int, R: int) -> int:
    """Rank whose key/value block rank r holds at step s."""
    return (r - s) % R


def _positions(ranges):
    return np.concatenate([np.arange(a, b) for a, b in ranges]) if ranges else np.zeros(0, int)


def step_partial(q, k, v, qpos, kpos, causal: bool, scale: float):
    """Partial (o, lse) of query rows qpos against key rows kpos, one (b, h) slice.

    q [N, D], k [N, D], v [N, D] fp64.  Rows with no visible key get the identity.
    """
    scores = scale * (q[qpos] @ k[kpos].T)
    visible = np.ones(scores.shape, bool)
    if causal:
        visible = kpos[None, :] <= qpos[:, None]
    masked = np.where(visible, scores, -np.inf)
    block_max = masked.max(axis=1)
    any_vis = visible.any(axis=1)
    shift = np.where(any_vis, block_max, 0.0)
    e = np.where(visible, np.exp(masked - shift[:, None]), 0.0)
    block_sum = e.sum(axis=1)
    block_out = e @ v[kpos]
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(any_vis[:, None], block_out / np.where(any_vis, block_sum, 1.0)[:, None], 0.0)
        lse = np.where(any_vis, shift + np.log(np.where(any_vis, block_sum, 1.0)), -np.inf)
    return o, lse


def ring_forward(q, k, v, R: int, layout: str, causal: bool, scale: float | None = None):
    """Ring attention over R simulated ranks.  q [B,Hq,N,D], k/v [B,Hkv,N,D] (fp64 view).

    Returns o [B,Hq,N,D] and lse [B,Hq,N] in natural sequence order.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    positions = rank_positions(N, R, layout)
    o_all = np.zeros((B, Hq, N, D))
    lse_all = np.full((B, Hq, N), -np.inf)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for r in range(R):
                qpos = positions[r]
                out = np.zeros((len(qpos), D))
                lse = np.full(len(qpos), -np.inf)
                for s in range(R):
                    kpos = positions[kv_source(r, s, R)]
                    bo, bl = step_partial(q[b, h], k[b, hk], v[b, hk], qpos, kpos, causal, scale)
                    out, lse = merge_sigmoid(out, lse, bo, bl)
                o_all[b, h, qpos] = out
                lse_all[b, h, qpos] = lse
    return o_all, lse_all


def zigzag_step_case(r: int, s: int, R: int) -> str:
    """The three forward cases of the zigzag ring on the Twinkle page.

    'local'      step 0: the rank's own chunks, causal
    'front_kv'   0 < s <= r: every query row against the front chunk of the held block
    'back_q'     s > r: only the back query chunk, against the whole held block
    """
    if s == 0:
        return "local"
    return "front_kv" if s <= r else "back_q"
