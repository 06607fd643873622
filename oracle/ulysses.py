"""The Ulysses all-to-all over sp ranks, written as the exchange itself.  TEST
INFRASTRUCTURE ONLY.

"序列并行与 Ring Attention：超长上下文训练技术解析", section "1. Ulysses (All-to-All)":
each rank starts with a sequence shard holding every head; the all-to-all scatters the
head axis and gathers the sequence axis, after which rank r holds heads
[r H/sp, (r+1) H/sp) for the whole sequence; the inverse exchange undoes it.
"""
from __future__ import annotations

import numpy as np


def seq_to_heads(x, sp: int):
    """[sp, S/sp, H, D] sequence shards -> [sp, S, H/sp, D] head shards."""
    x = np.asarray(x)
    n_ranks, ss, H, D = x.shape
    assert n_ranks == sp and H % sp == 0
    hs = H // sp
    out = np.empty((sp, sp * ss, hs, D), dtype=x.dtype)
    for dst in range(sp):            # every receiving rank ...
        for src in range(sp):        # ... gets, from every sending rank, its head slice
            out[dst, src * ss:(src + 1) * ss] = x[src, :, dst * hs:(dst + 1) * hs]
    return out


def heads_to_seq(y, sp: int):
    """The inverse: [sp, S, H/sp, D] head shards -> [sp, S/sp, H, D] sequence shards."""
    y = np.asarray(y)
    n_ranks, S, hs, D = y.shape
    assert n_ranks == sp and S % sp == 0
    ss = S // sp
    out = np.empty((sp, ss, hs * sp, D), dtype=y.dtype)
    for dst in range(sp):
        for src in range(sp):
            out[dst, :, src * hs:(src + 1) * hs] = y[src, dst * ss:(dst + 1) * ss]
    return out
