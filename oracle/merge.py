"""Log-sum-exp merge of two partial attention results, fp64.  TEST INFRASTRUCTURE ONLY.

A partial over a key set A is (o_A, lse_A) with
    o_A   = sum_{j in A} e^{s_j} v_j / sum_{j in A} e^{s_j}
    lse_A = ln sum_{j in A} e^{s_j}.
For disjoint A and B the partial over A u B is, by the definition above,
    lse = ln(e^{lse_A} + e^{lse_B})
    o   = (e^{lse_A} o_A + e^{lse_B} o_B) / e^{lse}.
The identity partial (empty key set) is (o = 0, lse = -inf); merging with it
changes nothing, and merging two identities gives the identity.

:func:`merge` writes that definition out with numpy's ``logaddexp``.
:func:`merge_sigmoid` is the sigmoid / log-sigmoid form of ``update_out_and_lse``
from "序列并行与 Ring Attention：超长上下文训练技术解析", section
"前向传播：ZigZag Ring FlashAttention"; it is the same quantity for finite
LSEs, and the identity element is handled explicitly (the page's form would
produce NaN from -inf - (-inf)).
"""
from __future__ import annotations

import numpy as np


def merge(o_a, lse_a, o_b, lse_b):
    """Merge partials: o_* [..., D], lse_* [...] (fp64).  Returns (o, lse)."""
    o_a = np.asarray(o_a, np.float64)
    o_b = np.asarray(o_b, np.float64)
    lse_a = np.asarray(lse_a, np.float64)
    lse_b = np.asarray(lse_b, np.float64)
    lse = np.logaddexp(lse_a, lse_b)
    empty = np.isneginf(lse)
    safe = np.where(empty, 0.0, lse)
    w_a = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - safe))
    w_b = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - safe))
    o = w_a[..., None] * o_a + w_b[..., None] * o_b
    o = np.where(empty[..., None], 0.0, o)
    return o, lse


def _log_sigmoid(x):
    return -np.logaddexp(0.0, -x)


def merge_sigmoid(o, lse, block_o, block_lse):
    """The page's sigmoid form: o <- o - sigma(lse_b - lse)(o - o_b); lse <- lse - log sigma(lse - lse_b)."""
    o = np.asarray(o, np.float64)
    block_o = np.asarray(block_o, np.float64)
    lse = np.asarray(lse, np.float64)
    block_lse = np.asarray(block_lse, np.float64)
    a_empty = np.isneginf(lse)
    b_empty = np.isneginf(block_lse)
    both = ~(a_empty | b_empty)
    la = np.where(both, lse, 0.0)
    lb = np.where(both, block_lse, 0.0)
    sig = 1.0 / (1.0 + np.exp(-(lb - la)))
    o_new = o - sig[..., None] * (o - block_o)
    lse_new = la - _log_sigmoid(la - lb)
    o_out = np.where(both[..., None], o_new, np.where(a_empty[..., None], block_o, o))
    lse_out = np.where(both, lse_new, np.where(a_empty, block_lse, lse))
    return o_out, lse_out
