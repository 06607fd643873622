"""Packed variable-length batches (cu_seqlens) through the C ABI, against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_long_context_gb300 import synth
from helpers import assert_close, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


def _cu(lengths, lead=0):
    cu = [lead]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


CASES = [
    # lengths, leading pad, trailing pad, Hq, Hkv, D, dtype, causal
    ([1, 127, 128, 129, 0, 300, 513], 0, 37, 4, 2, 128, torch.bfloat16, True),
    ([1000, 24, 256, 255], 5, 0, 2, 2, 128, torch.bfloat16, False),
    ([200, 64, 333], 0, 11, 4, 1, 64, torch.bfloat16, True),
    ([50, 0, 77, 3], 2, 9, 2, 1, 32, torch.bfloat16, True),     # CUDA-core path
    ([40, 65, 1], 1, 4, 2, 2, 16, torch.float32, True),          # fp32 path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}seq_D{c[5]}_{str(c[6])[6:]}_{'c' if c[7] else 'n'}")
def test_varlen_matches_oracle(ra, case):
    lengths, lead, trail, Hq, Hkv, D, dtype, causal = case
    cu = _cu(lengths, lead)
    T = cu[-1] + trail
    q, k, v = synth.make_qkv(1, Hq, Hkv, T, D, dtype, seed=T, device="cuda")
    o, lse = ra.attn_varlen_fwd(q, k, v, cu, causal=causal)
    ra.check()
    o_ref, l_ref = oracle.attention_varlen(to_oracle(q), to_oracle(k), to_oracle(v), cu, causal)
    og = o.float().cpu().numpy()
    lg = lse.cpu().numpy()
    pad = np.isneginf(l_ref[0, 0])
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref)), "padding rows must have LSE = -inf"
    assert np.all(og[:, :, pad] == 0), "padding rows must have O = 0"
    real = ~pad
    assert_close(og[:, :, real], lg[:, :, real], o_ref[:, :, real], l_ref[:, :, real], dtype,
                 f"varlen {case}")


def test_varlen_equals_each_sequence_alone(ra):
    lengths = [384, 129, 1, 700]
    cu = _cu(lengths)
    q, k, v = synth.make_qkv(1, 4, 2, cu[-1], 128, torch.bfloat16, seed=3, device="cuda")
    o, lse = ra.attn_varlen_fwd(q, k, v, cu, causal=True)
    for a, b in zip(cu[:-1], cu[1:]):
        oi, li = ra.attn_fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], causal=True)
        assert torch.equal(o[:, :, a:b], oi) and torch.equal(lse[:, :, a:b], li), (a, b)
    ra.check()


def test_varlen_many_sequences_span_launches(ra):
    """More sequences than one launch's segment table (128)."""
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(1, 200, size=300)]
    cu = _cu(lengths)
    q, k, v = synth.make_qkv(1, 2, 1, cu[-1], 128, torch.bfloat16, seed=8, device="cuda")
    o, lse = ra.attn_varlen_fwd(q, k, v, cu, causal=True)
    ra.check()
    rows = []
    for i in rng.choice(len(lengths), size=20, replace=False):
        a, b = cu[i], cu[i + 1]
        for r in {a, b - 1, (a + b) // 2}:
            for h in range(2):
                rows.append((0, h, r))
    rows = np.array(rows, np.int64)
    idx = torch.as_tensor(rows, device="cuda")
    og = o[idx[:, 0], idx[:, 1], idx[:, 2]].float().cpu().numpy()
    lg = lse[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    o_ref = np.zeros((len(rows), 128))
    l_ref = np.zeros(len(rows))
    seq_of = np.searchsorted(np.array(cu), rows[:, 2], side="right") - 1
    for n, (r, s) in enumerate(zip(rows, seq_of)):
        oi, li = oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), True, None,
                                  kv_lo=cu[s], kv_hi=cu[s + 1], rows=[r])
        o_ref[n], l_ref[n] = oi[0], li[0]
    assert_close(og, lg, o_ref, l_ref, torch.bfloat16, "300 sequences")


@pytest.mark.parametrize("cu", [[0], [3, 3, 3], [0, 0, 8]], ids=["no_sequences", "empty_sequences", "one_sequence_all_rows"])
def test_varlen_degenerate_tables(ra, cu):
    """No sequences, only empty ones (every row is padding: O = 0, LSE = -inf), and one
    sequence over the whole packed length (the single pass, bit for bit)."""
    T = 8
    q, k, v = synth.make_qkv(1, 2, 1, T, 128, torch.bfloat16, seed=12, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 2, T), 7.0, device="cuda")
    o, lse = ra.attn_varlen_fwd(q, k, v, cu, causal=True, o=o, lse=lse)
    ra.check()
    covered = torch.zeros(T, dtype=torch.bool)
    for a, b in zip(cu[:-1], cu[1:]):
        covered[a:b] = True
    pad = (~covered).nonzero().flatten().tolist()
    assert torch.all(o[:, :, pad] == 0).item()
    assert torch.all(torch.isneginf(lse[:, :, pad])).item()
    if covered.all():
        o1, l1 = ra.attn_fwd(q, k, v, causal=True)
        ra.check()
        assert torch.equal(o, o1) and torch.equal(lse, l1)
