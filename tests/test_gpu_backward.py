"""Gradients through the C ABI (ra_attn_bwd) against the fp64 gradient oracle."""
import numpy as np
import pytest
import torch

from exact_long_context_gb300 import synth
from helpers import EDGE_SCALE, assert_grad_close, edge_inputs, to_oracle
from oracle import backward as ob

pytestmark = pytest.mark.gpu

# Tolerances (helpers.assert_grad_close): max-abs error / max(1, max |reference|) over the
# tensor and, per row, against the row's own magnitude.  float32 arithmetic with fp32 inputs;
# with bf16 inputs/outputs the rounding of O (inside D = rowsum(dO * O)), of P and dS before
# the tensor-core products and of the stored gradients (2^-9 relative), the same bound as
# the forward's bf16 output.


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


CASES = [
    # B, Hq, Hkv, N, D, causal, dtype
    (1, 1, 1, 1, 16, True, torch.float32),
    (1, 2, 1, 33, 16, True, torch.float32),
    (2, 2, 2, 70, 64, False, torch.float32),
    (1, 4, 2, 129, 128, True, torch.float32),
    (1, 2, 2, 128, 128, True, torch.bfloat16),
    (1, 4, 1, 200, 128, True, torch.bfloat16),
    (2, 2, 2, 96, 64, False, torch.bfloat16),
    (1, 2, 1, 50, 32, True, torch.bfloat16),     # CUDA-core path (D = 32)
    (1, 4, 2, 1000, 128, True, torch.bfloat16),  # tensor cores: ragged tail, GQA
    (1, 2, 2, 512, 64, True, torch.bfloat16),
    (2, 2, 1, 384, 128, False, torch.bfloat16),
    # fewer rows than a warp's D-pass span, and one row per head (non-causal: under causality
    # row 0 sees one key, its exact dQ is 0 and only the bf16 rounding of O inside D is left)
    (2, 3, 3, 3, 64, False, torch.bfloat16),
    (3, 2, 1, 1, 128, False, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}-{c[2]}N{c[3]}D{c[4]}{'c' if c[5] else 'n'}{str(c[6])[6:]}")
def test_backward_matches_oracle(ra, case):
    B, Hq, Hkv, N, D, causal, dtype = case
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=N * 7 + D, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(N + 1)
    dout = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(dtype)
    o, lse = ra.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = ra.attn_bwd(q, k, v, o, lse, dout, causal=causal)
    ra.check()
    rq, rk, rv, _, _ = ob.attention_bwd(to_oracle(q), to_oracle(k), to_oracle(v), to_oracle(dout),
                                        causal)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        scaled, row, p999 = assert_grad_close(got, ref, dtype, name)
        print(case, name, f"scaled {scaled:.2e} row {row:.2e} p99.9 {p999:.2e}")


def test_backward_tensor_cores_match_cuda_cores(ra):
    """Same values through the tensor-core kernels (aligned) and the CUDA-core kernels
    (rows of 136 elements viewed as 128: strides not 16-byte multiples)."""
    B, Hq, Hkv, N, D = 1, 4, 2, 700, 128
    g = torch.Generator(device="cuda").manual_seed(4)
    raw = torch.randn(4, B, Hq, N, 136, generator=g, device="cuda").to(torch.bfloat16)
    q_u, do_u = raw[0][..., :D], raw[3][..., :D]
    k_u, v_u = raw[1][:, :Hkv, :, :D], raw[2][:, :Hkv, :, :D]
    q, k, v, do = (t.contiguous() for t in (q_u, k_u, v_u, do_u))
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    a = ra.attn_bwd(q, k, v, o, lse, do, causal=True)
    o_u = torch.empty(B, Hq, N, 136, dtype=torch.bfloat16, device="cuda")[..., :D]
    o_u.copy_(o)
    bq = torch.empty_like(raw[0])[..., :D]
    bk = torch.empty(B, Hkv, N, 136, dtype=torch.bfloat16, device="cuda")[..., :D]
    bv = torch.empty(B, Hkv, N, 136, dtype=torch.bfloat16, device="cuda")[..., :D]
    c = ra.attn_bwd(q_u, k_u, v_u, o_u, lse, do_u, causal=True, dq=bq, dk=bk, dv=bv)
    ra.check()
    for x, y, name in zip(a, c, ("dq", "dk", "dv")):
        err = (x.float() - y.float()).abs().max().item() / max(1.0, y.float().abs().max().item())
        assert err <= 2e-2, (name, err)


def test_backward_every_tile_runs_once_in_head_groups(ra):
    """A whole-sequence backward whose tiles go in head groups of single tiles from the
    kernels' work counters (dQ: groups of 12 and 4 query heads across the two batches;
    dK/dV: groups of 3, 3 and 2 (batch, KV head) units): gradients start as NaN and must all
    be written, sampled rows match the oracle, and every counter pair is back to zero."""
    B, Hq, Hkv, N, D = 2, 8, 4, 16384, 128
    dtype = torch.bfloat16
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=61, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(62)
    dout = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(dtype)
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    ra.attn_bwd(q, k, v, o, lse, dout, causal=True, dq=dq, dk=dk, dv=dv)
    ra.check()
    assert ra.work_counters_in_use() == 0
    for t in (dq, dk, dv):
        assert not torch.isnan(t).any().item()
    rng = np.random.default_rng(63)
    q_rows = np.array([(int(b), int(h), int(i)) for b, h, i in
                       zip(rng.integers(0, B, 6), rng.integers(0, Hq, 6), rng.integers(0, N, 6))]
                      + [(0, 0, 0), (1, Hq - 1, N - 1), (1, 4, 127), (0, 7, 128)])
    # keys near the end (few rows see them, so the oracle stays quick) in every group
    kv_rows = np.array([(b, hk, j) for b in range(B) for hk in range(Hkv) for j in (N - 1, N - 129 - hk)])
    args = [to_oracle(t) for t in (q, k, v, dout)]
    rq, rk, rv = ob.gradient_rows(*args, True, None, q_rows, kv_rows)
    for name, got, rows, ref in (("dq", dq, q_rows, rq), ("dk", dk, kv_rows, rk), ("dv", dv, kv_rows, rv)):
        sel = got[rows[:, 0], rows[:, 1], rows[:, 2]].float().cpu().numpy().astype(np.float64)
        scaled, row, p999 = assert_grad_close(sel, ref, dtype, f"{name} sampled")
        print(name, f"sampled: scaled {scaled:.2e} row {row:.2e} p99.9 {p999:.2e}")


def test_backward_empty_and_errors(ra):
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 0, device="cuda")
    ra.attn_bwd(q, q, q, q, lse, q, causal=True)
    ra.check()
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 8, device="cuda")
    with pytest.raises(ra.RaError):
        ra.attn_bwd(q, q, q, q, lse, q.float(), causal=True)  # dtype mismatch


@pytest.mark.parametrize("kind", ["uniform", "peaked", "ramp_up", "ramp_down"])
def test_backward_edge_cases(ra, kind):
    """Gradients on the softmax edge cases (scores all 0, very peaked, a running maximum
    that moves along the walk) through the single pass and the zigzag and striped ring
    schedules, with three query heads per KV head, against the fp64 gradients."""
    B, Hq, Hkv, N, D = 1, 6, 2, 768, 128
    scale = EDGE_SCALE[kind]
    q, k, v = edge_inputs(kind, B, Hq, Hkv, N, D, seed=43)
    g = torch.Generator(device="cuda").manual_seed(44)
    dout = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(torch.bfloat16)
    o, lse = ra.attn_fwd(q, k, v, causal=True, scale=scale)
    ref = ob.attention_bwd(to_oracle(q), to_oracle(k), to_oracle(v), to_oracle(dout), True, scale)[:3]
    runs = [("single pass", lambda: ra.attn_bwd(q, k, v, o, lse, dout, causal=True, scale=scale))]
    for R, layout in ((2, "zigzag"), (4, "striped")):
        runs.append((f"{layout} R{R}", lambda R=R, layout=layout:
                     ra.ring_sim_bwd(q, k, v, o, lse, dout, R, layout, True, scale=scale)))
    for run, fn in runs:
        grads = fn()
        ra.check()
        for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
            # nearly one-hot or uniform rows: per-row bound off (see helpers.assert_grad_close)
            scaled, row, p999 = assert_grad_close(got, r, torch.bfloat16, f"{kind} {run} {name}", per_row=False)
            print(kind, run, name, f"scaled {scaled:.2e} row {row:.2e} p99.9 {p999:.2e}")
