"""Gradients through the C ABI (ra_attn_bwd) against the fp64 gradient oracle."""
import numpy as np
import pytest
import torch

from exact_long_context_gb300 import synth
from helpers import to_oracle
from oracle import backward as ob

pytestmark = pytest.mark.gpu

# max-abs error / max(1, max |reference|): float32 arithmetic with fp32 inputs, and with
# bf16 inputs/outputs the rounding of O (inside D = rowsum(dO * O)) and of the stored
# gradients (2^-9 relative), the same bound as the forward's bf16 output.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


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
    (1, 2, 1, 50, 32, True, torch.bfloat16),
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
        got = got.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        err = np.max(np.abs(got - ref)) / max(1.0, np.max(np.abs(ref)))
        assert err <= TOL[dtype], f"{name}: scaled max-abs error {err:.3e}"
        print(case, name, f"{err:.2e}")


def test_backward_empty_and_errors(ra):
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 0, device="cuda")
    ra.attn_bwd(q, q, q, q, lse, q, causal=True)
    ra.check()
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 8, device="cuda")
    with pytest.raises(ra.RaError):
        ra.attn_bwd(q, q, q, q, lse, q.float(), causal=True)  # dtype mismatch
