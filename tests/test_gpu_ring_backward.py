"""Ring-scheduled gradients through the C ABI (ra_ring_sim_bwd) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_long_context_gb300 import synth
from helpers import GRAD_TOL, assert_grad_close, to_oracle
from oracle import backward as ob

pytestmark = pytest.mark.gpu

# Tolerances as for ra_attn_bwd (helpers.assert_grad_close): max-abs error / max(1, max
# |reference|) over the tensor and, per row, against the row's own magnitude.


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


def _inputs(B, Hq, Hkv, N, D, dtype, seed):
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dout = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(dtype)
    return q, k, v, dout


CASES = [
    # B, Hq, Hkv, N, D, R, layout, causal, dtype
    (1, 2, 1, 64, 16, 4, "zigzag", True, torch.float32),      # worked-example sized chunks of 8
    (1, 2, 2, 48, 16, 3, "striped", True, torch.float32),
    (1, 2, 1, 60, 32, 3, "contig", False, torch.float32),
    (1, 4, 2, 1024, 128, 4, "zigzag", True, torch.bfloat16),  # chunks of one tile
    (1, 4, 2, 768, 128, 4, "zigzag", True, torch.bfloat16),   # chunks of 96 rows: under a tile
    (1, 2, 2, 640, 128, 2, "contig", True, torch.bfloat16),   # 320-row blocks: ragged tiles
    (1, 4, 1, 600, 128, 3, "striped", True, torch.bfloat16),  # interleave of 200
    (1, 2, 2, 516, 128, 4, "striped", True, torch.bfloat16),  # 129 per rank: key tiles no row sees
    (2, 2, 2, 512, 64, 2, "zigzag", False, torch.bfloat16),
    (1, 2, 2, 480, 64, 5, "striped", False, torch.bfloat16),
    (1, 2, 1, 96, 32, 2, "zigzag", True, torch.bfloat16),     # CUDA-core path (D = 32)
    (1, 2, 2, 2048, 128, 8, "zigzag", True, torch.bfloat16),
    (1, 2, 1, 4096, 128, 2, "zigzag", True, torch.bfloat16),  # chunks of 8 tiles, 4 blocks
    (1, 2, 2, 3072, 64, 3, "contig", True, torch.bfloat16),
    # striped ranks of whole tiles: one fused launch per kernel walks every step
    (1, 4, 2, 1536, 128, 3, "striped", True, torch.bfloat16),   # 512 per rank, GQA
    (1, 2, 2, 1024, 64, 4, "striped", True, torch.bfloat16),    # 256 per rank, D = 64
    (2, 2, 1, 768, 128, 3, "striped", False, torch.bfloat16),   # non-causal, batch 2
    (1, 2, 2, 1024, 128, 8, "striped", True, torch.bfloat16),   # one tile per rank
]


def _id(c):
    return f"B{c[0]}H{c[1]}-{c[2]}N{c[3]}D{c[4]}R{c[5]}{c[6]}{'c' if c[7] else 'n'}{str(c[8])[6:]}"


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_ring_backward_matches_oracle(ra, case):
    B, Hq, Hkv, N, D, R, layout, causal, dtype = case
    q, k, v, dout = _inputs(B, Hq, Hkv, N, D, dtype, seed=N * 3 + R)
    o, lse = ra.ring_sim_fwd(q, k, v, R, layout, causal)
    dq, dk, dv = ra.ring_sim_bwd(q, k, v, o, lse, dout, R, layout, causal)
    ra.check()
    args = [to_oracle(t) for t in (q, k, v, dout)]
    if N <= 256:
        rq, rk, rv = ob.ring_backward(*args, R, layout, causal)
    else:
        rq, rk, rv, _, _ = ob.attention_bwd(*args, causal)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        scaled, row, p999 = assert_grad_close(got, ref, dtype, name)
        print(_id(case), name, f"scaled {scaled:.2e} row {row:.2e} p99.9 {p999:.2e}")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)])
@pytest.mark.parametrize("layout", ["contig", "zigzag", "striped"])
def test_ring_size_one_is_attn_bwd(ra, dtype, D, layout):
    """One simulated rank is the whole-sequence backward, bit for bit (same kernels, one
    segment)."""
    q, k, v, dout = _inputs(1, 4, 2, 384, D, dtype, seed=5)
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    a = ra.attn_bwd(q, k, v, o, lse, dout, causal=True)
    b = ra.ring_sim_bwd(q, k, v, o, lse, dout, 1, layout, True)
    ra.check()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_ring_backward_tensor_cores_match_cuda_cores(ra):
    """The tensor-core kernels (aligned rows) and the CUDA-core kernels (rows whose
    strides are not 16-byte multiples) give the same ring gradients."""
    B, Hq, Hkv, N, D, R = 1, 4, 2, 1024, 128, 4
    q, k, v, dout = _inputs(B, Hq, Hkv, N, D, torch.bfloat16, seed=9)
    o, lse = ra.ring_sim_fwd(q, k, v, R, "zigzag", True)
    a = ra.ring_sim_bwd(q, k, v, o, lse, dout, R, "zigzag", True)

    def unaligned(t):
        buf = torch.empty(*t.shape[:3], 136, dtype=t.dtype, device=t.device)[..., :D]
        buf.copy_(t)
        return buf

    qu, ku, vu, ou, du = (unaligned(t) for t in (q, k, v, o, dout))
    b = ra.ring_sim_bwd(qu, ku, vu, ou, lse, du, R, "zigzag", True,
                        dq=unaligned(q), dk=unaligned(k), dv=unaligned(v))
    ra.check()
    for x, y in zip(a, b):
        err = (x.float() - y.float()).abs().max().item() / max(1.0, y.float().abs().max().item())
        assert err <= 1e-2


@pytest.mark.parametrize("name", ["ring8_zigzag_h8n32k", "ring8_striped_h8n32k"])
def test_ring_backward_full_size_sampled(ra, name):
    """The 8-rank zigzag and striped rings over 32768 positions (8 heads, head_dim 128,
    bf16): sampled dQ rows and dK/dV rows against the oracle one by one, the ring against
    the single pass, and sum_j dV_j = sum_i dO_i (each row of P sums to one)."""
    w = synth.WORKLOADS[name]
    q, k, v = synth.workload_inputs(w, device="cuda")
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    g = torch.Generator(device="cuda").manual_seed(77)
    dout = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(torch.bfloat16)
    R, layout = w.ring_size, w.layout
    o, lse = ra.ring_sim_fwd(q, k, v, R, layout, True)
    dq, dk, dv = ra.ring_sim_bwd(q, k, v, o, lse, dout, R, layout, True)
    ra.check()
    rng = np.random.default_rng(8)
    # query rows anywhere; key rows of every KV head in the last chunk and at the start of
    # the second-to-last (zigzag: keys whose gradients two ring steps write, the back chunk
    # of rank 0 and the front of rank 1's), and one key of an early chunk (zigzag: chunk 2,
    # rank 2's front chunk, seen by nearly every row and written on every step that reaches
    # it); under the striped layout the same positions fall on every rank
    chunk = N // (2 * R)
    q_rows = np.array([(0, int(h), int(i)) for h, i in zip(rng.integers(0, Hq, 12), rng.integers(0, N, 12))]
                      + [(0, 0, 0), (0, Hq - 1, N - 1), (0, 3, chunk), (0, 5, chunk - 1)])
    kv_rows = [(0, hk, j) for hk in range(Hkv) for j in (N - 1, N - chunk, N - chunk - 1 - hk)]
    kv_rows += [(0, 0, 2 * chunk + 5)]
    kv_rows = np.array(kv_rows)
    args = [to_oracle(t) for t in (q, k, v, dout)]
    rq, rk, rv = ob.gradient_rows(*args, True, None, q_rows, kv_rows)
    for gname, got, rows, ref in (("dq", dq, q_rows, rq), ("dk", dk, kv_rows, rk), ("dv", dv, kv_rows, rv)):
        sel = got[rows[:, 0], rows[:, 1], rows[:, 2]].float().cpu().numpy().astype(np.float64)
        scaled, row, p999 = assert_grad_close(sel, ref, torch.bfloat16, f"{name} {gname} sampled")
        print(name, gname, f"sampled: scaled {scaled:.2e} row {row:.2e} p99.9 {p999:.2e}")
    # the ring against the single pass on the same forward outputs
    sq, sk, sv = ra.attn_bwd(q, k, v, o, lse, dout, causal=True)
    for x, y in ((dq, sq), (dk, sk), (dv, sv)):
        err = (x.float() - y.float()).abs().max().item() / max(1.0, y.float().abs().max().item())
        assert err <= GRAD_TOL[torch.bfloat16]
    # sum over keys of dV = sum over rows of dO, per KV head (G query heads each)
    G = Hq // Hkv
    lhs = dv.double().sum(dim=2)
    rhs = dout.double().view(B, Hkv, G, N, D).sum(dim=(2, 3))
    bound = 2.0 ** -8 * (dv.double().abs().sum(dim=2) + dout.double().abs().view(B, Hkv, G, N, D).sum(dim=(2, 3)))
    assert torch.all((lhs - rhs).abs() <= bound)


REPEAT_CASES = [
    # B, Hq, Hkv, N, D, R, layout: fused rings whose kernels hand tensor-memory slots between
    # several threads; a race there shows as a run that differs from the others
    (1, 2, 2, 1024, 64, 4, "striped"),
    (1, 2, 2, 1024, 128, 4, "striped"),
    (1, 4, 2, 2048, 64, 4, "zigzag"),
    (1, 2, 2, 1024, 64, 1, "contig"),
]


@pytest.mark.parametrize("case", REPEAT_CASES, ids=lambda c: f"N{c[3]}D{c[4]}R{c[5]}{c[6]}")
def test_ring_backward_is_repeatable(ra, case):
    """The same causal backward 60 times: every run finite and bit-identical to the first
    (each output element has one writer and a fixed order of additions, so any difference
    is a race)."""
    B, Hq, Hkv, N, D, R, layout = case
    q, k, v, dout = _inputs(B, Hq, Hkv, N, D, torch.bfloat16, seed=N * 3 + R)
    o, lse = ra.ring_sim_fwd(q, k, v, R, layout, True)
    first = None
    for i in range(60):
        grads = ra.ring_sim_bwd(q, k, v, o, lse, dout, R, layout, True)
        ra.check()
        for name, t in zip(("dq", "dk", "dv"), grads):
            assert torch.isfinite(t.float()).all().item(), f"run {i}: non-finite {name}"
        if first is None:
            first = [t.clone() for t in grads]
        else:
            for name, a, b in zip(("dq", "dk", "dv"), first, grads):
                assert torch.equal(a, b), f"run {i}: {name} differs from the first run"
