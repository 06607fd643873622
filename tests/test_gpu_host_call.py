"""ra_ring_sim_fwd_host: the same results as ra_ring_sim_fwd on device buffers, bit for
bit, through host buffers (its staged, head-group pipelined copies)."""
import ctypes

import pytest
import torch

from exact_long_context_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


CASES = [
    # B, Hq, Hkv, N, D, R, layout, causal, dtype
    (2, 4, 2, 1024, 128, 1, "contig", True, torch.bfloat16),
    (1, 8, 8, 2048, 128, 4, "zigzag", True, torch.bfloat16),
    (2, 6, 3, 768, 64, 3, "striped", True, torch.bfloat16),
    (1, 4, 1, 512, 128, 2, "contig", False, torch.bfloat16),
    (2, 2, 2, 96, 16, 4, "zigzag", True, torch.float32),
    (1, 24, 24, 256, 128, 1, "contig", True, torch.bfloat16),  # more KV heads than groups
    (2, 12, 6, 512, 128, 2, "zigzag", True, torch.bfloat16),  # one KV head per group, two batches
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}-{c[2]}N{c[3]}D{c[4]}R{c[5]}{c[6]}")
def test_host_call_equals_device_call(ra, case):
    B, Hq, Hkv, N, D, R, layout, causal, dtype = case
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=N + R, device="cuda")
    od, ld = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    oh, lh = ra.ring_sim_fwd_host(hq, hk, hv, R, layout, causal=causal)
    torch.cuda.synchronize()
    ra.check()
    assert torch.equal(oh, od.cpu())
    assert torch.equal(lh, ld.cpu())


def test_host_call_rejects_bad_arguments(ra):
    q, k, v = synth.make_qkv(1, 2, 2, 256, 128, torch.bfloat16, seed=1, device="cpu")
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ws = torch.empty(ra.ring_sim_fwd_host_workspace_bytes(hq, hk, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises(ra.RaError):  # workspace too small
        ra.ring_sim_fwd_host(hq, hk, hv, 1, workspace=ws[: ws.numel() // 2])
    with pytest.raises(ra.RaError):  # not contiguous
        ra.ring_sim_fwd_host(hq.transpose(1, 2).contiguous().transpose(1, 2), hk, hv, 1, workspace=ws)
    with pytest.raises(ValueError):  # device tensors where host ones belong
        ra.ring_sim_fwd_host(q.cuda(), k.cuda(), v.cuda(), 1, workspace=ws)
