"""The allocation-free ring entry point, ra_ring_sim_fwd_noalloc, through the C ABI.

It exists for callers that cannot have device memory allocated for them (a framework
whose memory pool owns the device, a latency-critical loop where cudaMalloc/cudaFree
would synchronise the device, a host application that passes a plugin only its input
and output buffers).  Its float32 running output lives in a fixed array inside the
library instead of a caller workspace, so this test checks that two calls in a row -
the second one finding the first one's leftovers in that shared array - each match
ra_ring_sim_fwd with a workspace, within the parity tolerances used elsewhere.

Collected last on purpose (file name), and self-contained so that it passes alone in a
fresh process as well as after the rest of the suite.
"""
import ctypes

import pytest
import torch

from exact_long_context_gb300 import synth
from helpers import BF16_LSE_REL, BF16_O_TOL, F32_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    L = ra_mod.lib()
    T = ctypes.POINTER(ra_mod.RaTensor)
    L.ra_ring_sim_fwd_noalloc.argtypes = [T, T, T, T, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_float, ctypes.c_void_p]
    L.ra_ring_sim_fwd_noalloc.restype = ctypes.c_int
    return ra_mod


def _noalloc(ra, q, k, v, R, layout, causal):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    d = [ra._desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"))]
    st = ra.lib().ra_ring_sim_fwd_noalloc(*(ctypes.byref(x) for x in d), lse.data_ptr(), R,
                                          ra.LAYOUTS[layout], int(causal), 0.0,
                                          torch.cuda.current_stream().cuda_stream)
    return st, o, lse


@pytest.mark.parametrize("case", [
    (1, 4, 2, 2048, 128, 4, "zigzag", True, torch.bfloat16),
    (1, 2, 1, 96, 16, 4, "contig", True, torch.float32),
], ids=["bf16_zigzag_R4", "f32_contig_R4"])
def test_noalloc_matches_workspace_entry_point_twice(ra, case):
    B, Hq, Hkv, N, D, R, layout, causal, dtype = case
    for call, seed in enumerate((21, 22)):
        q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=seed, device="cuda")
        st, o, lse = _noalloc(ra, q, k, v, R, layout, causal)
        assert st == ra.RA_OK, ra.lib().ra_last_error().decode()
        ref_o, ref_l = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
        ra.check()
        o_err = (o.float() - ref_o.float()).abs().max().item()
        if dtype == torch.bfloat16:
            l_err = ((lse - ref_l).abs() / ref_l.abs().clamp(min=1)).max().item()
            assert o_err <= BF16_O_TOL and l_err <= BF16_LSE_REL, (call, o_err, l_err)
        else:
            l_err = (lse - ref_l).abs().max().item()
            assert o_err <= F32_TOL and l_err <= F32_TOL, (call, o_err, l_err)


def test_noalloc_rejects_sizes_beyond_its_scratch(ra):
    # 1 x 8 x 16384 x 128 = 16 Mi floats of running output: twice the fixed 8 Mi
    q = torch.zeros(1, 8, 16384, 128, dtype=torch.bfloat16, device="cuda")
    st, _, _ = _noalloc(ra, q, q, q, 2, "contig", True)
    assert st == ra.RA_ERR_UNSUPPORTED
    assert "scratch" in ra.lib().ra_last_error().decode()
    small = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    st, _, _ = _noalloc(ra, small, small, small, 128, "contig", True)
    assert st == ra.RA_ERR_UNSUPPORTED
