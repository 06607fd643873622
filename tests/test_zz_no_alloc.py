"""The allocation-free ring entry point, ra_ring_sim_fwd_noalloc, through the C ABI.

It exists for callers that cannot have device memory allocated for them (a framework
whose memory pool owns the device, a latency-critical loop where cudaMalloc/cudaFree
would synchronise the device, a host application that passes a plugin only its input
and output buffers).  A call that runs the fused ring needs no scratch; the per-step
launches keep their float32 running output in a fixed array inside the library instead
of a caller workspace.  So this test checks that two calls in a row - the second one
finding the first one's leftovers in that shared array - each match the oracle, and
ra_ring_sim_fwd with a workspace, within the parity tolerances used elsewhere.

Collected last on purpose (file name), and self-contained so that it passes alone in a
fresh process as well as after the rest of the suite.
"""
import ctypes

import pytest
import torch

from exact_long_context_gb300 import synth
import oracle
from helpers import (BF16_LSE_REL, BF16_O_TOL, F32_TOL, assert_close, gather_rows, oracle_full,
                     sample_rows, to_oracle)

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


CASES = {
    # fused ring (no scratch): whole-tile chunks, a ragged chunk of 96 rows, batch 2 with
    # three query heads per KV head, D = 64, and 128 chunks in one launch
    "bf16_zigzag_R4": (1, 4, 2, 2048, 128, 4, "zigzag", True, torch.bfloat16),
    "bf16_zigzag_R5_ragged": (1, 2, 1, 960, 128, 5, "zigzag", True, torch.bfloat16),
    "bf16_zigzag_R3_b2_gqa3": (2, 6, 2, 768, 128, 3, "zigzag", True, torch.bfloat16),
    "bf16_zigzag_R4_d64": (1, 4, 2, 1024, 64, 4, "zigzag", True, torch.bfloat16),
    "bf16_zigzag_R64": (1, 2, 1, 2048, 128, 64, "zigzag", True, torch.bfloat16),
    # per-step launches over the fixed scratch array
    "f32_contig_R4": (1, 2, 1, 96, 16, 4, "contig", True, torch.float32),
    "f32_zigzag_R64": (1, 2, 1, 2048, 16, 64, "zigzag", True, torch.float32),
    "bf16_striped_R3_192": (1, 2, 1, 576, 128, 3, "striped", True, torch.bfloat16),
    "f32_noncausal_zigzag_R2": (1, 3, 3, 256, 32, 2, "zigzag", False, torch.float32),
    # exactly the scratch's 8 Mi floats of running output (accepted)
    "f32_contig_R2_at_limit": (2, 16, 16, 2048, 128, 2, "contig", True, torch.float32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(ra, name):
    B, Hq, Hkv, N, D, R, layout, causal, dtype = CASES[name]
    if name == "f32_contig_R2_at_limit":
        assert B * Hq * N * D == 8 * 1024 * 1024
    for call, seed in enumerate((21, 22)):
        q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=seed, device="cuda")
        st, o, lse = _noalloc(ra, q, k, v, R, layout, causal)
        assert st == ra.RA_OK, ra.lib().ra_last_error().decode()
        ref_o, ref_l = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
        ra.check()
        # against the library's workspace call
        o_err = (o.float() - ref_o.float()).abs().max().item()
        if dtype == torch.bfloat16:
            l_err = ((lse - ref_l).abs() / ref_l.abs().clamp(min=1)).max().item()
            assert o_err <= BF16_O_TOL and l_err <= BF16_LSE_REL, (call, o_err, l_err)
        else:
            l_err = (lse - ref_l).abs().max().item()
            assert o_err <= F32_TOL and l_err <= F32_TOL, (call, o_err, l_err)
        # against the oracle: every row, or sampled rows (chunk edges and random rows) at
        # the at-limit size
        chunk = N // (2 * R) if layout == "zigzag" else N // R
        if B * Hq * N <= 16384:
            ro, rl = oracle_full(q, k, v, causal)
            assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, dtype, f"{name} call {call}")
        else:
            rows = sample_rows(B, Hq, N, chunk=chunk, n_random=4, seed=seed,
                               heads=[(0, 0), (B - 1, Hq - 1)])
            ro, rl = oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), causal, rows=rows)
            og, lg = gather_rows(o, lse, rows)
            assert_close(og, lg, ro, rl, dtype, f"{name} call {call}")
    assert ra.work_counters_in_use() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(ra):
    # float32 runs keep a running output: 1 x 8 x 16384 x 128 = 16 Mi floats, twice the
    # fixed 8 Mi
    q = torch.zeros(1, 8, 16384, 128, dtype=torch.float32, device="cuda")
    st, _, _ = _noalloc(ra, q, q, q, 2, "contig", True)
    assert st == ra.RA_ERR_UNSUPPORTED
    assert "scratch" in ra.lib().ra_last_error().decode()
    # more than 64 per-step ranks
    small = torch.zeros(1, 1, 256, 16, dtype=torch.float32, device="cuda")
    st, _, _ = _noalloc(ra, small, small, small, 128, "contig", True)
    assert st == ra.RA_ERR_UNSUPPORTED
    # the same sizes in bf16 run the fused ring and need no scratch
    qb = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    st, o, lse = _noalloc(ra, qb, qb, qb, 128, "contig", True)
    assert st == ra.RA_OK, ra.lib().ra_last_error().decode()
    ra.check()
    # Q = 0: every visible score is 0, so row i's LSE is ln(i + 1) and O = 0 (V = 0)
    want = torch.log(torch.arange(1, 257, device="cuda", dtype=torch.float32))
    assert (lse[0, 0] - want).abs().max().item() <= 1e-3 * 6
    assert o.float().abs().max().item() == 0.0
