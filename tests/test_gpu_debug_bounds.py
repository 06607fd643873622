"""The bounds-checked debug build (libra_debug.so, RA_DEBUG_BOUNDS): its kernels check every
tile coordinate and row index against its tensor before a global-memory access, record
RA_ERR_BOUNDS and skip the access instead of trapping.

Run in a child process that loads the debug library (RA_LIBRARY=debug): its self-test's
failing check is reported as RA_ERR_BOUNDS, and on valid inputs - the single pass, fused
and per-step rings, packed sequences, the backward - no check fires and the results match
the oracle.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent('''
    import sys, torch
    sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
    from exact_long_context_gb300 import ra, synth
    from helpers import assert_close, oracle_full
    assert ra.LIB_PATH.endswith("libra_debug.so"), ra.LIB_PATH
    assert ra.lib().ra_debug_bounds_checked() == 1
    ra.bounds_selftest()
    try:
        ra.check()
        raise SystemExit("the failing bounds check was not reported")
    except ra.RaError as e:
        assert e.status == ra.RA_ERR_BOUNDS, e
    ra.check()  # cleared
    cases = [(1, 4, 2, 640, 128, 1, "contig", torch.bfloat16), (1, 2, 1, 768, 128, 3, "zigzag", torch.bfloat16),
             (1, 2, 2, 576, 128, 3, "striped", torch.bfloat16), (1, 2, 1, 512, 64, 2, "striped", torch.bfloat16),
             (2, 3, 1, 200, 32, 2, "zigzag", torch.float32)]
    for B, Hq, Hkv, N, D, R, layout, dt in cases:
        q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dt, seed=N, device="cuda")
        o, lse = ra.ring_sim_fwd(q, k, v, R, layout, causal=True)
        ra.check()
        ro, rl = oracle_full(q, k, v, True)
        assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, dt, f"{layout} R={R}")
        dout = torch.randn_like(q)
        ra.ring_sim_bwd(q, k, v, o, lse, dout, R, layout, causal=True)
        ra.check()
    q, k, v = synth.make_qkv(1, 2, 1, 700, 128, torch.bfloat16, seed=9, device="cuda")
    o, lse = ra.attn_varlen_fwd(q, k, v, [0, 300, 300, 650], causal=True)
    ra.check()
    print("DEBUG_BOUNDS_OK")
''').replace("ROOT", repr(ROOT))


def test_debug_build_reports_failed_checks_and_passes_valid_inputs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, ROOT)
    from exact_long_context_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, RA_LIBRARY="debug")
    res = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "DEBUG_BOUNDS_OK" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]
