"""Failure detection without a GPU fault.

Two forms, neither of which faults, traps or hangs the GPU:
- a kernel launch made to fail on the host (ra_debug_fail_next_launches): the call
  reports RA_ERR_CUDA with its message, nothing reaches the GPU, and the next call runs;
- the kernels' own bounded pipeline waits made to run out: the TMA producers pause 5 ms
  before their first copy (ra_debug_set_producer_delay_ns) under a 1 us wait limit
  (ra_debug_set_wait_limit_ns), so the consumers wait on barriers that nothing completes
  in time: each tensor-core kernel records
  RA_ERR_TIMEOUT in the device error word, winds down (its copies and MMAs in flight
  complete, tensor memory is released) and returns; the host reads the status, and the
  context stays usable.  The pages' ring loops wait without a limit (`op.wait()` in the
  `ring_attention_forward` listing of "Ring Attention 论文解析").
"""
import pytest
import torch

from exact_long_context_gb300 import synth
from helpers import assert_close, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    ra_mod.lib()
    return ra_mod


def _status(ra):
    try:
        ra.check()
        return ra.RA_OK
    except ra.RaError as e:
        return e.status


def test_injected_launch_failure_is_reported_and_the_next_call_runs(ra):
    q, k, v = synth.make_qkv(1, 2, 1, 256, 128, torch.bfloat16, seed=3, device="cuda")
    qf, kf, vf = (t.float() for t in (q, k, v))
    calls = {
        "attn_fwd (tensor cores)": lambda: ra.attn_fwd(q, k, v, causal=True),
        "ring_sim_fwd fused": lambda: ra.ring_sim_fwd(q, k, v, 2, "zigzag", causal=True),
        "ring_sim_fwd per step (float32)": lambda: ra.ring_sim_fwd(qf, kf, vf, 2, "zigzag", causal=True),
        "attn_varlen_fwd": lambda: ra.attn_varlen_fwd(q, k, v, [0, 100, 200], causal=True),
        "lse_merge": lambda: ra.lse_merge(torch.zeros(1, 2, 256, 128, device="cuda"),
                                          torch.zeros(1, 2, 256, device="cuda"), q,
                                          torch.zeros(1, 2, 256, device="cuda")),
        "ulysses_all_to_all": lambda: ra.ulysses_all_to_all(torch.zeros(2, 128, 2, 128, device="cuda"), 2, True),
    }
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    dout = torch.randn_like(q)
    calls["attn_bwd"] = lambda: ra.attn_bwd(q, k, v, o, lse, dout, causal=True)
    for name, call in calls.items():
        ra.fail_next_launches(1)
        with pytest.raises(ra.RaError) as ei:
            call()
        assert ei.value.status == ra.RA_ERR_CUDA, name
        assert "injected" in str(ei.value), (name, str(ei.value))
        assert _status(ra) == ra.RA_OK, name  # nothing reached the GPU
    ra.fail_next_launches(0)
    assert ra.work_counters_in_use() == 0
    o2, lse2 = ra.attn_fwd(q, k, v, causal=True)
    ra.check()
    ro, rl = oracle_full(q, k, v, True)
    assert_close(o2.float().cpu().numpy(), lse2.cpu().numpy(), ro, rl, torch.bfloat16, "after injection")


def test_kernel_waits_time_out_cleanly_and_the_context_survives(ra):
    """A paused producer under a short limit makes the tensor-core kernels' pipeline waits run
    out: each call either completes with the same result as under the default settings, or
    reports RA_ERR_TIMEOUT (at least one must), and afterwards a normal call matches the
    oracle."""
    B, Hq, Hkv, N, D = 1, 1, 1, 512, 128
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, torch.bfloat16, seed=5, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    o_ref, l_ref = ra.attn_fwd(q, k, v, causal=True)
    calls = {
        "attn_fwd": lambda: ra.attn_fwd(q, k, v, causal=True),
        "ring_sim_fwd fused R=2": lambda: ra.ring_sim_fwd(q, k, v, 2, "zigzag", causal=True),
        "attn_bwd": lambda: ra.attn_bwd(q, k, v, o_ref, l_ref, dout, causal=True),
        "ring_sim_bwd fused R=2": lambda: ra.ring_sim_bwd(q, k, v, o_ref, l_ref, dout, 2, "zigzag", causal=True),
    }
    want = {}
    for name, call in calls.items():  # results under the default limit
        want[name] = [t.clone() for t in call()]
        ra.check()
    got = {}
    try:
        ra.set_wait_limit_ns(1000)
        ra.set_producer_delay_ns(5_000_000)
        for name, call in calls.items():
            out = call()
            got[name] = (_status(ra), out)
    finally:
        ra.set_producer_delay_ns(0)
        ra.set_wait_limit_ns(-1)
    timeouts = [n for n, (st, _) in got.items() if st == ra.RA_ERR_TIMEOUT]
    for name, (st, out) in got.items():
        assert st in (ra.RA_OK, ra.RA_ERR_TIMEOUT), (name, st)
        if st == ra.RA_OK:  # a run that finished within the limit is the normal result
            for a, b in zip(out, want[name]):
                assert torch.equal(a, b), name
    assert timeouts, "no wait ran out behind a paused producer"
    # launches that ended on a timeout still released their work counters
    assert ra.work_counters_in_use() == 0
    # the context is usable and the default limit is back
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    assert _status(ra) == ra.RA_OK
    ro, rl = oracle_full(q, k, v, True)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, torch.bfloat16, "after the timeouts")
