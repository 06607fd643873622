"""GPU path (through the C ABI) against the oracle, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import merge as om
from exact_long_context_gb300 import synth
from helpers import (EDGE_SCALE, assert_close, edge_inputs, errors, gather_rows, oracle_full,
                     sample_rows, to_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    ra_mod.launch_count(reset=True)
    return ra_mod


def _full_compare(o, lse, q, k, v, causal, scale, dtype, what):
    o_ref, l_ref = oracle_full(q, k, v, causal, scale)
    return assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, dtype, what)


# ---------------------------------------------------------------- worked example (fp32)

def test_worked_example_ring4_fp32(ra):
    w = synth.WORKLOADS["tiny_ring4_fp32"]
    q, k, v = (t.cuda() for t in synth.workload_inputs(w))
    o, lse = ra.ring_sim_fwd(q, k, v, 4, "contig", causal=False, scale=w.scale)
    ra.check()
    err = _full_compare(o, lse, q, k, v, False, w.scale, torch.float32, "tiny ring4 fp32")
    print("tiny ring4 fp32 errors", err)
    o1, l1 = ra.attn_fwd(q, k, v, causal=False, scale=w.scale)
    ra.check()
    _full_compare(o1, l1, q, k, v, False, w.scale, torch.float32, "tiny single pass fp32")


# ---------------------------------------------------------------- small sweeps, full compare

SMALL_BF16 = [
    # B, Hq, Hkv, N, D, causal
    (1, 1, 1, 1, 128, True),
    (1, 1, 1, 7, 128, False),
    (1, 2, 1, 128, 128, True),
    (1, 2, 2, 256, 128, True),
    (2, 4, 2, 300, 128, True),
    (1, 4, 1, 384, 128, False),
    (1, 2, 2, 513, 128, True),
    (1, 8, 2, 1000, 128, True),
    (1, 2, 1, 200, 64, True),
    (2, 4, 4, 640, 64, False),
    (1, 4, 2, 1024, 64, True),
    (2, 6, 2, 700, 128, True),    # three query heads per KV head, batch 2
    (3, 3, 1, 257, 64, False),
]


@pytest.mark.parametrize("shape", SMALL_BF16, ids=lambda s: "x".join(map(str, s)))
def test_attn_bf16_small(ra, shape):
    B, Hq, Hkv, N, D, causal = shape
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, torch.bfloat16, seed=N + D, device="cuda")
    scale = 1.0 / math.sqrt(D)
    o, lse = ra.attn_fwd(q, k, v, causal=causal, scale=scale)
    ra.check()
    err = _full_compare(o, lse, q, k, v, causal, scale, torch.bfloat16, f"bf16 {shape}")
    print(shape, "errors", err)


SMALL_F32 = [
    (1, 1, 1, 1, 16, True),
    (1, 2, 1, 33, 16, True),
    (1, 2, 2, 100, 64, False),
    (2, 4, 2, 129, 128, True),
    (1, 3, 1, 70, 80, True),
    (1, 1, 1, 65, 1, False),
]


@pytest.mark.parametrize("shape", SMALL_F32, ids=lambda s: "x".join(map(str, s)))
def test_attn_f32_small(ra, shape):
    B, Hq, Hkv, N, D, causal = shape
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, torch.float32, seed=N, device="cuda")
    o, lse = ra.attn_fwd(q, k, v, causal=causal)
    ra.check()
    _full_compare(o, lse, q, k, v, causal, 1.0 / math.sqrt(D), torch.float32, f"f32 {shape}")


def test_bf16_other_head_sizes_use_cuda_cores(ra):
    for D in (16, 32, 96):
        q, k, v = synth.make_qkv(1, 2, 1, 150, D, torch.bfloat16, seed=D, device="cuda")
        o, lse = ra.attn_fwd(q, k, v, causal=True)
        ra.check()
        _full_compare(o, lse, q, k, v, True, 1.0 / math.sqrt(D), torch.bfloat16, f"bf16 D={D}")


def test_strided_inputs(ra):
    """[B, N, H, D] storage viewed as [B, H, N, D]; and an unaligned view (CUDA-core path)."""
    B, N, H, D = 1, 384, 4, 128
    g = torch.Generator(device="cuda").manual_seed(11)
    base = torch.randn(3, B, N, H, D, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = (base[i].transpose(1, 2) for i in range(3))
    o = torch.empty(B, N, H, D, dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    o, lse = ra.attn_fwd(q, k, v, causal=True, o=o)
    ra.check()
    _full_compare(o, lse, q, k, v, True, None, torch.bfloat16, "BNHD strides")
    # rows of 130 elements: not 16-byte aligned, so the tensor-core path is not taken
    raw = torch.randn(3, 1, 2, 200, 130, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = (raw[i][..., :128] for i in range(3))
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    ra.check()
    _full_compare(o, lse, q, k, v, True, None, torch.bfloat16, "unaligned strides")


def test_empty_and_degenerate(ra):
    q = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = ra.attn_fwd(q, q[:, :1], q[:, :1], causal=True)
    ra.check()
    assert o.numel() == 0
    q = torch.empty(0, 2, 64, 128, dtype=torch.bfloat16, device="cuda")
    ra.attn_fwd(q, q, q, causal=True)
    ra.check()
    # a single key: O = v_0
    q, k, v = synth.make_qkv(1, 2, 2, 1, 128, torch.bfloat16, seed=1, device="cuda")
    o, lse = ra.attn_fwd(q, k, v, causal=False)
    ra.check()
    assert torch.equal(o, v)


def test_launch_counts_are_native(ra):
    """One launch for the single pass and for a tensor-core ring of any layout (all steps
    in one launch); one per step on the CUDA-core path."""
    q, k, v = synth.make_qkv(1, 2, 1, 256, 128, torch.bfloat16, seed=3, device="cuda")
    before = ra.launch_count()
    ra.attn_fwd(q, k, v, causal=True)
    ra.ring_sim_fwd(q, k, v, 2, "zigzag", causal=True)
    ra.ring_sim_fwd(q, k, v, 4, "contig", causal=True)
    ra.check()
    assert ra.launch_count() - before == 1 + 1 + 1
    before = ra.launch_count()
    ra.ring_sim_fwd(q, k, v, 2, "striped", causal=True)
    qf, kf, vf = (t.float() for t in (q, k, v))
    ra.ring_sim_fwd(qf, kf, vf, 2, "zigzag", causal=True)
    ra.check()
    assert ra.launch_count() - before == 1 + 2


# ---------------------------------------------------------------- ring simulation

RING_SMALL = [
    # B, Hq, Hkv, N, D, R, layout, causal, dtype
    (1, 2, 1, 1024, 128, 2, "zigzag", True, torch.bfloat16),
    (1, 2, 2, 1024, 128, 4, "contig", True, torch.bfloat16),
    (1, 4, 2, 2048, 128, 8, "zigzag", True, torch.bfloat16),
    (1, 2, 1, 768, 128, 3, "zigzag", False, torch.bfloat16),
    (1, 2, 1, 960, 128, 5, "zigzag", True, torch.bfloat16),   # chunk 96: partial tiles
    (1, 2, 2, 640, 64, 5, "contig", True, torch.bfloat16),
    (1, 2, 1, 256, 32, 4, "zigzag", True, torch.bfloat16),   # CUDA-core path
    (1, 2, 1, 96, 16, 4, "zigzag", True, torch.float32),
    (1, 1, 1, 64, 16, 8, "contig", False, torch.float32),
    (1, 2, 1, 2048, 128, 4, "striped", True, torch.bfloat16),
    (1, 4, 2, 1024, 128, 8, "striped", True, torch.bfloat16),
    (1, 2, 2, 768, 64, 3, "striped", True, torch.bfloat16),
    (1, 2, 1, 1000, 128, 5, "striped", False, torch.bfloat16),   # 200 rows per rank: ragged
    # several 256-row blocks per chunk: the fused ring walks a diagonal prefix, then the
    # later steps' ranges
    (1, 2, 1, 4096, 128, 4, "contig", True, torch.bfloat16),
    (1, 2, 2, 4096, 128, 2, "zigzag", True, torch.bfloat16),
    (1, 2, 1, 3072, 64, 3, "zigzag", False, torch.bfloat16),
    (1, 2, 1, 96, 16, 4, "striped", True, torch.float32),
    # striped rings in one launch: each step a causal prefix with its own diagonal offset
    (1, 2, 1, 4096, 128, 4, "striped", True, torch.bfloat16),     # 1024 rows per rank
    (1, 4, 2, 2048, 128, 4, "striped", False, torch.bfloat16),
    (1, 2, 2, 1536, 64, 3, "striped", True, torch.bfloat16),      # 512 rows per rank, D = 64
    (1, 2, 1, 1152, 128, 3, "striped", True, torch.bfloat16),     # 384 rows: a 128-row last item
    (1, 2, 1, 256, 32, 8, "striped", True, torch.bfloat16),       # CUDA-core path
    # batch 2 and three query heads per KV head inside one fused launch
    (2, 6, 2, 1024, 128, 4, "zigzag", True, torch.bfloat16),
    (2, 3, 1, 2048, 128, 4, "striped", True, torch.bfloat16),
    (2, 6, 2, 768, 64, 3, "contig", False, torch.bfloat16),
]


@pytest.mark.parametrize("case", RING_SMALL, ids=lambda c: f"{c[6]}R{c[5]}N{c[3]}D{c[4]}{'c' if c[7] else 'n'}")
def test_ring_sim_small(ra, case):
    B, Hq, Hkv, N, D, R, layout, causal, dtype = case
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, dtype, seed=R * 100 + N, device="cuda")
    o, lse = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
    ra.check()
    err = _full_compare(o, lse, q, k, v, causal, 1.0 / math.sqrt(D), dtype, f"ring {case}")
    print(case, "errors", err)


FWD_REPEAT_CASES = [
    # B, Hq, Hkv, N, D, R, layout, causal: the single pass and fused rings, both head sizes
    (1, 4, 2, 2048, 128, 1, "contig", True),
    (1, 4, 2, 2048, 64, 4, "zigzag", True),
    (1, 2, 2, 1024, 128, 4, "striped", True),
    (1, 2, 2, 1024, 64, 4, "striped", True),
    (2, 6, 2, 1024, 128, 4, "zigzag", False),
]


@pytest.mark.parametrize("case", FWD_REPEAT_CASES, ids=lambda c: f"{c[6]}R{c[5]}N{c[3]}D{c[4]}{'c' if c[7] else 'n'}")
def test_forward_is_repeatable(ra, case):
    """The same forward 60 times: every run bit-identical to the first (the producer, the
    MMA thread and the softmax warps hand tensor-memory and shared-memory buffers to one
    another; each output row is written once from a fixed order of additions, so any
    difference is a race)."""
    B, Hq, Hkv, N, D, R, layout, causal = case
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, torch.bfloat16, seed=R * 10 + N, device="cuda")
    o0, l0 = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
    ra.check()
    assert torch.isfinite(o0.float()).all().item()
    for i in range(59):
        o, lse = ra.ring_sim_fwd(q, k, v, R, layout, causal=causal)
        ra.check()
        assert torch.equal(o, o0) and torch.equal(lse, l0), f"run {i + 1} differs from the first"


def test_ring_invariants_gpu(ra):
    """R = 1 vs R = 4 contig / zigzag / striped on the GPU: same result within rounding."""
    q, k, v = synth.make_qkv(1, 4, 2, 4096, 128, torch.bfloat16, seed=9, device="cuda")
    o1, l1 = ra.attn_fwd(q, k, v, causal=True)
    oc, lc = ra.ring_sim_fwd(q, k, v, 4, "contig", causal=True)
    oz, lz = ra.ring_sim_fwd(q, k, v, 4, "zigzag", causal=True)
    os_, ls = ra.ring_sim_fwd(q, k, v, 4, "striped", causal=True)
    ra.check()
    for o, l, name in ((oc, lc, "contig"), (oz, lz, "zigzag"), (os_, ls, "striped")):
        assert (o.float() - o1.float()).abs().max().item() <= 2e-2, name
        assert ((l - l1).abs() / l1.abs().clamp(min=1)).max().item() <= 1e-3, name


# ---------------------------------------------------------------- softmax edge cases

@pytest.mark.parametrize("kind", list(EDGE_SCALE))
def test_softmax_edge_cases(ra, kind):
    """Scores all equal, nearly flat (scale 0.01), very peaked (scale 4: score spread ~45,
    most exponentials underflow to 0) and a running maximum that moves along the key walk,
    through the single pass and the fused contiguous / zigzag / striped rings, each against
    the oracle on every element.

    Peaked rows make O nearly one row of V, up to ~5 in magnitude, where half a bf16 unit
    of the stored output is already 0.0156: these cases sit at 0.017-0.020 of the 2e-2
    bound (the kernel is deterministic, so the margin does not move between runs)."""
    B, Hq, Hkv, N, D = 2, 6, 2, 1024, 128
    scale = EDGE_SCALE[kind]
    q, k, v = edge_inputs(kind, B, Hq, Hkv, N, D, seed=41)
    o_ref, l_ref = oracle_full(q, k, v, True, scale)
    runs = [("single pass", lambda: ra.attn_fwd(q, k, v, causal=True, scale=scale))]
    for R, layout in ((4, "zigzag"), (2, "contig"), (4, "striped")):
        runs.append((f"{layout} R{R}",
                     lambda R=R, layout=layout: ra.ring_sim_fwd(q, k, v, R, layout, causal=True, scale=scale)))
    for name, fn in runs:
        o, lse = fn()
        ra.check()
        err = assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, torch.bfloat16,
                           f"{kind} {name}")
        print(kind, name, "errors", err)
    if kind == "uniform":
        # closed form: LSE of row i is ln(i + 1) (i + 1 keys, all scores 0)
        want = np.log(np.arange(1, N + 1, dtype=np.float64))
        assert np.max(np.abs(l_ref[0, 0] - want)) <= 1e-12


# ---------------------------------------------------------------- the workloads at full size

def _workload_case(ra, name, n_random, heads=None):
    w = synth.WORKLOADS[name]
    q, k, v = synth.workload_inputs(w, device="cuda")
    o, lse = ra.ring_sim_fwd(q, k, v, w.ring_size, w.layout, causal=w.causal, scale=w.scale)
    ra.check()
    assert torch.isfinite(o).all().item() and torch.isfinite(lse).all().item()
    chunk = w.N // (2 * w.ring_size) if w.layout == "zigzag" else w.N // w.ring_size
    rows = sample_rows(w.B, w.Hq, w.N, chunk=chunk, n_random=n_random, seed=w.seed, heads=heads)
    o_ref, l_ref = oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), w.causal, w.scale,
                                    rows=rows)
    og, lg = gather_rows(o, lse, rows)
    err = assert_close(og, lg, o_ref, l_ref, w.dtype, name)
    print(name, "oracle-sampled rows", len(rows), "errors", err)
    return q, k, v, o, lse


def test_workload_dense_causal_b2h32n4k(ra):
    w = synth.WORKLOADS["dense_causal_b2h32n4k"]
    q, k, v = synth.workload_inputs(w, device="cuda")
    o, lse = ra.attn_fwd(q, k, v, causal=True, scale=w.scale)
    ra.check()
    # whole heads compared element by element, plus sampled rows of every head
    for b, h in ((0, 0), (1, 31)):
        o_ref, l_ref = oracle.attention(to_oracle(q[b:b + 1, h:h + 1]), to_oracle(k[b:b + 1, h:h + 1]),
                                        to_oracle(v[b:b + 1, h:h + 1]), True, w.scale)
        assert_close(o[b:b + 1, h:h + 1].float().cpu().numpy(), lse[b:b + 1, h:h + 1].cpu().numpy(),
                     o_ref, l_ref, w.dtype, f"head {b},{h}")
    rows = sample_rows(w.B, w.Hq, w.N, chunk=256, n_random=4, seed=2)
    o_ref, l_ref = oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), True, w.scale, rows=rows)
    og, lg = gather_rows(o, lse, rows)
    print("dense causal errors", assert_close(og, lg, o_ref, l_ref, w.dtype, "dense sampled"))
    # ring_size = 1 through the ring entry point is the same call
    o2, l2 = ra.ring_sim_fwd(q, k, v, 1, "contig", causal=True, scale=w.scale)
    ra.check()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_workload_ring8_zigzag(ra):
    q, k, v, o, lse = _workload_case(ra, "ring8_zigzag_h8n32k", n_random=32)
    w = synth.WORKLOADS["ring8_zigzag_h8n32k"]
    oc, lc = ra.ring_sim_fwd(q, k, v, w.ring_size, "contig", causal=True, scale=w.scale)
    o1, l1 = ra.attn_fwd(q, k, v, causal=True, scale=w.scale)
    ra.check()
    for a, la, name in ((oc, lc, "contig"), (o1, l1, "single pass")):
        assert (a.float() - o.float()).abs().max().item() <= 2e-2, name
        assert ((la - lse).abs() / lse.abs().clamp(min=1)).max().item() <= 1e-3, name


@pytest.mark.parametrize("name", ["dense_causal_b2h32n4k_d64", "ring8_zigzag_h16n32k_d64"])
def test_workload_head_size_64(ra, name):
    """The dense and ring shapes at head size 64 (bench workloads): sampled rows against the
    oracle, and the ring against the single pass."""
    q, k, v, o, lse = _workload_case(ra, name, n_random=16, heads=[(0, 0), (0, 5), (0, 15)])
    w = synth.WORKLOADS[name]
    if w.ring_size > 1:
        o1, l1 = ra.attn_fwd(q, k, v, causal=True, scale=w.scale)
        ra.check()
        assert (o1.float() - o.float()).abs().max().item() <= 2e-2
        assert ((l1 - lse).abs() / lse.abs().clamp(min=1)).max().item() <= 1e-3


def test_workload_gqa_ring16(ra):
    _workload_case(ra, "gqa_ring16_zigzag_h32kv8n128k", n_random=8)


def test_workload_ring64_million(ra):
    w = synth.WORKLOADS["ring64_zigzag_h8kv2n1m"]
    heads = [(0, h) for h in range(w.Hq)]
    _workload_case(ra, "ring64_zigzag_h8kv2n1m", n_random=4, heads=heads)


WORK_ORDER_CASES = {
    # (B, Hq, Hkv, N, D, ring_size, layout): heads per group of consecutive work items
    # (K/V of a group within 48 MiB) and the groups' shapes
    "dense b2h32n4k: groups of 24, 24, 16 heads": (2, 32, 32, 4096, 128, 1, "contig"),
    "gqa b2 hq8 hkv4 n16k: groups of 12 and 4, across the batch": (2, 8, 4, 16384, 128, 1, "contig"),
    "fused ring8 zigzag h8n32k: groups of 3, 3, 2": (1, 8, 8, 32768, 128, 8, "zigzag"),
    "fused ring8 zigzag h16n32k d64: groups of 6, 6, 4": (1, 16, 16, 32768, 64, 8, "zigzag"),
    "fused ring4 striped h8n32k: groups of 3, 3, 2": (1, 8, 8, 32768, 128, 4, "striped"),
    # 160 zigzag chunks are more than one launch takes: one launch per step, tile-pair items
    "per-step ring80 zigzag h8n20k: tile pairs": (1, 8, 8, 20480, 128, 80, "zigzag"),
    # 10920-row ranks are not whole tiles: per-step launches of single blocks
    "per-step ring3 striped h8n32760: single blocks": (1, 8, 8, 32760, 128, 3, "striped"),
}


@pytest.mark.parametrize("name", list(WORK_ORDER_CASES))
def test_every_work_item_runs_once(ra, name):
    """O and the LSE start as NaN; every row must be written (each work item taken exactly
    once from the launch's work counter, in head groups), sampled rows match the oracle, and
    every counter pair is back to zero after the launch."""
    B, Hq, Hkv, N, D, R, layout = WORK_ORDER_CASES[name]
    q, k, v = synth.make_qkv(B, Hq, Hkv, N, D, torch.bfloat16, seed=41, device="cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device="cuda")
    if R > 1:
        ra.ring_sim_fwd(q, k, v, R, layout, causal=True, o=o, lse=lse)
    else:
        ra.attn_fwd(q, k, v, causal=True, o=o, lse=lse)
    ra.check()
    assert ra.work_counters_in_use() == 0
    assert not torch.isnan(o).any().item() and not torch.isnan(lse).any().item()
    chunk = N // (2 * R) if layout == "zigzag" else N // R
    rows = sample_rows(B, Hq, N, chunk=chunk, n_random=2, seed=41, heads=[(0, 0), (B - 1, Hq - 1)])
    o_ref, l_ref = oracle.attention(to_oracle(q), to_oracle(k), to_oracle(v), True, rows=rows)
    og, lg = gather_rows(o, lse, rows)
    assert_close(og, lg, o_ref, l_ref, torch.bfloat16, name)


# ---------------------------------------------------------------- LSE merge

@pytest.mark.parametrize("blk_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D,blk_offset", [(128, 0), (100, 0), (64, 0), (52, 0), (30, 0), (128, 4)])
def test_lse_merge(ra, blk_dtype, D, blk_offset):
    """D <= 128 with 16-byte rows takes the half-warp path (100 and 52: a lane with four
    values at the row's end); a block tensor offset by four elements (8 bytes for bf16)
    takes the one-warp-per-row path; D = 30 the scalar path."""
    B, H, N = 2, 3, 257
    g = torch.Generator(device="cuda").manual_seed(D)
    o_acc = torch.randn(B, H, N, D, generator=g, device="cuda")
    o_blk = torch.randn(B, H, N, D, generator=g, device="cuda").to(blk_dtype)
    if blk_offset:
        wide = torch.zeros(B, H, N, D + 2 * blk_offset, dtype=blk_dtype, device="cuda")
        wide[..., blk_offset:blk_offset + D] = o_blk
        o_blk = wide[..., blk_offset:blk_offset + D]
    lse_acc = torch.randn(B, H, N, generator=g, device="cuda") * 4
    lse_blk = torch.randn(B, H, N, generator=g, device="cuda") * 4
    lse_acc[0, 0, :10] = -math.inf
    lse_blk[0, 0, 5:15] = -math.inf
    o_acc[0, 0, :10] = 0  # identity partials carry o = 0
    ref_o, ref_l = om.merge(o_acc.cpu().double().numpy(), lse_acc.cpu().double().numpy(),
                            o_blk.float().cpu().double().numpy(), lse_blk.cpu().double().numpy())
    ra.lse_merge(o_acc, lse_acc, o_blk, lse_blk)
    ra.check()
    got_o = o_acc.cpu().double().numpy()
    got_l = lse_acc.cpu().double().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(ref_l))
    fin = ~np.isneginf(ref_l)
    assert np.max(np.abs(got_l[fin] - ref_l[fin])) <= 1e-5
    assert np.max(np.abs(got_o - ref_o)) <= 1e-5


# ---------------------------------------------------------------- device-side timeout path

def test_wait_timeout_is_reported_and_context_survives(ra):
    ra.wait_selftest(2_000_000)  # 2 ms on a barrier that nothing completes
    with pytest.raises(ra.RaError) as ei:
        ra.check()
    assert ei.value.status == ra.RA_ERR_TIMEOUT
    ra.check()  # the word was cleared
    q, k, v = synth.make_qkv(1, 1, 1, 128, 128, torch.bfloat16, seed=1, device="cuda")
    o, lse = ra.attn_fwd(q, k, v, causal=True)
    ra.check()
    assert torch.isfinite(o).all().item()
