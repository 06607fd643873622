"""Host-side checks of libra.so that need no GPU: exports, argument validation, ring plan."""
import ctypes
import math
import os
import re

import pytest

from oracle import ring as oring

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ra():
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "ra.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol(ra):
    names = header_symbols()
    assert {"ra_attn_fwd", "ra_lse_merge", "ra_ring_sim_fwd", "ra_ring_sim_workspace_bytes"} <= set(names)
    L = ctypes.CDLL(ra.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert ra.version() == 100


def _t(shape, dtype=1, data=0x10000, stride=None):
    d = ra_mod().RaTensor()
    d.data = data
    d.dtype = dtype
    if stride is None:
        stride = [shape[1] * shape[2] * shape[3], shape[2] * shape[3], shape[3], 1]
    for i in range(4):
        d.shape[i] = shape[i]
        d.stride[i] = stride[i]
    return d


def ra_mod():
    from exact_long_context_gb300 import ra as ra_m
    return ra_m


def _call(ra, q, k, v, o, lse=0x20000, causal=1, scale=0.0, R=1, layout=0, ws=None):
    L = ra.lib()
    P = ctypes.byref
    return L.ra_ring_sim_fwd(P(q) if q is not None else None, P(k), P(v), P(o), lse, R, layout,
                             causal, scale, ws, None)


def test_argument_errors_are_reported_without_touching_a_gpu(ra):
    S = (1, 4, 256, 128)
    KV = (1, 2, 256, 128)
    IA, UN = ra.RA_ERR_INVALID_ARG, ra.RA_ERR_UNSUPPORTED
    assert _call(ra, None, _t(KV), _t(KV), _t(S)) == IA
    assert _call(ra, _t(S), _t(KV), _t((1, 2, 255, 128)), _t(S)) == IA  # k/v differ
    assert _call(ra, _t(S), _t((1, 3, 256, 128)), _t((1, 3, 256, 128)), _t(S)) == IA  # Hq % Hkv
    assert _call(ra, _t(S), _t(KV), _t(KV), _t((1, 4, 256, 64))) == IA  # o shape
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S, dtype=0)) == IA  # mixed dtype
    assert _call(ra, _t(S, stride=[0, 0, 128, 2]), _t(KV), _t(KV), _t(S)) == IA  # stride[3]
    assert _call(ra, _t(S, data=0), _t(KV), _t(KV), _t(S)) == IA  # null data
    assert _call(ra, _t(S, data=0x10001), _t(KV), _t(KV), _t(S)) == IA  # misaligned bf16
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), lse=None) == IA
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), scale=math.nan) == IA
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=0) == IA
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=3) == IA  # 256 % 3
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=3, layout=1) == IA
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=256, layout=1) == IA  # 256 % 512
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=4, layout=7) == IA
    # workspace missing where the ring keeps a float32 running output: float32 inputs, a
    # striped rank that is not whole 128-row tiles, more chunks than one fused launch holds
    f32 = [_t(x, dtype=0) for x in (S, KV, KV, S)]
    assert _call(ra, *f32, R=4, ws=None) == IA
    assert _call(ra, _t(S), _t(KV), _t(KV), _t(S), R=4, layout=2, ws=None) == IA
    long_q, long_kv = (1, 4, 256 * 128, 128), (1, 2, 256 * 128, 128)
    assert _call(ra, _t(long_q), _t(long_kv), _t(long_kv), _t(long_q), R=128, layout=1, ws=None) == IA
    assert "workspace" in ra.lib().ra_last_error().decode()
    big = (1, 4, 256, 192)
    assert _call(ra, _t(big), _t((1, 2, 256, 192)), _t((1, 2, 256, 192)), _t(big)) == UN
    assert "D > 128" in ra.lib().ra_last_error().decode()
    bad = _t(S)
    bad.dtype = 9
    assert _call(ra, bad, _t(KV), _t(KV), _t(S)) == IA


def test_workspace_size(ra):
    q = _t((2, 8, 1024, 128))
    L = ra.lib()
    assert L.ra_ring_sim_workspace_bytes(ctypes.byref(q), 1) == 0
    assert L.ra_ring_sim_workspace_bytes(ctypes.byref(q), 4) == 2 * 8 * 1024 * 128 * 4
    assert L.ra_ring_sim_workspace_bytes(ctypes.byref(q), 0) == 0


def _ws_for(ra, q, kv, dtype=1, R=4, layout=0, causal=1, data=0x10000):
    L = ra.lib()
    P = ctypes.byref
    return L.ra_ring_sim_workspace_bytes_for(P(_t(q, dtype, data)), P(_t(kv, dtype)), P(_t(kv, dtype)),
                                             P(_t(q, dtype)), R, layout, causal)


def test_workspace_size_for_the_call(ra):
    """Zero exactly when the call runs the fused tensor-core ring (bf16, D 64 or 128, 16-byte
    aligned, contiguous or zigzag with at most 128 chunks, or striped ranks of whole 128-row
    tiles), whose running result stays in the kernel; the full float32 running output else."""
    full = lambda q: q[0] * q[1] * q[2] * q[3] * 4  # noqa: E731
    q, kv = (1, 8, 32768, 128), (1, 2, 32768, 128)
    for layout in (0, 1, 2):
        for causal in (0, 1):
            assert _ws_for(ra, q, kv, layout=layout, causal=causal) == 0
    assert _ws_for(ra, q, kv, R=64, layout=1) == 0  # 128 chunks: one launch
    assert _ws_for(ra, q, kv, R=128, layout=1) == full(q)  # 256 chunks: per-step launches
    assert _ws_for(ra, q, kv, R=128, layout=0) == 0  # 128 contiguous chunks
    assert _ws_for(ra, q, kv, R=1) == 0  # the single pass
    q64, kv64 = (1, 8, 4096, 64), (1, 8, 4096, 64)
    assert _ws_for(ra, q64, kv64, R=8, layout=1) == 0
    assert _ws_for(ra, q64, kv64, R=8, layout=1, dtype=0) == full(q64)  # float32: CUDA cores
    q96, kv96 = (1, 8, 4096, 96), (1, 8, 4096, 96)
    assert _ws_for(ra, q96, kv96, R=8, layout=1) == full(q96)  # D = 96: CUDA cores
    assert _ws_for(ra, q, kv, R=8, layout=1, data=0x10008) == full(q)  # base not 16-byte aligned
    qs, kvs = (1, 8, 8 * 192, 128), (1, 8, 8 * 192, 128)
    assert _ws_for(ra, qs, kvs, R=8, layout=2) == full(qs)  # striped ranks of 192 rows
    assert _ws_for(ra, qs, kvs, R=8, layout=1) == 0
    assert _ws_for(ra, q, kv, R=3, layout=1) == 0 and "ring" in ra.lib().ra_last_error().decode()


def test_merge_argument_errors(ra):
    L = ra.lib()
    a = _t((1, 2, 8, 16), dtype=0)
    b = _t((1, 2, 8, 16), dtype=1)
    wrong = _t((1, 2, 9, 16), dtype=1)
    assert L.ra_lse_merge(ctypes.byref(a), 0x20000, ctypes.byref(wrong), 0x30000, None) == ra.RA_ERR_INVALID_ARG
    assert L.ra_lse_merge(ctypes.byref(b), 0x20000, ctypes.byref(b), 0x30000, None) == ra.RA_ERR_INVALID_ARG
    assert L.ra_lse_merge(ctypes.byref(a), None, ctypes.byref(b), 0x30000, None) == ra.RA_ERR_INVALID_ARG


def _covered(plan_steps, N, causal):
    """For every query position, the list of key positions it is scheduled to see."""
    seen = {}
    for segs in plan_steps:
        for s in segs:
            rs, qr, kr, dg = s["rs"], s["q_rank"], s["kv_rank"], s["diag"]
            for i in range(*s["q"]):
                for a, b in s["kv"]:
                    for j in range(a, b):
                        if causal and j + dg > i:
                            continue
                        seen.setdefault(i * rs + qr, []).append(j * rs + kr)
    return seen


@pytest.mark.parametrize("layout", ["contig", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_plan_covers_every_visible_key_once(ra, layout, causal, R):
    N = 2 * R * 6
    steps = [ra.ring_sim_plan(N, R, layout, causal, s) for s in range(R)]
    seen = _covered(steps, N, causal)
    for i in range(N):
        keys = sorted(seen.get(i, []))
        want = list(range(0, i + 1)) if causal else list(range(N))
        assert keys == want, (i, keys[:10])
    # first/last flags: every query chunk has exactly one FIRST and one FINAL segment
    firsts, finals = {}, {}
    for segs in steps:
        for s in segs:
            key = (s["rank"], s["q"])
            firsts[key] = firsts.get(key, 0) + (s["flags"] & ra.SEG_FIRST > 0)
            finals[key] = finals.get(key, 0) + (s["flags"] & ra.SEG_FINAL > 0)
    assert set(firsts.values()) == {1} and set(finals.values()) == {1}
    # the rank partition matches the oracle's restatement
    held = oring.rank_positions(N, R, layout)
    for s in steps[0]:
        pos = [i * s["rs"] + s["q_rank"] for i in range(*s["q"])]
        assert set(pos) <= set(held[s["rank"]].tolist())


@pytest.mark.parametrize("R", [2, 3, 4, 8])
def test_plan_reproduces_the_zigzag_step_cases(ra, R):
    N = 2 * R * 4
    h = N // (2 * R)
    for s in range(R):
        by_rank = {}
        for seg in ra.ring_sim_plan(N, R, "zigzag", True, s):
            by_rank.setdefault(seg["rank"], []).append(seg)
        for r in range(R):
            case = oring.zigzag_step_case(r, s, R)
            segs = sorted(by_rank.get(r, []), key=lambda x: x["q"])
            src = oring.kv_source(r, s, R)
            front = (src * h, (src + 1) * h)
            back = ((2 * R - 1 - src) * h, (2 * R - src) * h)
            if case == "local":
                assert [x["q"] for x in segs] == [(r * h, (r + 1) * h), ((2 * R - 1 - r) * h, (2 * R - r) * h)]
            elif case == "front_kv":
                assert len(segs) == 2 and all(x["kv"] == [front] for x in segs)
            else:
                assert len(segs) == 1 and segs[0]["q"] == ((2 * R - 1 - r) * h, (2 * R - r) * h)
                assert segs[0]["kv"] == [front, back]


def test_plan_contig_causal_block_classes(ra, golden_dir):
    """Contiguous causal ring: rank r sees rank j's block iff j <= r (the page's three classes)."""
    rows = []
    for line in open(os.path.join(golden_dir, "causal_block_classes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            qb, kb, cls = line.split()
            rows.append((int(qb), int(kb), cls))
    R, c = 8, 16
    N = R * c
    for qb, kb, cls in rows:
        s = (qb - kb) % R  # the step at which rank qb holds block kb
        segs = [x for x in ra.ring_sim_plan(N, R, "contig", True, s) if x["rank"] == qb]
        if cls == "skip":
            assert segs == []
        else:
            assert len(segs) == 1 and segs[0]["kv"] == [(kb * c, (kb + 1) * c)]
            assert (kb == qb) == (cls == "diagonal")


def test_plan_striped_is_balanced(ra):
    """Striped ranks see (almost) the same number of causal pairs at every step."""
    R, N = 8, 8 * 64
    for s_ in range(R):
        segs = ra.ring_sim_plan(N, R, "striped", True, s_)
        assert len(segs) == R
        for g in segs:
            assert g["rs"] == R and g["diag"] == (1 if g["kv_rank"] > g["q_rank"] else 0)


def test_plan_rejects_bad_arguments(ra):
    with pytest.raises(ValueError):
        ra.ring_sim_plan(100, 3, "contig", True, 0)
    with pytest.raises(ValueError):
        ra.ring_sim_plan(96, 3, "zigzag", True, 3)


def test_varlen_argument_errors(ra):
    L = ra.lib()
    S = (1, 2, 100, 128)
    IA = ra.RA_ERR_INVALID_ARG

    def call(cu, n, shape=S):
        arr = (ctypes.c_int32 * max(1, len(cu)))(*cu)
        return L.ra_attn_varlen_fwd(ctypes.byref(_t(shape)), ctypes.byref(_t(shape)),
                                    ctypes.byref(_t(shape)), ctypes.byref(_t(shape)), 0x20000,
                                    ctypes.cast(arr, ctypes.c_void_p), n, 1, 0.0, None)
    assert call([0, 50, 40], 2) == IA      # decreasing
    assert call([0, 50, 101], 2) == IA     # beyond the packed length
    assert call([-1, 50], 1) == IA         # negative
    assert call([0, 50], -1) == IA
    assert call([0, 50], 1, shape=(2, 2, 100, 128)) == IA  # B must be 1
    assert L.ra_attn_varlen_fwd(ctypes.byref(_t(S)), ctypes.byref(_t(S)), ctypes.byref(_t(S)),
                                ctypes.byref(_t(S)), 0x20000, None, 3, 1, 0.0, None) == IA


@pytest.mark.parametrize("R", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("layout", ["contig", "zigzag", "striped"])
def test_backward_plan_covers_every_visible_pair_once(ra, layout, causal, R):
    """Over the ring steps, the dQ segments (kind 0) visit every visible (row, key) pair
    exactly once, and so do the dK/dV segments (kind 1); each fixed range has exactly one
    FIRST and one FINAL segment, on its first and last step; at step s the partner of a
    range of rank r (dQ) is rank (r - s) mod R, of a key range of rank j (dK/dV) rank
    (j + s) mod R."""
    N = 2 * R * 6
    held = oring.rank_positions(N, R, layout)
    rank_of = {}
    for r, pos in enumerate(held):
        for p in pos.tolist():
            rank_of[p] = r
    rs = R if layout == "striped" else 1

    def positions(a, b, rank):
        return [i * rs + rank for i in range(a, b)]

    for kind in (0, 1):
        seen = {}
        first, last, nfirst, nfinal = {}, {}, {}, {}
        for s in range(R):
            for g in ra.ring_sim_bwd_plan(N, R, layout, causal, s, kind):
                fixed = positions(g["f0"], g["f1"], g["f_rank"])
                streamed = positions(g["s0a"], g["s1a"], g["s_rank"]) + positions(g["s0b"], g["s1b"], g["s_rank"])
                fr = {rank_of[p] for p in fixed}
                sr = {rank_of[p] for p in streamed}
                assert len(fr) == 1 and len(sr) == 1
                fr, sr = fr.pop(), sr.pop()
                assert sr == ((fr - s) % R if kind == 0 else (fr + s) % R)
                for a in fixed:
                    for b in streamed:
                        row, key = (a, b) if kind == 0 else (b, a)
                        vis = (not causal) or key <= row
                        # the kernels' index rule (key index + diag <= row index) is the
                        # position rule
                        assert vis == ((not causal) or key // rs + g["diag"] <= row // rs)
                        if vis:
                            seen[(row, key)] = seen.get((row, key), 0) + 1
                rid = (fr, g["f0"])
                first.setdefault(rid, s)
                last[rid] = s
                nfirst[rid] = nfirst.get(rid, 0) + (g["flags"] & 1)
                nfinal[rid] = nfinal.get(rid, 0) + ((g["flags"] >> 1) & 1)
                assert bool(g["flags"] & 1) == (first[rid] == s)
        want = {(i, j) for i in range(N) for j in range(N) if (not causal or j <= i)}
        assert set(seen) == want and set(seen.values()) == {1}, kind
        assert set(nfirst.values()) == {1} and set(nfinal.values()) == {1}
        for s in range(R):
            for g in ra.ring_sim_bwd_plan(N, R, layout, causal, s, kind):
                rid = ({rank_of[p] for p in positions(g["f0"], g["f1"], g["f_rank"])}.pop(), g["f0"])
                assert bool(g["flags"] & 2) == (last[rid] == s)


def test_host_call_head_groups(ra):
    """The host-buffer call's head groups: every KV head in exactly one non-empty group, in
    order; equal sizes (within one head) unless the call is copy-bound with at least three
    heads per group, where sizes fall in proportion to ng, ng - 1, ..., 1 and the last group
    is the smallest (the dense workload's 32 heads in 8 groups: 7, 6, 6, 4, 4, 2, 2, 1)."""
    assert ra.host_group_bounds(32, 8, True) == [0, 7, 13, 19, 23, 27, 29, 31, 32]
    for hkv in range(1, 130):
        for ng in range(1, min(8, hkv) + 1):
            for copy_bound in (False, True):
                kb = ra.host_group_bounds(hkv, ng, copy_bound)
                assert kb[0] == 0 and kb[-1] == hkv and len(kb) == ng + 1
                sizes = [b - a for a, b in zip(kb, kb[1:])]
                assert min(sizes) >= 1, (hkv, ng, copy_bound, sizes)
                if copy_bound and ng >= 4 and hkv >= 3 * ng:
                    assert sizes[-1] == min(sizes) and sizes[0] == max(sizes), (hkv, ng, sizes)
                    assert all(a + 1 >= b for a, b in zip(sizes, sizes[1:])), (hkv, ng, sizes)
                    share = [hkv * (ng - g) / (ng * (ng + 1) / 2) for g in range(ng)]
                    assert all(abs(z - w) <= 1.0 for z, w in zip(sizes, share)), (hkv, ng, sizes)
                else:
                    assert max(sizes) - min(sizes) <= 1, (hkv, ng, copy_bound, sizes)
    with pytest.raises(ValueError):
        ra.host_group_bounds(4, 5, True)  # more groups than heads
    with pytest.raises(ValueError):
        ra.host_group_bounds(64, 9, True)  # more than the call's 8 groups
