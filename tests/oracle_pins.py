"""Pins of the oracle to facts outside itself.

Each ``pin_*`` function raises AssertionError when the oracle (the build selected by
``plant``; 0 is the real one) disagrees with something fixed by the pages or by
mathematics: a brute-force full-matrix softmax, the glossary page's worked example,
closed forms, invariants, the merge algebra and an independent ring restatement.
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
checks that every deliberately wrong build fails at least one of them.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from oracle import merge as om
from oracle import ring as oring

TOL = 1e-12


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def brute_force(q, k, v, causal, scale, kv_lo=0, kv_hi=None):
    """Full n x n score matrix, exp without a max shift, then normalise (fp64)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hq, N, D = q.shape
    G = Hq // k.shape[1]
    kx = np.repeat(k, G, axis=1)
    vx = np.repeat(v, G, axis=1)
    S = scale * np.einsum("bhid,bhjd->bhij", q, kx)
    kv_hi = N if kv_hi is None else kv_hi
    j = np.arange(N)[None, :]
    i = np.arange(N)[:, None]
    vis = (j >= kv_lo) & (j < kv_hi)
    if causal:
        vis = vis & (j <= i)
    P = np.where(vis, np.exp(S), 0.0)
    Z = P.sum(-1)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(Z[..., None] > 0, (P @ vx) / Z[..., None], 0.0)
        L = np.where(Z > 0, np.log(Z), -np.inf)
    return O, L


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isneginf(a) & np.isneginf(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b)), f"{what}: -inf pattern differs"
    with np.errstate(invalid="ignore"):
        d = np.abs(np.where(both_inf, 0.0, a - b))
    scale = np.maximum(1.0, np.abs(np.where(both_inf, 0.0, b)))
    err = float(np.max(d / scale)) if d.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


BRUTE_CASES = [
    # B, Hq, Hkv, N, D, causal
    (1, 1, 1, 1, 1, False),
    (1, 1, 1, 7, 4, True),
    (2, 2, 2, 33, 16, False),
    (1, 4, 2, 40, 8, True),
    (1, 4, 1, 17, 5, True),
    (2, 8, 2, 64, 16, False),
    (1, 6, 3, 29, 64, True),
]


def pin_brute_force(plant=0):
    for n, (B, Hq, Hkv, N, D, causal) in enumerate(BRUTE_CASES):
        q = _rand((B, Hq, N, D), 10 + n)
        k = _rand((B, Hkv, N, D), 20 + n)
        v = _rand((B, Hkv, N, D), 30 + n)
        scale = 0.7 / np.sqrt(D)
        o, l = oracle.attention(q, k, v, causal, scale, plant=plant)
        ob, lb = brute_force(q, k, v, causal, scale)
        _close(o, ob, what=f"brute O case {n}")
        _close(l, lb, what=f"brute LSE case {n}")
        # a key window [lo, hi) on top of causality
        lo, hi = N // 3, max(N // 3 + 1, (2 * N) // 3)
        o, l = oracle.attention(q, k, v, causal, scale, kv_lo=lo, kv_hi=hi, plant=plant)
        ob, lb = brute_force(q, k, v, causal, scale, lo, hi)
        _close(o, ob, what=f"brute windowed O case {n}")
        _close(l, lb, what=f"brute windowed LSE case {n}")


def read_golden(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            vals[key] = rest.strip()
    return vals


def pin_worked_example(golden_dir, plant=0):
    """The glossary page's 4-device simulation, regenerated from its seed."""
    import torch

    g = read_golden(os.path.join(golden_dir, "worked_example_ring4.txt"))
    n_dev, block, dim = int(g["n_devices"]), int(g["block"]), int(g["dim"])
    atol = float(g["atol"])
    torch.manual_seed(int(g["seed"]))
    qkv = torch.randn(3, n_dev * block, dim)
    q32, k32, v32 = (t.numpy() for t in qkv)
    q, k, v = (t.astype(np.float64) for t in (q32, k32, v32))
    scale = 1.0 / np.sqrt(dim)

    # the page's unshifted ring loop, in fp64: numerator / denominator per device
    ring = np.zeros((n_dev * block, dim))
    for i in range(n_dev):
        qi = q[i * block:(i + 1) * block]
        num = np.zeros((block, dim))
        den = np.zeros((block, 1))
        for step in range(n_dev):
            j = (i - step) % n_dev
            p = np.exp(qi @ k[j * block:(j + 1) * block].T * scale)
            num += p @ v[j * block:(j + 1) * block]
            den += p.sum(axis=1, keepdims=True)
        ring[i * block:(i + 1) * block] = num / den
    assert f"{block}x{block}" == g["score_block"]
    assert f"{n_dev * block}x{n_dev * block}" == g["full_matrix"]

    o, _ = oracle.attention(q32.reshape(1, 1, -1, dim), k32.reshape(1, 1, -1, dim),
                            v32.reshape(1, 1, -1, dim), False, scale, plant=plant)
    o = o.reshape(-1, dim)
    _close(o, ring, what="worked example: oracle vs the page's ring loop")
    # the page's claim: the ring result matches the full fp32 softmax at atol 1e-5
    full32 = torch.softmax(qkv[0] @ qkv[1].T / dim ** 0.5, dim=-1) @ qkv[2]
    claim = bool(np.allclose(ring, full32.numpy().astype(np.float64), rtol=1e-5, atol=atol))
    assert str(claim) == g["expected_allclose"]
    assert np.max(np.abs(o - full32.numpy())) <= atol, "oracle vs fp32 full softmax beyond atol"


def pin_closed_forms(plant=0):
    rng = np.random.default_rng(7)
    B, Hq, Hkv, N, D = 2, 4, 2, 23, 8
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    G = Hq // Hkv
    # Q = 0: uniform weights over the visible keys
    q0 = np.zeros((B, Hq, N, D))
    for causal in (False, True):
        o, l = oracle.attention(q0, k, v, causal, 0.3, plant=plant)
        for h in range(Hq):
            vk = v[:, h // G]
            if causal:
                cnt = np.arange(1, N + 1, dtype=np.float64)
                mean = np.cumsum(vk, axis=1) / cnt[None, :, None]
            else:
                cnt = np.full(N, float(N))
                mean = np.repeat(vk.mean(axis=1, keepdims=True), N, axis=1)
            _close(o[:, h], mean, what="Q=0 mean of visible V")
            _close(l[:, h], np.broadcast_to(np.log(cnt), (B, N)), what="Q=0 LSE = ln(count)")
    # V constant per KV head: O equals that constant
    q = rng.standard_normal((B, Hq, N, D))
    c = rng.standard_normal((B, Hkv, 1, D))
    vc = np.broadcast_to(c, (B, Hkv, N, D)).copy()
    for causal in (False, True):
        o, _ = oracle.attention(q, k, vc, causal, 0.5, plant=plant)
        for h in range(Hq):
            _close(o[:, h], np.broadcast_to(c[:, h // G], (B, N, D)), what="constant V")
    # causal row 0 sees only key 0: O_0 = v_0, LSE_0 = s_00
    scale = 0.37
    o, l = oracle.attention(q, k, v, True, scale, plant=plant)
    for h in range(Hq):
        _close(o[:, h, 0], v[:, h // G, 0], what="causal row 0 output")
        s00 = scale * np.einsum("bd,bd->b", q[:, h, 0], k[:, h // G, 0])
        _close(l[:, h, 0], s00, what="causal row 0 LSE")
    # a single key (N = 1)
    q1, k1, v1 = q[:, :, :1], k[:, :, :1], v[:, :, :1]
    o, l = oracle.attention(q1, k1, v1, False, scale, plant=plant)
    for h in range(Hq):
        _close(o[:, h, 0], v1[:, h // G, 0], what="single key output")
    # an empty key window: identity partial
    o, l = oracle.attention(q, k, v, False, scale, kv_lo=5, kv_hi=5, plant=plant)
    assert np.all(o == 0) and np.all(np.isneginf(l)), "empty window must give (0, -inf)"


def pin_invariants(plant=0):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, N, D = 1, 4, 2, 31, 16
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    for causal in (False, True):
        o, l = oracle.attention(q, k, v, causal, scale, plant=plant)
        kx = np.repeat(k, G, axis=1)
        s = scale * np.einsum("bhid,bhjd->bhij", q, kx)
        vis = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
        smax = np.where(vis, s, -np.inf).max(-1)
        cnt = vis.sum(-1)
        assert np.all(l >= smax - 1e-12), "LSE below the row max"
        assert np.all(l <= smax + np.log(cnt) + 1e-12), "LSE above max + ln(count)"
        # GQA: explicit repetition of KV heads gives the same result
        oe, le = oracle.attention(q, kx, np.repeat(v, G, axis=1), causal, scale, plant=plant)
        _close(o, oe, what="GQA vs repeated KV heads")
        _close(l, le, what="GQA LSE vs repeated KV heads")
    # non-causal: permuting keys (with their values) leaves every row unchanged
    perm = rng.permutation(N)
    o, l = oracle.attention(q, k, v, False, scale, plant=plant)
    op, lp = oracle.attention(q, k[:, :, perm], v[:, :, perm], False, scale, plant=plant)
    _close(o, op, what="key permutation")
    _close(l, lp, what="key permutation LSE")


def pin_merge(plant=0):
    rng = np.random.default_rng(5)
    B, Hq, Hkv, N, D = 1, 2, 1, 48, 8
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    scale = 1.0 / np.sqrt(D)
    cuts = [0, 5, 17, 18, 30, 48]
    for causal in (False, True):
        full_o, full_l = oracle.attention(q, k, v, causal, scale, plant=plant)
        parts = [oracle.attention(q, k, v, causal, scale, kv_lo=a, kv_hi=b, plant=plant)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        for trial in range(4):
            order = rng.permutation(len(parts))
            o = np.zeros_like(full_o)
            l = np.full_like(full_l, -np.inf)
            for idx in order:
                o, l = om.merge(o, l, *parts[idx])
            _close(o, full_o, what=f"merged blocks (order {order}) vs single pass")
            _close(l, full_l, what="merged LSE vs single pass")
            o2 = np.zeros_like(full_o)
            l2 = np.full_like(full_l, -np.inf)
            for idx in order:
                o2, l2 = om.merge_sigmoid(o2, l2, *parts[idx])
            _close(o2, full_o, tol=1e-11, what="sigmoid-form merge vs single pass")
            _close(l2, full_l, tol=1e-11, what="sigmoid-form merged LSE")
    # algebra: commutative, associative, identity
    a = (rng.standard_normal((9, D)), rng.standard_normal(9) * 3)
    b = (rng.standard_normal((9, D)), rng.standard_normal(9) * 3)
    c = (rng.standard_normal((9, D)), rng.standard_normal(9) * 3)
    ab = om.merge(*a, *b)
    _close(ab[0], om.merge(*b, *a)[0], what="commutative")
    _close(om.merge(*ab, *c)[0], om.merge(*a, *om.merge(*b, *c))[0], what="associative")
    ident = (np.zeros((9, D)), np.full(9, -np.inf))
    _close(om.merge(*a, *ident)[0], a[0], what="identity right")
    _close(om.merge(*ident, *a)[1], a[1], what="identity left")
    both = om.merge(*ident, *ident)
    assert np.all(both[0] == 0) and np.all(np.isneginf(both[1]))
    # the definition on one scalar pair
    o, l = om.merge(np.array([[1.0]]), np.array([0.0]), np.array([[3.0]]), np.array([np.log(3.0)]))
    _close(l, [np.log(4.0)], what="ln(e^0 + e^ln3) = ln 4")
    _close(o, [[(1.0 * 1 + 3.0 * 3) / 4]], what="weights 1/4, 3/4")


def pin_ring(plant=0):
    rng = np.random.default_rng(3)
    for (B, Hq, Hkv, N, D, R, layout, causal) in [
        (1, 2, 1, 32, 8, 4, "contig", False),
        (1, 2, 1, 32, 8, 4, "contig", True),
        (1, 2, 2, 48, 8, 3, "zigzag", True),
        (1, 4, 2, 64, 16, 4, "zigzag", True),
        (1, 2, 1, 40, 8, 5, "zigzag", False),
        (1, 1, 1, 16, 4, 1, "zigzag", True),
        (1, 2, 1, 64, 8, 8, "zigzag", True),
        (1, 2, 1, 36, 8, 4, "striped", True),
        (1, 4, 2, 40, 8, 8, "striped", True),
        (1, 2, 2, 30, 8, 3, "striped", False),
    ]:
        q = rng.standard_normal((B, Hq, N, D))
        k = rng.standard_normal((B, Hkv, N, D))
        v = rng.standard_normal((B, Hkv, N, D))
        scale = 1.0 / np.sqrt(D)
        o, l = oracle.attention(q, k, v, causal, scale, plant=plant)
        ro, rl = oring.ring_forward(q, k, v, R, layout, causal, scale)
        _close(ro, o, tol=1e-11, what=f"ring {layout} R={R} causal={causal} O")
        _close(rl, l, tol=1e-11, what=f"ring {layout} R={R} LSE")


def pin_zigzag_map(golden_dir):
    """The Twinkle page's 8-chunk / 4-GPU table and its three forward step cases."""
    want = {}
    with open(os.path.join(golden_dir, "zigzag_8chunks_4ranks.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                r, chunks = line.split(":")
                want[int(r)] = [int(c) for c in chunks.split()]
    ranges = oring.rank_ranges(8, 4, "zigzag")
    assert {r: [a for a, _ in rr] for r, rr in enumerate(ranges)} == want
    # the step cases follow from causality on global positions
    for R in (2, 3, 4, 8):
        N = 2 * R * 3
        ranges = oring.rank_ranges(N, R, "zigzag")
        h = N // (2 * R)
        for r in range(R):
            qf, qb = ranges[r]
            for s in range(R):
                src = oring.kv_source(r, s, R)
                kf, kb = ranges[src]
                case = oring.zigzag_step_case(r, s, R)

                def sees(qr, kr):  # does any row of qr see any key of kr (causal)?
                    return kr[0] <= qr[1] - 1

                def sees_all(qr, kr):
                    return kr[1] - 1 <= qr[0]

                if case == "local":
                    assert src == r
                elif case == "front_kv":
                    assert sees_all(qf, kf) and sees_all(qb, kf), (R, r, s)
                    assert not sees(qf, kb) and not sees(qb, kb), (R, r, s)
                else:
                    assert not sees(qf, kf) and not sees(qf, kb), (R, r, s)
                    assert sees_all(qb, kf) and sees_all(qb, kb), (R, r, s)
                assert kb[0] - kf[0] >= h


ALL_PINS = ["pin_brute_force", "pin_worked_example", "pin_closed_forms", "pin_invariants",
            "pin_merge", "pin_ring"]


def pin_varlen(plant=0):
    """Packed batch == block-diagonal brute force, and == each sequence run on its own."""
    rng = np.random.default_rng(17)
    cu = [3, 3, 10, 11, 30, 52]  # leading padding, an empty sequence, trailing padding
    T = 57
    Hq, Hkv, D = 4, 2, 8
    q = rng.standard_normal((1, Hq, T, D))
    k = rng.standard_normal((1, Hkv, T, D))
    v = rng.standard_normal((1, Hkv, T, D))
    scale = 0.41
    for causal in (False, True):
        o, l = oracle.attention_varlen(q, k, v, cu, causal, scale, plant=plant)
        # brute force with a block-diagonal mask
        G = Hq // Hkv
        kx = np.repeat(k, G, axis=1)
        vx = np.repeat(v, G, axis=1)
        S = scale * np.einsum("bhid,bhjd->bhij", q, kx)
        seq = np.full(T, -1)
        for i in range(len(cu) - 1):
            seq[cu[i]:cu[i + 1]] = i
        vis = (seq[:, None] == seq[None, :]) & (seq[:, None] >= 0)
        if causal:
            vis &= np.tril(np.ones((T, T), bool))
        Pm = np.where(vis, np.exp(S), 0.0)
        Z = Pm.sum(-1)
        with np.errstate(invalid="ignore", divide="ignore"):
            ob = np.where(Z[..., None] > 0, (Pm @ vx) / Z[..., None], 0.0)
            lb = np.where(Z > 0, np.log(Z), -np.inf)
        _close(o, ob, what=f"varlen brute causal={causal}")
        _close(l, lb, what=f"varlen brute LSE causal={causal}")
        # each sequence alone (sliced arrays, no window)
        for i in range(len(cu) - 1):
            a, b = cu[i], cu[i + 1]
            if b <= a:
                continue
            oi, li = oracle.attention(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], causal, scale,
                                      plant=plant)
            _close(o[:, :, a:b], oi, what=f"varlen seq {i} alone")
            _close(l[:, :, a:b], li, what=f"varlen seq {i} alone LSE")


ALL_PINS.append("pin_varlen")


def pin_backward():
    """The gradient oracle against torch autograd (fp64) and central finite differences."""
    import torch

    from oracle import backward as ob

    rng = np.random.default_rng(23)
    for (B, Hq, Hkv, N, D, causal) in [(1, 2, 1, 9, 4, True), (2, 4, 2, 13, 8, False),
                                        (1, 3, 3, 7, 5, True)]:
        q = rng.standard_normal((B, Hq, N, D))
        k = rng.standard_normal((B, Hkv, N, D))
        v = rng.standard_normal((B, Hkv, N, D))
        do = rng.standard_normal((B, Hq, N, D))
        scale = 0.6 / np.sqrt(D)
        dq, dk, dv, o, lse = ob.attention_bwd(q, k, v, do, causal, scale)
        # the forward it differentiates is the oracle's forward
        of, lf = oracle.attention(q, k, v, causal, scale)
        _close(o, of, what="backward oracle forward O")
        _close(lse, lf, what="backward oracle forward LSE")
        # autograd on an independent torch formulation
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        G = Hq // Hkv
        s = scale * torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(G, dim=1))
        if causal:
            s = s.masked_fill(~torch.tril(torch.ones(N, N, dtype=torch.bool)), float("-inf"))
        out = torch.softmax(s, dim=-1) @ tv.repeat_interleave(G, dim=1)
        (out * torch.tensor(do)).sum().backward()
        _close(dq, tq.grad.numpy(), tol=1e-11, what="dq vs autograd")
        _close(dk, tk.grad.numpy(), tol=1e-11, what="dk vs autograd")
        _close(dv, tv.grad.numpy(), tol=1e-11, what="dv vs autograd")
    # central finite differences of L = sum(dO * O) on a tiny case
    B, Hq, Hkv, N, D = 1, 2, 1, 5, 3
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    do = rng.standard_normal((B, Hq, N, D))
    dq, dk, dv, _, _ = ob.attention_bwd(q, k, v, do, True, 0.5)

    def loss(qq, kk, vv):
        o_, _ = oracle.attention(qq, kk, vv, True, 0.5)
        return float(np.sum(do * o_))

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = [q, k, v]; args_m = [q, k, v]
            pos = "qkv".index(name)
            args_p[pos] = xp; args_m[pos] = xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        _close(g, num, tol=1e-7, what=f"d{name} vs finite differences")


def pin_ring_backward():
    """The ring-scheduled gradients against the whole-sequence gradients and, step by
    step, against torch autograd taken with respect to the score matrix.

    - Summed over the R steps they equal ``attention_bwd`` (itself pinned to autograd
      and finite differences) for every layout, ring size, mask and head grouping.
    - Step s of rank r is the gradient through the scores of r's rows against the keys
      of rank (r - s) mod R only: dS and P of the full problem come from autograd on
      S = scale Q K^T (so the D = rowsum(dO * O) term is not retyped here), and the
      step's dQ / dK / dV are their products restricted to that block.
    - Zigzag steps follow the Twinkle page's three cases: for s > r the front query
      chunk of rank r adds nothing; for 0 < s <= r the back key chunk of the held
      block receives nothing.
    """
    import torch

    from oracle import backward as ob

    rng = np.random.default_rng(29)
    B, Hq, Hkv, D = 1, 4, 2, 8
    G = Hq // Hkv
    for (N, R, layout, causal) in [(24, 3, oring.CONTIG, True), (24, 3, oring.ZIGZAG, True),
                                   (24, 4, oring.STRIPED, True), (24, 2, oring.ZIGZAG, False),
                                   (20, 5, oring.STRIPED, False), (16, 1, oring.CONTIG, True),
                                   (32, 4, oring.ZIGZAG, True)]:
        q = rng.standard_normal((B, Hq, N, D))
        k = rng.standard_normal((B, Hkv, N, D))
        v = rng.standard_normal((B, Hkv, N, D))
        do = rng.standard_normal((B, Hq, N, D))
        scale = 0.7 / np.sqrt(D)
        dq, dk, dv, steps = ob.ring_backward(q, k, v, do, R, layout, causal, scale, steps=True)
        fq, fk, fv, _, _ = ob.attention_bwd(q, k, v, do, causal, scale)
        what = f"{layout} R={R} causal={causal}"
        _close(dq, fq, what="ring dq " + what)
        _close(dk, fk, what="ring dk " + what)
        _close(dv, fv, what="ring dv " + what)
        assert len(steps) == R
        # autograd with respect to the scaled scores
        tq, tk = torch.tensor(q), torch.tensor(k).repeat_interleave(G, dim=1)
        S = (scale * torch.einsum("bhid,bhjd->bhij", tq, tk)).detach().requires_grad_(True)
        Sm = S
        if causal:
            Sm = S.masked_fill(~torch.tril(torch.ones(N, N, dtype=torch.bool)), float("-inf"))
        Pt = torch.softmax(Sm, dim=-1)
        (Pt @ torch.tensor(v).repeat_interleave(G, dim=1) * torch.tensor(do)).sum().backward()
        dS = S.grad.numpy()
        Pf = Pt.detach().numpy()
        if layout == oring.STRIPED:
            pos = [np.arange(r, N, R) for r in range(R)]
        elif layout == oring.CONTIG:
            c = N // R
            pos = [np.arange(r * c, (r + 1) * c) for r in range(R)]
        else:
            h2 = N // (2 * R)
            pos = [np.concatenate([np.arange(r * h2, (r + 1) * h2),
                                   np.arange((2 * R - 1 - r) * h2, (2 * R - r) * h2)]) for r in range(R)]
        for s_, (sq, sk, sv) in enumerate(steps):
            eq = np.zeros_like(q)
            ek = np.zeros_like(k)
            ev = np.zeros_like(v)
            for r in range(R):
                j = (r - s_) % R  # the block rank r holds at step s (glossary worked example)
                qp, kp = pos[r], pos[j]
                for h in range(Hq):
                    blk = dS[0, h][np.ix_(qp, kp)]
                    pb = Pf[0, h][np.ix_(qp, kp)]
                    eq[0, h, qp] += scale * blk @ k[0, h // G, kp]
                    ek[0, h // G, kp] += scale * blk.T @ q[0, h, qp]
                    ev[0, h // G, kp] += pb.T @ do[0, h, qp]
            _close(sq, eq, tol=1e-11, what=f"step {s_} dq " + what)
            _close(sk, ek, tol=1e-11, what=f"step {s_} dk " + what)
            _close(sv, ev, tol=1e-11, what=f"step {s_} dv " + what)
            if layout == oring.ZIGZAG and causal:
                h2 = N // (2 * R)
                for r in range(R):
                    j = (r - s_) % R
                    case = oring.zigzag_step_case(r, s_, R)
                    if case == "back_q":
                        assert not np.any(sq[:, :, r * h2:(r + 1) * h2]), what
                    if case == "front_kv":
                        back = slice((2 * R - 1 - j) * h2, (2 * R - j) * h2)
                        assert not np.any(sk[:, :, back]) or R == 1, what


def pin_gradient_rows():
    """Gradient rows computed one by one equal the rows of the whole-problem gradients."""
    from oracle import backward as ob

    rng = np.random.default_rng(31)
    for causal, (B, Hq, Hkv, N, D) in [(True, (2, 4, 2, 37, 8)), (False, (1, 3, 1, 29, 5)),
                                       (True, (1, 2, 2, 1, 4))]:
        q = rng.standard_normal((B, Hq, N, D))
        k = rng.standard_normal((B, Hkv, N, D))
        v = rng.standard_normal((B, Hkv, N, D))
        do = rng.standard_normal((B, Hq, N, D))
        fq, fk, fv, _, _ = ob.attention_bwd(q, k, v, do, causal, 0.45)
        qr = np.array([(b, h, i) for b in range(B) for h in range(Hq) for i in {0, N // 2, N - 1}])
        kr = np.array([(b, h, j) for b in range(B) for h in range(Hkv) for j in {0, N // 3, N - 1}])
        gq, gk, gv = ob.gradient_rows(q, k, v, do, causal, 0.45, qr, kr)
        _close(gq, fq[qr[:, 0], qr[:, 1], qr[:, 2]], what="dq rows")
        _close(gk, fk[kr[:, 0], kr[:, 1], kr[:, 2]], what="dk rows")
        _close(gv, fv[kr[:, 0], kr[:, 1], kr[:, 2]], what="dv rows")


def pin_ulysses():
    """The all-to-all restatement: round trip, element formula, labelled example."""
    from oracle import ulysses as ou

    rng = np.random.default_rng(31)
    for sp, S, H, D in [(1, 8, 4, 3), (2, 8, 4, 3), (4, 12, 8, 2), (8, 16, 8, 5)]:
        x = rng.standard_normal((sp, S // sp, H, D))
        y = ou.seq_to_heads(x, sp)
        assert y.shape == (sp, S, H // sp, D)
        assert np.array_equal(ou.heads_to_seq(y, sp), x), "round trip"
        ss, hs = S // sp, H // sp
        for _ in range(50):
            r, s, j = rng.integers(sp), rng.integers(S), rng.integers(hs)
            assert np.array_equal(y[r, s, j], x[s // ss, s % ss, r * hs + j])
    # labelled: value = 1000 * position + head; rank r must hold the whole sequence of
    # its heads, positions in order
    sp, S, H = 4, 8, 8
    lab = np.zeros((sp, S // sp, H, 1))
    for r in range(sp):
        for i in range(S // sp):
            for h in range(H):
                lab[r, i, h, 0] = 1000 * (r * (S // sp) + i) + h
    y = ou.seq_to_heads(lab, sp)
    for r in range(sp):
        want = np.array([[1000 * p + h for h in range(r * 2, r * 2 + 2)] for p in range(S)])
        assert np.array_equal(y[r, :, :, 0], want)
