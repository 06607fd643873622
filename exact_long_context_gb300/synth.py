"""Seeded synthetic inputs.  Holds no attention arithmetic: random draws and shapes only.

Recipe: Q, K, V are drawn in that order; each tensor is filled head by head,
(b, h) in row-major order, with an N x D block of float32 standard normals from a
``torch.Generator`` seeded with the workload's seed on the requested device, then
rounded once to the workload dtype (bfloat16 round-to-nearest-even, or kept fp32).
The tiny workload instead draws ``torch.randn(3, 32, 16)`` after
``torch.manual_seed(0)`` on the CPU, exactly as the worked example of the "Ring
Attention" glossary page (ultralytics.com) does, and splits it into q, k, v.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    dtype: torch.dtype
    causal: bool
    ring_size: int
    layout: str  # "contig" or "zigzag"
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        """Causal-adjusted attention FLOPs: 4*B*Hq*N^2*D, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.D
        return f / 2 if self.causal else f


WORKLOADS = {
    "tiny_ring4_fp32": Workload("tiny_ring4_fp32", 1, 1, 1, 32, 16, torch.float32, False, 4,
                                "contig", 0),
    "dense_causal_b2h32n4k": Workload("dense_causal_b2h32n4k", 2, 32, 32, 4096, 128,
                                      torch.bfloat16, True, 1, "contig", 2),
    "ring8_zigzag_h8n32k": Workload("ring8_zigzag_h8n32k", 1, 8, 8, 32768, 128, torch.bfloat16,
                                    True, 8, "zigzag", 3),
    # the same inputs as the zigzag ring: an A/B of the two partitions
    "ring8_contig_h8n32k": Workload("ring8_contig_h8n32k", 1, 8, 8, 32768, 128, torch.bfloat16,
                                    True, 8, "contig", 3),
    "ring8_striped_h8n32k": Workload("ring8_striped_h8n32k", 1, 8, 8, 32768, 128, torch.bfloat16,
                                     True, 8, "striped", 3),
    "gqa_ring16_zigzag_h32kv8n128k": Workload("gqa_ring16_zigzag_h32kv8n128k", 1, 32, 8, 131072,
                                              128, torch.bfloat16, True, 16, "zigzag", 4),
    "ring64_zigzag_h8kv2n1m": Workload("ring64_zigzag_h8kv2n1m", 1, 8, 2, 1048576, 128,
                                       torch.bfloat16, True, 64, "zigzag", 5),
    # head size 64 (the other tensor-core head size): the dense and ring shapes at D = 64
    "dense_causal_b2h32n4k_d64": Workload("dense_causal_b2h32n4k_d64", 2, 32, 32, 4096, 64,
                                          torch.bfloat16, True, 1, "contig", 6),
    "ring8_zigzag_h16n32k_d64": Workload("ring8_zigzag_h16n32k_d64", 1, 16, 16, 32768, 64,
                                         torch.bfloat16, True, 8, "zigzag", 7),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of variable-length sequences (cu_seqlens).

    Sequence lengths are drawn log-uniformly in [min_len, max_len] with numpy's
    default_rng(seed) until ``total`` tokens are filled (the last one is cut to fit).
    """
    name: str
    Hq: int
    Hkv: int
    D: int
    dtype: torch.dtype
    causal: bool
    total: int
    min_len: int
    max_len: int
    seed: int
    B: int = 1
    ring_size: int = 1
    layout: str = "packed"

    @property
    def N(self) -> int:
        return self.total

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def lengths(self):
        import numpy as np

        rng = np.random.default_rng(self.seed)
        out, used = [], 0
        while used < self.total:
            n = int(round(math.exp(rng.uniform(math.log(self.min_len), math.log(self.max_len)))))
            n = min(n, self.total - used)
            out.append(n)
            used += n
        return out

    def cu_seqlens(self):
        cu = [0]
        for n in self.lengths():
            cu.append(cu[-1] + n)
        return cu

    def flops(self) -> float:
        f = sum(4.0 * self.Hq * n * n * self.D for n in self.lengths())
        return f / 2 if self.causal else f


VARLEN_WORKLOADS = {
    "varlen_causal_h32kv8_128k": VarlenWorkload("varlen_causal_h32kv8_128k", 32, 8, 128,
                                                torch.bfloat16, True, 131072, 256, 16384, 6),
}


def _fill(shape, gen, device, dtype):
    B, H, N, D = shape
    out = torch.empty(shape, dtype=dtype, device=device)
    for b in range(B):
        for h in range(H):
            blk = torch.randn((N, D), generator=gen, device=device, dtype=torch.float32)
            out[b, h].copy_(blk)  # copy_ rounds to the target dtype (RNE for bfloat16)
    return out


def make_qkv(B, Hq, Hkv, N, D, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Seeded q [B,Hq,N,D], k and v [B,Hkv,N,D] (see the module recipe)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _fill((B, Hq, N, D), gen, device, dtype)
    k = _fill((B, Hkv, N, D), gen, device, dtype)
    v = _fill((B, Hkv, N, D), gen, device, dtype)
    return q, k, v


def worked_example_qkv():
    """The glossary page's worked-example inputs as [1, 1, 32, 16] float32 tensors."""
    torch.manual_seed(0)
    q, k, v = torch.randn(3, 32, 16)
    return (q.reshape(1, 1, 32, 16).contiguous(), k.reshape(1, 1, 32, 16).contiguous(),
            v.reshape(1, 1, 32, 16).contiguous())


def workload_inputs(w, device="cpu"):
    if w.name == "tiny_ring4_fp32":
        q, k, v = worked_example_qkv()
        return q.to(device), k.to(device), v.to(device)
    if isinstance(w, VarlenWorkload):
        return make_qkv(1, w.Hq, w.Hkv, w.total, w.D, w.dtype, w.seed, device)
    return make_qkv(w.B, w.Hq, w.Hkv, w.N, w.D, w.dtype, w.seed, device)
