"""The Ulysses exchange through the C ABI: exact against the oracle's restatement, and
scatter-heads -> per-rank attention -> gather-sequence equals plain attention."""
import numpy as np
import pytest
import torch

from exact_long_context_gb300 import synth
from oracle import ulysses as ou

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_long_context_gb300 import build
    build.build()
    from exact_long_context_gb300 import ra as ra_mod
    return ra_mod


@pytest.mark.parametrize("sp,S,H,D,dtype", [
    (2, 256, 4, 128, torch.bfloat16), (4, 1024, 8, 64, torch.bfloat16), (8, 512, 8, 128, torch.float32),
    (4, 96, 4, 24, torch.bfloat16), (1, 64, 2, 16, torch.float32), (3, 99, 6, 7, torch.float32),
])
def test_transform_is_exact(ra, sp, S, H, D, dtype):
    g = torch.Generator(device="cuda").manual_seed(S + H)
    x = torch.randn(sp, S // sp, H, D, generator=g, device="cuda").to(dtype)
    y = ra.ulysses_all_to_all(x, sp, to_heads=True)
    back = ra.ulysses_all_to_all(y, sp, to_heads=False)
    ra.check()
    view = (lambda t: t.cpu().view(torch.int16).numpy()) if dtype == torch.bfloat16 else (lambda t: t.cpu().numpy())
    assert np.array_equal(view(y), ou.seq_to_heads(view(x), sp))
    assert torch.equal(back, x)


@pytest.mark.parametrize("sp,Hq,Hkv", [(2, 8, 4), (4, 8, 4), (4, 16, 4)])
def test_ulysses_attention_equals_plain_attention(ra, sp, Hq, Hkv):
    S, D = 2048, 128
    q, k, v = synth.make_qkv(1, Hq, Hkv, S, D, torch.bfloat16, seed=sp * 10 + Hq, device="cuda")
    # the sequence axis sharded over sp ranks: [sp, S/sp, H, D]
    shard = lambda t: t[0].transpose(0, 1).reshape(sp, S // sp, t.shape[1], D).contiguous()
    qh, kh, vh = (ra.ulysses_all_to_all(shard(t), sp, to_heads=True) for t in (q, k, v))
    # each rank: whole sequence, H/sp heads -> attention over [B = sp, H/sp, S, D] views
    oh = torch.empty_like(qh)
    lse = torch.empty(sp, Hq // sp, S, device="cuda")
    ra.attn_fwd(qh.transpose(1, 2), kh.transpose(1, 2), vh.transpose(1, 2), causal=True,
                o=oh.transpose(1, 2), lse=lse)
    o_seq = ra.ulysses_all_to_all(oh, sp, to_heads=False)  # back to sequence shards
    o_ref, lse_ref = ra.attn_fwd(q, k, v, causal=True)
    ra.check()
    o_full = o_seq.reshape(S, Hq, D).transpose(0, 1).unsqueeze(0)
    assert torch.equal(o_full, o_ref)
    assert torch.equal(lse.reshape(Hq, S).unsqueeze(0), lse_ref)
