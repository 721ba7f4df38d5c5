"""GPU parity of the strided entry point (dit_attn_fwd_strided) against the fp64 oracle.

The token-major BSND layout ([B, N, H, D] in memory) is how the pages' sequence-parallel
code holds activations (MindIE-SD parallelism docs; valdrada.cn Wan2.2, CP section).  The
oracle always computes on contiguous BHND copies of the same bf16 values, so a layout or
stride mistake anywhere in the kernel's addressing shows as a mismatch.  Same tolerances as
the contiguous path: O max-abs 1e-2 / mean-abs 1e-3, LSE 1e-3 (bf16 output: one bf16 ulp).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import ditattn as da
from diffusion_transformer_long_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def bf16_ulp(x):
    a = np.abs(x).astype(np.float64)
    return np.power(2.0, np.floor(np.log2(np.maximum(a, 1e-30))) - 7)


def check(o, lse, o_ref, lse_ref, what, bf16_out=False):
    o = o.double().cpu().numpy()
    err = np.abs(o - o_ref)
    bound = np.maximum(1e-2, bf16_ulp(o_ref)) if bf16_out else 1e-2
    assert (err <= bound).all(), f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= 1e-3, f"{what}: mean-abs {err.mean():.3e}"
    lerr = np.abs(lse.double().cpu().numpy() - lse_ref).max()
    assert lerr <= 1e-3, f"{what}: lse {lerr:.3e}"


def rand_bhnd(B, H, N, D, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, H, N, D, generator=g) * scale).to(torch.bfloat16)


def as_bsnd(x):
    """A [B, H, N, D] logical view over token-major memory holding the same values."""
    return x.transpose(1, 2).contiguous().to(DEV).transpose(1, 2)


@pytest.mark.parametrize("B,H,N,D", [(1, 2, 129, 64), (2, 3, 300, 128), (1, 24, 1000, 128),
                                     (2, 1, 513, 64)])
def test_bsnd_everywhere(B, H, N, D):
    q, k, v = (rand_bhnd(B, H, N, D, seed=N + i, scale=1.3) for i in range(3))
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = as_bsnd(q), as_bsnd(k), as_bsnd(v)
    assert qd.stride(2) == H * D and qd.stride(3) == 1  # token-major rows
    out_mem = torch.full((B, N, H, D), math.nan, device=DEV)
    o, lse = da.attn_fwd_strided(qd, kd, vd, out=out_mem.transpose(1, 2), scale=scale)
    da.check()
    assert torch.isfinite(out_mem).all()
    check(o, lse, o_ref, lse_ref, f"BSND {B}x{H}x{N}x{D}")


def test_mixed_layouts_bf16_out_and_padded_rows():
    """q token-major, k/v head-major with padded rows (row stride D + 64), bf16 output
    token-major with padded heads: every view addressed through its own strides."""
    B, H, N, D = 2, 3, 700, 128
    q, k, v = (rand_bhnd(B, H, N, D, seed=40 + i, scale=1.5) for i in range(3))
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd = as_bsnd(q)
    kpad = torch.zeros(B, H, N, D + 64, dtype=torch.bfloat16, device=DEV)
    vpad = torch.zeros(B, H, N, D + 64, dtype=torch.bfloat16, device=DEV)
    kpad[..., :D] = k.to(DEV)
    vpad[..., :D] = v.to(DEV)
    out_mem = torch.zeros(B, N, H, D + 128, dtype=torch.bfloat16, device=DEV)
    out = out_mem[..., :D].transpose(1, 2)
    o, lse = da.attn_fwd_strided(qd, kpad[..., :D], vpad[..., :D], out=out, scale=scale)
    da.check()
    assert (out_mem[..., D:] == 0).all()  # padding untouched
    check(o, lse, o_ref, lse_ref, "mixed layouts, bf16 out", bf16_out=True)


def test_contiguous_strides_match_dedicated_entry_points_bitwise():
    w = synth.WORKLOADS["flux"]
    q, k, v = (t.to(DEV) for t in synth.make_qkv(w))
    o1, l1 = da.attn_fwd(q, k, v, scale=w.scale)
    o2, l2 = da.attn_fwd_strided(q, k, v, scale=w.scale)
    s, n = 1152, 1152
    o3, l3 = da.attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], scale=w.scale)
    o4, l4 = da.attn_fwd_strided(q, k[:, :, s:s + n], v[:, :, s:s + n], scale=w.scale)
    da.check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o3, o4) and torch.equal(l3, l4)


def test_bsnd_chunk_views_merge_to_full_attention():
    """Ring chunks as token-range views of token-major K/V, merged by the LSE merge."""
    B, H, N, D = 1, 4, 900, 128
    q, k, v = (rand_bhnd(B, H, N, D, seed=60 + i) for i in range(3))
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = as_bsnd(q), as_bsnd(k), as_bsnd(v)
    chunks = (200, 333, 367)
    parts = torch.empty(len(chunks), B, H, N, D, device=DEV)
    lses = torch.empty(len(chunks), B, H, N, device=DEV)
    s = 0
    for c, n in enumerate(chunks):
        da.attn_fwd_strided(qd, kd[:, :, s:s + n], vd[:, :, s:s + n], out=parts[c], lse=lses[c],
                            scale=scale)
        s += n
    o, lse = da.attn_lse_merge(parts, lses)
    da.check()
    check(o, lse, o_ref, lse_ref, "BSND chunk views + merge")
