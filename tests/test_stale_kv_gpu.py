"""GPU parity of stale-KV attention (dit_attn_stale_kv_fwd) against the fp64 oracle.

Displaced patch parallelism (PipeFusion / DistriFusion: arganzheng.life multi-GPU diffusion
parallelism, section 6 PipeFusion; xllm-io review of PipeFusion, method section) keeps a
KV buffer of all N tokens from the previous diffusion step; a patch's fresh K/V rows
replace their stale rows and the patch's queries attend to the whole buffer.  The oracle
applies the same row replacement to CPU copies of the buffers, then computes plain
attention over them; the buffers must equal that replacement bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import ditattn as da

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("B,H,N,m,row0,D", [
    (1, 2, 1024, 256, 256, 128), (1, 3, 1000, 250, 750, 64), (2, 2, 777, 130, 0, 128),
    (1, 24, 4608, 1152, 2304, 128), (1, 1, 300, 300, 0, 128), (1, 2, 513, 1, 512, 64)])
def test_stale_kv_patch_vs_oracle(B, H, N, m, row0, D):
    k_buf, v_buf = rand((B, H, N, D), seed=1), rand((B, H, N, D), seed=2)
    q = rand((B, H, m, D), seed=3, scale=1.3)
    k_new, v_new = rand((B, H, m, D), seed=4, scale=1.3), rand((B, H, m, D), seed=5)
    scale = 1 / math.sqrt(D)
    k_ref, v_ref = k_buf.clone(), v_buf.clone()
    k_ref[:, :, row0:row0 + m] = k_new
    v_ref[:, :, row0:row0 + m] = v_new
    o_ref, lse_ref = oracle.attention(q, k_ref, v_ref, scale)
    kb, vb = k_buf.to(DEV), v_buf.to(DEV)
    o, lse = da.stale_kv_attention(q.to(DEV), k_new.to(DEV), v_new.to(DEV), kb, vb, row0,
                                   scale=scale)
    da.check()
    assert torch.equal(kb.cpu(), k_ref) and torch.equal(vb.cpu(), v_ref)
    err = np.abs(o.double().cpu().numpy() - o_ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, (err.max(), err.mean())
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3


def test_stale_rows_matter():
    """With stale rows that differ from the fresh ones, the result differs from attention over
    an all-fresh buffer, and matches it when the stale rows are replaced everywhere."""
    B, H, N, m, D = 1, 2, 512, 128, 128
    k_fresh, v_fresh = rand((B, H, N, D), seed=6), rand((B, H, N, D), seed=7)
    q = rand((B, H, m, D), seed=8)
    kb = rand((B, H, N, D), seed=9).to(DEV)
    vb = rand((B, H, N, D), seed=10).to(DEV)
    row0 = 128
    kf, vf = k_fresh.to(DEV), v_fresh.to(DEV)
    o_stale, _ = da.stale_kv_attention(q.to(DEV), kf[:, :, row0:row0 + m].contiguous(),
                                       vf[:, :, row0:row0 + m].contiguous(), kb, vb, row0)
    o_fresh, _ = da.attn_chunk_fwd(q.to(DEV), kf, vf)
    da.check()
    assert (o_stale - o_fresh).abs().max().item() > 1e-2
    for r in range(0, N, m):  # refresh every patch: the buffer becomes all fresh
        da.stale_kv_attention(q.to(DEV), kf[:, :, r:r + m].contiguous(),
                              vf[:, :, r:r + m].contiguous(), kb, vb, r)
    o_all, _ = da.stale_kv_attention(q.to(DEV), kf[:, :, row0:row0 + m].contiguous(),
                                     vf[:, :, row0:row0 + m].contiguous(), kb, vb, row0)
    da.check()
    assert torch.equal(kb, kf) and torch.equal(vb, vf)
    assert torch.equal(o_all, o_fresh)
