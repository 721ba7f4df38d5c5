"""GPU parity of split-KV attention (dit_attn_chunk_fwd_splitkv) against the fp64 oracle.

Every (head, Q pair) work item is split over contiguous ranges of the key tiles; the fp32
partials land in a caller-provided workspace and are merged exactly (the LSE combination the
Ring section of arganzheng.life's multi-GPU diffusion parallelism page implies).  The
result must be full attention over all keys, within the path's tolerances (O max-abs 1e-2,
mean-abs 1e-3, LSE 1e-3), and match the unsplit pass to fp32 merge rounding.
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


def check(o, lse, o_ref, lse_ref, what, bf16_out=False):
    o = o.double().cpu().numpy()
    err = np.abs(o - o_ref)
    if bf16_out:
        ulp = np.power(2.0, np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 7)
        assert (err <= np.maximum(1e-2, ulp)).all(), f"{what}: max-abs {err.max():.3e}"
    else:
        assert err.max() <= 1e-2, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= 1e-3, f"{what}: mean-abs {err.mean():.3e}"
    lerr = np.abs(lse.double().cpu().numpy() - lse_ref).max()
    assert lerr <= 1e-3, f"{what}: lse {lerr:.3e}"


@pytest.mark.parametrize("B,H,Nq,nkv,D,splits", [
    (1, 2, 300, 2000, 128, 3), (2, 3, 129, 1000, 64, 7), (1, 4, 1000, 5000, 128, 5),
    (1, 1, 64, 8192, 128, 64), (1, 2, 513, 300, 128, 3), (2, 1, 1, 1200, 64, 2)])
def test_splitkv_vs_oracle(B, H, Nq, nkv, D, splits):
    q = rand((B, H, Nq, D), seed=Nq, scale=1.4)
    k, v = rand((B, H, nkv, D), seed=nkv, scale=1.4), rand((B, H, nkv, D), seed=nkv + 1)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = da.attn_chunk_fwd_splitkv(qd, kd, vd, scale=scale, splits=splits)
    o1, l1 = da.attn_chunk_fwd(qd, kd, vd, scale=scale)
    da.check()
    check(o, lse, o_ref, lse_ref, f"split-KV S={splits} {B}x{H}x{Nq}x{nkv}x{D}")
    # Split and unsplit passes round P to bf16 against different running maxima, so they
    # differ by that rounding (largest for these x1.4 scores); the oracle check is the gate.
    assert (o - o1).abs().max().item() <= 5e-3 and (lse - l1).abs().max().item() <= 1e-4


def test_splitkv_bf16_out_views_and_workspace_bounds():
    B, H, Nq, N, D, S = 1, 3, 500, 3000, 128, 4
    q = rand((B, H, Nq, D), seed=1)
    k, v = rand((B, H, N, D), seed=2), rand((B, H, N, D), seed=3)
    s0, n = 700, 1900  # a chunk view of the keys
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, kv_start=s0, kv_len=n)
    need = da.lib().dit_attn_splitkv_workspace_bytes(B, H, Nq, D, S)
    pad = 4096
    ws = torch.full((need + pad,), 0xAB, dtype=torch.uint8, device=DEV)
    kd, vd = k.to(DEV), v.to(DEV)
    o, lse = da.attn_chunk_fwd_splitkv(q.to(DEV), kd[:, :, s0:s0 + n], vd[:, :, s0:s0 + n],
                                       scale=scale, out_dtype=torch.bfloat16, splits=S,
                                       workspace=ws)
    da.check()
    assert (ws[need:] == 0xAB).all()  # nothing written past the declared workspace
    check(o, lse, o_ref, lse_ref, "split-KV bf16 out over a chunk view", bf16_out=True)


def test_suggestion_and_capped_grid():
    """The suggestion splits a few-query problem, and a capped persistent grid (each CTA
    walking many items whose key ranges differ by a tile) gives the same result."""
    B, H, Nq, N, D = 1, 2, 256, 27280, 128
    assert da.lib().dit_attn_splitkv_suggest(B, H, Nq, N) > 1
    assert da.lib().dit_attn_splitkv_suggest(1, 24, 27280, 27280) == 1
    q = rand((B, H, Nq, D), seed=4)
    k, v = rand((B, H, N, D), seed=5), rand((B, H, N, D), seed=6)
    o_ref, lse_ref = oracle.attention(q, k, v, 1 / math.sqrt(D))
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = da.attn_chunk_fwd_splitkv(qd, kd, vd)  # suggested split count
    da.set_grid_limit(3)
    try:
        o3, l3 = da.attn_chunk_fwd_splitkv(qd, kd, vd, splits=7)
        da.check()
    finally:
        da.set_grid_limit(0)
    check(o, lse, o_ref, lse_ref, "suggested split")
    check(o3, l3, o_ref, lse_ref, "split 7 on 3 CTAs")


@pytest.mark.parametrize("limit", [0, 3])
def test_short_ranges_staged_partials_on_capped_grid(limit):
    """Split ranges of at most 16 key tiles take the short-item form, whose fp32 partials go
    out through the partly staged TMA stores (the output map's range dimension): 16 ranges of
    13-14 tiles over 27280 keys, the grid capped so that each CTA walks many items of
    different ranges; ragged query count."""
    B, H, Nq, N, D, S = 1, 3, 333, 27280, 128, 16
    q = rand((B, H, Nq, D), seed=12)
    k, v = rand((B, H, N, D), seed=13), rand((B, H, N, D), seed=14)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    da.set_grid_limit(limit)
    try:
        o, lse = da.attn_chunk_fwd_splitkv(qd, kd, vd, scale=scale, splits=S)
        ob, lb = da.attn_chunk_fwd_splitkv(qd, kd, vd, scale=scale, splits=S,
                                           out_dtype=torch.bfloat16)
        da.check()
    finally:
        da.set_grid_limit(0)
    check(o, lse, o_ref, lse_ref, f"split {S} short ranges, grid {limit}")
    check(ob, lb, o_ref, lse_ref, f"split {S} short ranges bf16 out, grid {limit}", bf16_out=True)


def test_stale_kv_with_splits():
    B, H, N, m, row0, D = 1, 4, 4096, 512, 1024, 128
    k_buf, v_buf = rand((B, H, N, D), seed=7), rand((B, H, N, D), seed=8)
    q = rand((B, H, m, D), seed=9, scale=1.3)
    k_new, v_new = rand((B, H, m, D), seed=10, scale=1.3), rand((B, H, m, D), seed=11)
    k_ref, v_ref = k_buf.clone(), v_buf.clone()
    k_ref[:, :, row0:row0 + m] = k_new
    v_ref[:, :, row0:row0 + m] = v_new
    o_ref, lse_ref = oracle.attention(q, k_ref, v_ref, 1 / math.sqrt(D))
    kb, vb = k_buf.to(DEV), v_buf.to(DEV)
    o, lse = da.stale_kv_attention(q.to(DEV), k_new.to(DEV), v_new.to(DEV), kb, vb, row0,
                                   splits=None)
    da.check()
    assert torch.equal(kb.cpu(), k_ref) and torch.equal(vb.cpu(), v_ref)
    check(o, lse, o_ref, lse_ref, "stale-KV, suggested splits")


def test_split_suggestion_follows_the_cost_estimate():
    """The suggestion keeps patches whose items already fill the grid unsplit (FLUX, CFG and
    Wan2.1 patch shapes, where splitting measured slower), and splits a Wan2.2 patch (336
    items of 214 tiles: 3 waves unsplit) into 3 or 4 ranges."""
    L = da.lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with torch.cuda.device(0):
        assert L.dit_attn_splitkv_suggest(1, 24, 1152, 4608) == 1     # FLUX patch
        assert L.dit_attn_splitkv_suggest(2, 24, 1536, 4608) == 1     # CFG patch
        assert L.dit_attn_splitkv_suggest(1, 40, 9450, 75600) == 1    # Wan2.1 patch
        s = L.dit_attn_splitkv_suggest(1, 24, 3410, 27280)            # Wan2.2 patch
        if sms == 152:
            assert s in (3, 4)
        assert 1 <= s <= 16
        assert L.dit_attn_splitkv_suggest(1, 1, 64, 128) == 1         # one key tile: no split
