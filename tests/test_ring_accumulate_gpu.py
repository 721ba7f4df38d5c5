"""GPU parity of the hop-by-hop ring (dit_attn_chunk_fwd_accumulate) against the fp64 oracle.

One hop merges the attention of the queries against one KV chunk into a running (O, lse):
  M = max(lse_run, lse_c), lse' = M + ln(e^(lse_run-M) + e^(lse_c-M)),
  O' = e^(lse_run-lse') O_run + e^(lse_c-lse') O_c
(arganzheng.life multi-GPU diffusion parallelism, section 4.2 Ring: online-softmax
accumulation over the ring rounds).  The expected value of one hop is the oracle's own
two-way LSE merge of the given running state with the oracle's attention over the chunk.
Tolerances as for the chunk partials: O max-abs 1e-2 / mean-abs 1e-3, LSE 1e-3; a merge
of exact partials adds only fp32 rounding.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import ditattn as da

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


def rand_qkv(B, H, N, D, seed, nk=None, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    nk = N if nk is None else nk
    q = (torch.randn(B, H, N, D, generator=g) * scale).to(torch.bfloat16)
    k = (torch.randn(B, H, nk, D, generator=g) * scale).to(torch.bfloat16)
    v = torch.randn(B, H, nk, D, generator=g).to(torch.bfloat16)
    return q, k, v


def check(o, lse, o_ref, lse_ref, what):
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    err = np.abs(o - o_ref)
    assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_ABS, f"{what}: lse {np.abs(lse - lse_ref).max():.3e}"


def running_state(B, H, N, D, seed, lse_of_chunk):
    """A random running (O, lse): lse_run around the chunk's own LSE, with rows far below it,
    far above it, and empty (-inf, O_run = NaN, which must never be read)."""
    g = torch.Generator().manual_seed(seed)
    o_run = torch.randn(B, H, N, D, generator=g)
    lse_run = torch.from_numpy(lse_of_chunk).float() + torch.randn(B, H, N, generator=g) * 2
    lse_run[..., 0::7] -= 60.0   # negligible running weight
    lse_run[..., 3::7] += 60.0   # negligible chunk weight
    lse_run[..., 5::11] = -math.inf
    o_run[..., 5::11, :] = math.nan
    return o_run, lse_run


@pytest.mark.parametrize("B,H,N,n_kv,D", [
    (1, 1, 1, 1, 64), (1, 2, 129, 200, 128), (2, 1, 333, 128, 64), (1, 3, 700, 315, 128),
    (2, 2, 1000, 513, 128)])
def test_one_hop_vs_oracle_merge(B, H, N, n_kv, D):
    q, k, v = rand_qkv(B, H, N, D, seed=N + n_kv, nk=n_kv, scale=1.4)
    scale = 1 / math.sqrt(D)
    o_c, lse_c = oracle.attention(q, k, v, scale)
    o_run, lse_run = running_state(B, H, N, D, seed=D + N, lse_of_chunk=lse_c)
    o_prev = np.nan_to_num(o_run.double().numpy())  # empty rows carry weight 0
    o_ref, lse_ref = oracle.lse_merge(np.stack([o_prev, o_c]),
                                      np.stack([lse_run.double().numpy(), lse_c]))
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = o_run.to(DEV), lse_run.to(DEV)
    da.attn_chunk_fwd_accumulate(qd, kd, vd, o, lse, scale=scale)
    da.check()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check(o, lse, o_ref, lse_ref, f"one hop {B}x{H}x{N}, n_kv={n_kv}, D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_ring_any_order_and_mixed_start(D):
    """All chunks folded in, in two different orders, from an empty state and from a first
    chunk computed by dit_attn_chunk_fwd, with one chunk as a packed buffer: every result is
    the full attention."""
    B, H, N = 2, 2, 700
    chunks = (1, 127, 128, 129, 315)
    starts = np.cumsum((0,) + chunks[:-1])
    q, k, v = rand_qkv(B, H, N, D, seed=31 + D, scale=1.5)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))

    def fold(order, first_plain):
        o = torch.empty(B, H, N, D, device=DEV)
        lse = torch.full((B, H, N), -math.inf, device=DEV)
        for i, c in enumerate(order):
            s, n = int(starts[c]), chunks[c]
            kc, vc = kd[:, :, s:s + n], vd[:, :, s:s + n]
            if c == 3:  # packed chunk buffer, head stride n_kv*D
                kc, vc = kc.contiguous(), vc.contiguous()
            if i == 0 and first_plain:
                da.attn_chunk_fwd(qd, kc, vc, out=o, lse=lse, scale=scale)
            else:
                da.attn_chunk_fwd_accumulate(qd, kc, vc, o, lse, scale=scale)
        da.check()
        return o, lse

    o1, l1 = fold((0, 1, 2, 3, 4), first_plain=False)
    o2, l2 = fold((4, 2, 0, 3, 1), first_plain=True)
    check(o1, l1, o_ref, lse_ref, f"ring in order D={D}")
    check(o2, l2, o_ref, lse_ref, f"ring reordered D={D}")
    assert (o1 - o2).abs().max().item() <= 2e-3


def test_equals_separate_merge_and_fused():
    B, H, N, D = 1, 4, 2000, 128
    q, k, v = (t.to(DEV) for t in rand_qkv(B, H, N, D, seed=8))
    chunks = (500, 500, 500, 500)
    o_f, l_f = da.attn_fwd(q, k, v)
    o_m, l_m = da.chunk_attention(q, k, v, chunks)
    o_r, l_r = da.ring_attention(q, k, v, chunks)
    da.check()
    for o, l in ((o_f, l_f), (o_m, l_m)):
        d = (o_r - o).abs()
        assert d.max().item() <= 2e-3 and d.mean().item() <= 1e-4
        assert (l_r - l).abs().max().item() <= 1e-4


CANARY = -1.2345e30


def test_canaries_and_16_byte_aligned_running_output():
    """Running state as slices of larger buffers, o_run 16- but not 32-byte aligned: nothing
    outside is touched and the result equals the 32-byte-aligned one."""
    B, H, N, D, pad = 1, 2, 333, 128, 1028  # pad*4 = 16 (mod 32)
    q, k, v = (t.to(DEV) for t in rand_qkv(B, H, N, D, seed=77))
    n_o, n_l = B * H * N * D, B * H * N
    big = torch.full((n_o + 2 * pad,), CANARY, device=DEV)
    big_l = torch.full((n_l + 2 * pad,), CANARY, device=DEV)
    o = big[pad:pad + n_o].view(B, H, N, D)
    lse = big_l[pad:pad + n_l].view(B, H, N)
    assert o.data_ptr() % 32 == 16
    chunks = (100, 133, 100)
    da.ring_attention(q, k, v, chunks, o_run=o, lse_run=lse)
    o_al, l_al = da.ring_attention(q, k, v, chunks)
    da.check()
    for buf, n in ((big, n_o), (big_l, n_l)):
        assert (buf[:pad] == CANARY).all() and (buf[pad + n:] == CANARY).all()
    assert torch.equal(o, o_al) and torch.equal(lse, l_al)
    o_ref, lse_ref = oracle.attention(*(t.cpu() for t in (q, k, v)), 1 / math.sqrt(D))
    check(o, lse, o_ref, lse_ref, "16-byte-aligned running output")
