"""All virtual ranks of the ring decomposition in one launch (dit_attn_chunks_fwd).

The batched launch must give, bit for bit, the partials of one dit_attn_chunk_fwd per chunk
(the same tiles are computed in the same order; keys past a chunk's end are masked, so their
probabilities are exactly 0 whether the rows hold the next chunk or zero fill), and merged by
dit_attn_lse_merge it must match the fp64 oracle within the parity tolerances.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import ditattn as da
from diffusion_transformer_long_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3
DEV = torch.device("cuda:0")


def rand_qkv(B, H, nq, nk, D, seed, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, nq, D, generator=g) * amp).to(torch.bfloat16)
    k = (torch.randn(B, H, nk, D, generator=g) * amp).to(torch.bfloat16)
    v = torch.randn(B, H, nk, D, generator=g).to(torch.bfloat16)
    return q, k, v


def per_chunk(q, k, v, chunks, scale, dtype):
    p = len(chunks)
    B, H, Nq, D = q.shape
    parts = torch.empty(p, B, H, Nq, D, device=DEV, dtype=dtype)
    lses = torch.empty(p, B, H, Nq, device=DEV)
    s = 0
    for c, n in enumerate(chunks):
        da.attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], out=parts[c], lse=lses[c],
                          scale=scale)
        s += n
    return parts, lses


def check(o, lse, o_ref, lse_ref, what):
    o = o.double().cpu().numpy()
    err = np.abs(o - o_ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"{what}: {err.max():.3e} {err.mean():.3e}"
    lerr = np.abs(lse.double().cpu().numpy() - lse_ref).max()
    assert lerr <= LSE_ABS, f"{what}: lse {lerr:.3e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunks", [(700,), (1, 127, 128, 129, 315), (300, 400), (90, 610)])
def test_batched_equals_per_chunk_and_oracle(D, dtype, chunks):
    B, H, Nq, nk = 2, 2, 333, sum(chunks)
    q, k, v = rand_qkv(B, H, Nq, nk, D, seed=len(chunks) * 7 + D, amp=1.5)
    scale = 1 / math.sqrt(D)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    pb, lb = da.attn_chunks_fwd(qd, kd, vd, chunks, scale=scale, partial_dtype=dtype)
    pc, lc = per_chunk(qd, kd, vd, chunks, scale, dtype)
    da.check()
    assert torch.equal(pb, pc) and torch.equal(lb, lc)
    o, lse = da.attn_lse_merge(pb, lb)
    da.check()
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    check(o, lse, o_ref, lse_ref, f"batched {chunks} D={D} {dtype}")
    s = 0
    for c, n in enumerate(chunks[:2]):
        oc, lc_ref = oracle.attention(q, k, v, scale, kv_start=s, kv_len=n)
        if dtype == torch.float32:
            check(pb[c], lb[c], oc, lc_ref, f"chunk {c}")
        s += n


def test_chunks_need_not_cover_all_keys():
    q, k, v = rand_qkv(1, 3, 200, 1000, 128, seed=11)
    scale = 1 / math.sqrt(128)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    # chunks [0, 300) and [300, 650) of 1000 keys: the rows past 650 are never attended
    pb, lb = da.attn_chunks_fwd(qd, kd, vd, [300, 350], scale=scale)
    o, lse = da.attn_lse_merge(pb, lb)
    da.check()
    o_ref, lse_ref = oracle.attention(q, k, v, scale, kv_start=0, kv_len=650)
    check(o, lse, o_ref, lse_ref, "chunks over the first 650 keys")


def test_chunk_attention_batched_flag():
    w = synth.WORKLOADS["cfg"]  # uneven 1000/1536/2072 split, outlier keys
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = da.chunk_attention(qd, kd, vd, w.alt_chunks, scale=w.scale)
    o2, l2 = da.chunk_attention(qd, kd, vd, w.alt_chunks, scale=w.scale, batched=True)
    da.check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_wan22_size_batched_equals_per_chunk():
    w = synth.WORKLOADS["wan22"]
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    del q, k, v
    pb, lb = da.attn_chunks_fwd(qd, kd, vd, w.chunks, scale=w.scale)
    pc, lc = per_chunk(qd, kd, vd, w.chunks, w.scale, torch.float32)
    da.check()
    assert torch.equal(pb, pc) and torch.equal(lb, lc)


@pytest.mark.parametrize("p", [1, 64])
def test_chunk_count_limits(p):
    D, nk = 64, 700
    q, k, v = rand_qkv(1, 2, 150, nk, D, seed=p)
    scale = 1 / math.sqrt(D)
    base, rem = divmod(nk, p)
    chunks = [base + (1 if c < rem else 0) for c in range(p)]
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    pb, lb = da.attn_chunks_fwd(qd, kd, vd, chunks, scale=scale)
    pc, lc = per_chunk(qd, kd, vd, chunks, scale, torch.float32)
    o, lse = da.attn_lse_merge(pb, lb)
    da.check()
    assert torch.equal(pb, pc) and torch.equal(lb, lc)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    check(o, lse, o_ref, lse_ref, f"p={p}")


def test_chunk_table_not_starting_at_key_zero():
    """The C ABI takes any increasing table inside [0, n_kv]: chunks [100, 400) and
    [400, 650) of 700 keys."""
    import ctypes
    D, nk = 128, 700
    q, k, v = rand_qkv(2, 1, 300, nk, D, seed=5)
    scale = 1 / math.sqrt(D)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    parts = torch.empty(2, 2, 1, 300, D, device=DEV)
    lses = torch.empty(2, 2, 1, 300, device=DEV)
    starts = (ctypes.c_int * 3)(100, 400, 650)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = da.lib().dit_attn_chunks_fwd(ptr(qd), ptr(kd), ptr(vd), ptr(parts), ptr(lses), 2, 1, 300,
                                      nk, D, nk * D, 2, starts, scale, 0,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == da.DIT_OK
    o, lse = da.attn_lse_merge(parts, lses)
    da.check()
    o_ref, lse_ref = oracle.attention(q, k, v, scale, kv_start=100, kv_len=550)
    check(o, lse, o_ref, lse_ref, "chunks over keys [100, 650)")
