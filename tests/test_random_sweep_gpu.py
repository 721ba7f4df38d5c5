"""GPU parity over a seeded sweep of random shapes and entry points, each compared in full with
the fp64 oracle.

Every case draws B, H, D, the query and key counts (ragged, from 1 row up), the input amplitude
and, where the entry point has them, a random chunk split, split-KV count or patch position;
the case list is fixed by the seed, so a failure names a reproducible configuration.
Tolerances are those of the other parity tests: max-abs 1e-2, mean-abs 1e-3, LSE 1e-3 (a bf16
output is allowed one bf16 ulp of the oracle value where that is larger; a merge of bf16
partials, one bf16 ulp of each partial weighted by its merge weight, from the oracle's own
partials, where that is larger).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import ditattn as da

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3
DEV = torch.device("cuda:0")
PATHS = ("fused", "fused_bf16", "chunks_f32", "chunks_bf16", "ring", "splitkv", "bsnd",
         "batched", "cross", "stale")


def _cases(n=100, seed=2026):
    rs = np.random.RandomState(seed)
    out = []
    for i in range(n):
        path = PATHS[i % len(PATHS)]
        B, H = int(rs.randint(1, 3)), int(rs.randint(1, 4))
        D = int(rs.choice([64, 128]))
        nq = int(rs.choice([rs.randint(1, 130), rs.randint(1, 1400)]))
        nk = nq if path in PATHS[:8] else int(rs.randint(1, 3000))
        if path == "stale":
            nk = max(nk, nq)
        amp = float(rs.choice([0.5, 1.0, 2.0] if path in ("chunks_bf16", "batched")
                              else [0.5, 1.0, 2.0, 3.0]))
        p = int(rs.randint(1, min(6, nk) + 1))
        cuts = np.sort(rs.choice(np.arange(1, nk), size=p - 1, replace=False)) if p > 1 else []
        chunks = tuple(int(x) for x in np.diff(np.concatenate([[0], cuts, [nk]])))
        splits = int(rs.randint(2, 7))
        row0 = int(rs.randint(0, max(nk - nq, 0) + 1))
        out.append(dict(path=path, B=B, H=H, D=D, nq=nq, nk=nk, amp=amp, chunks=chunks,
                        splits=splits, row0=row0, seed=int(rs.randint(1 << 30))))
    return out


CASES = _cases()


def _ulp_bf16(x):
    a = np.abs(x).astype(np.float64)
    return np.power(2.0, np.floor(np.log2(np.maximum(a, 1e-30))) - 7)


def _bf16_partials_bound(q, k, v, scale, chunks, lse_ref):
    """Error a merge of bf16-rounded partials may carry: each partial O_c is rounded once to
    bf16 (up to half an ulp of O_c), and the merge weights it by exp(lse_c - lse); one full
    ulp per partial is allowed.  The partials and weights come from the oracle."""
    bound, s = 0.0, 0
    for n in chunks:
        oc, lc = oracle.attention(q, k, v, scale, kv_start=s, kv_len=n)
        bound = bound + np.exp(lc - lse_ref)[..., None] * _ulp_bf16(oc)
        s += n
    return bound


def _check(o, lse, o_ref, lse_ref, what, bf16_out=False, extra_bound=None):
    o = o.detach().double().cpu().numpy()
    lse = lse.detach().double().cpu().numpy()
    err = np.abs(o - o_ref)
    bound = np.maximum(MAX_ABS, _ulp_bf16(o_ref)) if bf16_out else MAX_ABS
    if extra_bound is not None:
        bound = np.maximum(bound, extra_bound)
    assert (err <= bound).all(), f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    lerr = np.abs(lse - lse_ref).max()
    assert lerr <= LSE_ABS, f"{what}: lse {lerr:.3e}"


@pytest.mark.parametrize("case", CASES, ids=lambda c: "{path}-B{B}H{H}D{D}-q{nq}-k{nk}".format(**c))
def test_random_case(case):
    c = case
    B, H, D, nq, nk = c["B"], c["H"], c["D"], c["nq"], c["nk"]
    g = torch.Generator().manual_seed(c["seed"])
    q = (torch.randn(B, H, nq, D, generator=g) * c["amp"]).to(torch.bfloat16)
    k = (torch.randn(B, H, nk, D, generator=g) * c["amp"]).to(torch.bfloat16)
    v = torch.randn(B, H, nk, D, generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    what = f"{c}"
    path = c["path"]

    if path == "stale":
        m = nq
        k_new = (torch.randn(B, H, m, D, generator=g) * c["amp"]).to(torch.bfloat16)
        v_new = torch.randn(B, H, m, D, generator=g).to(torch.bfloat16)
        r0 = c["row0"]
        k_upd, v_upd = k.clone(), v.clone()
        k_upd[:, :, r0:r0 + m] = k_new
        v_upd[:, :, r0:r0 + m] = v_new
        o_ref, lse_ref = oracle.attention(q, k_upd, v_upd, scale)
        kb, vb = k.to(DEV), v.to(DEV)
        o, lse = da.stale_kv_attention(q.to(DEV), k_new.to(DEV), v_new.to(DEV), kb, vb, r0,
                                       scale=scale, splits=None)
        da.check()
        assert torch.equal(kb.cpu(), k_upd) and torch.equal(vb.cpu(), v_upd), what
        _check(o, lse, o_ref, lse_ref, what)
        return

    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    extra = None
    if path == "fused":
        o, lse = da.attn_fwd(qd, kd, vd, scale=scale)
    elif path == "fused_bf16":
        o, lse = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=torch.bfloat16)
    elif path == "chunks_f32":
        o, lse = da.chunk_attention(qd, kd, vd, c["chunks"], scale=scale)
    elif path == "chunks_bf16":
        o, lse = da.chunk_attention(qd, kd, vd, c["chunks"], scale=scale,
                                    partial_dtype=torch.bfloat16)
        extra = _bf16_partials_bound(q, k, v, scale, c["chunks"], lse_ref)
    elif path == "ring":
        o, lse = da.ring_attention(qd, kd, vd, c["chunks"], scale=scale)
    elif path in ("splitkv", "cross"):
        splits = min(c["splits"], (nk + 127) // 128) if path == "splitkv" else None
        o, lse = da.attn_chunk_fwd_splitkv(qd, kd, vd, scale=scale, splits=splits)
    elif path == "batched":
        partial_dtype = torch.bfloat16 if c["seed"] % 2 else torch.float32
        o, lse = da.chunk_attention(qd, kd, vd, c["chunks"], scale=scale, batched=True,
                                    partial_dtype=partial_dtype)
        if partial_dtype == torch.bfloat16:
            extra = _bf16_partials_bound(q, k, v, scale, c["chunks"], lse_ref)
    elif path == "bsnd":
        qs, ks, vs = (x.transpose(1, 2).contiguous().transpose(1, 2) for x in (qd, kd, vd))
        out = torch.empty(B, nq, H, D, device=DEV).transpose(1, 2)
        o, lse = da.attn_fwd_strided(qs, ks, vs, out=out, scale=scale)
    else:
        raise AssertionError(path)
    da.check()
    _check(o, lse, o_ref, lse_ref, what, bf16_out=(path == "fused_bf16"), extra_bound=extra)
