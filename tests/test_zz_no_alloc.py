"""The no-allocation split-KV entry point (dit_attn_chunk_fwd_splitkv_noalloc), whose fp32
partials live in the library's fixed device scratch array instead of a caller workspace.

Two calls in a row (different inputs, the second reusing the scratch the first wrote) must
equal dit_attn_chunk_fwd_splitkv with a caller workspace bit for bit: same kernels, same
partial layout.  Collected last so that it also runs after every other test in one process;
it passes alone in a fresh process too.  Requests whose partials exceed the scratch are
rejected before anything is launched.
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


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    B, H, Nq, N, D, S = 1, 4, 600, 6000, 128, 5
    results = []
    for seed in (1, 2):
        q = rand((B, H, Nq, D), seed=seed, scale=1.2).to(DEV)
        k = rand((B, H, N, D), seed=seed + 10, scale=1.2).to(DEV)
        v = rand((B, H, N, D), seed=seed + 20).to(DEV)
        out = torch.empty(B, H, Nq, D, device=DEV)
        lse = torch.empty(B, H, Nq, device=DEV)
        da.attn_chunk_fwd_splitkv_noalloc(q, k, v, out, lse, splits=S)
        results.append((q, k, v, out, lse))
    da.check()
    for q, k, v, out, lse in results:
        o_ws, l_ws = da.attn_chunk_fwd_splitkv(q, k, v, splits=S)
        da.check()
        assert torch.equal(out, o_ws) and torch.equal(lse, l_ws)
    q, k, v, out, lse = results[1]
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D))
    err = np.abs(out.double().cpu().numpy() - o_ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3


def test_bf16_output_and_unsplit_calls():
    B, H, Nq, N, D = 2, 2, 300, 2500, 64
    q, k, v = (rand((B, H, n, D), seed=30 + i).to(DEV) for i, n in enumerate((Nq, N, N)))
    for S in (1, 3):
        out = torch.empty(B, H, Nq, D, device=DEV, dtype=torch.bfloat16)
        lse = torch.empty(B, H, Nq, device=DEV)
        da.attn_chunk_fwd_splitkv_noalloc(q, k, v, out, lse, splits=S)
        o_ws, l_ws = da.attn_chunk_fwd_splitkv(q, k, v, out_dtype=torch.bfloat16, splits=S)
        da.check()
        assert torch.equal(out, o_ws) and torch.equal(lse, l_ws)


def test_request_beyond_the_scratch_is_rejected():
    B, H, Nq, N, D, S = 1, 24, 27280, 27280, 128, 8
    assert da.lib().dit_attn_splitkv_workspace_bytes(B, H, Nq, D, S) > (128 << 20)
    q = torch.zeros(B, H, Nq, D, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(B, H, Nq, D, device=DEV)
    lse = torch.empty(B, H, Nq, device=DEV)
    with pytest.raises(da.DitError) as e:
        da.attn_chunk_fwd_splitkv_noalloc(q, q.clone(), q.clone(), out, lse, splits=S)
    assert e.value.status == da.DIT_ERR_UNSUPPORTED
    da.check()
