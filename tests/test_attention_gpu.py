"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (from the arithmetic: bf16 inputs, fp32 accumulation, bf16 P for
the second GEMM): output max-abs <= 1e-2, mean-abs <= 1e-3 and LSE abs <= 1e-3
for fp32 outputs.  A bf16 output is additionally allowed its own rounding: one
bf16 ulp of the oracle value where that exceeds 1e-2.

Small and FLUX-sized workloads are compared in full; Wan-sized ones on a
seeded sample of query rows (all heads x 128 rows incl. the first/last 16),
each sampled row exact in the oracle because rows are independent.
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


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.power(2.0, e - 7)


def assert_parity(o, lse, o_ref, lse_ref, what, bf16_out=False):
    o = o.detach().double().cpu().numpy()
    lse = lse.detach().double().cpu().numpy()
    err = np.abs(o - o_ref)
    if bf16_out:
        bound = np.maximum(MAX_ABS, bf16_ulp(o_ref))
        assert (err <= bound).all(), f"{what}: bf16 out error {float((err - bound).max())} over bound"
    else:
        assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    lerr = np.abs(lse - lse_ref).max()
    assert lerr <= LSE_ABS, f"{what}: lse {lerr:.3e}"
    return float(err.max()), float(err.mean()), float(lerr)


def to_dev(*ts):
    return [t.to(DEV) for t in ts]


def pick(o, lse, rows):
    if rows is None:
        return o, lse
    idx = torch.as_tensor(rows, device=o.device)
    return o.index_select(2, idx), lse.index_select(2, idx)


# ----------------------------------------------------------------- workloads
WORKLOAD_ROWS = {"tiny": None, "flux": None, "wan22": 128, "wan21": 128, "cfg": 512}


@pytest.fixture(scope="module", params=list(synth.WORKLOADS))
def workload(request):
    w = synth.WORKLOADS[request.param]
    q, k, v = synth.make_qkv(w)
    nrows = WORKLOAD_ROWS[w.name]
    rows = None if nrows is None else synth.sample_rows(w.N, nrows, seed=w.seed)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, rows=rows)
    qd, kd, vd = to_dev(q, k, v)
    del q, k, v
    yield w, qd, kd, vd, rows, o_ref, lse_ref
    del qd, kd, vd
    torch.cuda.empty_cache()


def test_fused_fp32(workload):
    w, q, k, v, rows, o_ref, lse_ref = workload
    o, lse = da.attn_fwd(q, k, v, scale=w.scale)
    da.check()
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} fused fp32")


def test_fused_bf16_out(workload):
    w, q, k, v, rows, o_ref, lse_ref = workload
    o, lse = da.attn_fwd(q, k, v, scale=w.scale, out_dtype=torch.bfloat16)
    da.check()
    assert o.dtype == torch.bfloat16
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} fused bf16", bf16_out=True)


def test_chunk_merge_fp32_partials(workload):
    w, q, k, v, rows, o_ref, lse_ref = workload
    o, lse = da.chunk_attention(q, k, v, w.chunks, scale=w.scale)
    da.check()
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} p={w.p} chunk+merge")
    if w.alt_chunks:
        o, lse = da.chunk_attention(q, k, v, w.alt_chunks, scale=w.scale)
        da.check()
        assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} uneven chunk+merge")


def test_chunk_merge_bf16_partials(workload):
    w, q, k, v, rows, o_ref, lse_ref = workload
    o, lse = da.chunk_attention(q, k, v, w.chunks, scale=w.scale, partial_dtype=torch.bfloat16)
    da.check()
    # bf16 partials carry one bf16 rounding of each O_c: allow one ulp of the result
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} bf16 partials", bf16_out=True)


def test_ring_accumulate(workload):
    """Hop-by-hop ring: every chunk folded into the running (O, lse) by
    dit_attn_chunk_fwd_accumulate.  The running output starts as NaN with lse = -inf, which
    also checks that empty rows' O_run is never read."""
    w, q, k, v, rows, o_ref, lse_ref = workload
    B, H, N, D = q.shape
    for chunks, what in ((w.chunks, f"p={w.p}"), (w.alt_chunks, "uneven")):
        if not chunks:
            continue
        o_run = torch.full((B, H, N, D), math.nan, device=DEV)
        o, lse = da.ring_attention(q, k, v, chunks, scale=w.scale, o_run=o_run)
        da.check()
        assert o.data_ptr() == o_run.data_ptr()
        assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} ring accumulate {what}")


def test_chunk_partials_match_oracle_chunks(workload):
    """Each virtual rank's partial (O_c, lse_c) against the oracle over that chunk alone."""
    w, q, k, v, rows, _, _ = workload
    if w.name not in ("tiny", "wan22"):
        pytest.skip("per-chunk check on two workloads")
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    for c, (s, n) in enumerate(zip(synth.chunk_starts(w.chunks), w.chunks)):
        if c not in (0, len(w.chunks) - 1):
            continue
        o, lse = da.attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], scale=w.scale)
        da.check()
        o_ref, lse_ref = oracle.attention(qc, kc, vc, w.scale, kv_start=s, kv_len=n, rows=rows)
        assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"{w.name} chunk {c}")


# ----------------------------------------------------------------- edge cases
def rand_qkv(B, H, N, D, seed, nk=None, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    nk = N if nk is None else nk
    q = (torch.randn(B, H, N, D, generator=g) * scale).to(torch.bfloat16)
    k = (torch.randn(B, H, nk, D, generator=g) * scale).to(torch.bfloat16)
    v = torch.randn(B, H, nk, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("B,H,N,D", [
    (1, 1, 1, 64), (1, 1, 1, 128), (1, 1, 7, 128), (1, 2, 129, 64), (2, 1, 200, 128),
    (1, 1, 255, 128), (1, 3, 257, 64), (1, 1, 300, 128), (2, 3, 384, 128), (1, 1, 513, 64),
    (1, 2, 1000, 128)])
def test_ragged_shapes_full(B, H, N, D):
    q, k, v = rand_qkv(B, H, N, D, seed=N + D)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = da.attn_fwd(qd, kd, vd, scale=scale)
    da.check()
    assert_parity(o, lse, o_ref, lse_ref, f"fused {B}x{H}x{N}x{D}")


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_chunks_views_and_packed(D):
    N, chunks = 700, (1, 127, 128, 129, 315)
    q, k, v = rand_qkv(2, 2, N, D, seed=D, scale=1.5)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = da.chunk_attention(qd, kd, vd, chunks, scale=scale)
    da.check()
    assert_parity(o, lse, o_ref, lse_ref, f"ragged chunks D={D}")
    # a packed chunk buffer, as a ring hop would receive it (head stride n_kv*D)
    s = 1 + 127
    kp = kd[:, :, s:s + 128].contiguous()
    vp = vd[:, :, s:s + 128].contiguous()
    op, lp = da.attn_chunk_fwd(qd, kp, vp, scale=scale)
    ov, lv = da.attn_chunk_fwd(qd, kd[:, :, s:s + 128], vd[:, :, s:s + 128], scale=scale)
    da.check()
    assert torch.equal(op, ov) and torch.equal(lp, lv)
    oc, lc = oracle.attention(q, k, v, scale, kv_start=s, kv_len=128)
    assert_parity(op, lp, oc, lc, "packed chunk")


def test_query_and_key_counts_differ():
    """N_q != n_kv (one chunk shorter than the queries), e.g. text K/V of 512 tokens."""
    q, _, _ = rand_qkv(1, 2, 1300, 128, seed=5)
    _, k, v = rand_qkv(1, 2, 512, 128, seed=6)
    scale = 1 / math.sqrt(128)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = da.attn_chunk_fwd(qd, kd, vd, scale=scale)
    da.check()
    assert_parity(o, lse, o_ref, lse_ref, "N_q=1300, n_kv=512")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_cross_attention_512_keys_full_shape(out_dtype):
    """The short-KV shape at full size, in the launch bench.py times: all 27280 Wan2.2 queries
    of 24 heads against the first 512 rows of K and V (views with the full buffer's head
    stride).  Items have 4 key tiles, so this is the short-item (soft-drain) form; sampled
    rows (all heads, first/last 16 included) against the oracle."""
    w = synth.WORKLOADS["wan22"]
    q, k, v = synth.make_qkv(w)
    n_txt = 512
    rows = synth.sample_rows(w.N, 256, seed=w.seed + 1)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, kv_start=0, kv_len=n_txt, rows=rows)
    qd, kd, vd = to_dev(q, k, v)
    del q, k, v
    o, lse = da.attn_chunk_fwd(qd, kd[:, :, :n_txt], vd[:, :, :n_txt], scale=w.scale,
                               out_dtype=out_dtype)
    da.check()
    assert o.dtype == out_dtype and o.shape == qd.shape
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, f"cross 27280x512 {out_dtype}",
                  bf16_out=out_dtype == torch.bfloat16)


def test_two_million_keys_ragged():
    """A sequence far longer than the pages' workloads: N = 2^21 + 37 tokens (8193 query pairs
    and key tiles per head, a 37-key ragged tail), D = 64, fused and as 3 uneven chunks merged
    by LSE; sampled rows (first/last 16 included) against the oracle."""
    n = (1 << 21) + 37
    c0, c1 = 700_001, 650_000
    w = synth.Workload("long2m", 1, 1, n, 64, 11, "iid", (c0, c1, n - c0 - c1))
    q, k, v = synth.make_qkv(w)
    rows = synth.sample_rows(n, 48, seed=w.seed)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, rows=rows)
    qd, kd, vd = to_dev(q, k, v)
    del q, k, v
    o, lse = da.attn_fwd(qd, kd, vd, scale=w.scale)
    da.check()
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, "fused 2M")
    del o, lse
    o, lse = da.chunk_attention(qd, kd, vd, list(w.chunks), scale=w.scale, batched=True)
    da.check()
    assert_parity(*pick(o, lse, rows), o_ref, lse_ref, "3 chunks 2M")
    del o, lse, qd, kd, vd
    torch.cuda.empty_cache()


# ----------------------------------------------------------------- closed forms / invariants
@pytest.fixture(scope="module")
def flux_inputs():
    w = synth.WORKLOADS["flux"]
    q, k, v = synth.make_qkv(w)
    return w, *to_dev(q, k, v)


def test_q_zero_gives_mean_of_v(flux_inputs):
    w, q, k, v = flux_inputs
    o, lse = da.attn_fwd(torch.zeros_like(q), k, v, scale=w.scale)
    da.check()
    mean_v = v.double().mean(dim=2, keepdim=True).expand_as(o)
    assert (o.double() - mean_v).abs().max().item() <= 1e-3
    assert (lse.double() - math.log(w.N)).abs().max().item() <= 1e-4


def test_v_ones_gives_ones(flux_inputs):
    w, q, k, v = flux_inputs
    o, _ = da.attn_fwd(q, k, torch.ones_like(v), scale=w.scale)
    o2, _ = da.chunk_attention(q, k, torch.ones_like(v), w.chunks, scale=w.scale)
    da.check()
    assert (o - 1).abs().max().item() <= 2e-3
    assert (o2 - 1).abs().max().item() <= 2e-3


def test_kv_permutation_invariance(flux_inputs):
    w, q, k, v = flux_inputs
    perm = torch.randperm(w.N, generator=torch.Generator().manual_seed(9)).to(DEV)
    o1, l1 = da.attn_fwd(q, k, v, scale=w.scale)
    o2, l2 = da.attn_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), scale=w.scale)
    da.check()
    d = (o1 - o2).abs()
    assert d.max().item() <= 2e-3 and d.mean().item() <= 1e-4
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_fused_equals_chunk_merge(flux_inputs):
    w, q, k, v = flux_inputs
    o1, l1 = da.attn_fwd(q, k, v, scale=w.scale)
    for p in (1, 2, 3, 7):
        o2, l2 = da.chunk_attention(q, k, v, synth.even_chunks(w.N, p), scale=w.scale)
        da.check()
        d = (o1 - o2).abs()
        assert d.max().item() <= 2e-3 and d.mean().item() <= 1e-4, p
        assert (l1 - l2).abs().max().item() <= 1e-4, p


def test_heads_independent(flux_inputs):
    w, q, k, v = flux_inputs
    o, lse = da.attn_fwd(q, k, v, scale=w.scale)
    h = 5
    o1, l1 = da.attn_fwd(q[:, h:h + 1].contiguous(), k[:, h:h + 1].contiguous(),
                         v[:, h:h + 1].contiguous(), scale=w.scale)
    da.check()
    assert torch.equal(o1[:, 0], o[:, h]) and torch.equal(l1[:, 0], lse[:, h])


# ----------------------------------------------------------------- merge kernel alone
@pytest.mark.parametrize("pdt,odt", [(torch.float32, torch.float32), (torch.bfloat16, torch.float32),
                                     (torch.float32, torch.bfloat16), (torch.bfloat16, torch.bfloat16)])
@pytest.mark.parametrize("p,D", [(1, 128), (3, 64), (8, 128), (13, 128)])
def test_merge_kernel_vs_oracle(p, D, pdt, odt):
    g = torch.Generator().manual_seed(p * 100 + D)
    B, H, N = 2, 3, 77
    parts = torch.randn(p, B, H, N, D, generator=g).to(pdt)
    lses = (torch.randn(p, B, H, N, generator=g) * 6).float()
    if p > 1:
        lses[0, 0, 0, :5] = -math.inf  # a chunk that saw nothing contributes nothing
    o_ref, l_ref = oracle.lse_merge(parts.double().numpy(), lses.double().numpy())
    o, l = da.attn_lse_merge(parts.to(DEV), lses.to(DEV), out_dtype=odt)
    da.check()
    tol = 1e-5 if odt == torch.float32 else None
    od = o.double().cpu().numpy()
    if tol is not None:
        assert np.abs(od - o_ref).max() <= 1e-5 * max(1.0, np.abs(o_ref).max())
    else:
        assert (np.abs(od - o_ref) <= bf16_ulp(o_ref) * 0.5 + 1e-5).all()
    assert np.abs(l.double().cpu().numpy() - l_ref).max() <= 1e-5


def test_merge_all_minus_inf_row():
    parts = torch.randn(3, 1, 1, 4, 64, device=DEV)
    lses = torch.full((3, 1, 1, 4), -math.inf, device=DEV)
    o, l = da.attn_lse_merge(parts, lses)
    da.check()
    assert (o == 0).all() and torch.isneginf(l).all()


# ----------------------------------------------------------------- buffers and failures
CANARY = -1.2345e30


def test_canaries_untouched():
    """Outputs written through slices of larger buffers: nothing outside is touched."""
    B, H, N, D, pad = 1, 2, 333, 128, 1024
    q, k, v = to_dev(*rand_qkv(B, H, N, D, seed=77))
    n_out = B * H * N * D
    big = torch.full((n_out + 2 * pad,), CANARY, device=DEV)
    big_l = torch.full((B * H * N + 2 * pad,), CANARY, device=DEV)
    out = big[pad:pad + n_out].view(B, H, N, D)
    lse = big_l[pad:pad + B * H * N].view(B, H, N)
    da.attn_fwd(q, k, v, out=out, lse=lse)
    parts = torch.full((3 * n_out + 2 * pad,), CANARY, device=DEV)
    lses = torch.full((3 * B * H * N + 2 * pad,), CANARY, device=DEV)
    P = parts[pad:pad + 3 * n_out].view(3, B, H, N, D)
    L = lses[pad:pad + 3 * B * H * N].view(3, B, H, N)
    s = 0
    for c, n in enumerate((100, 133, 100)):
        da.attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], out=P[c], lse=L[c])
        s += n
    mo = torch.full((n_out + 2 * pad,), CANARY, device=DEV)
    ml = torch.full((B * H * N + 2 * pad,), CANARY, device=DEV)
    da.attn_lse_merge(P, L, out=mo[pad:pad + n_out].view(B, H, N, D),
                      lse=ml[pad:pad + B * H * N].view(B, H, N))
    da.check()
    for buf, n in ((big, n_out), (big_l, B * H * N), (parts, 3 * n_out), (lses, 3 * B * H * N),
                   (mo, n_out), (ml, B * H * N)):
        assert (buf[:pad] == CANARY).all() and (buf[pad + n:] == CANARY).all()
        assert torch.isfinite(buf[pad:pad + n]).all()
    assert torch.allclose(mo[pad:pad + n_out].view(B, H, N, D), out, atol=2e-3)


def test_timeout_is_reported_and_context_survives():
    """Failure injection: K/V copies are never issued, the bounded wait (~10 ms) expires, the
    kernel exits cleanly and dit_attn_check reports DIT_ERR_TIMEOUT; later calls work."""
    q, k, v = to_dev(*rand_qkv(1, 1, 256, 128, seed=3))
    da.check()
    da.inject_stall(True, 20_000_000)
    try:
        da.attn_fwd(q, k, v)
        with pytest.raises(da.DitError) as e:
            da.check()
        assert e.value.status == da.DIT_ERR_TIMEOUT
    finally:
        da.inject_stall(False)
    da.check()  # status was cleared
    o, lse = da.attn_fwd(q, k, v)
    da.check()
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(128))
    assert_parity(o, lse, o_ref, lse_ref, "after timeout")


def test_device_validation_errors():
    q, k, v = to_dev(*rand_qkv(1, 1, 64, 128, seed=1))
    L = da.lib()
    out = torch.empty(1, 1, 64, 128, device=DEV)
    lse = torch.empty(1, 1, 64, device=DEV)
    st = L.dit_attn_fwd(da._ptr(q), da._ptr(k), da._ptr(v), da._ptr(out), da._ptr(lse), 1, 1, 64,
                        96, 0.1, 0, None)
    assert st == da.DIT_ERR_UNSUPPORTED
    st = L.dit_attn_fwd(da._ptr(q), da._ptr(k), da._ptr(v), da._ptr(q), da._ptr(lse), 1, 1, 64,
                        128, 0.1, 0, None)
    assert st == da.DIT_ERR_INVALID_ARG  # output aliases an input


@pytest.mark.parametrize("limit", [1, 3])
def test_persistent_grid_many_items_per_cta(limit):
    """A capped persistent grid makes every CTA walk many (head, Q-pair) work items, carrying
    barrier phases, Q refills and O hand-offs across items; results must not change."""
    da.set_grid_limit(limit)
    try:
        for D in (64, 128):
            q, k, v = rand_qkv(2, 3, 700, D, seed=11 + D, scale=1.3)
            scale = 1 / math.sqrt(D)
            o_ref, lse_ref = oracle.attention(q, k, v, scale)
            qd, kd, vd = to_dev(q, k, v)
            o, lse = da.attn_fwd(qd, kd, vd, scale=scale)
            ob, lb = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=torch.bfloat16)
            oc, lc = da.chunk_attention(qd, kd, vd, (1, 127, 128, 129, 315), scale=scale)
            orr, lrr = da.ring_attention(qd, kd, vd, (1, 127, 128, 129, 315), scale=scale)
            da.check()
            assert_parity(o, lse, o_ref, lse_ref, f"grid={limit} D={D} fused")
            assert_parity(ob, lb, o_ref, lse_ref, f"grid={limit} D={D} bf16", bf16_out=True)
            assert_parity(oc, lc, o_ref, lse_ref, f"grid={limit} D={D} chunks")
            assert_parity(orr, lrr, o_ref, lse_ref, f"grid={limit} D={D} ring accumulate")
    finally:
        da.set_grid_limit(0)


@pytest.mark.parametrize("D", [64, 128])
def test_canaries_untouched_bf16_short_items(D):
    """Short items with bf16 output store O with TMA stores clipped at the last query row:
    outputs written through slices of larger buffers (fused, one chunk, all chunks in one
    launch; ragged N) match the oracle and touch nothing outside."""
    B, H, N, pad = 2, 2, 333, 4096
    q, k, v = rand_qkv(B, H, N, D, seed=78 + D)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    n_out = B * H * N * D
    big = torch.full((n_out + 2 * pad,), CANARY, device=DEV, dtype=torch.bfloat16)
    out = big[pad:pad + n_out].view(B, H, N, D)
    o, lse = da.attn_fwd(qd, kd, vd, out=out, scale=scale, out_dtype=torch.bfloat16)
    one = torch.full((n_out + 2 * pad,), CANARY, device=DEV, dtype=torch.bfloat16)
    oc, lc = da.attn_chunk_fwd(qd, kd[:, :, 100:300], vd[:, :, 100:300],
                               out=one[pad:pad + n_out].view(B, H, N, D), scale=scale,
                               out_dtype=torch.bfloat16)
    chunks = (100, 133, 100)
    parts = torch.full((3 * n_out + 2 * pad,), CANARY, device=DEV, dtype=torch.bfloat16)
    P = parts[pad:pad + 3 * n_out].view(3, B, H, N, D)
    _, L = da.attn_chunks_fwd(qd, kd, vd, chunks, partials=P, scale=scale,
                              partial_dtype=torch.bfloat16)
    da.check()
    for buf, n in ((big, n_out), (one, n_out), (parts, 3 * n_out)):
        assert (buf[:pad] == CANARY).all() and (buf[pad + n:] == CANARY).all()
    assert_parity(o, lse, o_ref, lse_ref, f"D={D} bf16 short fused", bf16_out=True)
    oc_ref, lc_ref = oracle.attention(q, k, v, scale, kv_start=100, kv_len=200)
    assert_parity(oc, lc, oc_ref, lc_ref, f"D={D} bf16 short chunk", bf16_out=True)
    om, lm = da.attn_lse_merge(P, L)
    da.check()
    assert_parity(om, lm, o_ref, lse_ref, f"D={D} bf16 short chunks merged", bf16_out=True)


def test_concurrent_launches_on_two_streams():
    """A fused pass and a batched chunk pass launched at the same time on two streams (their
    CTAs share the SMs): both results are bitwise those of the launches run one after the
    other."""
    w = synth.WORKLOADS["flux"]
    q, k, v = to_dev(*synth.make_qkv(w))
    o_ref, l_ref = da.attn_fwd(q, k, v, scale=w.scale)
    p_ref, pl_ref = da.attn_chunks_fwd(q, k, v, w.chunks, scale=w.scale)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            o, l = da.attn_fwd(q, k, v, scale=w.scale)
        with torch.cuda.stream(s2):
            pp, pl = da.attn_chunks_fwd(q, k, v, w.chunks, scale=w.scale)
        outs.append((o, l, pp, pl))
    torch.cuda.synchronize()
    da.check()
    for o, l, pp, pl in outs:
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
        assert torch.equal(pp, p_ref) and torch.equal(pl, pl_ref)


def outlier_qkv(B, H, N, D, seed):
    """CFG-stress-like inputs (the cfg workload's recipe at another shape): Q, K x gain and a
    fraction of keys x outlier gain, so the running max keeps rising and O is rescaled on most
    tiles."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, D, generator=g) * synth.CFG_QK_GAIN
    k = torch.randn(B, H, N, D, generator=g) * synth.CFG_QK_GAIN
    v = torch.randn(B, H, N, D, generator=g)
    n_out = int(synth.CFG_OUTLIER_FRACTION * N)
    for b in range(B):
        for h in range(H):
            idx = torch.randperm(N, generator=g)[:n_out]
            k[b, h, idx] *= synth.CFG_OUTLIER_GAIN
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


@pytest.mark.parametrize("limit", [0, 1, 3])
def test_rescale_on_capped_grid(limit):
    """Inputs whose running max keeps rising, so O is rescaled (and P published whole) on
    most tiles: items of more than 16 key tiles (fused, and all chunks in one launch), with
    every CTA walking many items when the grid is capped."""
    B, H, N, D = 2, 3, 2500, 128
    q, k, v = outlier_qkv(B, H, N, D, seed=31)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    da.set_grid_limit(limit)
    try:
        o, lse = da.attn_fwd(qd, kd, vd, scale=scale)
        ob, lb = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=torch.bfloat16)
        oc, lc = da.chunk_attention(qd, kd, vd, (2100, 400), scale=scale)
        da.check()
    finally:
        da.set_grid_limit(0)
    assert_parity(o, lse, o_ref, lse_ref, f"grid={limit} outliers fused")
    assert_parity(ob, lb, o_ref, lse_ref, f"grid={limit} outliers bf16", bf16_out=True)
    assert_parity(oc, lc, o_ref, lse_ref, f"grid={limit} outliers chunks")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_output_16_byte_aligned_not_32(dtype):
    """The epilogue writes 32-byte vectors when the output is 32-byte aligned and falls back to
    16-byte vectors otherwise; both must give the same result and touch nothing outside."""
    B, H, N, D = 1, 2, 300, 128
    q, k, v = rand_qkv(B, H, N, D, seed=21)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    qd, kd, vd = to_dev(q, k, v)
    n = B * H * N * D
    shift = 16 // torch.empty((), dtype=dtype).element_size()  # 16 bytes
    big = torch.full((n + 64,), 7.0, device=DEV, dtype=dtype)
    out = big[shift:shift + n].view(B, H, N, D)
    assert out.data_ptr() % 32 == 16
    o, lse = da.attn_fwd(qd, kd, vd, out=out, scale=scale)
    o_al, _ = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=dtype)
    da.check()
    assert torch.equal(o, o_al)
    assert (big[:shift] == 7.0).all() and (big[shift + n:] == 7.0).all()
    assert_parity(o, lse, o_ref, lse_ref, f"16B-aligned {dtype}", bf16_out=dtype == torch.bfloat16)


# ----------------------------------------------------------------- host tensors, pipelined
@pytest.mark.parametrize("pinned", [True, False])
def test_host_tensors_pipelined_over_head_groups(pinned):
    """attention() on host tensors runs head groups through host_pipeline (upload, compute and
    download overlapped); heads are independent, so every path must equal the device call on
    the same data bit for bit, and the fused result must match the oracle."""
    B, H, N, D = 2, 7, 600, 128
    q, k, v = rand_qkv(B, H, N, D, seed=91)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    assert da.head_groups(B * H) == [(0, 1), (1, 3), (3, 11), (11, 13), (13, 14)]
    qd, kd, vd = to_dev(q, k, v)
    chunks = [200, 150, 250]
    for kw in (dict(), dict(chunks=chunks), dict(chunks=chunks, accumulate=True),
               dict(out_dtype=torch.bfloat16)):
        o_h, l_h = da.attention(q, k, v, **kw)
        o_d, l_d = da.attention(qd, kd, vd, **kw)
        da.check()
        assert not o_h.is_cuda and o_h.is_pinned()
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu()), kw
    o_ref, lse_ref = oracle.attention(q, k, v, 1 / math.sqrt(D))
    o_h, l_h = da.attention(q, k, v)
    assert_parity(o_h, l_h, o_ref, lse_ref, "host pipelined fused")


@pytest.mark.parametrize("amp", [8.0, 30.0])
def test_extreme_logits_every_path(amp):
    """Q and K scaled so that scaled scores reach ~amp^2 (about 3000 for amp = 30): the
    softmax is one-hot per row and any missing max subtraction overflows fp32.  Every path
    must match the oracle (which subtracts the exact max in fp64).

    O is held to the usual tolerances.  The LSE of such rows is about the top score, whose
    fp32 accumulation over D products of magnitude ~1e4 (the tensor core's fp32 sum) carries
    a few fp32 ulps of error at |lse| ~ 3000 (one ulp = 2.4e-4), so beyond the workloads'
    range the LSE bound is 1e-3 plus 16 fp32 ulps of |lse|."""
    B, H, N, D = 1, 2, 900, 128
    q, k, v = rand_qkv(B, H, N, D, seed=int(amp), scale=amp)
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = oracle.attention(q, k, v, scale)
    assert np.abs(lse_ref).max() > (500 if amp > 10 else 20)
    qd, kd, vd = to_dev(q, k, v)
    chunks = (300, 257, 343)
    for name, (o, lse) in {
        "fused": da.attn_fwd(qd, kd, vd, scale=scale),
        "chunk+merge": da.chunk_attention(qd, kd, vd, chunks, scale=scale),
        "ring": da.ring_attention(qd, kd, vd, chunks, scale=scale),
        "split-kv": da.attn_chunk_fwd_splitkv(qd, kd, vd, scale=scale, splits=3),
    }.items():
        da.check()
        assert torch.isfinite(o).all() and torch.isfinite(lse).all(), name
        ulp = np.power(2.0, np.floor(np.log2(np.maximum(np.abs(lse_ref), 1e-30))) - 23)
        lerr = np.abs(lse.double().cpu().numpy() - lse_ref)
        assert (lerr <= 1e-3 + 16 * ulp).all(), f"amp {amp} {name}: lse {lerr.max():.3e}"
        err = np.abs(o.double().cpu().numpy() - o_ref)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"amp {amp} {name}: {err.max()}"


@pytest.mark.parametrize("D,dtype", [(64, torch.float32), (128, torch.float32),
                                     (64, torch.bfloat16), (128, torch.bfloat16)])
def test_fused_without_lse(D, dtype):
    """lse = NULL: the pass skips the LSE and its unrounded row sum; O is bitwise the same
    (it is normalised by the rounded sum either way), on the plain and strided entry points."""
    q, k, v = rand_qkv(2, 3, 517, D, seed=D + 3, scale=1.5)
    scale = 1 / math.sqrt(D)
    qd, kd, vd = to_dev(q, k, v)
    o1, l1 = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=dtype)
    o2, l2 = da.attn_fwd(qd, kd, vd, scale=scale, out_dtype=dtype, with_lse=False)
    q_s, k_s, v_s = (da.bhnd_to_bsnd(t) for t in (qd, kd, vd))
    o3 = torch.empty(2, 517, 3, D, device=DEV, dtype=dtype).transpose(1, 2)
    with torch.cuda.device(DEV):
        qs, ks, vs, os_ = (da.view_strides(t) for t in (q_s.transpose(1, 2), k_s.transpose(1, 2),
                                                         v_s.transpose(1, 2), o3))
        import ctypes
        st = da.lib().dit_attn_fwd_strided(
            ctypes.c_void_p(q_s.data_ptr()), ctypes.byref(qs), ctypes.c_void_p(k_s.data_ptr()),
            ctypes.byref(ks), ctypes.c_void_p(v_s.data_ptr()), ctypes.byref(vs),
            ctypes.c_void_p(o3.data_ptr()), ctypes.byref(os_), None, 2, 3, 517, 517, D, scale,
            0 if dtype == torch.float32 else 1,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == da.DIT_OK
    da.check()
    assert l2 is None
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
