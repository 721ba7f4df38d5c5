"""Pins for the fp64 oracle: it is checked against things other than itself.

* 50-digit decimal brute force straight from the softmax definition (no max
  shift, no log-space tricks) on tiny inputs;
* closed forms: Q = 0, V = 1, N = 1, equal keys, V = I, a two-key example;
* invariants: chunk merge == full attention for every p and uneven splits,
  merge associativity, KV permutation, key shift, linearity in V, head
  independence;
* a NumPy/SciPy float64 cross-check on the tiny workload.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_long_gb300 import synth


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def decimal_attention(q, k, v, scale):
    """Brute force for one head: q [n,D], k,v [m,D] (bf16 tensors) -> (o [n,D], lse [n])."""
    getcontext().prec = 50
    Q = [[Decimal(float(x)) for x in row] for row in q.float().tolist()]
    K = [[Decimal(float(x)) for x in row] for row in k.float().tolist()]
    V = [[Decimal(float(x)) for x in row] for row in v.float().tolist()]
    sc = Decimal(float(scale))
    outs, lses = [], []
    for qi in Q:
        w = [(sc * sum(a * b for a, b in zip(qi, kj))).exp() for kj in K]
        l = sum(w)
        outs.append([float(sum(w[j] * V[j][d] for j in range(len(K))) / l) for d in range(len(Q[0]))])
        lses.append(float(l.ln()))
    return np.array(outs), np.array(lses)


@pytest.mark.parametrize("n,m,d,scale,seed", [
    (1, 1, 1, 1.0, 0), (3, 5, 2, 0.7071067811865476, 1), (5, 8, 4, 0.5, 2),
    (8, 7, 3, 1.3, 3), (4, 6, 4, 2.5, 4)])
def test_decimal_brute_force(n, m, d, scale, seed):
    q = rand_bf16((1, 1, n, d), seed)
    k = rand_bf16((1, 1, m, d), seed + 100)
    v = rand_bf16((1, 1, m, d), seed + 200)
    o, lse = oracle.attention(q, k, v, scale)
    o_ref, lse_ref = decimal_attention(q[0, 0], k[0, 0], v[0, 0], scale)
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=0, atol=1e-12)


def test_decimal_brute_force_chunk_and_rows():
    """A KV sub-range and a row subset, against the brute force on the same sub-range."""
    q = rand_bf16((1, 1, 6, 4), 7)
    k = rand_bf16((1, 1, 9, 4), 8)
    v = rand_bf16((1, 1, 9, 4), 9)
    o, lse = oracle.attention(q, k, v, 0.5, kv_start=3, kv_len=4, rows=[5, 0, 2])
    o_ref, lse_ref = decimal_attention(q[0, 0, [5, 0, 2]], k[0, 0, 3:7], v[0, 0, 3:7], 0.5)
    np.testing.assert_allclose(o[0, 0], o_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0, 0], lse_ref, atol=1e-12, rtol=0)


def test_two_key_closed_form():
    """q.k0 = 0 and q.k1 = 1 with scale 1: weights 1 : e, so o = (v0 + e v1) / (1 + e)."""
    q = bf16([[[[1.0, 0.0]]]])
    k = bf16([[[[0.0, 3.0], [1.0, -2.0]]]])
    v = bf16([[[[2.0, -1.0], [0.5, 4.0]]]])
    o, lse = oracle.attention(q, k, v, 1.0)
    e = math.e
    np.testing.assert_allclose(o[0, 0, 0], [(2.0 + e * 0.5) / (1 + e), (-1.0 + e * 4.0) / (1 + e)],
                               atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(1 + e)) < 1e-15


def test_q_zero_gives_mean_of_v():
    k = rand_bf16((1, 2, 37, 16), 1)
    v = rand_bf16((1, 2, 37, 16), 2)
    q = torch.zeros((1, 2, 5, 16), dtype=torch.bfloat16)
    o, lse = oracle.attention(q, k, v, 0.25)
    mean_v = v.double().mean(dim=2, keepdim=True).numpy()
    np.testing.assert_allclose(o, np.broadcast_to(mean_v, o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(37), atol=1e-14)


def test_v_ones_gives_ones():
    q = rand_bf16((2, 1, 9, 8), 3, 3.0)
    k = rand_bf16((2, 1, 33, 8), 4, 3.0)
    v = torch.ones((2, 1, 33, 8), dtype=torch.bfloat16)
    o, _ = oracle.attention(q, k, v, 0.9)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_single_key():
    q = rand_bf16((1, 1, 4, 8), 5)
    k = rand_bf16((1, 1, 1, 8), 6)
    v = rand_bf16((1, 1, 1, 8), 7)
    o, lse = oracle.attention(q, k, v, 0.3)
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(v[0, 0].double().numpy(), (4, 8)))
    exact = [0.3 * sum(float(a) * float(b) for a, b in zip(q[0, 0, i].float(), k[0, 0, 0].float()))
             for i in range(4)]
    np.testing.assert_allclose(lse[0, 0], exact, atol=1e-15)


def test_equal_keys():
    q = rand_bf16((1, 1, 3, 8), 8)
    krow = rand_bf16((1, 1, 1, 8), 9)
    k = krow.expand(1, 1, 20, 8).contiguous()
    v = rand_bf16((1, 1, 20, 8), 10)
    o, lse = oracle.attention(q, k, v, 0.5)
    mean_v = v[0, 0].double().mean(dim=0).numpy()
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(mean_v, (3, 8)), atol=1e-14)
    s = [0.5 * sum(float(a) * float(b) for a, b in zip(q[0, 0, i].float(), krow[0, 0, 0].float()))
         for i in range(3)]
    np.testing.assert_allclose(lse[0, 0], np.array(s) + math.log(20), atol=1e-13)


def test_identity_values_expose_probabilities():
    """V = I (N = D = 64): o_ij is the softmax weight p_ij; rows sum to one, p_ij = exp(s_ij - lse_i)."""
    q = rand_bf16((1, 1, 64, 64), 11)
    k = rand_bf16((1, 1, 64, 64), 12)
    v = torch.eye(64, dtype=torch.bfloat16).reshape(1, 1, 64, 64)
    o, lse = oracle.attention(q, k, v, 0.125)
    P = o[0, 0]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14)
    assert (P > 0).all()
    i, j = 17, 42
    s = 0.125 * sum(float(a) * float(b) for a, b in zip(q[0, 0, i].float(), k[0, 0, j].float()))
    assert abs(P[i, j] - math.exp(s - lse[0, 0, i])) < 1e-14


def merge_chunks(q, k, v, scale, chunks):
    parts, lses, s = [], [], 0
    for c in chunks:
        o, l = oracle.attention(q, k, v, scale, kv_start=s, kv_len=c)
        parts.append(o)
        lses.append(l)
        s += c
    return oracle.lse_merge(np.stack(parts), np.stack(lses))


@pytest.mark.parametrize("chunks", [
    (64,), (32, 32), (22, 21, 21), (16, 16, 16, 16), synth.even_chunks(64, 7),
    synth.even_chunks(64, 8), (1,) * 64, (1, 63), (50, 3, 11), (5, 40, 1, 18)])
def test_chunk_merge_equals_full(chunks):
    q = rand_bf16((1, 2, 24, 16), 20, 2.0)
    k = rand_bf16((1, 2, 64, 16), 21, 2.0)
    v = rand_bf16((1, 2, 64, 16), 22)
    o_full, lse_full = oracle.attention(q, k, v, 0.25)
    o_m, lse_m = merge_chunks(q, k, v, 0.25, chunks)
    np.testing.assert_allclose(o_m, o_full, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse_m, lse_full, atol=1e-13, rtol=0)


def test_merge_associative_and_minus_inf():
    g = np.random.default_rng(0)
    parts = g.standard_normal((4, 10, 8))
    lses = g.standard_normal((4, 10)) * 5
    o_all, l_all = oracle.lse_merge(parts, lses)
    o01, l01 = oracle.lse_merge(parts[:2], lses[:2])
    o23, l23 = oracle.lse_merge(parts[2:], lses[2:])
    o_tree, l_tree = oracle.lse_merge(np.stack([o01, o23]), np.stack([l01, l23]))
    np.testing.assert_allclose(o_tree, o_all, atol=1e-13)
    np.testing.assert_allclose(l_tree, l_all, atol=1e-13)
    # a chunk with lse = -inf contributes nothing; all -inf gives o = 0, lse = -inf
    lses2 = lses.copy()
    lses2[1] = -np.inf
    o_a, l_a = oracle.lse_merge(parts, lses2)
    o_b, l_b = oracle.lse_merge(parts[[0, 2, 3]], lses[[0, 2, 3]])
    np.testing.assert_allclose(o_a, o_b, atol=1e-14)
    np.testing.assert_allclose(l_a, l_b, atol=1e-14)
    o_n, l_n = oracle.lse_merge(parts[:2], np.full((2, 10), -np.inf))
    assert (o_n == 0).all() and np.isneginf(l_n).all()


def test_kv_permutation_invariance():
    q = rand_bf16((1, 1, 12, 16), 30)
    k = rand_bf16((1, 1, 50, 16), 31)
    v = rand_bf16((1, 1, 50, 16), 32)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(3))
    o1, l1 = oracle.attention(q, k, v, 0.3)
    o2, l2 = oracle.attention(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), 0.3)
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-13)


def test_key_shift():
    """k_j -> k_j + c leaves o unchanged and shifts lse by scale * q.c (integer data: exact in bf16)."""
    g = torch.Generator().manual_seed(40)
    q = torch.randint(-3, 4, (1, 1, 10, 8), generator=g).to(torch.bfloat16)
    k = torch.randint(-8, 9, (1, 1, 30, 8), generator=g).to(torch.bfloat16)
    v = torch.randint(-8, 9, (1, 1, 30, 8), generator=g).to(torch.bfloat16)
    c = torch.randint(-5, 6, (8,), generator=g).to(torch.bfloat16)
    o1, l1 = oracle.attention(q, k, v, 0.1)
    o2, l2 = oracle.attention(q, (k.float() + c.float()).to(torch.bfloat16), v, 0.1)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    shift = 0.1 * (q.double() @ c.double()).numpy()
    np.testing.assert_allclose(l2 - l1, shift, atol=1e-12)


def test_linear_in_v():
    g = torch.Generator().manual_seed(50)
    q = rand_bf16((1, 1, 7, 8), 51)
    k = rand_bf16((1, 1, 25, 8), 52)
    v1 = torch.randint(-4, 5, (1, 1, 25, 8), generator=g).to(torch.bfloat16)
    v2 = torch.randint(-4, 5, (1, 1, 25, 8), generator=g).to(torch.bfloat16)
    v3 = (2 * v1.float() - 3 * v2.float()).to(torch.bfloat16)  # exact: small integers
    o1, _ = oracle.attention(q, k, v1, 0.4)
    o2, _ = oracle.attention(q, k, v2, 0.4)
    o3, _ = oracle.attention(q, k, v3, 0.4)
    np.testing.assert_allclose(o3, 2 * o1 - 3 * o2, atol=1e-12)


def test_heads_independent():
    q = rand_bf16((2, 3, 9, 8), 60)
    k = rand_bf16((2, 3, 21, 8), 61)
    v = rand_bf16((2, 3, 21, 8), 62)
    o, l = oracle.attention(q, k, v, 0.35)
    for b in range(2):
        for h in range(3):
            oh, lh = oracle.attention(q[b:b + 1, h:h + 1].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                                      v[b:b + 1, h:h + 1].contiguous(), 0.35)
            np.testing.assert_array_equal(oh[0, 0], o[b, h])
            np.testing.assert_array_equal(lh[0, 0], l[b, h])


def test_thread_count_does_not_change_result():
    q = rand_bf16((1, 2, 40, 16), 70)
    k = rand_bf16((1, 2, 70, 16), 71)
    v = rand_bf16((1, 2, 70, 16), 72)
    o1, l1 = oracle.attention(q, k, v, 0.25, threads=1)
    o4, l4 = oracle.attention(q, k, v, 0.25, threads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(l1, l4)


def test_numpy_scipy_cross_check_tiny_workload():
    sp = pytest.importorskip("scipy.special")
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(w)
    rows = synth.sample_rows(w.N, 64)
    o, lse = oracle.attention(q, k, v, w.scale, rows=rows)
    Q, K, V = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for b in range(w.B):
        for h in range(w.H):
            s = w.scale * (Q[b, h, rows] @ K[b, h].T)
            ls = sp.logsumexp(s, axis=1)
            np.testing.assert_allclose(lse[b, h], ls, atol=1e-12)
            np.testing.assert_allclose(o[b, h], np.exp(s - ls[:, None]) @ V[b, h], atol=1e-12)


def test_bad_arguments_rejected():
    q = rand_bf16((1, 1, 4, 8), 0)
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, 1.0, kv_start=2, kv_len=5)
    with pytest.raises(RuntimeError):
        oracle.attention(q, q, q, 1.0, rows=[7])
