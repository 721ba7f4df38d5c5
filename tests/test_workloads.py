"""The synthetic workloads match the shapes the pages print (tests/golden/page_shapes.json)."""
import json
import math
import os

import torch

from diffusion_transformer_long_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_shapes.json")))


def test_flux_shape():
    g, w = GOLDEN["flux_1024"], synth.WORKLOADS["flux"]
    assert w.N == g["N"] and w.H * w.D == g["d_model"]
    assert g["N"] * g["d_model"] * 2 == g["tensor_bytes_bf16"]
    assert round(g["tensor_bytes_bf16"] / 1e6) == g["tensor_mb_printed"]  # decimal MB
    assert w.p == g["ring_degree"] and set(w.chunks) == {g["gemm_rows_per_rank_printed"]}
    assert synth.WORKLOADS["cfg"].N == g["N"] and synth.WORKLOADS["cfg"].H * 128 == g["d_model"]


def test_wan21_shape():
    g, w = GOLDEN["wan21_720p_81f"], synth.WORKLOADS["wan21"]
    assert w.N == g["N"] and w.H * w.D == g["d_model"]
    assert round(g["N"] * g["d_model"] * 2 / 1e6) == g["tensor_mb_printed"]
    assert w.p == g["ring_degree"] and sum(w.chunks) == w.N
    assert [p for p in range(1, 9) if w.H % p == 0] == g["ulysses_degrees_dividing_40_heads_printed"]


def test_wan22_token_count_derivation():
    g, w = GOLDEN["wan22_ti2v_5b"], synth.WORKLOADS["wan22"]
    lat_t = (g["video"]["frames"] - 1) // g["vae_stride"][0] + 1
    lat_h = g["video"]["height"] // g["vae_stride"][1]
    lat_w = g["video"]["width"] // g["vae_stride"][2]
    assert [lat_t, lat_h, lat_w] == g["latent"][2:]
    grid = [lat_t // g["patch"][0], lat_h // g["patch"][1], lat_w // g["patch"][2]]
    assert grid == g["tokens_grid"]
    assert math.prod(grid) == g["N"] == w.N
    assert (w.H, w.D) == (g["heads"], g["head_dim"]) and w.H * w.D == g["d_model"]
    assert w.chunks == (3410,) * 8
    u = GOLDEN["wan22_ulysses_2"]
    assert w.N // 2 == u["tokens_per_rank_before_a2a"] and w.H // 2 == u["heads_per_rank_after_a2a"]


def test_workload_flops_and_chunks():
    for w in synth.WORKLOADS.values():
        assert sum(w.chunks) == w.N
        assert w.flops == 4.0 * w.B * w.H * w.N * w.N * w.D
        assert abs(w.scale - 1 / math.sqrt(w.D)) < 1e-15
    assert sum(synth.WORKLOADS["cfg"].alt_chunks) == synth.WORKLOADS["cfg"].N


def test_generators_are_seeded_and_shaped():
    w = synth.WORKLOADS["tiny"]
    a = synth.make_qkv(w)
    b = synth.make_qkv(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and tuple(x.shape) == (w.B, w.H, w.N, w.D)
        assert torch.equal(x, y)


def test_flux_rows_are_rms_normalised():
    w = synth.WORKLOADS["flux"]
    small = synth.Workload("flux_small", 1, 2, 64, 128, w.seed, w.kind, (64,))
    q, k, v = synth.make_qkv(small)
    rms = q.float().pow(2).mean(-1).sqrt()
    assert torch.allclose(rms, torch.ones_like(rms), atol=2e-2)
    assert not torch.allclose(v.float().pow(2).mean(-1).sqrt(), torch.ones(1), atol=1e-3)


def test_cfg_outliers():
    small = synth.Workload("cfg_small", 2, 2, 400, 128, 4, "cfg_stress", (400,))
    q, k, v = synth.make_qkv(small)
    norms = k.float().norm(dim=-1)  # ~4*sqrt(128) = 45 normally, ~453 for outliers
    n_big = (norms > 200).sum(dim=-1)
    assert (n_big == 20).all()
    assert abs(q.float().std().item() - 4.0) < 0.2
