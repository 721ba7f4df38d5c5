"""Seeded synthetic inputs shaped like the pages' DiT attention workloads.

This module holds no attention arithmetic: it only draws Q, K, V and names the
workloads.  Both the CUDA path's tests/bench and the oracle's tests consume
what it returns, so the two sides always see identical bf16 bits.

Recipe (every config): ``torch.Generator().manual_seed(seed)``, then float32
``randn`` for Q, K and V in that order, the config's transform in float32,
then a round-to-nearest-even cast to bf16.  Layout [B, H, N, D], contiguous.

Workload shapes and where they come from:
  tiny   B1 H2  N1024  D64   iid N(0,1)                       (CPU-oracle-sized case)
  flux   B1 H24 N4608  D128  Q, K rows RMS-normalised, V N(0,1)
         FLUX.1-dev 1024^2: 4096 image + 512 text tokens, d = 3072 = 24 x 128
         (arganzheng.life multi-GPU diffusion parallelism, section 1.1 table)
  wan22  B1 H24 N27280 D128  iid N(0,1)
         Wan2.2 TI2V-5B 704x1280x121 frames: VAE stride (4,16,16) and patch
         (1,2,2) give 31 x 22 x 40 = 27280 tokens, 24 heads x 128
         ("AIGC distributed inference ... from Wan2.2", model parameters)
  wan21  B1 H40 N75600 D128  iid N(0,1)
         Wan2.1-14B 720p 81 frames: N = 75600, d = 5120 = 40 x 128
         (arganzheng.life, section 1.1 table)
  cfg    B2 H24 N4608  D128  cond/uncond stacked on the batch (MindIE-SD
         parallelism docs, CFG fusion); Q and K x4, 5% of each head's K rows
         x10 more (large-norm outliers)
Chunking follows the Ring degree the pages use: p = 4 for FLUX, p = 8 for Wan
(arganzheng.life, section 1.1 table); tiny uses p = 4; cfg uses 3 equal chunks
and an uneven 1000/1536/2072 split.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    seed: int
    kind: str                 # "iid" | "rmsnorm_qk" | "cfg_stress"
    chunks: tuple             # KV chunk lengths (sum = N), one per virtual ring rank
    alt_chunks: tuple = field(default=())

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H*N^2*D: the two GEMMs of attention (softmax not counted)."""
        return 4.0 * self.B * self.H * self.N * self.N * self.D

    @property
    def p(self) -> int:
        return len(self.chunks)


def even_chunks(n: int, p: int) -> tuple:
    """Split n rows into p consecutive chunks whose lengths differ by at most one."""
    if p < 1 or p > n:
        raise ValueError("need 1 <= p <= n")
    base, extra = divmod(n, p)
    return tuple(base + (1 if c < extra else 0) for c in range(p))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1024, 64, 0, "iid", even_chunks(1024, 4)),
    "flux": Workload("flux", 1, 24, 4608, 128, 1, "rmsnorm_qk", even_chunks(4608, 4)),
    "wan22": Workload("wan22", 1, 24, 27280, 128, 2, "iid", even_chunks(27280, 8)),
    "wan21": Workload("wan21", 1, 40, 75600, 128, 3, "iid", even_chunks(75600, 8)),
    "cfg": Workload("cfg", 2, 24, 4608, 128, 4, "cfg_stress", even_chunks(4608, 3),
                    alt_chunks=(1000, 1536, 2072)),
}

RMS_EPS = 1e-6
CFG_QK_GAIN = 4.0
CFG_OUTLIER_FRACTION = 0.05
CFG_OUTLIER_GAIN = 10.0


def make_qkv(w: Workload):
    """Seeded bf16 Q, K, V [B, H, N, D] (contiguous, CPU) for workload w."""
    g = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.kind == "rmsnorm_qk" and which in ("q", "k"):
            x = x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + RMS_EPS)
        elif w.kind == "cfg_stress" and which in ("q", "k"):
            x = x * CFG_QK_GAIN
        out.append(x)
    q, k, v = out
    if w.kind == "cfg_stress":
        n_out = int(math.floor(CFG_OUTLIER_FRACTION * w.N))
        for b in range(w.B):
            for h in range(w.H):
                idx = torch.randperm(w.N, generator=g)[:n_out]
                k[b, h, idx] = k[b, h, idx] * CFG_OUTLIER_GAIN
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v))


def sample_rows(n: int, count: int = 128, edge: int = 16, seed: int = 0) -> list:
    """Seeded sorted query-row sample: the first and last `edge` rows plus random interior rows."""
    if n <= count:
        return list(range(n))
    head = list(range(edge))
    tail = list(range(n - edge, n))
    g = torch.Generator().manual_seed(1000 + seed)
    interior = torch.randperm(n - 2 * edge, generator=g)[: count - 2 * edge] + edge
    return sorted(head + tail + interior.tolist())


def chunk_starts(chunks) -> list:
    """First key row of each chunk."""
    s, out = 0, []
    for c in chunks:
        out.append(s)
        s += c
    return out
