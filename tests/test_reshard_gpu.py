"""GPU checks of the strided layout copy (dit_layout_copy): bit-exact against PyTorch CPU
indexing of the same values.

Covers the token-major <-> head-major transpose, padded strides, fp32 and bf16, and the
local halves of the Ulysses re-shard (arganzheng.life multi-GPU diffusion parallelism,
section 4.1 Ulysses; valdrada.cn Wan2.2, CP section): p virtual ranks pack their token
shards by head group, a simulated all-to-all hands buffer r of rank s to rank r, and each
rank unpacks all tokens of its heads.  The round trip must reproduce the exact head
slices of the full sequence.
"""
import pytest
import torch

from diffusion_transformer_long_gb300 import ditattn as da

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def rand(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,N,H,D", [(1, 1, 1, 64), (2, 333, 3, 128), (1, 4608, 24, 128),
                                     (2, 129, 5, 64)])
def test_bsnd_bhnd_round_trip_bit_exact(dtype, B, N, H, D):
    x = rand((B, N, H, D), dtype, seed=N * H + D)
    xd = x.to(DEV)
    y = da.bsnd_to_bhnd(xd)
    z = da.bhnd_to_bsnd(y)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), x.transpose(1, 2).contiguous())
    assert torch.equal(z.cpu(), x)


def test_padded_and_sliced_views():
    B, H, N, D = 2, 4, 300, 128
    x = rand((B, H, N, D + 64), torch.bfloat16, seed=1)
    src = x.to(DEV)[..., :D]                                   # padded rows
    big = torch.zeros(B, N + 10, H, D + 128, dtype=torch.bfloat16, device=DEV)
    dst = big[:, 5:5 + N, :, :D].transpose(1, 2)               # token-major window
    da.layout_copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), x[..., :D])
    assert (big[:, :5] == 0).all() and (big[:, 5 + N:] == 0).all() and (big[..., D:] == 0).all()


def test_kv_buffer_row_update_in_place():
    B, H, N, m, D, row0 = 1, 3, 1000, 200, 128, 417
    buf = rand((B, H, N, D), torch.bfloat16, seed=2)
    new = rand((B, H, m, D), torch.bfloat16, seed=3)
    bd = buf.to(DEV)
    da.layout_copy(new.to(DEV), bd[:, :, row0:row0 + m])
    torch.cuda.synchronize()
    ref = buf.clone()
    ref[:, :, row0:row0 + m] = new
    assert torch.equal(bd.cpu(), ref)


@pytest.mark.parametrize("p", [2, 4, 8])
def test_ulysses_pack_all_to_all_unpack(p):
    B, N, H, D = 1, 27280 // 20, 24, 128   # Wan2.2-like head count, a short sequence
    N -= N % p
    x = rand((B, N, H, D), torch.bfloat16, seed=p)
    xd = x.to(DEV)
    n, hp = N // p, H // p
    send = [da.ulysses_pack(xd[:, s * n:(s + 1) * n].contiguous(), p) for s in range(p)]
    # the all-to-all: rank r receives buffer r of every rank s, in rank order
    recv = [torch.stack([send[s][r] for s in range(p)]) for r in range(p)]
    full = [da.ulysses_unpack(recv[r]) for r in range(p)]
    torch.cuda.synchronize()
    for r in range(p):
        assert torch.equal(full[r].cpu(), x[:, :, r * hp:(r + 1) * hp])
