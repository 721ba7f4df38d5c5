"""C-ABI boundary checks that need no GPU: the library builds, loads and exports
every entry point include/ditattn.h declares, and argument validation rejects
bad calls with the documented status before any CUDA call is made."""
import ctypes
import math
import os
import re
import subprocess

import pytest
import torch

from diffusion_transformer_long_gb300 import build as dbuild
from diffusion_transformer_long_gb300 import ditattn as da

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ditattn.h")


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return da.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(dit_\w+)\s*\(", text, flags=re.M))


def test_header_matches_binding():
    assert declared_functions() == set(da.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", da.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_version_and_status_strings(lib):
    assert lib.dit_version() == 100
    assert da.status_string(da.DIT_OK) == "ok"
    assert da.status_string(da.DIT_ERR_TIMEOUT) == "device wait timed out"
    assert da.status_string(99) == "unknown status"


# Fake, well-separated, 256-byte-aligned "device" addresses: validation never dereferences them.
Q, K, V, OUT, LSE = (ctypes.c_void_p(a) for a in (1 << 40, 2 << 40, 3 << 40, 4 << 40, 5 << 40))


def fwd(lib, q=Q, k=K, v=V, out=OUT, lse=LSE, B=1, H=2, N=256, D=128, scale=0.088, dt=0):
    return lib.dit_attn_fwd(q, k, v, out, lse, B, H, N, D, scale, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), da.DIT_ERR_INVALID_ARG), (dict(H=-1), da.DIT_ERR_INVALID_ARG),
    (dict(N=0), da.DIT_ERR_INVALID_ARG), (dict(D=0), da.DIT_ERR_INVALID_ARG),
    (dict(D=96), da.DIT_ERR_UNSUPPORTED), (dict(D=256), da.DIT_ERR_UNSUPPORTED),
    (dict(q=None), da.DIT_ERR_INVALID_ARG), (dict(out=None), da.DIT_ERR_INVALID_ARG),
    (dict(k=ctypes.c_void_p((2 << 40) + 8)), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((4 << 40) + 4)), da.DIT_ERR_INVALID_ARG),
    (dict(lse=ctypes.c_void_p((5 << 40) + 2)), da.DIT_ERR_INVALID_ARG),
    (dict(scale=0.0), da.DIT_ERR_INVALID_ARG), (dict(scale=-1.0), da.DIT_ERR_INVALID_ARG),
    (dict(scale=math.inf), da.DIT_ERR_INVALID_ARG), (dict(scale=math.nan), da.DIT_ERR_INVALID_ARG),
    (dict(dt=7), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((1 << 40) + 4096)), da.DIT_ERR_INVALID_ARG),   # out inside q
    (dict(lse=ctypes.c_void_p((4 << 40) + 1024)), da.DIT_ERR_INVALID_ARG),   # lse inside out
    (dict(B=1 << 16, H=1 << 16), da.DIT_ERR_INVALID_ARG),                    # B*H overflows int
])
def test_fwd_validation(lib, kw, status):
    assert fwd(lib, **kw) == status


def chunk(lib, n_kv=100, hs=256 * 128, D=128, **kw):
    args = dict(q=Q, k=K, v=V, out=OUT, lse=LSE, B=1, H=2, N=256, scale=0.088, dt=0)
    args.update(kw)
    return lib.dit_attn_chunk_fwd(args["q"], args["k"], args["v"], args["out"], args["lse"],
                                  args["B"], args["H"], args["N"], n_kv, D, hs, args["scale"],
                                  args["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(n_kv=0), da.DIT_ERR_INVALID_ARG),
    (dict(lse=None), da.DIT_ERR_INVALID_ARG),                 # a chunk's LSE is its output
    (dict(n_kv=300, hs=256 * 128), da.DIT_ERR_INVALID_ARG),   # stride shorter than the chunk
    (dict(hs=256 * 128 + 4), da.DIT_ERR_INVALID_ARG),         # stride not 16-byte aligned
    (dict(hs=1 << 39), da.DIT_ERR_INVALID_ARG),
    (dict(D=80), da.DIT_ERR_UNSUPPORTED),
    (dict(k=ctypes.c_void_p((2 << 40) + 2)), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((2 << 40) + 64)), da.DIT_ERR_INVALID_ARG),     # out inside k
])
def test_chunk_validation(lib, kw, status):
    assert chunk(lib, **kw) == status


def chunks_batched(lib, starts=(0, 40, 100), n_kv=100, hs=256 * 128, D=128, p=None, **kw):
    args = dict(q=Q, k=K, v=V, out=OUT, lse=LSE, B=1, H=2, N=256, scale=0.088, dt=0)
    args.update(kw)
    p = len(starts) - 1 if p is None else p
    arr = (ctypes.c_int * max(1, len(starts)))(*starts) if starts is not None else None
    return lib.dit_attn_chunks_fwd(args["q"], args["k"], args["v"], args["out"], args["lse"],
                                   args["B"], args["H"], args["N"], n_kv, D, hs, p, arr,
                                   args["scale"], args["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(starts=None, p=2), da.DIT_ERR_INVALID_ARG),                 # no chunk table
    (dict(starts=(0,), p=0), da.DIT_ERR_INVALID_ARG),                 # p = 0
    (dict(starts=tuple(range(66)), n_kv=100, p=65), da.DIT_ERR_INVALID_ARG),   # p > 64
    (dict(starts=(0, 40, 40)), da.DIT_ERR_INVALID_ARG),               # empty chunk
    (dict(starts=(0, 60, 40)), da.DIT_ERR_INVALID_ARG),               # decreasing
    (dict(starts=(-1, 40, 100)), da.DIT_ERR_INVALID_ARG),             # before the first key
    (dict(starts=(0, 40, 101)), da.DIT_ERR_INVALID_ARG),              # past n_kv
    (dict(n_kv=0), da.DIT_ERR_INVALID_ARG), (dict(D=96), da.DIT_ERR_UNSUPPORTED),
    (dict(dt=5), da.DIT_ERR_INVALID_ARG),
    # the second partial block (256 rows x 2 heads x 128 x 4 B past OUT) would overlap LSE
    (dict(lse=ctypes.c_void_p((4 << 40) + 2 * 256 * 128 * 4 + 256)), da.DIT_ERR_INVALID_ARG),
    # the second chunk's LSE rows overlap a partial block placed right after them
    (dict(out=ctypes.c_void_p((5 << 40) + 2 * 256 * 4 + 256)), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((2 << 40) + 64)), da.DIT_ERR_INVALID_ARG),     # partials inside k
])
def test_chunks_batched_validation(lib, kw, status):
    assert chunks_batched(lib, **kw) == status


def test_chunks_batched_binding_rejects_host_tensors():
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        da.attn_chunks_fwd(x, x, x, [4, 4])


def accumulate(lib, n_kv=100, hs=256 * 128, D=128, **kw):
    args = dict(q=Q, k=K, v=V, out=OUT, lse=LSE, B=1, H=2, N=256, scale=0.088)
    args.update(kw)
    return lib.dit_attn_chunk_fwd_accumulate(args["q"], args["k"], args["v"], args["out"],
                                             args["lse"], args["B"], args["H"], args["N"], n_kv, D,
                                             hs, args["scale"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(n_kv=0), da.DIT_ERR_INVALID_ARG), (dict(N=0), da.DIT_ERR_INVALID_ARG),
    (dict(n_kv=300, hs=256 * 128), da.DIT_ERR_INVALID_ARG),   # stride shorter than the chunk
    (dict(hs=256 * 128 + 4), da.DIT_ERR_INVALID_ARG),
    (dict(D=96), da.DIT_ERR_UNSUPPORTED),
    (dict(out=None), da.DIT_ERR_INVALID_ARG), (dict(lse=None), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((4 << 40) + 8)), da.DIT_ERR_INVALID_ARG),     # o_run not 16-aligned
    (dict(lse=ctypes.c_void_p((5 << 40) + 2)), da.DIT_ERR_INVALID_ARG),
    (dict(scale=math.nan), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((3 << 40) + 64)), da.DIT_ERR_INVALID_ARG),     # o_run inside v
    (dict(lse=ctypes.c_void_p((4 << 40) + 1024)), da.DIT_ERR_INVALID_ARG),  # lse_run inside o_run
])
def test_accumulate_validation(lib, kw, status):
    assert accumulate(lib, **kw) == status


def test_accumulate_binding_checks_running_state(lib):
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):           # host tensors
        da.attn_chunk_fwd_accumulate(x, x, x, o, torch.zeros(1, 1, 8))
    with pytest.raises(ValueError):           # chunk lengths must cover the keys
        da.ring_attention(x, x, x, [3, 4])


def strided(lib, qs=None, ks=None, vs=None, os_=None, out=OUT, B=2, H=3, N=256, n_kv=100, D=128,
            dt=0):
    def ref(x):
        return None if x is None else ctypes.byref(da.Strides(*x))
    return lib.dit_attn_fwd_strided(Q, ref(qs), K, ref(ks), V, ref(vs), out, ref(os_), LSE, B, H, N,
                                    n_kv, D, 0.088, dt, None)


BSND = (256 * 3 * 128, 128, 3 * 128)  # [B, N, H, D] memory, B=2 H=3 N=256 D=128


@pytest.mark.parametrize("kw,status", [
    (dict(qs=(0, 128, 384)), da.DIT_ERR_INVALID_ARG),                 # zero stride
    (dict(ks=(-8, 128, 384)), da.DIT_ERR_INVALID_ARG),                # negative stride
    (dict(vs=(98304, 132, 384)), da.DIT_ERR_INVALID_ARG),             # not a multiple of 8
    (dict(qs=(1 << 39, 128, 384)), da.DIT_ERR_INVALID_ARG),
    (dict(os_=(98304, 128, 64)), da.DIT_ERR_INVALID_ARG),             # out rows overlap
    (dict(os_=(256 * 128, 128, 3 * 128)), da.DIT_ERR_INVALID_ARG),   # out batches overlap
    (dict(out=ctypes.c_void_p((1 << 40) + 256)), da.DIT_ERR_INVALID_ARG),  # out inside q's range
    (dict(D=96), da.DIT_ERR_UNSUPPORTED), (dict(n_kv=0), da.DIT_ERR_INVALID_ARG),
    (dict(dt=5), da.DIT_ERR_INVALID_ARG),
])
def test_strided_validation(lib, kw, status):
    assert strided(lib, **kw) == status


def test_strided_size_one_dimensions_take_any_stride(lib):
    # B = 1, H = 1: their strides address nothing; validation must not reject them (the call
    # then fails only at launch, here without a GPU).
    st = strided(lib, qs=(0, 3, 128), ks=(0, 1, 128), vs=(5, 5, 128), os_=(0, 0, 128), B=1, H=1)
    assert st not in (da.DIT_ERR_INVALID_ARG, da.DIT_ERR_UNSUPPORTED)


def copy(lib, src=Q, ss=None, dst=OUT, ds=None, B=2, H=3, N=256, D=128, dt=1):
    def ref(x):
        return None if x is None else ctypes.byref(da.Strides(*x))
    return lib.dit_layout_copy(src, ref(ss), dst, ref(ds), B, H, N, D, dt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(src=None), da.DIT_ERR_INVALID_ARG), (dict(N=0), da.DIT_ERR_INVALID_ARG),
    (dict(D=32), da.DIT_ERR_UNSUPPORTED), (dict(dt=9), da.DIT_ERR_INVALID_ARG),
    (dict(dst=ctypes.c_void_p((4 << 40) + 8)), da.DIT_ERR_INVALID_ARG),
    (dict(ss=(1, 128, 384)), da.DIT_ERR_INVALID_ARG),
    (dict(ds=(98304, 128, 64)), da.DIT_ERR_INVALID_ARG),               # dst rows overlap
    (dict(dst=ctypes.c_void_p((1 << 40) + 4096)), da.DIT_ERR_INVALID_ARG),  # dst inside src
    (dict(N=65535 * 128 + 1), da.DIT_ERR_UNSUPPORTED),                 # copy grid too tall
])
def test_layout_copy_validation(lib, kw, status):
    assert copy(lib, **kw) == status


def stale(lib, q=Q, kn=K, vn=V, kb=ctypes.c_void_p(6 << 40), vb=ctypes.c_void_p(7 << 40), out=OUT,
          lse=LSE, B=1, H=2, m=256, N=1024, D=128, row0=256, splits=1, ws=None, ws_bytes=0):
    return lib.dit_attn_stale_kv_fwd(q, kn, vn, kb, vb, out, lse, B, H, m, N, D, row0, 0.088, 0,
                                     splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(m=0), da.DIT_ERR_INVALID_ARG), (dict(row0=-1), da.DIT_ERR_INVALID_ARG),
    (dict(row0=769), da.DIT_ERR_INVALID_ARG),                          # patch past the buffer
    (dict(m=1025), da.DIT_ERR_INVALID_ARG), (dict(D=80), da.DIT_ERR_UNSUPPORTED),
    (dict(kn=None), da.DIT_ERR_INVALID_ARG),
    (dict(kb=ctypes.c_void_p((7 << 40) + 4096)), da.DIT_ERR_INVALID_ARG),   # k_buf inside v_buf
    (dict(kn=ctypes.c_void_p((6 << 40) + 1024)), da.DIT_ERR_INVALID_ARG),   # k_new inside k_buf
    (dict(out=ctypes.c_void_p((2 << 40) + 64)), da.DIT_ERR_INVALID_ARG),    # out inside k_new
    (dict(splits=9), da.DIT_ERR_INVALID_ARG),                               # > 8 key tiles
    (dict(splits=2), da.DIT_ERR_INVALID_ARG),                               # no workspace
])
def test_stale_kv_validation(lib, kw, status):
    assert stale(lib, **kw) == status


WS = ctypes.c_void_p(8 << 40)


def splitkv(lib, n_kv=1000, splits=3, ws=WS, ws_bytes=None, B=1, H=2, N=256, D=128, out=OUT):
    if ws_bytes is None:
        ws_bytes = lib.dit_attn_splitkv_workspace_bytes(B, H, N, D, splits)
    return lib.dit_attn_chunk_fwd_splitkv(Q, K, V, out, LSE, B, H, N, n_kv, D, N * D * 8, 0.088, 0,
                                          splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(splits=0), da.DIT_ERR_INVALID_ARG), (dict(splits=65, n_kv=65 * 128), da.DIT_ERR_INVALID_ARG),
    (dict(splits=9, n_kv=1000), da.DIT_ERR_INVALID_ARG),                  # 8 key tiles only
    (dict(ws=None), da.DIT_ERR_INVALID_ARG),
    (dict(ws=ctypes.c_void_p((8 << 40) + 128)), da.DIT_ERR_INVALID_ARG),  # not 256-byte aligned
    (dict(ws_bytes=1000), da.DIT_ERR_INVALID_ARG),                        # too small
    (dict(ws=ctypes.c_void_p((4 << 40) + 256)), da.DIT_ERR_INVALID_ARG),  # workspace inside out
    (dict(D=96), da.DIT_ERR_UNSUPPORTED),
])
def test_splitkv_validation(lib, kw, status):
    assert splitkv(lib, **kw) == status


def test_noalloc_splitkv_rejects_beyond_scratch_before_any_cuda_call(lib):
    # Wan2.2-sized queries with 8 key splits need 2.7 GB of partials; the scratch is 128 MiB.
    B, H, N, D = 1, 24, 27280, 128
    st = lib.dit_attn_chunk_fwd_splitkv_noalloc(Q, K, V, OUT, LSE, B, H, N, N, D, N * D, 0.088, 0,
                                                8, None)
    assert st == da.DIT_ERR_UNSUPPORTED
    assert lib.dit_attn_chunk_fwd_splitkv_noalloc(Q, K, V, OUT, LSE, B, H, N, N, D, N * D, 0.088,
                                                  0, 0, None) == da.DIT_ERR_INVALID_ARG


def test_splitkv_workspace_bytes(lib):
    f = lib.dit_attn_splitkv_workspace_bytes
    assert f(1, 2, 256, 128, 1) == 0 and f(0, 2, 256, 128, 3) == 0
    rows = 1 * 2 * 256
    o = 3 * rows * 128 * 4
    assert f(1, 2, 256, 128, 3) == (o + 255) // 256 * 256 + 3 * rows * 4
    rows = 3 * 5 * 77
    o = 4 * rows * 64 * 4
    assert f(3, 5, 77, 64, 4) == (o + 255) // 256 * 256 + 4 * rows * 4
    assert lib.dit_attn_splitkv_suggest(1, 24, 3410, 27280) == 1  # no GPU here: no SM count


def merge(lib, p=4, parts=Q, lses=K, out=OUT, lse=LSE, B=1, H=2, N=256, D=128, pdt=0, odt=0):
    return lib.dit_attn_lse_merge(parts, lses, p, out, lse, B, H, N, D, pdt, odt, None)


@pytest.mark.parametrize("kw,status", [
    (dict(p=0), da.DIT_ERR_INVALID_ARG), (dict(N=0), da.DIT_ERR_INVALID_ARG),
    (dict(D=32), da.DIT_ERR_UNSUPPORTED), (dict(parts=None), da.DIT_ERR_INVALID_ARG),
    (dict(parts=ctypes.c_void_p((1 << 40) + 8)), da.DIT_ERR_INVALID_ARG),
    (dict(lses=ctypes.c_void_p((2 << 40) + 1)), da.DIT_ERR_INVALID_ARG),
    (dict(pdt=3), da.DIT_ERR_INVALID_ARG), (dict(odt=-1), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((1 << 40) + 4096)), da.DIT_ERR_INVALID_ARG),   # out inside partials
    (dict(lse=ctypes.c_void_p((2 << 40) + 16)), da.DIT_ERR_INVALID_ARG),     # lse inside lses
])
def test_merge_validation(lib, kw, status):
    assert merge(lib, **kw) == status


def test_binding_rejects_host_tensors_and_bad_dtypes(lib):
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        da.attn_fwd(x, x, x)
    with pytest.raises(TypeError):
        da._dt(torch.float16)


def test_kv_head_stride_of_views():
    full = torch.zeros(2, 3, 40, 64)
    assert da.kv_head_stride(full[:, :, 5:17]) == 40 * 64
    assert da.kv_head_stride(torch.zeros(1, 1, 9, 64)) == 9 * 64
    assert da.kv_head_stride(torch.zeros(4, 1, 9, 64)[:, :, 2:5]) == 9 * 64
    with pytest.raises(ValueError):
        da.kv_head_stride(full.transpose(2, 3))


def noalloc(lib, n_kv=1000, splits=3, out=OUT, lse=LSE, q=Q, B=1, H=2, N=256, D=128):
    return lib.dit_attn_chunk_fwd_splitkv_noalloc(q, K, V, out, lse, B, H, N, n_kv, D, N * D * 8,
                                                  0.088, 0, splits, None)


@pytest.mark.parametrize("kw,status", [
    (dict(splits=0), da.DIT_ERR_INVALID_ARG),
    (dict(splits=65, n_kv=65 * 128), da.DIT_ERR_INVALID_ARG),      # more than 64 splits
    (dict(splits=9, n_kv=1000), da.DIT_ERR_INVALID_ARG),           # more splits than key tiles
    (dict(lse=None), da.DIT_ERR_INVALID_ARG),
    (dict(out=None), da.DIT_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((1 << 40) + 4096)), da.DIT_ERR_INVALID_ARG),   # out inside q
    (dict(lse=ctypes.c_void_p((4 << 40) + 1024)), da.DIT_ERR_INVALID_ARG),   # lse inside out
    (dict(D=96), da.DIT_ERR_UNSUPPORTED),
    # partials of 24 heads x 27280 rows x 8 splits exceed the 128 MiB scratch
    (dict(B=1, H=24, N=27280, n_kv=27280 * 8, splits=8), da.DIT_ERR_UNSUPPORTED),
])
def test_noalloc_splitkv_validation(lib, kw, status):
    assert noalloc(lib, **kw) == status


CPU = torch.device("cpu")


@pytest.mark.parametrize("bad", [
    dict(out=torch.zeros(1, 2, 8, 32)),                                 # wrong shape
    dict(out=torch.zeros(1, 2, 8, 64, dtype=torch.float16)),            # wrong dtype
    dict(out=torch.zeros(1, 2, 64, 8).transpose(2, 3)),                 # not contiguous
    dict(lse=torch.zeros(1, 2, 8, dtype=torch.bfloat16)),               # lse not fp32
    dict(lse=torch.zeros(1, 2, 9)),                                     # lse wrong shape
    dict(lse=torch.zeros(1, 2, 16)[:, :, ::2]),                         # lse not contiguous
    dict(out=[0.0] * 4),                                                # not a tensor
])
def test_binding_rejects_bad_caller_outputs(bad):
    kw = dict(out=None, lse=None)
    kw.update(bad)
    with pytest.raises(ValueError):
        da._check_out(kw["out"], kw["lse"], (1, 2, 8, 64), CPU)


def test_binding_output_checks_accept_good_outputs_and_views():
    da._check_out(torch.zeros(1, 2, 8, 64), torch.zeros(1, 2, 8), (1, 2, 8, 64), CPU)
    da._check_out(torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16), None, (1, 2, 8, 64), CPU)
    # a token-major view is fine where the entry point takes strides
    bsnd = torch.zeros(1, 8, 2, 64).transpose(1, 2)
    da._check_out(bsnd, None, (1, 2, 8, 64), CPU, contiguous=False)
    with pytest.raises(ValueError):
        da._check_out(bsnd, None, (1, 2, 8, 64), CPU)
    with pytest.raises(ValueError):          # a tensor on another device
        da._check_out(torch.zeros(1, 2, 8, 64), None, (1, 2, 8, 64), torch.device("cuda", 0))
