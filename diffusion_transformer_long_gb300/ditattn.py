"""Python binding of the ditattn C ABI (include/ditattn.h): argument marshalling only.

Every step of attention runs in the library's CUDA kernels; this module checks
shapes/dtypes, allocates outputs with PyTorch when the caller does not pass
them, and hands raw pointers plus the current CUDA stream to the C entry
points.  There is no CPU fallback: without the built library or a CUDA device
every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_CUDA, DIT_ERR_TIMEOUT = range(5)
DIT_F32, DIT_BF16 = 0, 1

EXPORTED_SYMBOLS = ("dit_attn_fwd", "dit_attn_fwd_strided", "dit_attn_chunk_fwd", "dit_attn_chunks_fwd",
                    "dit_attn_chunk_fwd_accumulate", "dit_attn_lse_merge", "dit_layout_copy",
                    "dit_attn_stale_kv_fwd", "dit_attn_chunk_fwd_splitkv",
                    "dit_attn_splitkv_workspace_bytes", "dit_attn_splitkv_suggest",
                    "dit_attn_chunk_fwd_splitkv_noalloc",
                    "dit_attn_check", "dit_test_inject_stall", "dit_test_set_grid_limit",
                    "dit_status_string", "dit_version")


class Strides(ctypes.Structure):
    """dit_strides: element strides (b, h, n) of a [B, H, N, D] view with contiguous D."""
    _fields_ = [("b", ctypes.c_longlong), ("h", ctypes.c_longlong), ("n", ctypes.c_longlong)]

_lib = None


class DitError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libditattn.so (built in-tree by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        P, I, LL, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
        L.dit_attn_fwd.restype = I
        L.dit_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, F, I, P]
        SP = ctypes.POINTER(Strides)
        L.dit_attn_fwd_strided.restype = I
        L.dit_attn_fwd_strided.argtypes = [P, SP, P, SP, P, SP, P, SP, P, I, I, I, I, I, F, I, P]
        L.dit_attn_stale_kv_fwd.restype = I
        L.dit_attn_stale_kv_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P,
                                            ctypes.c_size_t, P]
        L.dit_attn_chunk_fwd_splitkv.restype = I
        L.dit_attn_chunk_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, LL, F, I, I, P,
                                                 ctypes.c_size_t, P]
        L.dit_attn_chunk_fwd_splitkv_noalloc.restype = I
        L.dit_attn_chunk_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, LL, F, I,
                                                         I, P]
        L.dit_attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
        L.dit_attn_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
        L.dit_attn_splitkv_suggest.restype = I
        L.dit_attn_splitkv_suggest.argtypes = [I, I, I, I]
        L.dit_layout_copy.restype = I
        L.dit_layout_copy.argtypes = [P, SP, P, SP, I, I, I, I, I, P]
        L.dit_attn_chunk_fwd.restype = I
        L.dit_attn_chunk_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, LL, F, I, P]
        L.dit_attn_chunks_fwd.restype = I
        L.dit_attn_chunks_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, LL, I, ctypes.POINTER(I), F,
                                          I, P]
        L.dit_attn_chunk_fwd_accumulate.restype = I
        L.dit_attn_chunk_fwd_accumulate.argtypes = [P, P, P, P, P, I, I, I, I, I, LL, F, P]
        L.dit_attn_lse_merge.restype = I
        L.dit_attn_lse_merge.argtypes = [P, P, I, P, P, I, I, I, I, I, I, P]
        L.dit_attn_check.restype = I
        L.dit_attn_check.argtypes = [P]
        L.dit_test_inject_stall.restype = None
        L.dit_test_inject_stall.argtypes = [I, LL]
        L.dit_test_set_grid_limit.restype = None
        L.dit_test_set_grid_limit.argtypes = [I]
        L.dit_status_string.restype = ctypes.c_char_p
        L.dit_status_string.argtypes = [I]
        L.dit_version.restype = I
        L.dit_version.argtypes = []
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dit_status_string(int(status)).decode()


def _dt(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return DIT_F32
    if dtype == torch.bfloat16:
        return DIT_BF16
    raise TypeError(f"unsupported output dtype {dtype}; use torch.float32 or torch.bfloat16")


def _stream(device: torch.device, stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, D]")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [B, H, N, D]")


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _check_out(out, lse, shape, device, out_name="out", lse_name="lse", contiguous=True):
    """Caller-provided outputs: `out` a [shape] fp32 or bf16 tensor and `lse` a contiguous fp32
    [shape[:-1]] tensor, both on `device` (the C ABI cannot see buffer sizes, so a wrong shape,
    dtype, layout or device must be stopped here).  `contiguous=False` lets `out` be any view
    whose last dimension is contiguous (the strided entry point checks the strides itself)."""
    shape = tuple(int(x) for x in shape)
    if out is not None:
        if not isinstance(out, torch.Tensor) or out.device != device:
            raise ValueError(f"{out_name} must be a tensor on {device}")
        if tuple(out.shape) != shape:
            raise ValueError(f"{out_name} must have shape {list(shape)}, got {list(out.shape)}")
        if out.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"{out_name} must be float32 or bfloat16, got {out.dtype}")
        if contiguous and not out.is_contiguous():
            raise ValueError(f"{out_name} must be contiguous")
        if not contiguous and out.stride(-1) != 1:
            raise ValueError(f"{out_name} must have a contiguous last dimension")
    if lse is not None:
        if not isinstance(lse, torch.Tensor) or lse.device != device:
            raise ValueError(f"{lse_name} must be a tensor on {device}")
        if tuple(lse.shape) != shape[:-1]:
            raise ValueError(f"{lse_name} must have shape {list(shape[:-1])}, "
                             f"got {list(lse.shape)}")
        if lse.dtype != torch.float32:
            raise ValueError(f"{lse_name} must be float32, got {lse.dtype}")
        if not lse.is_contiguous():
            raise ValueError(f"{lse_name} must be contiguous")


def attn_fwd(q, k, v, out=None, lse=None, scale=None, out_dtype=torch.float32, stream=None,
             with_lse=True):
    """Fused attention over all keys.  q, k, v: CUDA bf16 [B, H, N, D] contiguous.

    Returns (out [B, H, N, D] of out_dtype, lse fp32 [B, H, N]); with_lse=False skips the
    LSE (the library gets NULL) and returns (out, None).
    """
    _check_qkv(q, k, v)
    if not (k.is_contiguous() and v.is_contiguous()) or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("k and v must be contiguous with q's shape")
    B, H, N, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check_out(out, lse, (B, H, N, D), q.device)
    if out is None:
        out = torch.empty((B, H, N, D), device=q.device, dtype=out_dtype)
    if lse is None and with_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        st = lib().dit_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                _ptr(lse) if with_lse else None, B, H, N, D, scale,
                                _dt(out.dtype), _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_fwd")
    return out, (lse if with_lse else None)


def view_strides(x: torch.Tensor) -> Strides:
    """dit_strides of a [B, H, N, D] tensor view whose last dimension is contiguous (e.g. a
    token-major [B, N, H, D] tensor passed as x.transpose(1, 2))."""
    if x.dim() != 4 or x.stride(3) != 1:
        raise ValueError("expected a [B, H, N, D] view with contiguous last dimension")
    return Strides(*(int(s) for s in x.stride()[:3]))


def attn_fwd_strided(q, k, v, out=None, lse=None, scale=None, out_dtype=torch.float32,
                     stream=None):
    """Attention over arbitrary strided [B, H, N, D] views (last dimension contiguous): q is
    [B, H, N_q, D], k and v [B, H, n_kv, D].  A BSND tensor x ([B, N, H, D] in memory) is passed as
    x.transpose(1, 2), and `out` may be such a view too.  Returns (out, lse fp32 [B, H, N_q])."""
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4:
            raise ValueError("q, k, v must be 4-D bf16 CUDA tensor views")
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v must be [B, H, n_kv, D] matching q")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, Nq, D), device=q.device, dtype=out_dtype)
    _check_out(out, lse, (B, H, Nq, D), q.device, contiguous=False)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    qs, ks, vs, os_ = (view_strides(t) for t in (q, k, v, out))
    with torch.cuda.device(q.device):
        st = lib().dit_attn_fwd_strided(_ptr(q), ctypes.byref(qs), _ptr(k), ctypes.byref(ks),
                                        _ptr(v), ctypes.byref(vs), _ptr(out), ctypes.byref(os_),
                                        _ptr(lse), B, H, Nq, k.shape[2], D, scale, _dt(out.dtype),
                                        _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_fwd_strided")
    return out, lse


def layout_copy(src, dst, stream=None):
    """dst[...] = src[...] for two [B, H, N, D] views of the same shape and dtype (bf16 or fp32,
    last dimension contiguous), by the library's strided copy kernel.  Returns dst."""
    if not (src.is_cuda and dst.is_cuda) or src.device != dst.device:
        raise ValueError("src and dst must be CUDA tensors on one device")
    if src.shape != dst.shape or src.dtype != dst.dtype or src.dim() != 4:
        raise ValueError("src and dst must be [B, H, N, D] views of one shape and dtype")
    B, H, N, D = src.shape
    ss, ds = view_strides(src), view_strides(dst)
    with torch.cuda.device(src.device):
        st = lib().dit_layout_copy(_ptr(src), ctypes.byref(ss), _ptr(dst), ctypes.byref(ds), B, H,
                                   N, D, _dt(src.dtype), _stream(src.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_layout_copy")
    return dst


def bsnd_to_bhnd(x, out=None, stream=None):
    """Token-major [B, N, H, D] -> contiguous head-major [B, H, N, D]."""
    B, N, H, D = x.shape
    if out is None:
        out = torch.empty((B, H, N, D), device=x.device, dtype=x.dtype)
    layout_copy(x.transpose(1, 2), out, stream=stream)
    return out


def bhnd_to_bsnd(x, out=None, stream=None):
    """Head-major [B, H, N, D] -> contiguous token-major [B, N, H, D]."""
    B, H, N, D = x.shape
    if out is None:
        out = torch.empty((B, N, H, D), device=x.device, dtype=x.dtype)
    layout_copy(x, out.transpose(1, 2), stream=stream)
    return out


def ulysses_pack(x_local, p, out=None, stream=None):
    """Send buffers of one rank's Ulysses all-to-all: its token shard x_local [B, N/p, H, D]
    (token-major) split by head groups into out [p, B, N/p, H/p, D], out[r] = the heads
    r*H/p .. (r+1)*H/p that rank r will own.  One strided copy per destination rank."""
    B, n, H, D = x_local.shape
    if H % p:
        raise ValueError("Ulysses needs the head count divisible by the degree")
    hp = H // p
    if out is None:
        out = torch.empty((p, B, n, hp, D), device=x_local.device, dtype=x_local.dtype)
    for r in range(p):
        layout_copy(x_local[:, :, r * hp:(r + 1) * hp].transpose(1, 2), out[r].transpose(1, 2),
                    stream=stream)
    return out


def ulysses_unpack(recv, out=None, stream=None):
    """Receive side: recv [p, B, N/p, H/p, D], recv[r] = the token shard of rank r for this
    rank's head group, assembled into all tokens of those heads, out [B, N, H/p, D]
    (token-major; pass out.transpose(1, 2) to the attention as a [B, H/p, N, D] view)."""
    p, B, n, hp, D = recv.shape
    if out is None:
        out = torch.empty((B, p * n, hp, D), device=recv.device, dtype=recv.dtype)
    for r in range(p):
        layout_copy(recv[r].transpose(1, 2), out[:, r * n:(r + 1) * n].transpose(1, 2),
                    stream=stream)
    return out


def splitkv_plan(B, H, n_q, n_kv, D, device, splits=None, workspace=None):
    """(splits, workspace) for a split-KV call: the library's suggestion when splits is None,
    and a fresh torch workspace of the required size unless one is given."""
    with torch.cuda.device(device):
        if splits is None:
            splits = int(lib().dit_attn_splitkv_suggest(B, H, n_q, n_kv))
        need = int(lib().dit_attn_splitkv_workspace_bytes(B, H, n_q, D, splits))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if need and (workspace.numel() * workspace.element_size() < need or not workspace.is_cuda):
        raise ValueError(f"workspace must be a CUDA buffer of at least {need} bytes")
    return splits, workspace


def attn_chunk_fwd_splitkv(q, k, v, out=None, lse=None, scale=None, out_dtype=torch.float32,
                           splits=None, workspace=None, stream=None):
    """dit_attn_chunk_fwd with each (head, Q pair) split over key ranges into fp32 partials in
    `workspace` and merged (for few queries against many keys).  splits=None asks the library;
    the workspace is allocated with torch unless given.  Returns (out, lse)."""
    _check_qkv(q, k, v)
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v chunk must be [B, H, n_kv, D] matching q")
    hs = kv_head_stride(k)
    if kv_head_stride(v) != hs:
        raise ValueError("k and v chunks must have the same head stride")
    n_kv = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check_out(out, lse, (B, H, Nq, D), q.device)
    if out is None:
        out = torch.empty((B, H, Nq, D), device=q.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    splits, workspace = splitkv_plan(B, H, Nq, n_kv, D, q.device, splits, workspace)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(q.device):
        st = lib().dit_attn_chunk_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                              Nq, n_kv, D, hs, scale, _dt(out.dtype), splits,
                                              ws_ptr, ws_bytes, _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_chunk_fwd_splitkv")
    return out, lse


def attn_chunk_fwd_splitkv_noalloc(q, k, v, out, lse, scale=None, splits=None, stream=None):
    """Split-KV attention into the caller's out / lse with the library's fixed device scratch:
    no allocation on this path (out and lse are required).  splits=None asks the library.
    Calls overlapping in time race on the one scratch array."""
    _check_qkv(q, k, v)
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v chunk must be [B, H, n_kv, D] matching q")
    hs = kv_head_stride(k)
    if kv_head_stride(v) != hs:
        raise ValueError("k and v chunks must have the same head stride")
    n_kv = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None or lse is None:
        raise ValueError("out and lse are required: this path allocates nothing")
    _check_out(out, lse, (B, H, Nq, D), q.device)
    with torch.cuda.device(q.device):
        if splits is None:
            splits = int(lib().dit_attn_splitkv_suggest(B, H, Nq, n_kv))
        st = lib().dit_attn_chunk_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                                      _ptr(lse), B, H, Nq, n_kv, D, hs, scale,
                                                      _dt(out.dtype), splits,
                                                      _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_chunk_fwd_splitkv_noalloc")
    return out, lse


def stale_kv_attention(q, k_new, v_new, k_buf, v_buf, row0, out=None, lse=None, scale=None,
                       out_dtype=torch.float32, splits=1, workspace=None, stream=None):
    """One patch of displaced patch parallelism: the patch's fresh K/V rows [row0, row0 + m)
    overwrite their stale rows of the KV buffers (in place), then its m queries attend to all N
    buffer rows.  q, k_new, v_new [B, H, m, D]; k_buf, v_buf [B, H, N, D]; all bf16, contiguous.
    splits: key ranges of the attention (1: none; None: the library's suggestion).
    Returns (out [B, H, m, D], lse fp32 [B, H, m])."""
    for t in (q, k_new, v_new, k_buf, v_buf):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q, k_new, v_new, k_buf, v_buf must be contiguous 4-D bf16 CUDA tensors")
    B, H, m, D = q.shape
    N = k_buf.shape[2]
    if k_new.shape != q.shape or v_new.shape != q.shape or v_buf.shape != k_buf.shape \
            or tuple(k_buf.shape[:2]) != (B, H) or k_buf.shape[3] != D:
        raise ValueError("shape mismatch between the patch and the KV buffers")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check_out(out, lse, (B, H, m, D), q.device)
    if out is None:
        out = torch.empty((B, H, m, D), device=q.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, m), device=q.device, dtype=torch.float32)
    splits, workspace = splitkv_plan(B, H, m, N, D, q.device, splits, workspace)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(q.device):
        st = lib().dit_attn_stale_kv_fwd(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_buf),
                                         _ptr(v_buf), _ptr(out), _ptr(lse), B, H, m, N, D,
                                         int(row0), scale, _dt(out.dtype), splits, ws_ptr,
                                         ws_bytes, _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_stale_kv_fwd")
    return out, lse


def kv_head_stride(k: torch.Tensor) -> int:
    """Elements between consecutive (b, h) heads of a [B, H, n, D] K/V view (rows D apart)."""
    B, H, n, D = k.shape
    if k.stride(3) != 1 or (n > 1 and k.stride(2) != D):
        raise ValueError("K/V rows must be contiguous and D elements apart")
    if B > 1 and H > 1:
        if k.stride(0) != H * k.stride(1):
            raise ValueError("K/V heads must be evenly spaced across the batch")
        return k.stride(1)
    if H > 1:
        return k.stride(1)
    if B > 1:
        return k.stride(0)
    return n * D  # a single head: the stride is never used


def attn_chunk_fwd(q, k, v, out=None, lse=None, scale=None, out_dtype=torch.float32, stream=None):
    """Attention of q against one KV chunk (a view such as k[:, :, s:s+n] or a packed buffer).

    Returns (partial out [B, H, N_q, D] of out_dtype, lse fp32 [B, H, N_q]).
    """
    _check_qkv(q, k, v)
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v chunk must be [B, H, n_kv, D] matching q")
    hs = kv_head_stride(k)
    if kv_head_stride(v) != hs:
        raise ValueError("k and v chunks must have the same head stride")
    n_kv = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check_out(out, lse, (B, H, Nq, D), q.device)
    if out is None:
        out = torch.empty((B, H, Nq, D), device=q.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        st = lib().dit_attn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq,
                                      n_kv, D, hs, scale, _dt(out.dtype),
                                      _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_chunk_fwd")
    return out, lse


def _chunk_plan(q, k, v, chunks, partials, lses, partial_dtype):
    """Shared argument handling of the all-chunks-in-one-launch calls: (hs, starts, partials,
    lses) with the host chunk-start table and the partial buffers (allocated unless given)."""
    _check_qkv(q, k, v)
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v must be [B, H, n_kv, D] matching q")
    if any(int(n) < 1 for n in chunks) or sum(int(n) for n in chunks) > k.shape[2]:
        raise ValueError("chunk lengths must be positive and fit in the keys")
    hs = kv_head_stride(k)
    if kv_head_stride(v) != hs:
        raise ValueError("k and v must have the same head stride")
    p = len(chunks)
    starts = (ctypes.c_int * (p + 1))()
    acc = 0
    for c, n in enumerate(chunks):
        starts[c] = acc
        acc += int(n)
    starts[p] = acc
    _check_out(partials, lses, (p, B, H, Nq, D), q.device, "partials", "lses")
    if partials is None:
        partials = torch.empty((p, B, H, Nq, D), device=q.device, dtype=partial_dtype)
    if lses is None:
        lses = torch.empty((p, B, H, Nq), device=q.device, dtype=torch.float32)
    return hs, starts, partials, lses


def attn_chunks_fwd(q, k, v, chunks, partials=None, lses=None, scale=None,
                    partial_dtype=torch.float32, stream=None):
    """Every chunk's partial (O_c, lse_c) of the ring decomposition in one launch
    (dit_attn_chunks_fwd): chunk c is keys [s_c, s_c + chunks[c]) of k / v, s_c the sum of the
    earlier lengths.  Returns (partials [p, B, H, N_q, D] of partial_dtype, lses [p, B, H, N_q])."""
    hs, starts, partials, lses = _chunk_plan(q, k, v, chunks, partials, lses, partial_dtype)
    B, H, Nq, D = q.shape
    p = len(chunks)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib().dit_attn_chunks_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(partials), _ptr(lses), B, H,
                                       Nq, k.shape[2], D, hs, p, starts, scale, _dt(partials.dtype),
                                       _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_chunks_fwd")
    return partials, lses


def attn_chunk_fwd_accumulate(q, k, v, o_run, lse_run, scale=None, stream=None):
    """One ring hop with the merge fused in: the attention of q against one KV chunk (a view such
    as k[:, :, s:s+n] or a packed buffer) merged in place into the running o_run (fp32
    [B, H, N_q, D]) and lse_run (fp32 [B, H, N_q]).  Rows with lse_run = -inf are empty: their
    o_run is not read.  Returns (o_run, lse_run)."""
    _check_qkv(q, k, v)
    B, H, Nq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != D:
        raise ValueError("k/v chunk must be [B, H, n_kv, D] matching q")
    hs = kv_head_stride(k)
    if kv_head_stride(v) != hs:
        raise ValueError("k and v chunks must have the same head stride")
    if (o_run.dtype != torch.float32 or tuple(o_run.shape) != (B, H, Nq, D)
            or not o_run.is_contiguous() or o_run.device != q.device):
        raise ValueError("o_run must be a contiguous fp32 [B, H, N_q, D] tensor on q's device")
    if (lse_run.dtype != torch.float32 or tuple(lse_run.shape) != (B, H, Nq)
            or not lse_run.is_contiguous() or lse_run.device != q.device):
        raise ValueError("lse_run must be a contiguous fp32 [B, H, N_q] tensor on q's device")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib().dit_attn_chunk_fwd_accumulate(_ptr(q), _ptr(k), _ptr(v), _ptr(o_run),
                                                 _ptr(lse_run), B, H, Nq, k.shape[2], D, hs, scale,
                                                 _stream(q.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_chunk_fwd_accumulate")
    return o_run, lse_run


def attn_lse_merge(partials, lses, out=None, lse=None, out_dtype=torch.float32, stream=None):
    """Merge p partials [p, B, H, N, D] (fp32 or bf16) with lses fp32 [p, B, H, N]."""
    if not partials.is_cuda or partials.dim() != 5 or not partials.is_contiguous():
        raise ValueError("partials must be a contiguous CUDA tensor [p, B, H, N, D]")
    if lses.dtype != torch.float32 or tuple(lses.shape) != tuple(partials.shape[:4]) \
            or not lses.is_contiguous():
        raise ValueError("lses must be contiguous fp32 [p, B, H, N]")
    p, B, H, N, D = partials.shape
    _check_out(out, lse, (B, H, N, D), partials.device)
    if out is None:
        out = torch.empty((B, H, N, D), device=partials.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty((B, H, N), device=partials.device, dtype=torch.float32)
    with torch.cuda.device(partials.device):
        st = lib().dit_attn_lse_merge(_ptr(partials), _ptr(lses), p, _ptr(out), _ptr(lse), B, H, N,
                                      D, _dt(partials.dtype), _dt(out.dtype),
                                      _stream(partials.device, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_lse_merge")
    return out, lse


def check(device=None, stream=None):
    """Synchronise and raise DitError if a kernel reported a timed-out wait."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib().dit_attn_check(_stream(dev, stream))
    if st != DIT_OK:
        raise DitError(st, "dit_attn_check")


def inject_stall(enable: bool, wait_limit_cycles: int = 0):
    """TEST ONLY: make later attention launches time out on their first K/V wait (see header)."""
    lib().dit_test_inject_stall(1 if enable else 0, int(wait_limit_cycles))


def set_grid_limit(max_ctas: int):
    """TEST ONLY: cap the persistent attention grid (0 restores one CTA per SM)."""
    lib().dit_test_set_grid_limit(int(max_ctas))


def chunk_attention(q, k, v, chunks, scale=None, out_dtype=torch.float32,
                    partial_dtype=torch.float32, partials=None, lses=None, stream=None,
                    batched=False):
    """Ring decomposition on one GPU: one dit_attn_chunk_fwd per KV chunk (virtual rank), or
    with batched=True all chunks in one dit_attn_chunks_fwd launch (bitwise the same partials),
    then one dit_attn_lse_merge.  `chunks` lists the chunk lengths (sum = N_kv).  Returns
    (out, lse)."""
    B, H, Nq, D = q.shape
    if sum(chunks) != k.shape[2]:
        raise ValueError("chunk lengths must sum to the number of keys")
    p = len(chunks)
    if partials is None:
        partials = torch.empty((p, B, H, Nq, D), device=q.device, dtype=partial_dtype)
    if lses is None:
        lses = torch.empty((p, B, H, Nq), device=q.device, dtype=torch.float32)
    if batched:
        attn_chunks_fwd(q, k, v, chunks, partials=partials, lses=lses, scale=scale, stream=stream)
    else:
        s = 0
        for c, n in enumerate(chunks):
            attn_chunk_fwd(q, k[:, :, s:s + n], v[:, :, s:s + n], out=partials[c], lse=lses[c],
                           scale=scale, stream=stream)
            s += n
    return attn_lse_merge(partials, lses, out_dtype=out_dtype, stream=stream)


def ring_attention(q, k, v, chunks, scale=None, o_run=None, lse_run=None, stream=None):
    """Ring decomposition on one GPU with the merge fused into each hop: the running (o_run,
    lse_run) starts empty (lse_run = -inf) and every KV chunk (virtual rank) is folded in by one
    dit_attn_chunk_fwd_accumulate.  `chunks` lists the chunk lengths (sum = N_kv).  Returns
    (o_run fp32, lse_run)."""
    B, H, Nq, D = q.shape
    if sum(chunks) != k.shape[2] or any(n < 1 for n in chunks):
        raise ValueError("chunk lengths must be positive and sum to the number of keys")
    if o_run is None:
        o_run = torch.empty((B, H, Nq, D), device=q.device, dtype=torch.float32)
    if lse_run is None:
        lse_run = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    lse_run.fill_(float("-inf"))
    s = 0
    for n in chunks:
        attn_chunk_fwd_accumulate(q, k[:, :, s:s + n], v[:, :, s:s + n], o_run, lse_run,
                                  scale=scale, stream=stream)
        s += n
    return o_run, lse_run


def head_groups(n_heads, groups=5):
    """Split n_heads heads into consecutive groups for host pipelining: small first and last
    groups (so that the first compute starts, and the last copy-back ends, early) around a
    large middle one.  groups=5 (the default) gives about 1/12, 1/6, 1/2, 1/6, 1/12 of the
    heads (2, 4, 12, 4, 2 for 24 heads: the fastest end-to-end split measured for the Wan2.2
    shape among eight tried); groups=3 gives about 1/6, 2/3, 1/6.  Returns [(h0, h1), ...]."""
    if groups >= 5 and n_heads >= 5:
        e1, e2 = max(1, n_heads // 12), max(1, n_heads // 6)
        sizes = [e1, e2, n_heads - 2 * (e1 + e2), e2, e1]
    elif groups >= 3 and n_heads >= 3:
        edge = max(1, n_heads // 6)
        sizes = [edge, n_heads - 2 * edge, edge]
    elif groups >= 2 and n_heads >= 2:
        sizes = [n_heads // 2, n_heads - n_heads // 2]
    else:
        sizes = [n_heads]
    out, h = [], 0
    for n in sizes:
        out.append((h, h + n))
        h += n
    return out


_PIPE_STREAMS = {}


def _pipeline_streams(dev: torch.device):
    """Upload and download streams of host_pipeline, created once per device."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _PIPE_STREAMS:
        _PIPE_STREAMS[key] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    return _PIPE_STREAMS[key]


def host_pipeline(fn, inputs, outputs, groups, device=None):
    """Runs fn over head groups with host<->device copies overlapped with compute.

    inputs / outputs: host tensors (pinned for the copies to overlap) whose first dimension is
    the flattened (batch, head) index; groups: [(h0, h1), ...] ranges of it.  For each group,
    its input slices are copied to the device on one stream, fn(*device_input_slices) runs on
    the current stream and returns device tensors shaped like the output slices, and those are
    copied back on a third stream: group g+1's upload and group g-1's download overlap group g's
    compute.  Returns outputs once every copy has landed.  (Alternating the groups over two
    compute streams, so that one group's kernels fill the previous group's last wave, measured
    slower.)"""
    dev = torch.device("cuda") if device is None else torch.device(device)
    comp = torch.cuda.current_stream(dev)
    up, down = _pipeline_streams(dev)
    d_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in inputs]
    up.wait_stream(comp)  # the device buffers were allocated on the compute stream
    keep = []
    for h0, h1 in groups:
        with torch.cuda.stream(up):
            for dt, ht in zip(d_in, inputs):
                dt[h0:h1].copy_(ht[h0:h1], non_blocking=True)
        comp.wait_stream(up)
        res = fn(*(dt[h0:h1] for dt in d_in))
        down.wait_stream(comp)
        with torch.cuda.stream(down):
            for ht, r in zip(outputs, res):
                ht[h0:h1].copy_(r, non_blocking=True)
        keep.append(res)  # device results stay alive until their copies are done
    down.synchronize()
    return outputs


def attention(q, k, v, scale=None, chunks=None, out_dtype=torch.float32,
              partial_dtype=torch.float32, device=None, accumulate=False, with_lse=True):
    """User-level call.  Accepts CUDA tensors, or CPU tensors (pinned for the copies to overlap)
    that are processed in head groups through host_pipeline, results returned in pinned host
    memory.  chunks=None runs the fused pass; a list of chunk lengths runs the p-chunk ring
    decomposition, merged by a separate LSE-merge pass or, with accumulate=True, hop by hop
    inside each chunk pass (fp32 output).  with_lse=False (fused pass on device tensors only)
    skips the LSE and returns (out, None)."""
    if not with_lse and (chunks is not None or not q.is_cuda):
        raise ValueError("with_lse=False applies to the fused pass on device tensors")
    if not q.is_cuda:
        # Host tensors: pipelined over head groups (uploads, compute and downloads overlap).
        B, H, Nq, D = q.shape
        o_dtype = torch.float32 if (accumulate and chunks is not None) else out_dtype
        out_h = torch.empty((B * H, Nq, D), dtype=o_dtype, pin_memory=True)
        lse_h = torch.empty((B * H, Nq), dtype=torch.float32, pin_memory=True)

        def per_group(qg, kg, vg):
            o, l = attention(qg.unsqueeze(0), kg.unsqueeze(0), vg.unsqueeze(0), scale=scale,
                             chunks=chunks, out_dtype=out_dtype, partial_dtype=partial_dtype,
                             accumulate=accumulate)
            return o[0], l[0]

        flat = [t.reshape(B * H, *t.shape[2:]) for t in (q, k, v)]
        host_pipeline(per_group, flat, [out_h, lse_h], head_groups(B * H), device)
        return out_h.view(B, H, Nq, D), lse_h.view(B, H, Nq)
    if chunks is None:
        out, lse = attn_fwd(q, k, v, scale=scale, out_dtype=out_dtype, with_lse=with_lse)
    elif accumulate:
        if out_dtype != torch.float32:
            raise ValueError("the hop-by-hop ring accumulates in fp32")
        out, lse = ring_attention(q, k, v, chunks, scale=scale)
    else:
        out, lse = chunk_attention(q, k, v, chunks, scale=scale, out_dtype=out_dtype,
                                   partial_dtype=partial_dtype)
    return out, lse
