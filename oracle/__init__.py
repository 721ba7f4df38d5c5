"""fp64 CPU oracle for DiT attention, KV-chunk attention and the LSE merge.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py``
may import this package.  The product path never calls it, and it shares no
code with the CUDA path: the arithmetic lives in ``attn_oracle.c`` (plain
loops, IEEE fp64, compiled with ``-ffp-contract=off`` so x86 and Arm give the
same bits); this module only marshals arrays.

Definitions (see the header of ``attn_oracle.c`` for the sources):
    s_ij = scale * q_i . k_j,  m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i)
    lse_i = m_i + ln l_i,      o_i = sum_j exp(s_ij - m_i) v_j / l_i
    merge: lse = M + ln sum_c exp(lse_c - M),  o = sum_c exp(lse_c - lse) o_c

Parity pins (tests/test_oracle.py): 50-digit decimal brute force straight from
the softmax definition, closed forms (Q = 0, V = 1, N = 1, equal keys, V = I),
invariants (chunk merge = full attention for every p, merge associativity, KV
permutation, key shift, linearity in V, head independence) and a NumPy /
SciPy float64 cross-check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (atomically) and return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB_PATH)
    except subprocess.CalledProcessError as e:  # pragma: no cover - toolchain failure
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed: {e.stderr}") from e
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                         ctypes.c_double, _P, _I64, _P, _P, ctypes.c_int]
        lib.oracle_lse_merge.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P]
        lib.oracle_threads_used.restype = ctypes.c_int
        lib.oracle_threads_used.argtypes = [ctypes.c_int, _I64]
        _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array (accepts torch bf16 or uint16 numpy)."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # local: only needed for torch inputs
    if x.dtype != torch.bfloat16:
        raise TypeError("torch inputs must be bfloat16")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def attention(q, k, v, scale: float, kv_start: int = 0, kv_len: int | None = None,
              rows=None, threads: int = 0):
    """Attention of query rows of q [B,H,Nq,D] over keys [kv_start, kv_start+kv_len) of k,v [B,H,Nk,D].

    Returns (out, lse): fp64 arrays [B,H,R,D] and [B,H,R] where R = len(rows)
    (all Nq rows when rows is None).
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if qb.ndim != 4 or kb.ndim != 4 or kb.shape != vb.shape:
        raise ValueError("expected q [B,H,Nq,D] and k, v [B,H,Nk,D]")
    B, H, Nq, D = qb.shape
    Nk = kb.shape[2]
    if kb.shape[0] != B or kb.shape[1] != H or kb.shape[3] != D:
        raise ValueError("q and k/v disagree on B, H or D")
    if kv_len is None:
        kv_len = Nk - kv_start
    if kv_start < 0 or kv_len < 1 or kv_start + kv_len > Nk:
        raise ValueError("KV range out of bounds")
    if rows is None:
        rows_arr = None
        R = Nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = int(rows_arr.shape[0])
    out = np.empty((B, H, R, D), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    lib = _load()
    koff = kv_start * D * 2  # bytes
    rc = lib.oracle_attention(
        qb.ctypes.data, kb.ctypes.data + koff, vb.ctypes.data + koff,
        B * H, Nq, kv_len, D, Nq * D, Nk * D, float(scale),
        None if rows_arr is None else rows_arr.ctypes.data, R,
        out.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed with {rc}")
    return out, lse


def lse_merge(partials, lses):
    """Merge p partials: partials [p, ..., D], lses [p, ...] -> (out [..., D], lse [...]) in fp64."""
    P = np.ascontiguousarray(np.asarray(partials, dtype=np.float64))
    L = np.ascontiguousarray(np.asarray(lses, dtype=np.float64))
    if P.ndim < 2 or L.shape != P.shape[:-1]:
        raise ValueError("partials must be [p, ..., D] and lses [p, ...]")
    p, D = P.shape[0], P.shape[-1]
    rows = int(np.prod(P.shape[1:-1], dtype=np.int64)) if P.ndim > 2 else 1
    out = np.empty(P.shape[1:], dtype=np.float64)
    lse = np.empty(L.shape[1:], dtype=np.float64)
    rc = _load().oracle_lse_merge(P.ctypes.data, L.ctypes.data, p, rows, D,
                                  out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_lse_merge failed with {rc}")
    return out, lse


def threads_used(threads: int, items: int) -> int:
    """Worker threads oracle attention starts for a `threads` request over `items` rows."""
    return int(_load().oracle_threads_used(int(threads), int(items)))
