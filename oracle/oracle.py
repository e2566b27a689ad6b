"""Plain fp64 CPU oracle for the exact softmax attention forward and backward,
and for causal linear attention (the second workload).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference leg import this module.  The product path
(the CUDA library and its Python binding) never does, and shares no code with
it.

The arithmetic lives in attn_oracle.c (plain loops, fp64, pthreads over rows);
this file compiles it with gcc on first use and marshals numpy arrays.  Each
function states the passage it follows in its docstring.

Parity status: every function here is pinned by tests/test_oracle.py against
closed forms, brute force, invariants the pages state, and an independent
library restatement (numpy/torch fp64 softmax); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, pthreads)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.fattn_oracle_forward.restype = ctypes.c_int
    lib.fattn_oracle_forward.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fattn_oracle_backward.restype = ctypes.c_int
    lib.fattn_oracle_backward.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fattn_oracle_linear.restype = ctypes.c_int
    lib.fattn_oracle_linear.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.fattn_oracle_probs.restype = ctypes.c_int
    lib.fattn_oracle_probs.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
    ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def forward(q, k, v, scale: float, causal: bool, key_len=None, rows=None, threads: int | None = None,
            _lib_override=None):
    """Exact attention forward in fp64, the plain definition.

    q, k, v: uint16 bf16 bit patterns, shape [B, H, N, d].
    key_len: int32 [B] or None.  rows: optional flat row ids (b*H+h)*N+i.
    Returns (o, lse): o float64 [B,H,N,d] (or [len(rows), d]), lse float64.

    Follows "understand-flashattention", forward-pass formulas (S = Q K^T,
    P = softmax(S), O = P V) and the logsumexp derivation (L = m + log l);
    scale then mask as in "PyTorch profiling part 3: attention", section
    "Naive attention"; an all-masked row gives 0 / -inf as in its section
    "The safe softmax".
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, N, d]")
    B, H, N, d = q.shape
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(key_len, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_len must have shape [B]")
    r = None
    if rows is not None:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = r.size
        o = np.empty((n_rows, d), dtype=np.float64)
        lse = np.empty((n_rows,), dtype=np.float64)
    else:
        n_rows = B * H * N
        o = np.empty((B, H, N, d), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64)
    rc = (_lib_override or _load()).fattn_oracle_forward(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, N, d, float(scale), int(bool(causal)),
        kl.ctypes.data if kl is not None else None, r.ctypes.data if r is not None else None,
        n_rows, o.ctypes.data, lse.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle forward failed with code {rc}")
    return o, lse


def backward(q, k, v, dout, scale: float, causal: bool, key_len=None, heads=None, threads: int | None = None,
             _lib_override=None):
    """Exact attention backward in fp64: (dQ, dK, dV) for the loss gradient dout = dL/dO.

    q, k, v, dout: uint16 bf16 bit patterns, shape [B, H, N, d].  key_len:
    int32 [B] or None.  heads: optional flat head ids b*H+h; the result then
    has shape [len(heads), N, d] per tensor, else [B, H, N, d].

    Follows "understand-flashattention", section "Attention forward and
    backward formulas", backward pass steps 1-5 (dV = P^T dO, dP = dO V^T,
    dS_ij = P_ij (dP_ij - sum_k dP_ik P_ik), dQ = dS K, dK = dS^T Q), with the
    softmax scale of S = scale * Q K^T carried into dQ and dK by the chain rule,
    and P the forward's masked softmax (forward()).
    """
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q, k, v, dout must share the shape [B, H, N, d]")
    B, H, N, d = q.shape
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(key_len, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_len must have shape [B]")
    hs = None
    if heads is not None:
        hs = np.ascontiguousarray(heads, dtype=np.int64)
        n_heads = hs.size
        shape = (n_heads, N, d)
    else:
        n_heads = B * H
        shape = (B, H, N, d)
    dq = np.empty(shape, dtype=np.float64)
    dk = np.empty(shape, dtype=np.float64)
    dv = np.empty(shape, dtype=np.float64)
    rc = (_lib_override or _load()).fattn_oracle_backward(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, H, N, d, float(scale),
        int(bool(causal)), kl.ctypes.data if kl is not None else None, hs.ctypes.data if hs is not None else None,
        n_heads, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle backward failed with code {rc}")
    return dq, dk, dv


def probs(q, k, scale: float, causal: bool, key_len=None, b: int = 0, h: int = 0, _lib_override=None):
    """The full P (softmax of the masked, scaled scores) and S of one head, fp64.

    Same definition as forward(); for small N only (N*N doubles each).
    "understand-flashattention", forward-pass formulas and the numerically
    stable softmax section.
    """
    q, k = _bits(q), _bits(k)
    B, H, N, d = q.shape
    kl = None if key_len is None else np.ascontiguousarray(key_len, dtype=np.int32)
    p = np.empty((N, N), dtype=np.float64)
    s = np.empty((N, N), dtype=np.float64)
    rc = (_lib_override or _load()).fattn_oracle_probs(
        q.ctypes.data, k.ctypes.data, B, H, N, d, float(scale), int(bool(causal)),
        kl.ctypes.data if kl is not None else None, b, h, p.ctypes.data, s.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle probs failed with code {rc}")
    return p, s


def linear(q, k, v, key_len=None, eps: float = 1e-6, threads: int | None = None, _lib_override=None):
    """Causal linear attention in fp64 (the "Linear Attention CUDA kernel"
    page: phi = elu + 1 on queries and keys, keys past key_len[b] zeroed, the
    running outer-product state of its CPU causal dot product, and the
    normaliser 1 / (phi(q_i) . cumsum(phi(k))_i + eps) of
    CausalLinearAttention.forward).

    q, k: float32 [B, H, N, E]; v: float32 [B, H, N, M]; key_len: int32 [B]
    or None.  Returns float64 [B, H, N, M].
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B, H, N, E] and v [B, H, N, M]")
    B, H, N, E = q.shape
    M = v.shape[3]
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(key_len, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_len must have shape [B]")
    out = np.empty((B, H, N, M), dtype=np.float64)
    rc = (_lib_override or _load()).fattn_oracle_linear(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, N, E, M, kl.ctypes.data if kl is not None else None,
        float(eps), out.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle linear failed with code {rc}")
    return out


class Oracle:
    """forward()/probs() bound to one compiled copy of attn_oracle.c (the test
    suite uses this to run its pins against deliberately broken copies)."""

    def __init__(self, lib_path: str):
        self._lib = _bind(lib_path)

    def forward(self, *a, **kw):
        return forward(*a, _lib_override=self._lib, **kw)

    def linear(self, *a, **kw):
        return linear(*a, _lib_override=self._lib, **kw)

    def probs(self, *a, **kw):
        return probs(*a, _lib_override=self._lib, **kw)

    def backward(self, *a, **kw):
        return backward(*a, _lib_override=self._lib, **kw)


def compile_source(src_path: str, out_path: str) -> str:
    """Compile a copy of the oracle source (same flags as build())."""
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", src_path, "-o", out_path, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out_path
