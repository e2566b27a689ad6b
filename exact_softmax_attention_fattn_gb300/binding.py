"""Thin ctypes binding over libfattn.so (include/fattn.h).

Argument marshalling only: every step of the attention forward runs in the
CUDA kernel behind `fattn_fwd`, every step of the backward in the kernels
behind `fattn_bwd`.  PyTorch supplies device memory and the
current stream.  If the library is not built, or no GPU is present, calls
raise FattnError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "_lib", "libfattn.so")

FATTN_OK = 0
FATTN_ERR_INVALID_ARG = 1
FATTN_ERR_UNSUPPORTED = 2
FATTN_ERR_CUDA = 3
FATTN_ERR_TIMEOUT = 4

EXPORTED = ("fattn_fwd", "fattn_fwd_splitkv", "fattn_fwd_host", "fattn_fwd_noalloc", "fattn_splitkv_plan",
            "fattn_unit_schedule", "fattn_bwd", "fattn_linear_fwd", "fattn_set_kernel_events",
            "fattn_status_string", "fattn_last_error", "fattn_version", "fattn_tensor_map_stats")

_lock = threading.Lock()
_lib = None


_STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
                 4: "kernel wait timed out"}


class FattnError(RuntimeError):
    """A non-zero status from libfattn (the status code is in .status)."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS_NAMES.get(status, 'unknown status')} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfattn.so once; raise FattnError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise FattnError(FATTN_ERR_CUDA, f"{_LIB_PATH} is not built; run "
                                 "`python -m exact_softmax_attention_fattn_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            lib.fattn_fwd.restype = ctypes.c_int
            lib.fattn_fwd.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p,
            ]
            lib.fattn_fwd_splitkv.restype = ctypes.c_int
            lib.fattn_fwd_splitkv.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
            ]
            lib.fattn_fwd_host.restype = ctypes.c_int
            lib.fattn_fwd_host.argtypes = lib.fattn_fwd.argtypes
            lib.fattn_fwd_noalloc.restype = ctypes.c_int
            lib.fattn_fwd_noalloc.argtypes = lib.fattn_fwd.argtypes
            lib.fattn_linear_fwd.restype = ctypes.c_int
            lib.fattn_linear_fwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + [
                ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]
            lib.fattn_set_kernel_events.restype = ctypes.c_int
            lib.fattn_set_kernel_events.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            lib.fattn_splitkv_plan.restype = ctypes.c_int
            lib.fattn_splitkv_plan.argtypes = [ctypes.c_int] * 6
            lib.fattn_unit_schedule.restype = ctypes.c_longlong
            lib.fattn_unit_schedule.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_longlong]
            lib.fattn_bwd.restype = ctypes.c_int
            lib.fattn_bwd.argtypes = [ctypes.c_void_p] * 9 + [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p,
            ]
            lib.fattn_status_string.restype = ctypes.c_char_p
            lib.fattn_status_string.argtypes = [ctypes.c_int]
            lib.fattn_last_error.restype = ctypes.c_int
            lib.fattn_last_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
            lib.fattn_version.restype = ctypes.c_int
            lib.fattn_version.argtypes = []
            lib.fattn_tensor_map_stats.restype = ctypes.c_int
            lib.fattn_tensor_map_stats.argtypes = [ctypes.POINTER(ctypes.c_longlong)] * 2
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().fattn_status_string(int(status)).decode()


def fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int, N: int, d: int,
            scale: float, causal: bool, key_len_ptr: int | None, stream: int | None, n_splits: int | None = None) -> int:
    """fattn_fwd (n_splits None) or fattn_fwd_splitkv with raw addresses; returns the status code."""
    if n_splits is None:
        return load_library().fattn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N), int(d),
                                        float(scale), int(bool(causal)), key_len_ptr, stream)
    return load_library().fattn_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N), int(d),
                                            float(scale), int(bool(causal)), key_len_ptr, int(n_splits), stream)


def fwd_host_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int, N: int, d: int,
                 scale: float, causal: bool, key_len_ptr: int | None, stream: int | None) -> int:
    """fattn_fwd_host with raw HOST addresses; returns the status code."""
    return load_library().fattn_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N), int(d),
                                         float(scale), int(bool(causal)), key_len_ptr, stream)


def noalloc_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int, N: int, d: int,
                scale: float, causal: bool, key_len_ptr: int | None, stream: int | None) -> int:
    """fattn_fwd_noalloc (the forward on the library's static scratch, never
    split) with raw device addresses; returns the status code."""
    return load_library().fattn_fwd_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N), int(d),
                                            float(scale), int(bool(causal)), key_len_ptr, stream)


def linear_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, B: int, H: int, N: int, E: int, M: int,
               key_len_ptr: int | None, eps: float, stream: int | None) -> int:
    """fattn_linear_fwd with raw addresses; returns the status code."""
    return load_library().fattn_linear_fwd(q_ptr, k_ptr, v_ptr, out_ptr, int(B), int(H), int(N), int(E), int(M),
                                           key_len_ptr, float(eps), stream)


def linear_forward(q, k, v, key_len=None, eps: float = 1e-6, out=None, stream=None):
    """Causal linear attention (fattn_linear_fwd) on fp32 device tensors
    q, k [B, H, N, E] and v [B, H, N, M]: returns (or fills) out [B, H, N, M],
    enqueued on `stream` (default: the current stream)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.float32 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of rank 4")
    B, H, N, E = q.shape
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("k must be shaped like q, v like q up to its last dimension")
    M = v.shape[3]
    if out is None:
        out = torch.empty((B, H, N, M), dtype=torch.float32, device=q.device)
    elif out.shape != (B, H, N, M) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor [B, H, N, M]")
    kl_ptr = None
    if key_len is not None:
        kl = torch.as_tensor(key_len, dtype=torch.int32).to(q.device).contiguous()
        if kl.shape != (B,):
            raise ValueError("key_len must hold B values")
        kl_ptr = kl.data_ptr()
    with torch.cuda.device(q.device):
        handle = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
        st = linear_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, E, M, kl_ptr, eps, handle)
    if st != FATTN_OK:
        raise FattnError(st, "fattn_linear_fwd")
    return out


def set_kernel_events(start=None, stop=None) -> None:
    """fattn_set_kernel_events with two torch.cuda.Event objects (created with
    enable_timing=True and recorded once, so that their CUDA events exist), or
    None, None to clear: the calling thread's next calls record them around
    their dominant kernel."""
    load_library().fattn_set_kernel_events(None if start is None else start.cuda_event,
                                           None if stop is None else stop.cuda_event)


def splitkv_plan(B: int, H: int, N: int, causal: bool, num_sms: int, n_splits: int = 0) -> int:
    """fattn_splitkv_plan: key splits per query block the forward uses; host only."""
    return load_library().fattn_splitkv_plan(int(B), int(H), int(N), int(bool(causal)), int(num_sms),
                                             int(n_splits))


def unit_schedule(B: int, H: int, N: int, num_ctas: int) -> list[int] | None:
    """fattn_unit_schedule: the forward's unit per (round, CTA) for a causal call
    with all keys visible, as a flat list [round * G + cta], or None where the
    library keeps the snake order; host only."""
    lib = load_library()
    n = lib.fattn_unit_schedule(int(B), int(H), int(N), int(num_ctas), None, 0)
    if n <= 0:
        return None
    buf = (ctypes.c_int * n)()
    if lib.fattn_unit_schedule(int(B), int(H), int(N), int(num_ctas), buf, n) != n:
        raise FattnError(FATTN_ERR_INVALID_ARG, "fattn_unit_schedule")
    return list(buf)


def bwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, do_ptr: int, lse_ptr: int, dq_ptr: int, dk_ptr: int,
            dv_ptr: int, B: int, H: int, N: int, d: int, scale: float, causal: bool, key_len_ptr: int | None,
            stream: int | None) -> int:
    """fattn_bwd with raw addresses; returns the status code."""
    return load_library().fattn_bwd(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, int(B),
                                    int(H), int(N), int(d), float(scale), int(bool(causal)), key_len_ptr, stream)


def tensor_map_stats() -> tuple[int, int]:
    """fattn_tensor_map_stats: (reused, freshly encoded) tensor maps since load."""
    hits, misses = ctypes.c_longlong(0), ctypes.c_longlong(0)
    load_library().fattn_tensor_map_stats(ctypes.byref(hits), ctypes.byref(misses))
    return hits.value, misses.value


def last_error(stream=None) -> tuple[int, list[int]]:
    """fattn_last_error on `stream` (a torch.cuda.Stream, a raw handle or None
    for the current stream): (status, [status, role, barrier, unit])."""
    import torch

    if stream is None:
        handle = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, int):
        handle = stream
    else:
        handle = stream.cuda_stream
    detail = (ctypes.c_int * 4)()
    st = load_library().fattn_last_error(handle, detail)
    return st, list(detail)


def _check_qkv(q, k, v):
    import torch

    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be torch.bfloat16")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, N, d]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")


def forward_into(q, k, v, o, lse, causal: bool = False, scale: float | None = None, key_len=None,
                 stream=None, n_splits: int | None = None) -> None:
    """Run the kernel on device tensors, writing `o` (bf16 [B,H,N,d]) and `lse`
    (fp32 [B,H,N]) in place; enqueued on `stream` (default: current stream).
    n_splits: None (fattn_fwd, the library's split-KV choice) or a split count
    for fattn_fwd_splitkv (0 = the library's choice, 1 = no split)."""
    import torch

    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    kl_ptr = None
    if key_len is not None:
        if key_len.dtype != torch.int32 or key_len.shape != (B,) or key_len.device != q.device:
            raise ValueError("key_len must be an int32 tensor [B] on q's device")
        kl_ptr = key_len.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q.device):
        handle = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
        st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, scale,
                     causal, kl_ptr, handle, n_splits)
    if st != FATTN_OK:
        raise FattnError(st, "fattn_fwd" if n_splits is None else "fattn_fwd_splitkv")


def backward_into(q, k, v, o, lse, dout, dq, dk, dv, causal: bool = False, scale: float | None = None,
                  key_len=None, stream=None) -> None:
    """Gradients of the forward on device tensors: writes dq, dk, dv (bf16, shaped
    like q) from dout = dL/dO and the forward's o and lse; enqueued on `stream`."""
    import torch

    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    for name, t in (("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    kl_ptr = None
    if key_len is not None:
        if key_len.dtype != torch.int32 or key_len.shape != (B,) or key_len.device != q.device:
            raise ValueError("key_len must be an int32 tensor [B] on q's device")
        kl_ptr = key_len.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q.device):
        handle = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
        st = bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, causal, kl_ptr, handle)
    if st != FATTN_OK:
        raise FattnError(st, "fattn_bwd")


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, key_len=None):
    """dQ, dK, dV of bf16 [B, H, N, d] device tensors (enqueued on the current stream)."""
    import torch

    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    backward_into(q, k, v, o, lse, dout, dq, dk, dv, causal=causal, scale=scale, key_len=key_len)
    return dq, dk, dv


def forward(q, k, v, causal: bool = False, scale: float | None = None, key_len=None, n_splits: int | None = None):
    """O, LSE = attention forward of bf16 [B, H, N, d] tensors.

    Device tensors: the kernel is enqueued on the current stream and the call
    returns without synchronising.  Host tensors (pinned for speed): one
    fattn_fwd_host call on the current CUDA device (host <-> device copies
    overlapped with the kernels, chunk by chunk) into pinned host O and LSE;
    the call synchronises before returning them (n_splits must be None).
    `key_len` may be a tensor, a sequence of ints or None.
    """
    import torch

    if q.device.type == "cpu":
        if not torch.cuda.is_available():
            raise FattnError(FATTN_ERR_CUDA, "no CUDA device")
        if n_splits is not None:
            raise ValueError("n_splits applies to device tensors only")
        _check_qkv(q, k, v)
        B, H, N, d = q.shape
        kl_h = None if key_len is None else torch.as_tensor(key_len, dtype=torch.int32).cpu().contiguous()
        if kl_h is not None and kl_h.shape != (B,):
            raise ValueError("key_len must hold B values")
        o_h = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        l_h = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
        dev = torch.device("cuda", torch.cuda.current_device())
        stream = torch.cuda.current_stream(dev)
        st = fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_h.data_ptr(), l_h.data_ptr(), B, H, N, d,
                          1.0 / math.sqrt(d) if scale is None else scale, causal,
                          None if kl_h is None else kl_h.data_ptr(), stream.cuda_stream)
        if st != FATTN_OK:
            raise FattnError(st, "fattn_fwd_host")
        stream.synchronize()
        return o_h, l_h
    dev, qd, kd, vd = q.device, q, k, v
    _check_qkv(qd, kd, vd)
    kl = None
    if key_len is not None:
        kl = torch.as_tensor(key_len, dtype=torch.int32).to(dev, non_blocking=True).contiguous()
    B, H, N, _ = qd.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    forward_into(qd, kd, vd, o, lse, causal=causal, scale=scale, key_len=kl, n_splits=n_splits)
    return o, lse
