"""fattn_fwd_noalloc: the forward for callers that may not allocate device
memory -- code inside a framework that owns every device allocation through
its own arena, or a latency-critical path that must not take the driver's
allocation locks.  Its scratch (V in the P V operand type and the per-tile
storage modes) is a static device array inside the library instead of a
per-call pool allocation.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It passes alone in a fresh
process and after the other tests alike.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300 import binding
from exact_softmax_attention_fattn_gb300.inputs import Workload, make_inputs
from tests.gpu_helpers import bits_to_device, compare

pytestmark = pytest.mark.gpu


def _noalloc():
    lib = binding.load_library()
    fn = lib.fattn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int,
                                                                ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _check(w, dev, key_len=None):
    """Two no-alloc calls in a row through the same static scratch: each
    bit-identical to the forward without split-KV (fattn_fwd_splitkv with one
    split: the same kernels; the no-alloc entry point never splits), and each
    within the tolerances of the fp64 oracle on every element."""
    import torch

    x = make_inputs(w)
    q, k, v = (bits_to_device(a, dev) for a in (x.q, x.k, x.v))
    kl = None if key_len is None else torch.from_numpy(np.asarray(key_len, np.int32)).to(dev)
    B, H, N, d = x.q.shape
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    binding.forward_into(q, k, v, o_ref, lse_ref, causal=w.causal, scale=w.softmax_scale, key_len=kl, n_splits=1)
    fn = _noalloc()
    stream = torch.cuda.current_stream(dev).cuda_stream
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                w.softmax_scale, int(w.causal), None if kl is None else kl.data_ptr(), stream)
        assert st == binding.FATTN_OK, binding.status_string(st)
        outs.append((o, lse))
    st, detail = binding.last_error(torch.cuda.current_stream(dev))
    assert st == binding.FATTN_OK, f"kernel reported {binding.status_string(st)} {detail}"
    torch.cuda.synchronize(dev)
    o_or, l_or = oracle.forward(x.q, x.k, x.v, w.softmax_scale, w.causal,
                                key_len=None if key_len is None else np.asarray(key_len, np.int32))
    for o, lse in outs:
        np.testing.assert_array_equal(o.view(torch.int16).cpu().numpy(), o_ref.view(torch.int16).cpu().numpy())
        np.testing.assert_array_equal(lse.cpu().numpy(), lse_ref.cpu().numpy())
        compare(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), o_or, l_or,
                what=f"no-alloc {w.name}")


def test_noalloc_matches_fattn_fwd_and_the_oracle(cuda_device):
    _check(Workload("na128", 2, 4, 1000, 128, True, 40), cuda_device)
    # a different problem next, through the same scratch: key padding, peaky logits
    _check(Workload("na64", 3, 2, 700, 64, False, 41, qk_sigma=2.0), cuda_device, key_len=[700, 5, 333])
    # the 256-column kernel (its own pre-pass thread count and V tensor-map box), key padding
    _check(Workload("na256", 1, 2, 700, 256, False, 42), cuda_device, key_len=[650])


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    import torch

    fn = _noalloc()
    buf = torch.zeros(1024, dtype=torch.uint8, device=cuda_device)
    ptr = buf.data_ptr()
    # B*H = 64 at N = 4096, d = 128: the V copy alone fills the 64 MiB, the tile modes do not fit
    st = fn(ptr, ptr, ptr, ptr, ptr, 64, 1, 4096, 128, 0.088, 1, None, torch.cuda.current_stream().cuda_stream)
    assert st == binding.FATTN_ERR_UNSUPPORTED
