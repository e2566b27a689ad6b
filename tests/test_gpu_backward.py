"""CUDA backward vs the fp64 oracle, element by element, on seeded inputs.

The GPU forward supplies O and LSE (as a training step would); the GPU
backward's dQ, dK, dV are compared with the oracle's exact gradients of the
same bf16 inputs.  The pages state no tolerance for gradients; the bar in
check() is derived from the kernels' arithmetic.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300 import binding
from exact_softmax_attention_fattn_gb300.inputs import Workload, make_inputs
from tests.gpu_helpers import bits_to_device

pytestmark = pytest.mark.gpu


def run_gpu_backward(x, g, dev, causal, scale, key_len=None):
    import torch

    q, k, v, go = (bits_to_device(a, dev) for a in (x.q, x.k, x.v, g))
    kl = None if key_len is None else torch.from_numpy(np.asarray(key_len, np.int32)).to(dev)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    binding.forward_into(q, k, v, o, lse, causal=causal, scale=scale, key_len=kl)
    poison = float("nan")
    dq, dk, dv = (torch.full_like(q, poison) for _ in range(3))
    binding.backward_into(q, k, v, o, lse, go, dq, dk, dv, causal=causal, scale=scale, key_len=kl)
    torch.cuda.synchronize(dev)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    return tuple(t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv))


def check(ours, ref, what, max_rel=2.0 ** -6, mean_rel=2.0 ** -7):
    """Per tensor: max |diff| <= 2^-6 * S and mean |diff| <= 2^-7 * S_mean, where S
    is the tensor's own max |ref|, floored at 2^-8 of the largest of the three
    (an exactly-zero gradient, e.g. dQ and dK at N = 1, is judged against the
    size of the others), and S_mean likewise with mean |ref|.

    Derivation: every gradient element carries three roundings of relative
    size <= 2^-9 -- the bf16 output, P or dS rounded to bf16 before its MMA
    (the B operands dO, Q, K are bf16), and D = rowsum(dO * O) formed from the
    forward's bf16 O.  Added coherently that is 3 * 2^-9 ~ 5.9e-3 of the
    tensor's scale, under the 2^-6 bar with a 2.6x margin; their mean is about
    3 * 2^-10, under the 2^-7 bar with a 2.7x margin.  (Measured on GB300:
    max 2.6e-3 to 6.7e-3, mean 2.2e-3 to 3.8e-3 over the cases below.)"""
    report = []
    floor = 2.0 ** -8 * max(np.max(np.abs(r)) for r in ref)
    floor_mean = 2.0 ** -8 * max(np.mean(np.abs(r)) for r in ref)
    for name, a, r in zip(("dq", "dk", "dv"), ours, ref):
        assert np.all(np.isfinite(a)), f"{what}: {name} has non-finite values"
        scale_max = max(np.max(np.abs(r)), floor, 1e-30)
        scale_mean = max(np.mean(np.abs(r)), floor_mean, 1e-30)
        e_max = np.max(np.abs(a - r)) / scale_max
        e_mean = np.mean(np.abs(a - r)) / scale_mean
        report.append(f"{name} max {e_max:.2e} mean {e_mean:.2e}")
        assert e_max <= max_rel and e_mean <= mean_rel, f"{what}: {name} max_rel {e_max:.3g} mean_rel {e_mean:.3g}"
    print(what, " | ".join(report))


def cases(B, H, N, d, causal, seed, sigma=1.0):
    x = make_inputs(Workload("bwd", B, H, N, d, causal, seed, qk_sigma=sigma))
    g = make_inputs(Workload("bwd_g", B, H, N, d, causal, seed + 1000)).v
    return x, g


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 300])
def test_backward_ragged(cuda_device, d, causal, N):
    x, g = cases(2, 2, N, d, causal, 200 + N)
    scale = 1.0 / np.sqrt(d)
    ours = run_gpu_backward(x, g, cuda_device, causal, scale)
    ref = oracle.backward(x.q, x.k, x.v, g, scale, causal)
    check(ours, ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_key_padding(cuda_device, d, causal):
    x, g = cases(4, 2, 300, d, causal, 77, sigma=2.0)
    kl = [0, 1, 129, 300]
    scale = 1.0 / np.sqrt(d)
    ours = run_gpu_backward(x, g, cuda_device, causal, scale, key_len=kl)
    ref = oracle.backward(x.q, x.k, x.v, g, scale, causal, key_len=kl)
    check(ours, ref, f"key_len d={d} causal={causal}")
    # the batch with key_len = 0: every gradient is exactly zero
    for a in ours:
        assert np.all(a[0] == 0)


def test_backward_medium(cuda_device):
    x, g = cases(2, 4, 1024, 128, True, 88)
    scale = 1.0 / np.sqrt(128)
    ours = run_gpu_backward(x, g, cuda_device, True, scale)
    ref = oracle.backward(x.q, x.k, x.v, g, scale, True)
    check(ours, ref, "B2 H4 N1024 d128 causal")


def test_backward_headline_shape_sampled_heads(cuda_device):
    x, g = cases(2, 16, 4096, 128, True, 2)
    scale = 1.0 / np.sqrt(128)
    ours = run_gpu_backward(x, g, cuda_device, True, scale)
    heads = [0, 31]
    ref = oracle.backward(x.q, x.k, x.v, g, scale, True, heads=heads)
    sel = tuple(a.reshape(32, 4096, 128)[heads] for a in ours)
    check(sel, ref, "B2 H16 N4096 d128 causal, heads 0 and 31")
