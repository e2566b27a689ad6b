"""Causal linear attention (fattn_linear_fwd) vs the fp64 oracle on seeded
fp32 inputs, element by element.

The pages state no tolerance for this method.  The kernels sum in fp32: a
chunk's 64 rows, the prefix over at most ceil(N/64) chunks and E-term dot
products, about (64 + N/64 + E) roundings of relative size 2^-24 in the
numerator and the denominator (all of whose terms are positive weights), so
the output, a weighted average of value rows, is off by at most about
2 * 200 * 2^-24 ~ 2.4e-5 of the largest |v| at N = 4096, E = 64.  The bar,
max |diff| <= 2e-4 * max|v| and mean |diff| <= 1e-5 * max|v|, leaves a
margin of ~8x on the bound (errors measured are far below it).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300 import binding
from exact_softmax_attention_fattn_gb300.inputs import LINEAR_WORKLOADS, LinearWorkload, make_linear_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096


def run_gpu(x, dev, key_len=None, eps=1e-6, shift=0):
    """shift: extra floats before `out` (4 puts it on a 16- but not a 32-byte
    boundary)."""
    import torch

    q, k, v = (torch.from_numpy(a).to(dev) for a in (x.q, x.k, x.v))
    B, H, N, E = q.shape
    M = v.shape[3]
    buf = torch.full((B * H * N * M + 2 * GUARD + shift,), float("nan"), dtype=torch.float32, device=dev)
    out = buf[GUARD + shift:GUARD + shift + B * H * N * M].view(B, H, N, M)
    binding.linear_forward(q, k, v, key_len=key_len, eps=eps, out=out)
    torch.cuda.synchronize(dev)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    assert bool(torch.isnan(buf[:GUARD + shift]).all()) and bool(torch.isnan(buf[-GUARD:]).all()), "store outside out"
    return out.cpu().numpy().astype(np.float64)


def check(ours, ref, v, what):
    scale = float(np.max(np.abs(v)))
    d = np.abs(ours - ref)
    assert np.all(np.isfinite(ours)), f"{what}: non-finite output"
    assert d.max() <= 2e-4 * scale and d.mean() <= 1e-5 * scale, (
        f"{what}: max|d| {d.max():.3e} mean|d| {d.mean():.3e} (scale {scale:.3f})")


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 130, 300])
@pytest.mark.parametrize("E,M", [(4, 4), (32, 32), (48, 64), (64, 64), (128, 32), (64, 128)])
def test_linear_shapes(cuda_device, N, E, M):
    x = make_linear_inputs(LinearWorkload("lin", 2, 2, N, E, M, 300 + N + E + M))
    check(run_gpu(x, cuda_device), oracle.linear(x.q, x.k, x.v), x.v, f"N={N} E={E} M={M}")


@pytest.mark.parametrize("E,M", [(32, 32), (64, 64)])
def test_linear_key_lengths(cuda_device, E, M):
    """key_len {0, 1, 64, 65, 200, 300, -5, 1000}: an empty entry (output 0),
    chunk edges, out-of-range lengths clamped."""
    kl = [0, 1, 64, 65, 200, 300, -5, 1000]
    x = make_linear_inputs(LinearWorkload("lin_kl", 8, 2, 300, E, M, 77))
    ours = run_gpu(x, cuda_device, key_len=kl)
    check(ours, oracle.linear(x.q, x.k, x.v, key_len=kl), x.v, f"key_len E={E} M={M}")
    assert np.all(ours[0] == 0.0)


@pytest.mark.parametrize("shift", [4, 8])
@pytest.mark.parametrize("E,M", [(64, 64), (32, 40), (16, 12)])
def test_linear_output_alignment(cuda_device, shift, E, M):
    """Output rows on 16- and 32-byte boundaries, M a multiple of 8 or not:
    the oracle's result, and nothing stored outside `out`."""
    x = make_linear_inputs(LinearWorkload("lin_al", 1, 2, 300, E, M, 79 + shift + E + M))
    check(run_gpu(x, cuda_device, shift=shift), oracle.linear(x.q, x.k, x.v), x.v,
          f"shift={shift} E={E} M={M}")


def test_linear_eps(cuda_device):
    x = make_linear_inputs(LinearWorkload("lin_eps", 1, 2, 200, 64, 64, 78))
    for eps in (0.0, 1e-3, 10.0):
        check(run_gpu(x, cuda_device, eps=eps), oracle.linear(x.q, x.k, x.v, eps=eps), x.v, f"eps={eps}")


@pytest.mark.parametrize("name", sorted(LINEAR_WORKLOADS))
def test_linear_workloads_sampled_heads(cuda_device, name):
    """The measured workloads at full size; the oracle on two heads in full."""
    w = LINEAR_WORKLOADS[name]
    x = make_linear_inputs(w)
    ours = run_gpu(x, cuda_device, key_len=x.key_len)
    for bh in (0, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        kl = None if x.key_len is None else x.key_len[b:b + 1]
        ref = oracle.linear(x.q[sl], x.k[sl], x.v[sl], key_len=kl)
        check(ours[sl], ref, x.v[sl], f"{name} head {bh}")
