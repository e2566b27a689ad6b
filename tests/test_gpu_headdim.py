"""Head dims other than 64 and 128 against the fp64 oracle.

A head dim d (a multiple of 8) runs in the 64- or 128-column kernels (d <=
128) or the one-query-tile 256-column kernel (136..256), with the columns
past d read as zeros by the tensor maps: they add nothing to Q K^T, give
zero output columns that are never stored, and the rows in memory stay d
elements long.  Forward (unsplit and split-KV) at the forward's bars,
backward at the derived gradient bar (from 136 the three-pass 256-column
backward), with poisoned guard bands around the outputs.  Small problems at d > 128 split the key range on their
own (fewer query tiles than SMs), so the plain large-d cases below run the
split path too.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300.inputs import Workload, make_inputs
from tests.gpu_helpers import compare, run_gpu
from tests.test_gpu_backward import check as check_grads

pytestmark = pytest.mark.gpu

DIMS = [8, 16, 32, 48, 72, 80, 96, 112, 120]


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [129, 300])
def test_forward_head_dims(cuda_device, d, causal, N):
    x = make_inputs(Workload("hd", 2, 2, N, d, causal, 500 + d + N))
    o_g, l_g = run_gpu(x, cuda_device)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, causal)
    compare(o_g, l_g, o_r, l_r, f"d={d} N={N} causal={causal}")


@pytest.mark.parametrize("d", [32, 96])
def test_forward_head_dims_key_padding_and_split(cuda_device, d):
    x = make_inputs(Workload("hd_kl", 4, 2, 700, d, True, 600 + d, qk_sigma=2.0))
    kl = [0, 1, 129, 700]
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, True, key_len=kl)
    for n_splits in (1, 3):
        o_g, l_g = run_gpu(x, cuda_device, key_len=kl, n_splits=n_splits)
        compare(o_g, l_g, o_r, l_r, f"d={d} key_len splits={n_splits}")


def guarded_backward(x, g, dev, causal, scale):
    """The backward with dQ, dK, dV inside poisoned guard bands of their own."""
    import torch

    from exact_softmax_attention_fattn_gb300 import binding
    from tests.gpu_helpers import GUARD, POISON_BF16, bits_to_device

    q, k, v, go = (bits_to_device(a, dev) for a in (x.q, x.k, x.v, g))
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    binding.forward_into(q, k, v, o, lse, causal=causal, scale=scale)
    n = q.numel()
    bufs = [torch.full((n + 2 * GUARD,), POISON_BF16, dtype=torch.int16, device=dev) for _ in range(3)]
    grads = [b[GUARD:GUARD + n].view(torch.bfloat16).view(B, H, N, d) for b in bufs]
    binding.backward_into(q, k, v, o, lse, go, *grads, causal=causal, scale=scale)
    torch.cuda.synchronize(dev)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    for name, b in zip(("dq", "dk", "dv"), bufs):
        assert bool(torch.all(b[:GUARD] == POISON_BF16)) and bool(torch.all(b[-GUARD:] == POISON_BF16)), (
            f"a store landed outside {name}")
    return tuple(t.float().cpu().numpy().astype(np.float64) for t in grads)


@pytest.mark.parametrize("d", [16, 32, 96, 120, 136, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_head_dims(cuda_device, d, causal):
    x = make_inputs(Workload("hd_bwd", 2, 2, 300, d, causal, 700 + d))
    g = make_inputs(Workload("hd_bwd_g", 2, 2, 300, d, causal, 1700 + d)).v
    scale = 1.0 / np.sqrt(d)
    ours = guarded_backward(x, g, cuda_device, causal, scale)
    ref = oracle.backward(x.q, x.k, x.v, g, scale, causal)
    check_grads(ours, ref, f"backward d={d} causal={causal}")


LARGE = [136, 192, 256]


@pytest.mark.parametrize("d", LARGE)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 129, 300])
def test_forward_large_head_dims(cuda_device, d, causal, N):
    """The 64-key tiles of the 256-column kernel: N around one and two key tiles."""
    x = make_inputs(Workload("hd_large", 2, 2, N, d, causal, 800 + d + N))
    o_g, l_g = run_gpu(x, cuda_device)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, causal)
    compare(o_g, l_g, o_r, l_r, f"d={d} N={N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_forward_d256_key_padding_peaky(cuda_device, causal):
    """Key lengths {0, 1, 65, 700} (a fully masked batch entry) with Q, K ~
    N(0, 2^2): the rescale of the 256-column O runs."""
    x = make_inputs(Workload("hd256_kl", 4, 2, 700, 256, causal, 901, qk_sigma=2.0))
    kl = [0, 1, 65, 700]
    o_g, l_g = run_gpu(x, cuda_device, key_len=kl)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, causal, key_len=kl)
    compare(o_g, l_g, o_r, l_r, f"d=256 key_len causal={causal}")


def test_forward_d256_long(cuda_device):
    """B1 H4 N4096 d256 causal: many CTAs and key tiles, sampled heads in full."""
    x = make_inputs(Workload("hd256_long", 1, 4, 4096, 256, True, 902))
    o_g, l_g = run_gpu(x, cuda_device)
    rows = np.concatenate([h * 4096 + np.arange(4096) for h in (0, 3)]).astype(np.int64)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, True, rows=rows)
    compare(o_g.reshape(-1, 256)[rows], l_g.reshape(-1)[rows], o_r, l_r, "d=256 N=4096 causal")


@pytest.mark.parametrize("d", [136, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_large_head_dims_split(cuda_device, d, causal):
    """Explicit split counts at d > 128 (runs of 64-key tiles, fp32 partials,
    the combine), with key padding that leaves some runs empty and some rows
    with no visible key in a run: kl = 0 (nothing visible), 1, 65, 700."""
    x = make_inputs(Workload("hd_large_split", 4, 2, 700, d, causal, 950 + d, qk_sigma=2.0))
    kl = [0, 1, 65, 700]
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, causal, key_len=kl)
    for n_splits in (1, 2, 3, 11):
        o_g, l_g = run_gpu(x, cuda_device, key_len=kl, n_splits=n_splits)
        compare(o_g, l_g, o_r, l_r, f"d={d} causal={causal} key_len splits={n_splits}")


@pytest.mark.parametrize("d", [200, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_large_head_dims_key_padding(cuda_device, d, causal):
    """The 256-column backward with key lengths {0, 1, 129, 300}: a batch
    entry with no visible key (dQ = dK = dV = 0 there), keys past key_len
    (dK = dV = 0), N = 300 ragged over three 128-row tiles, Q, K ~ N(0, 2^2)."""
    import torch

    from exact_softmax_attention_fattn_gb300 import binding
    from tests.gpu_helpers import bits_to_device

    B, H, N = 4, 1, 300
    x = make_inputs(Workload("hd_bwd_kl", B, H, N, d, causal, 960 + d, qk_sigma=2.0))
    g = make_inputs(Workload("hd_bwd_kl_g", B, H, N, d, causal, 1960 + d)).v
    kl = np.array([0, 1, 129, 300], np.int32)
    scale = 1.0 / np.sqrt(d)
    dev = cuda_device
    q, k, v, go = (bits_to_device(a, dev) for a in (x.q, x.k, x.v, g))
    kl_t = torch.from_numpy(kl).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    binding.forward_into(q, k, v, o, lse, causal=causal, scale=scale, key_len=kl_t)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    binding.backward_into(q, k, v, o, lse, go, dq, dk, dv, causal=causal, scale=scale, key_len=kl_t)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    ours = tuple(t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv))
    ref = oracle.backward(x.q, x.k, x.v, g, scale, causal, key_len=kl)
    check_grads(ours, ref, f"backward d={d} causal={causal} key_len")
