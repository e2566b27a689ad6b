"""The forward on HOST buffers (fattn_fwd_host through binding.forward with
CPU tensors) against the fp64 oracle: one chunk for small problems; batch
chunks (B >= 4) and head chunks (B < 4) with copies overlapped with the
kernels for large ones; pinned and pageable inputs give the same bits."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300 import binding
from exact_softmax_attention_fattn_gb300.inputs import Workload, make_inputs
from tests.gpu_helpers import compare

pytestmark = pytest.mark.gpu


def host_tensors(x, pinned):
    import torch

    ts = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) for a in (x.q, x.k, x.v)]
    return [t.pin_memory() if pinned else t for t in ts]


def sampled_rows(B, H, N, heads, n_rand, seed):
    rows = [h * N + np.arange(N) for h in heads]
    rows.append(np.random.default_rng(seed).integers(0, B * H * N, size=n_rand))
    return np.unique(np.concatenate(rows)).astype(np.int64)


@pytest.mark.parametrize("shape,causal,keylen,sample", [
    ((1, 1, 128, 64), False, None, None),             # one chunk
    ((2, 3, 700, 96), True, [0, 333], None),          # one chunk, key padding incl. an empty batch entry
    ((8, 4, 2048, 128), False, "range", (2, 3000)),   # 8 batch chunks of 1 entry
    ((1, 8, 8192, 128), True, None, (2, 2000)),       # 8 head chunks of 1 head
    ((2, 4, 4096, 256), True, None, (2, 2000)),       # head chunks, the 256-column kernel
])
def test_host_forward_matches_oracle(cuda_device, shape, causal, keylen, sample):
    B, H, N, d = shape
    x = make_inputs(Workload("host", B, H, N, d, causal, 950 + N + d))
    kl = None
    if keylen == "range":
        kl = list(np.random.default_rng(5).integers(N // 2, N + 1, size=B))
    elif keylen is not None:
        kl = keylen
    qh, kh, vh = host_tensors(x, pinned=True)
    o, lse = binding.forward(qh, kh, vh, causal=causal, key_len=kl)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    o_g = o.float().numpy().astype(np.float64)
    l_g = lse.numpy().astype(np.float64)
    scale = 1.0 / np.sqrt(d)
    if sample is None:
        o_r, l_r = oracle.forward(x.q, x.k, x.v, scale, causal, key_len=kl)
        compare(o_g, l_g, o_r, l_r, f"host {shape}")
    else:
        rows = sampled_rows(B, H, N, [0, B * H - 1], sample[1], seed=N)
        o_r, l_r = oracle.forward(x.q, x.k, x.v, scale, causal, key_len=kl, rows=rows)
        compare(o_g.reshape(-1, d)[rows], l_g.reshape(-1)[rows], o_r, l_r, f"host {shape}")
        # every chunk wrote its rows: nothing left unwritten
        assert np.all(np.isfinite(o_g))


def test_pageable_and_pinned_inputs_agree(cuda_device):
    x = make_inputs(Workload("host_pg", 1, 8, 4096, 128, True, 960))
    a = binding.forward(*host_tensors(x, pinned=True), causal=True)
    b = binding.forward(*host_tensors(x, pinned=False), causal=True)
    np.testing.assert_array_equal(a[0].view(dtype=a[0].dtype).float().numpy(), b[0].float().numpy())
    np.testing.assert_array_equal(a[1].numpy(), b[1].numpy())


def test_host_entry_point_rejects_device_buffers(cuda_device):
    import torch

    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=cuda_device)
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device=cuda_device)
    st = binding.fwd_host_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(), 1, 1, 128, 64,
                              0.125, False, None, None)
    assert st == binding.FATTN_ERR_INVALID_ARG
