"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Small and ragged shapes are compared in full; the five measured workloads run
at full size in the same launch configuration the benchmark times and are
compared on sampled rows (every row of some heads, tile-boundary rows and
random rows of the others).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300.inputs import WORKLOADS, Workload, f32_to_bf16_bits, make_inputs
from tests.gpu_helpers import compare, run_gpu

pytestmark = pytest.mark.gpu


def full_check(x, dev, causal=None, scale=None, key_len="default", what=""):
    w = x.w
    causal = w.causal if causal is None else causal
    scale = w.softmax_scale if scale is None else scale
    kl = x.key_len if isinstance(key_len, str) else key_len
    o_g, l_g = run_gpu(x, dev, causal=causal, scale=scale, key_len=kl)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, scale, causal, key_len=kl)
    return compare(o_g, l_g, o_r, l_r, what or w.name)


@pytest.mark.parametrize("name", ["b1h1n128d64", "b1h1n128d64_causal"])
def test_small_workload_full(cuda_device, name):
    x = make_inputs(WORKLOADS[name])
    full_check(x, cuda_device)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 3, 127, 128, 129, 255, 256, 257, 300, 383, 513])
def test_ragged_lengths(cuda_device, d, causal, N):
    x = make_inputs(Workload("ragged", 2, 2, N, d, causal, 100 + N))
    full_check(x, cuda_device, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(cuda_device, d, causal):
    B, N = 8, 700
    x = make_inputs(Workload("kl", B, 2, N, d, causal, 7, qk_sigma=2.0))
    kl = np.array([0, 1, 2, 127, 128, 129, 700, 350], np.int32)
    full_check(x, cuda_device, key_len=kl, what=f"key_len d={d} causal={causal}")


def test_key_len_out_of_range_clamped(cuda_device):
    x = make_inputs(Workload("klc", 3, 1, 200, 64, False, 8))
    kl = np.array([-5, 1000, 200], np.int32)
    full_check(x, cuda_device, key_len=kl)


def test_fully_masked_rows_are_zero_and_neg_inf(cuda_device):
    x = make_inputs(Workload("fm", 2, 3, 300, 128, True, 9))
    kl = np.array([0, 0], np.int32)
    o, lse = run_gpu(x, cuda_device, key_len=kl)
    assert np.all(o == 0.0)
    assert np.all(np.isneginf(lse))


@pytest.mark.parametrize("d", [64, 128])
def test_scale_zero_is_uniform_attention(cuda_device, d):
    x = make_inputs(Workload("s0", 1, 2, 260, d, True, 10))
    full_check(x, cuda_device, scale=0.0)


@pytest.mark.parametrize("d", [64, 128])
def test_q_zero_gives_prefix_mean(cuda_device, d):
    x = make_inputs(Workload("q0", 1, 2, 384, d, True, 11))
    x.q[...] = 0
    o, lse = run_gpu(x, cuda_device)
    counts = np.arange(1, 385, dtype=np.float64)
    np.testing.assert_allclose(lse[0], np.broadcast_to(np.log(counts), (2, 384)), rtol=0, atol=1e-3)
    vf = oracle.forward(x.q, x.k, x.v, 1.0, True)[0]
    assert np.max(np.abs(o - vf)) <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
def test_constant_v_returned(cuda_device, d):
    x = make_inputs(Workload("cv", 2, 2, 333, d, False, 12, qk_sigma=2.0))
    c = f32_to_bf16_bits(np.linspace(-2.0, 2.0, d).astype(np.float32))
    x.v[...] = c
    o, _ = run_gpu(x, cuda_device)
    cf = (c.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.max(np.abs(o - cf)) <= 1e-2


def test_peaky_logits_rescaling(cuda_device):
    """Scores with std 8 force many rescales of the running max."""
    x = make_inputs(Workload("peaky", 2, 2, 1024, 128, False, 13, qk_sigma=2.0, scale=0.25))
    full_check(x, cuda_device)


def test_large_scores_stay_finite(cuda_device):
    x = make_inputs(Workload("big", 1, 2, 512, 64, True, 14, qk_sigma=4.0, scale=1.0))
    full_check(x, cuda_device)


def _scaled_v(x, factors):
    """Multiply V's 128-row tiles by powers of two (exact in bf16)."""
    from exact_softmax_attention_fattn_gb300.inputs import bf16_bits_to_f32

    v = bf16_bits_to_f32(x.v).copy()
    for t, f in enumerate(factors):
        v[:, :, 128 * t:128 * (t + 1)] *= f
    x.v[...] = f32_to_bf16_bits(v)
    return x


@pytest.mark.parametrize("factor", [2.0 ** 17, 2.0 ** -12])
def test_v_tiles_outside_fp16_range_use_bf16(cuda_device, factor):
    """V tiles too large (> 65504) or too small (< 2^-8) for fp16 P V keep
    bf16 operands; O scales exactly with V, so compare O / factor."""
    x = make_inputs(Workload("vr", 2, 2, 300, 128, True, 16))
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, True)
    _scaled_v(x, [factor] * 3)
    o_g, l_g = run_gpu(x, cuda_device)
    compare(o_g / factor, l_g, o_r, l_r, f"V x {factor}")


def test_v_tiles_mixed_storage(cuda_device):
    """One head whose V tiles alternate between bf16 and fp16 storage."""
    x = make_inputs(Workload("vm", 1, 2, 640, 64, False, 17))
    _scaled_v(x, [1.0, 2.0 ** -10, 1.0, 2.0 ** -10, 1.0])
    full_check(x, cuda_device)


def test_repeated_calls_identical(cuda_device):
    x = make_inputs(Workload("rep", 2, 4, 1000, 128, True, 15))
    a = run_gpu(x, cuda_device)
    b = run_gpu(x, cuda_device)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def sample_rows(w: Workload, n_full_heads: int, n_random: int, seed: int) -> np.ndarray:
    """All rows of the first and last n_full_heads heads, plus tile-boundary and random rows elsewhere."""
    BH, N = w.B * w.H, w.N
    rows = []
    heads = list(range(min(n_full_heads, BH))) + list(range(max(BH - n_full_heads, n_full_heads), BH))
    for bh in heads:
        rows.append(bh * N + np.arange(N))
    rng = np.random.default_rng(seed)
    edges = np.unique(np.clip(np.concatenate([np.arange(0, N, 128) + o for o in (-1, 0, 1, 127)]), 0, N - 1))
    for bh in rng.choice(BH, size=min(8, BH), replace=False):
        rows.append(bh * N + edges)
    rows.append(rng.integers(0, BH * N, size=n_random))
    return np.unique(np.concatenate(rows)).astype(np.int64)


@pytest.mark.parametrize("name,n_full,n_rand", [
    ("b4h8n1024d64_causal", 32, 0),
    ("b2h16n4096d128_causal", 2, 4000),
    ("b1h32n16384d128_causal", 0, 1500),
    ("b8h16n2048d128_keylen", 2, 4000),
])
def test_measured_workloads_sampled(cuda_device, name, n_full, n_rand):
    w = WORKLOADS[name]
    x = make_inputs(w)
    o_g, l_g = run_gpu(x, cuda_device, check_guards=False)
    rows = sample_rows(w, n_full, n_rand, seed=w.seed)
    o_r, l_r = oracle.forward(x.q, x.k, x.v, w.softmax_scale, w.causal, key_len=x.key_len, rows=rows)
    compare(o_g.reshape(-1, w.d)[rows], l_g.reshape(-1)[rows], o_r, l_r, name)
    # every output finite (no fully masked rows in these workloads)
    assert np.all(np.isfinite(o_g)) and np.all(np.isfinite(l_g))


def test_kernel_event_hook(cuda_device):
    """fattn_set_kernel_events: the library records the caller's events around
    the attention kernel; its time is positive and inside the whole call's."""
    import torch

    from exact_softmax_attention_fattn_gb300 import binding
    from tests.gpu_helpers import bits_to_device

    x = make_inputs(Workload("hook", 2, 8, 2048, 128, True, 77))
    q, k, v = (bits_to_device(a, cuda_device) for a in (x.q, x.k, x.v))
    o = torch.empty_like(q)
    lse = torch.empty((2, 8, 2048), dtype=torch.float32, device=cuda_device)
    stream = torch.cuda.current_stream(cuda_device)
    ks, ke, cs, ce = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    ks.record(stream)
    ke.record(stream)
    torch.cuda.synchronize(cuda_device)
    binding.set_kernel_events(ks, ke)
    cs.record(stream)
    binding.forward_into(q, k, v, o, lse, causal=True)
    ce.record(stream)
    binding.set_kernel_events(None, None)
    torch.cuda.synchronize(cuda_device)
    t_kernel, t_call = ks.elapsed_time(ke), cs.elapsed_time(ce)
    assert 0.0 < t_kernel <= t_call, (t_kernel, t_call)
    # cleared: a later call leaves the events where they were
    binding.forward_into(q, k, v, o, lse, causal=True)
    torch.cuda.synchronize(cuda_device)
    assert ks.elapsed_time(ke) == t_kernel


@pytest.mark.parametrize("off_elems", [0, 8])
def test_output_alignment_16_and_32_bytes(cuda_device, off_elems):
    """O at a 32-byte boundary (rows stored 32 bytes at a time) and at an odd
    16-byte boundary (16-byte stores): the same values."""
    import torch

    from exact_softmax_attention_fattn_gb300 import binding
    from tests.gpu_helpers import bits_to_device

    x = make_inputs(Workload("align", 1, 2, 300, 128, True, 41))
    q, k, v = (bits_to_device(a, cuda_device) for a in (x.q, x.k, x.v))
    n = q.numel()
    buf = torch.zeros(n + 64, dtype=torch.int16, device=cuda_device)
    base = (-buf.data_ptr() // 2) % 16  # first element at a 32-byte boundary
    o = buf[base + off_elems:base + off_elems + n].view(torch.bfloat16).view(q.shape)
    assert o.data_ptr() % 32 == (0 if off_elems == 0 else 16)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device=cuda_device)
    binding.forward_into(q, k, v, o, lse, causal=True, scale=x.w.softmax_scale)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, detail
    o_r, l_r = oracle.forward(x.q, x.k, x.v, x.w.softmax_scale, True)
    compare(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), o_r, l_r,
            f"O offset {off_elems} elements")
