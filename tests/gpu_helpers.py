"""Shared plumbing for the GPU tests: move seeded bf16 bit patterns to the
device, call the C ABI through the binding, compare with the oracle."""
from __future__ import annotations

from typing import NamedTuple

import numpy as np

# Tolerances of the attention forward against the fp64 oracle on the same
# bf16 inputs: max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3.
#
# O is delivered in bf16, rounded once from the kernel's fp32 result.  A
# result within 1e-2 of the exact value before that rounding lands within
# 1e-2 + half a bf16 ulp of it after.  Where |O| < 4 half an ulp is at most
# 2^-8... 2^-7 and 1e-2 itself is met by a correctly rounded result, so the
# bar is 1e-2 as stated.  Where |O| >= 4 the bf16 spacing is 2^-5, so even the
# exact result rounded can miss by 2^-6 = 0.0156 > 1e-2; there the bar is
# 1e-2 + half an ulp of the exact value (0.0256 in [4, 8)), the bound the
# stated tolerance implies for a bf16 output.  The mean and LSE bars are the
# stated ones.  compare() counts the elements that needed the wider bar.
MAX_ABS_O = 1e-2
MEAN_ABS_O = 1e-3
MAX_ABS_LSE = 1e-3

# every passing compare() call of this process: (what, ParityStats), summarised at the end of a pytest run
PARITY_LOG: list = []

POISON_BF16 = 0x7FC1  # a NaN pattern the kernel never writes
GUARD = 4096  # elements of canary before and after each output


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0**-126)
    return np.exp2(np.floor(np.log2(ax)) - 7.0)


def bits_to_device(bits: np.ndarray, dev):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev)
    return t.view(torch.bfloat16)


def guarded_outputs(B, H, N, d, dev):
    """O and LSE views inside poisoned guard bands (to catch stray stores)."""
    import torch

    n_o = B * H * N * d
    o_buf = torch.full((n_o + 2 * GUARD,), POISON_BF16, dtype=torch.int16, device=dev)
    l_buf = torch.full((B * H * N + 2 * GUARD,), -12345.0, dtype=torch.float32, device=dev)
    o = o_buf[GUARD:GUARD + n_o].view(torch.bfloat16).view(B, H, N, d)
    lse = l_buf[GUARD:GUARD + B * H * N].view(B, H, N)
    return o_buf, l_buf, o, lse


def guards_intact(o_buf, l_buf) -> bool:
    import torch

    ok_o = bool(torch.all(o_buf[:GUARD] == POISON_BF16)) and bool(torch.all(o_buf[-GUARD:] == POISON_BF16))
    ok_l = bool(torch.all(l_buf[:GUARD] == -12345.0)) and bool(torch.all(l_buf[-GUARD:] == -12345.0))
    return ok_o and ok_l


def run_gpu(x, dev, causal=None, scale=None, key_len="default", check_guards=True, n_splits=None):
    """Run the kernel on Inputs x; returns (o float64 numpy, lse float64 numpy)."""
    import torch

    from exact_softmax_attention_fattn_gb300 import binding

    w = x.w
    causal = w.causal if causal is None else causal
    scale = w.softmax_scale if scale is None else scale
    kl = x.key_len if isinstance(key_len, str) else key_len
    q, k, v = (bits_to_device(a, dev) for a in (x.q, x.k, x.v))
    B, H, N, d = x.q.shape
    o_buf, l_buf, o, lse = guarded_outputs(B, H, N, d, dev)
    kl_t = None if kl is None else torch.from_numpy(np.asarray(kl, dtype=np.int32)).to(dev)
    binding.forward_into(q, k, v, o, lse, causal=causal, scale=scale, key_len=kl_t, n_splits=n_splits)
    st, detail = binding.last_error()
    assert st == binding.FATTN_OK, f"kernel reported {binding.status_string(st)} {detail}"
    torch.cuda.synchronize()
    if check_guards:
        assert guards_intact(o_buf, l_buf), "a store landed outside O or LSE"
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


class ParityStats(NamedTuple):
    max_o: float            # max |dO| over all elements
    mean_o: float           # mean |dO|
    max_l: float            # max |dLSE| over rows with a visible key
    n_elements: int
    n_over_1e2: int         # elements with |dO| > 1e-2 (only possible where |O| >= 4)
    worst_over_ulps: float  # the largest of those errors, in bf16 ulps of the exact value (0 if none)


def parity_bar(o_ref: np.ndarray) -> np.ndarray:
    """Per-element max |dO| bar: 1e-2, plus half a bf16 ulp of the exact value where |O| >= 4."""
    return MAX_ABS_O + 0.5 * bf16_ulp(o_ref) * (np.abs(o_ref) >= 4.0)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", log=True) -> ParityStats:
    """Assert the tolerances; -inf LSE (fully masked rows) must match exactly.
    Returns the error statistics, including how many elements needed the
    wider bar at |O| >= 4 and the worst of them in ulps."""
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), ninf_ref), f"{what}: -inf LSE pattern differs"
    assert not np.any(np.isnan(lse_gpu)), f"{what}: NaN LSE"
    d_o = np.abs(o_gpu - o_ref)
    mean_o = float(d_o.mean()) if d_o.size else 0.0
    bar = parity_bar(o_ref)
    excess = d_o - bar
    max_o = float(d_o.max()) if d_o.size else 0.0
    worst = int(np.argmax(excess)) if d_o.size else 0
    fin = ~ninf_ref
    max_l = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if np.any(fin) else 0.0
    over = d_o > MAX_ABS_O
    n_over = int(np.count_nonzero(over))
    worst_ulps = float((d_o[over] / bf16_ulp(o_ref[over])).max()) if n_over else 0.0
    stats = ParityStats(max_o, mean_o, max_l, int(d_o.size), n_over, worst_ulps)
    assert d_o.size == 0 or excess.flat[worst] <= 0.0, (
        f"{what}: |dO| = {d_o.flat[worst]:.3e} at |O| = {abs(o_ref.flat[worst]):.3f} "
        f"(bar {bar.flat[worst]:.3e}; max|dO| {max_o:.3e})")
    assert mean_o <= MEAN_ABS_O, f"{what}: mean|dO| = {mean_o:.3e}"
    assert max_l <= MAX_ABS_LSE, f"{what}: max|dLSE| = {max_l:.3e}"
    if log:
        PARITY_LOG.append((what, stats))  # comparisons of the kernel's output that passed
    print(f"parity {what}: max|dO| {max_o:.3e} mean|dO| {mean_o:.3e} max|dLSE| {max_l:.3e}; "
          f"{n_over} of {d_o.size} elements over 1e-2 (worst {worst_ulps:.2f} ulp)")
    return stats
