"""Shared plumbing for the GPU tests: move seeded bf16 bit patterns to the
device, call the C ABI through the binding, compare with the oracle."""
from __future__ import annotations

import numpy as np

# Tolerances of the attention forward against the fp64 oracle on the same
# bf16 inputs: max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3.
#
# O is delivered in bf16.  Where |O| >= 4 the spacing of bf16 values is 2^-5,
# so rounding even the exact result can miss it by 2^-6 = 0.0156 > 1e-2: no
# bf16 output can meet 1e-2 there.  On those elements the bar is one bf16
# unit in the last place of the exact value (2^-5 in [4, 8)); everywhere else
# it is 1e-2 as stated.  The mean and LSE bars are unchanged.
MAX_ABS_O = 1e-2
MEAN_ABS_O = 1e-3
MAX_ABS_LSE = 1e-3

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


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Assert the tolerances; -inf LSE (fully masked rows) must match exactly."""
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), ninf_ref), f"{what}: -inf LSE pattern differs"
    assert not np.any(np.isnan(lse_gpu)), f"{what}: NaN LSE"
    d_o = np.abs(o_gpu - o_ref)
    mean_o = float(d_o.mean()) if d_o.size else 0.0
    bar = np.maximum(MAX_ABS_O, bf16_ulp(o_ref) * (np.abs(o_ref) >= 4.0))
    excess = d_o - bar
    max_o = float(d_o.max()) if d_o.size else 0.0
    worst = int(np.argmax(excess)) if d_o.size else 0
    fin = ~ninf_ref
    max_l = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if np.any(fin) else 0.0
    assert d_o.size == 0 or excess.flat[worst] <= 0.0, (
        f"{what}: |dO| = {d_o.flat[worst]:.3e} at |O| = {abs(o_ref.flat[worst]):.3f} "
        f"(bar {bar.flat[worst]:.3e}; max|dO| {max_o:.3e})")
    assert mean_o <= MEAN_ABS_O, f"{what}: mean|dO| = {mean_o:.3e}"
    assert max_l <= MAX_ABS_LSE, f"{what}: max|dLSE| = {max_l:.3e}"
    return max_o, mean_o, max_l
