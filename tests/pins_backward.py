"""Pins of the backward oracle: checks that fix dQ, dK, dV by something other
than the oracle's own formulas.  Each takes an Oracle (the real one, or a
deliberately broken copy) and raises AssertionError on a mismatch.

The gradients are of a scalar loss L through O, with dout = dL/dO
("understand-flashattention", backward pass steps 1-5, scale carried by the
chain rule through S = scale * Q K^T).
"""
from __future__ import annotations

import numpy as np

from exact_softmax_attention_fattn_gb300.inputs import Workload, bf16_bits_to_f32, make_inputs


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def _inputs(B, H, N, d, causal, seed, sigma=1.0):
    x = make_inputs(Workload("bwd", B, H, N, d, causal, seed, qk_sigma=sigma))
    g = make_inputs(Workload("bwd_g", B, H, N, d, causal, seed + 1000)).v  # dL/dO ~ N(0, 1)
    return x, g


def _np_forward(q, k, v, scale, causal, key_len):
    """Textbook softmax(mask(scale Q K^T)) V in fp64 (rows with no visible key: 0)."""
    B, H, N, d = q.shape
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((B, 1, N, N), dtype=bool)
    if causal:
        vis &= (j <= i)[None, None]
    if key_len is not None:
        kl = np.clip(np.asarray(key_len), 0, N)
        vis &= (j[None, None] < kl[:, None, None, None])
    s = np.where(vis, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(vis, np.exp(s - m), 0.0)
    den = e.sum(-1, keepdims=True)
    p = np.divide(e, den, out=np.zeros_like(e), where=den > 0)
    return np.einsum("bhij,bhjd->bhid", p, v)


def bwd_matches_torch_autograd(orc):
    """PyTorch's CPU fp64 autograd of the textbook forward, an independent library path."""
    import torch

    for causal, key_len in ((False, [70, 33]), (True, None), (True, [51, 70])):
        x, g = _inputs(2, 2, 70, 16, causal, 31)
        scale = 0.3
        q, k, v, go = (torch.tensor(_f64(a), requires_grad=True) for a in (x.q, x.k, x.v, g))
        N = q.shape[2]
        mask = torch.ones(2, 1, N, N, dtype=torch.bool)
        if causal:
            mask &= torch.tril(torch.ones(N, N, dtype=torch.bool))
        if key_len is not None:
            mask &= torch.arange(N)[None, None, None, :] < torch.tensor(key_len)[:, None, None, None]
        s = scale * q @ k.transpose(-1, -2)
        s = s.masked_fill(~mask, float("-inf"))
        o = torch.softmax(s, dim=-1) @ v
        (o * go.detach()).sum().backward()
        dq, dk, dv = orc.backward(x.q, x.k, x.v, g, scale, causal, key_len=key_len)
        for name, ours, ref in (("dq", dq, q.grad), ("dk", dk, k.grad), ("dv", dv, v.grad)):
            ref = ref.numpy()
            err = np.max(np.abs(ours - ref)) / max(1.0, np.max(np.abs(ref)))
            assert err <= 1e-10, f"{name} differs from torch autograd by {err:.3g} (causal={causal}, key_len={key_len})"


def bwd_matches_finite_differences(orc):
    """Central differences of the fp64 forward (first checked against the forward oracle)."""
    for causal, key_len in ((False, None), (True, None), (False, [3])):
        x, g = _inputs(1, 1, 5, 3, causal, 41, sigma=1.5)
        scale = 0.7
        q, k, v, go = (_f64(a) for a in (x.q, x.k, x.v, g))
        o_ref, _ = orc.forward(x.q, x.k, x.v, scale, causal, key_len=key_len)
        o_np = _np_forward(q, k, v, scale, causal, key_len)
        assert np.max(np.abs(o_np - o_ref)) <= 1e-12, "fp64 textbook forward disagrees with the forward oracle"
        loss = lambda q_, k_, v_: float(np.sum(_np_forward(q_, k_, v_, scale, causal, key_len) * go))  # noqa: E731
        dq, dk, dv = orc.backward(x.q, x.k, x.v, g, scale, causal, key_len=key_len)
        h = 1e-6
        for name, ours, which in (("dq", dq, 0), ("dk", dk, 1), ("dv", dv, 2)):
            fd = np.zeros_like(q)
            for idx in np.ndindex(q.shape):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += h
                args_m[which][idx] -= h
                fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.max(np.abs(ours - fd))
            assert err <= 1e-6, f"{name} differs from central differences by {err:.3g} (causal={causal}, key_len={key_len})"


def bwd_invariants(orc):
    """Sum_j dK_j = 0 (a shift of every key adds a per-row constant to the
    visible scores, which the softmax ignores); Sum_j dV_j = sum of dO over the
    rows with a visible key (rows of P sum to 1); a row with no visible key
    contributes nothing and gets dQ = 0."""
    x, g = _inputs(2, 2, 300, 32, True, 51)
    key_len = [300, 0]
    dq, dk, dv = orc.backward(x.q, x.k, x.v, g, 0.25, True, key_len=key_len)
    go = _f64(g)
    mag = np.max(np.abs(dk)) + 1.0
    assert np.max(np.abs(dk[0].sum(axis=1))) <= 1e-10 * mag * 300, "sum over keys of dK is not zero"
    assert np.max(np.abs(dv[0].sum(axis=1) - go[0].sum(axis=1))) <= 1e-9, "sum of dV rows != sum of dO rows"
    assert np.all(dq[1] == 0) and np.all(dk[1] == 0) and np.all(dv[1] == 0), "fully masked batch has gradients"


def bwd_constant_v_and_zero_scale(orc):
    """Constant V rows make O independent of Q and K, so dQ = dK = 0.  Scale 0
    makes P uniform over each row's visible keys: dQ = dK = 0 and
    dV_j = sum over rows i that see j of dO_i / (number of keys row i sees)."""
    x, g = _inputs(1, 2, 130, 16, True, 61)
    c = x.v[:, :, :1, :].copy()
    x.v[...] = c
    dq, dk, _ = orc.backward(x.q, x.k, x.v, g, 0.4, True)
    assert np.max(np.abs(dq)) <= 1e-12 and np.max(np.abs(dk)) <= 1e-12, "constant V still has dQ / dK"
    x, g = _inputs(1, 2, 130, 16, False, 62)
    key_len = [97]
    dq, dk, dv = orc.backward(x.q, x.k, x.v, g, 0.0, False, key_len=key_len)
    assert np.all(dq == 0) and np.all(dk == 0), "scale 0 still has dQ / dK"
    go = _f64(g)
    expect = np.zeros_like(go)
    expect[:, :, :97, :] = go.sum(axis=2, keepdims=True) / 97.0
    assert np.max(np.abs(dv - expect)) <= 1e-12, "scale-0 dV is not the uniform average"


def bwd_row_term_from_output(orc):
    """The reformulation the GPU kernels use: P recomputed from the forward's
    log-sum-exp (P = exp(S - LSE), "recomputing P needs logsumexp") and the
    row term of dS taken as D_i = dO_i . O_i instead of sum_k dP_ik P_ik
    (equal, since O_i = sum_k P_ik V_k).  A numpy backward built that way from
    the oracle's own forward O and LSE equals the oracle's backward."""
    for causal, key_len in ((True, None), (False, [90, 41]), (True, [77, 0])):
        x, g = _inputs(2, 2, 90, 16, causal, 71)
        scale = 0.3
        o, lse = orc.forward(x.q, x.k, x.v, scale, causal, key_len=key_len)
        dq, dk, dv = orc.backward(x.q, x.k, x.v, g, scale, causal, key_len=key_len)
        q, k, v, go = (_f64(a) for a in (x.q, x.k, x.v, g))
        N = q.shape[2]
        vis = np.ones((2, 1, N, N), dtype=bool)
        if causal:
            vis &= np.tril(np.ones((N, N), dtype=bool))[None, None]
        if key_len is not None:
            vis &= np.arange(N)[None, None, None, :] < np.asarray(key_len)[:, None, None, None]
        s = scale * np.einsum("bhid,bhjd->bhij", q, k)
        finite = np.isfinite(lse)  # rows with a visible key
        lse0 = np.where(finite, lse, 0.0)[..., None]
        p = np.where(vis & finite[..., None], np.exp(np.where(vis, s, 0.0) - lse0), 0.0)
        row = np.einsum("bhim,bhim->bhi", go, o)
        ds = p * (np.einsum("bhim,bhjm->bhij", go, v) - row[..., None])
        ref = (scale * np.einsum("bhij,bhjd->bhid", ds, k), scale * np.einsum("bhij,bhid->bhjd", ds, q),
               np.einsum("bhij,bhim->bhjm", p, go))
        for name, ours, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            err = np.max(np.abs(ours - want)) / max(1.0, np.max(np.abs(want)))
            assert err <= 1e-10, f"{name} from the output-based row term differs by {err:.3g}"


ALL_PINS = [
    ("torch_autograd", bwd_matches_torch_autograd),
    ("finite_differences", bwd_matches_finite_differences),
    ("invariants", bwd_invariants),
    ("constant_v_zero_scale", bwd_constant_v_and_zero_scale),
    ("row_term_from_output", bwd_row_term_from_output),
]
