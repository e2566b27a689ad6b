"""Pins of the causal linear attention oracle: checks that fix its result by
something other than its own running-state loop.  Each takes an Oracle (the
real one, or a deliberately broken copy) and raises AssertionError on a
mismatch.  ("Linear Attention CUDA kernel" page: phi = elu + 1, the key-length
mask on K, the causal dot product and the normaliser of
CausalLinearAttention.forward.)"""
from __future__ import annotations

import numpy as np

from exact_softmax_attention_fattn_gb300.inputs import LinearWorkload, make_linear_inputs


def _inputs(B, H, N, E, M, seed):
    x = make_linear_inputs(LinearWorkload("pin", B, H, N, E, M, seed))
    return x.q, x.k, x.v


def _phi(x):
    x = x.astype(np.float64)
    return np.where(x > 0, x + 1.0, np.expm1(np.minimum(x, 0.0)) + 1.0)


def lin_matches_quadratic_form(orc):
    """The page's quadratic form: V' = (phi(Q) phi(K)^T, lower-triangular) V,
    times Z = 1 / (phi(Q) . cumsum(phi(K)) + eps), written with numpy matrix
    products and a cumulative sum (no running state)."""
    for N, E, M, kl in ((37, 8, 5, None), (64, 16, 16, [40, 64]), (5, 3, 7, [0, 2])):
        B = 1 if kl is None else len(kl)
        q, k, v = _inputs(B, 2, N, E, M, 100 + N)
        eps = 1e-6
        ours = orc.linear(q, k, v, key_len=kl, eps=eps)
        qt, kt, vv = _phi(q), _phi(k), v.astype(np.float64)
        if kl is not None:
            mask = (np.arange(N)[None, :] < np.asarray(kl)[:, None]).astype(np.float64)
            kt = kt * mask[:, None, :, None]
        a = np.einsum("bhie,bhje->bhij", qt, kt) * np.tril(np.ones((N, N)))
        num = np.einsum("bhij,bhjm->bhim", a, vv)
        z = 1.0 / (np.einsum("bhie,bhie->bhi", qt, np.cumsum(kt, axis=2)) + eps)
        ref = num * z[..., None]
        err = np.max(np.abs(ours - ref)) / max(1.0, np.max(np.abs(ref)))
        assert err <= 1e-12, f"quadratic form differs by {err:.3g} (N={N}, key_len={kl})"


def lin_feature_map_values(orc):
    """One row, E = M = 1: out = v * phi(q) phi(k) / (phi(q) phi(k) + eps), so
    phi is read back exactly: phi(0) = 1, phi(1) = 2, phi(-1) = 1/e, phi(3) = 4."""
    eps = 1e-6
    for qv, kv, want in ((0.0, 0.0, 1.0), (1.0, 0.0, 2.0), (-1.0, 0.0, np.exp(-1.0)), (0.0, 3.0, 4.0)):
        q = np.full((1, 1, 1, 1), qv, np.float32)
        k = np.full((1, 1, 1, 1), kv, np.float32)
        v = np.full((1, 1, 1, 1), 1.0, np.float32)
        out = orc.linear(q, k, v, eps=eps)[0, 0, 0, 0]
        prod = out * eps / (1.0 - out)  # solve out = p / (p + eps) for p = phi(q) phi(k)
        assert abs(prod - want) <= 1e-9 * max(1.0, want), f"phi({qv}) phi({kv}) read back as {prod}, want {want}"


def lin_masks_and_invariants(orc):
    """key_len 0: every mapped key is zero, so the numerator is 0 and out = 0.
    Constant V rows (= c): out = c * t / (t + eps) with t = phi(q) . cumsum.
    V scaled by 2 (exactly, in float32): out scaled by 2.  Causality: changing the last row of K and
    V changes only the last output row."""
    q, k, v = _inputs(2, 2, 50, 8, 6, 7)
    out = orc.linear(q, k, v, key_len=[0, 50])
    assert np.all(out[0] == 0.0), "key_len 0 still has output"
    c = np.arange(1, 7, dtype=np.float32)
    vc = np.broadcast_to(c, v.shape).copy()
    oc = orc.linear(q, k, vc)
    qt, kt = _phi(q), _phi(k)
    t = np.einsum("bhie,bhie->bhi", qt, np.cumsum(kt, axis=2))
    want = c[None, None, None, :] * (t / (t + 1e-6))[..., None]
    assert np.max(np.abs(oc - want)) <= 1e-10 * np.max(np.abs(want)), "constant V not returned"
    o2x = orc.linear(q, k, 2.0 * v)
    o1 = orc.linear(q, k, v)
    assert np.max(np.abs(o2x - 2.0 * o1)) <= 1e-12 * np.max(np.abs(o2x)), "not linear in V"
    k2, v2 = k.copy(), v.copy()
    k2[:, :, -1] += 1.0
    v2[:, :, -1] -= 2.0
    o2 = orc.linear(q, k2, v2)
    assert np.array_equal(o2[:, :, :-1], o1[:, :, :-1]), "a later row changed an earlier output"
    assert not np.allclose(o2[:, :, -1], o1[:, :, -1]), "the last row ignored its own key and value"


def lin_first_row_closed_form(orc):
    """Row 0 sees only itself: out_0 = v_0 * (phi(q_0).phi(k_0)) / (phi(q_0).phi(k_0) + eps)."""
    q, k, v = _inputs(1, 3, 4, 5, 4, 9)
    eps = 1e-3
    out = orc.linear(q, k, v, eps=eps)
    p = np.sum(_phi(q[:, :, 0]) * _phi(k[:, :, 0]), axis=-1)
    want = v[:, :, 0].astype(np.float64) * (p / (p + eps))[..., None]
    assert np.max(np.abs(out[:, :, 0] - want)) <= 1e-12, "first row differs from its closed form"


def lin_chunked_regrouping(orc):
    """The regrouping the GPU kernels compute, restated in numpy: the rows cut
    into chunks of C; per chunk, tril(phi(Q_c) phi(K_c)^T) V_c plus phi(Q_c)
    times the state of all earlier chunks, over the row sums of the same
    lower triangle plus phi(Q_c) . (earlier key sums) + eps; then the chunk's
    own share (phi(K_c)^T V_c, column sums of phi(K_c)) joins the state.  The
    same sums as the running state, regrouped: equal to rounding for any C,
    including chunks cut across the key-length mask and a ragged last chunk."""
    for N, E, M, kl, C in ((130, 8, 6, [100], 64), (37, 4, 5, None, 5), (9, 3, 2, [4, 9], 1),
                           (200, 16, 8, [150, 200], 64)):
        B = 1 if kl is None else len(kl)
        q, k, v = _inputs(B, 2, N, E, M, 200 + N)
        eps = 1e-3
        ours = orc.linear(q, k, v, key_len=kl, eps=eps)
        qt, kt, vv = _phi(q), _phi(k), v.astype(np.float64)
        if kl is not None:
            mask = (np.arange(N)[None, :] < np.asarray(kl)[:, None]).astype(np.float64)
            kt = kt * mask[:, None, :, None]
        ref = np.zeros(vv.shape)
        state = np.zeros((B, 2, E, M))
        ksum = np.zeros((B, 2, E))
        for c0 in range(0, N, C):
            c1 = min(N, c0 + C)
            qc, kc, vc = qt[:, :, c0:c1], kt[:, :, c0:c1], vv[:, :, c0:c1]
            a = np.einsum("bhie,bhje->bhij", qc, kc) * np.tril(np.ones((c1 - c0, c1 - c0)))
            num = np.einsum("bhij,bhjm->bhim", a, vc) + np.einsum("bhie,bhem->bhim", qc, state)
            den = a.sum(axis=3) + np.einsum("bhie,bhe->bhi", qc, ksum) + eps
            ref[:, :, c0:c1] = num / den[..., None]
            state = state + np.einsum("bhje,bhjm->bhem", kc, vc)
            ksum = ksum + kc.sum(axis=2)
        err = np.max(np.abs(ours - ref)) / max(1.0, np.max(np.abs(ref)))
        assert err <= 1e-12, f"chunked form differs by {err:.3g} (N={N}, C={C}, key_len={kl})"


ALL_PINS = [
    ("quadratic_form", lin_matches_quadratic_form),
    ("feature_map_values", lin_feature_map_values),
    ("masks_and_invariants", lin_masks_and_invariants),
    ("first_row_closed_form", lin_first_row_closed_form),
    ("chunked_regrouping", lin_chunked_regrouping),
]
