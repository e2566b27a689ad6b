"""The oracle's pins as plain functions of an oracle object.

Each pin raises AssertionError when the oracle disagrees with a fact the pages
or the mathematics fix.  test_oracle.py runs them against the real oracle;
test_oracle_mutants.py runs them against copies with planted mistakes and
requires every copy to fail at least one.
"""
from __future__ import annotations

import math

import numpy as np

from exact_softmax_attention_fattn_gb300.inputs import Workload, f32_to_bf16_bits, make_inputs
from tests._ref_helpers import brute_row, online_blocks, to_f64, torch_reference

TIGHT = 1e-12


def _bits(a) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def pin_n1(orc):
    """N = 1: the one key has weight 1, so O = v_0 and LSE = scale * q.k."""
    w = Workload("n1", 2, 3, 1, 8, False, 21)
    x = make_inputs(w)
    sc = 0.37
    for causal in (False, True):
        o, lse = orc.forward(x.q, x.k, x.v, sc, causal)
        np.testing.assert_array_equal(o, to_f64(x.v))
        qk = np.einsum("bhnd,bhnd->bhn", to_f64(x.q), to_f64(x.k))
        np.testing.assert_allclose(lse, sc * qk, rtol=0, atol=TIGHT)


def pin_n2_logistic(orc):
    """N = 2, no mask: p_0 = 1/(1+exp(s_1-s_0)) and LSE = logaddexp(s_0, s_1)."""
    w = Workload("n2", 1, 4, 2, 16, False, 22)
    x = make_inputs(w)
    sc = 0.25
    o, lse = orc.forward(x.q, x.k, x.v, sc, False)
    qf, kf, vf = to_f64(x.q), to_f64(x.k), to_f64(x.v)
    for h in range(4):
        for i in range(2):
            s0 = sc * math.fsum(qf[0, h, i] * kf[0, h, 0])
            s1 = sc * math.fsum(qf[0, h, i] * kf[0, h, 1])
            p0 = 1.0 / (1.0 + math.exp(s1 - s0))
            exp_o = p0 * vf[0, h, 0] + (1.0 - p0) * vf[0, h, 1]
            np.testing.assert_allclose(o[0, h, i], exp_o, rtol=0, atol=1e-12)
            assert abs(lse[0, h, i] - np.logaddexp(s0, s1)) < 1e-12


def pin_causal_row0(orc):
    """Causal row 0 sees only key 0: O = v_0 exactly, LSE = s_00."""
    w = Workload("r0", 2, 2, 33, 16, True, 23)
    x = make_inputs(w)
    o, lse = orc.forward(x.q, x.k, x.v, 0.2, True)
    np.testing.assert_array_equal(o[:, :, 0, :], to_f64(x.v)[:, :, 0, :])
    s00 = 0.2 * np.einsum("bhd,bhd->bh", to_f64(x.q)[:, :, 0], to_f64(x.k)[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=TIGHT)


def pin_q_zero(orc, mode: str):
    """Q = 0 makes every score 0: O_i is the plain mean of the visible v_j and
    LSE_i = ln(#visible) ("understand-flashattention", logsumexp derivation
    with S = 0)."""
    B, H, N, d = 3, 2, 45, 8
    w = Workload("q0", B, H, N, d, False, 24)
    x = make_inputs(w)
    q0 = np.zeros_like(x.q)
    causal = mode in ("causal", "causal_keylen")
    kl = np.array([45, 17, 1], np.int32) if "keylen" in mode else None
    o, lse = orc.forward(q0, x.k, x.v, 0.3, causal, key_len=kl)
    vf = to_f64(x.v)
    for b in range(B):
        klen = N if kl is None else int(kl[b])
        for i in range(N):
            cnt = min(klen, i + 1) if causal else klen
            exp_o = vf[b, :, :cnt, :].mean(axis=1)
            np.testing.assert_allclose(o[b, :, i, :], exp_o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, :, i], math.log(cnt), rtol=0, atol=1e-13)


def pin_constant_v(orc):
    """Every v_j equal to c gives O_i = c on every row with a visible key."""
    w = Workload("cv", 2, 2, 50, 16, False, 25, qk_sigma=3.0)
    x = make_inputs(w)
    c = _bits(np.linspace(-3.0, 3.0, 16))
    v = np.broadcast_to(c, x.v.shape).copy()
    for causal, kl in ((False, None), (True, None), (True, np.array([50, 7], np.int32))):
        o, _ = orc.forward(x.q, x.k, v, 0.125, causal, key_len=kl)
        np.testing.assert_allclose(o, np.broadcast_to(to_f64(c), o.shape), rtol=0, atol=1e-12)


def pin_linear_v(orc):
    """O is affine in V: O(a V + b) = a O(V) + b (rows of P sum to one)."""
    w = Workload("lin", 1, 2, 40, 8, True, 26)
    x = make_inputs(w)
    rng = np.random.default_rng(0)
    v_small = rng.integers(-8, 9, size=x.v.shape).astype(np.float32) / 4.0
    v1 = _bits(v_small)
    v2 = _bits(2.0 * v_small + 1.0)  # exact in bf16
    o1, l1 = orc.forward(x.q, x.k, v1, 0.3, True)
    o2, l2 = orc.forward(x.q, x.k, v2, 0.3, True)
    np.testing.assert_allclose(o2, 2.0 * o1 + 1.0, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(l1, l2)


def pin_permutation(orc):
    """Without masks, permuting the keys (K and V rows together) changes
    nothing, and permuting the queries permutes the outputs."""
    w = Workload("perm", 1, 2, 31, 16, False, 27)
    x = make_inputs(w)
    o, lse = orc.forward(x.q, x.k, x.v, 0.25, False)
    pk = np.random.default_rng(1).permutation(31)
    o2, l2 = orc.forward(x.q, x.k[:, :, pk], x.v[:, :, pk], 0.25, False)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)
    pq = np.random.default_rng(2).permutation(31)
    o3, l3 = orc.forward(x.q[:, :, pq], x.k, x.v, 0.25, False)
    np.testing.assert_array_equal(o3, o[:, :, pq])
    np.testing.assert_array_equal(l3, lse[:, :, pq])


def pin_lse_bounds(orc):
    """max_vis s <= LSE <= max_vis s + ln(#visible)."""
    w = Workload("lb", 2, 2, 64, 16, True, 28, qk_sigma=2.0)
    x = make_inputs(w)
    kl = np.array([64, 20], np.int32)
    sc = 0.25
    _, lse = orc.forward(x.q, x.k, x.v, sc, True, key_len=kl)
    s = sc * np.einsum("bhid,bhjd->bhij", to_f64(x.q), to_f64(x.k))
    for b in range(2):
        for i in range(64):
            cnt = min(int(kl[b]), i + 1)
            mx = s[b, :, i, :cnt].max(axis=-1)
            assert np.all(lse[b, :, i] >= mx - 1e-12)
            assert np.all(lse[b, :, i] <= mx + math.log(cnt) + 1e-12)


def pin_probs(orc):
    """Rows of P sum to one ("understand-flashattention", numerically stable
    softmax) and P_ij = exp(S_ij - L_i) (its "recomputing P needs
    logsumexp" section); masked entries are exactly zero."""
    w = Workload("pr", 2, 2, 48, 16, True, 29, qk_sigma=2.0)
    x = make_inputs(w)
    kl = np.array([48, 30], np.int32)
    sc = 0.3
    _, lse = orc.forward(x.q, x.k, x.v, sc, True, key_len=kl)
    for b in range(2):
        for h in range(2):
            p, s = orc.probs(x.q, x.k, sc, True, key_len=kl, b=b, h=h)
            np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=TIGHT)
            ii, jj = np.meshgrid(np.arange(48), np.arange(48), indexing="ij")
            vis = (jj <= ii) & (jj < kl[b])
            assert np.all(p[~vis] == 0.0)
            pe = np.exp(s - lse[b, h][:, None])
            np.testing.assert_allclose(p[vis], pe[vis], rtol=1e-12, atol=0)
            sd = sc * to_f64(x.q)[b, h] @ to_f64(x.k)[b, h].T
            np.testing.assert_allclose(s, sd, rtol=0, atol=1e-12)


def pin_online_recurrence(orc, causal: bool, use_kl: bool):
    """The two-block derivation of "understand-flashattention" (steps 1-8),
    run blockwise in fp64 at every split point and at several block sizes,
    reaches the oracle's one-shot result."""
    B, H, N, d = 2, 1, 40, 8
    w = Workload("ol", B, H, N, d, False, 30, qk_sigma=2.5)
    x = make_inputs(w)
    kl = np.array([40, 13], np.int32) if use_kl else None
    sc = 0.35
    o, lse = orc.forward(x.q, x.k, x.v, sc, causal, key_len=kl)
    qf, kf, vf = to_f64(x.q), to_f64(x.k), to_f64(x.v)
    for b in range(B):
        s = sc * qf[b, 0] @ kf[b, 0].T
        klen = N if kl is None else int(kl[b])
        for i in range(N):
            row = s[i].copy()
            vis = np.arange(N) < klen
            if causal:
                vis &= np.arange(N) <= i
            row[~vis] = -np.inf
            splittings = [[t] for t in range(1, N)] + [list(range(bs, N, bs)) for bs in (3, 7, 16)]
            for splits in splittings:
                ob, lb = online_blocks(row, vf[b, 0], splits)
                np.testing.assert_allclose(ob, o[b, 0, i], rtol=0, atol=1e-12)
                assert abs(lb - lse[b, 0, i]) <= 1e-12 * max(1.0, abs(lb))


def pin_torch(orc, causal: bool, use_kl: bool):
    """Library restatement: torch fp64 softmax(scale Q K^T + bias) V."""
    w = Workload("tc", 2, 3, 200, 32, False, 31, qk_sigma=1.5)
    x = make_inputs(w)
    kl = np.array([200, 77], np.int32) if use_kl else None
    sc = 1.0 / math.sqrt(32)
    o, lse = orc.forward(x.q, x.k, x.v, sc, causal, key_len=kl)
    ot, lt = torch_reference(x.q, x.k, x.v, sc, causal, kl)
    np.testing.assert_allclose(o, ot, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lt, rtol=0, atol=1e-12)


def pin_brute(orc):
    """Pure-Python loops (math.fsum) on tiny inputs, every row."""
    w = Workload("bf", 2, 2, 6, 3, False, 32, qk_sigma=2.0)
    x = make_inputs(w)
    kl = np.array([4, 6], np.int32)
    for causal in (False, True):
        for key_len in (None, kl):
            o, lse = orc.forward(x.q, x.k, x.v, 0.7, causal, key_len=key_len)
            for b in range(2):
                for h in range(2):
                    for i in range(6):
                        ob, lb = brute_row(x.q, x.k, x.v, b, h, i, 0.7, causal, key_len)
                        np.testing.assert_allclose(o[b, h, i], ob, rtol=0, atol=1e-13)
                        assert abs(lse[b, h, i] - lb) < 1e-13


def pin_fully_masked(orc):
    """A row with no visible key gives O = 0 and LSE = -inf ("PyTorch
    profiling part 3: attention", section "The safe softmax")."""
    w = Workload("fm", 3, 2, 20, 8, False, 33)
    x = make_inputs(w)
    kl = np.array([0, 5, 0], np.int32)
    for causal in (False, True):
        o, lse = orc.forward(x.q, x.k, x.v, 0.5, causal, key_len=kl)
        assert np.all(o[0] == 0.0) and np.all(o[2] == 0.0)
        assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
        assert np.all(np.isfinite(lse[1])) and np.all(np.isfinite(o[1]))
        assert np.any(o[1] != 0.0)


def pin_masked_keys_irrelevant(orc):
    """Masked keys do not touch the result, even when their scores are huge:
    the max is taken over the visible scores only, which is what keeps the
    softmax stable ("understand-flashattention", numerically stable softmax)."""
    B, H, N, d = 2, 1, 12, 8
    w = Workload("mk", B, H, N, d, False, 34)
    x = make_inputs(w)
    kl = np.array([5, 12], np.int32)
    q = _bits(np.full((B, H, N, d), 8.0))
    k_small = x.k
    k_huge = k_small.copy()
    k_huge[0, :, 5:, :] = _bits(np.full((H, N - 5, d), 64.0))  # padded keys of batch 0
    for causal in (False, True):
        o1, l1 = orc.forward(q, k_small, x.v, 1.0, causal, key_len=kl)
        o2, l2 = orc.forward(q, k_huge, x.v, 1.0, causal, key_len=kl)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
    # causal: later keys with huge scores are invisible to earlier queries
    k_late = k_small.copy()
    k_late[1, :, 6:, :] = _bits(np.full((H, N - 6, d), 64.0))
    o1, l1 = orc.forward(q, k_small, x.v, 1.0, True)
    o2, l2 = orc.forward(q, k_late, x.v, 1.0, True)
    np.testing.assert_array_equal(o1[1, :, :6], o2[1, :, :6])
    np.testing.assert_array_equal(l1[1, :, :6], l2[1, :, :6])


def pin_block_merge(orc):
    """Merging the final states of key blocks, as the split-KV combine does:
    for a partition of the keys into blocks, each block's normalised output
    O_t and log-sum-exp L_t (the oracle on that block alone: its keys and
    values moved to the front, the rest masked by key_len) give the whole
    result as L = log sum_t e^(L_t), O = sum_t e^(L_t - L) O_t
    ("understand-flashattention", complete derivation for two blocks, applied
    to the blocks' final statistics)."""
    B, H, N, d = 1, 2, 50, 16
    x = make_inputs(Workload("bm", B, H, N, d, False, 35, qk_sigma=2.0))
    sc = 0.3
    o, lse = orc.forward(x.q, x.k, x.v, sc, False)
    for cuts in ([1], [17], [49], [10, 30], [5, 6, 40]):
        edges = [0] + cuts + [N]
        outs, lses = [], []
        for s, e in zip(edges[:-1], edges[1:]):
            kb, vb = np.zeros_like(x.k), np.zeros_like(x.v)
            kb[:, :, : e - s] = x.k[:, :, s:e]
            vb[:, :, : e - s] = x.v[:, :, s:e]
            ob, lb = orc.forward(x.q, kb, vb, sc, False, key_len=np.full(B, e - s, np.int32))
            outs.append(np.asarray(ob, np.float64))
            lses.append(np.asarray(lb, np.float64))
        big_l = np.logaddexp.reduce(np.stack(lses), axis=0)
        big_o = sum(np.exp(lt - big_l)[..., None] * ot for lt, ot in zip(lses, outs))
        np.testing.assert_allclose(big_o, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(big_l, lse, rtol=1e-12, atol=0)


ALL_PINS = [
    ("n1", pin_n1),
    ("n2_logistic", pin_n2_logistic),
    ("causal_row0", pin_causal_row0),
    ("q_zero_causal", lambda orc: pin_q_zero(orc, "causal")),
    ("q_zero_keylen", lambda orc: pin_q_zero(orc, "keylen")),
    ("q_zero_causal_keylen", lambda orc: pin_q_zero(orc, "causal_keylen")),
    ("constant_v", pin_constant_v),
    ("linear_v", pin_linear_v),
    ("permutation", pin_permutation),
    ("lse_bounds", pin_lse_bounds),
    ("probs", pin_probs),
    ("online", lambda orc: pin_online_recurrence(orc, True, True)),
    ("torch", lambda orc: pin_torch(orc, True, True)),
    ("brute", pin_brute),
    ("fully_masked", pin_fully_masked),
    ("masked_keys_irrelevant", pin_masked_keys_irrelevant),
    ("block_merge", pin_block_merge),
]
