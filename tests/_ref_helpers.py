"""Independent restatements used only to pin the oracle (test code).

Nothing here is imported by the product path.  These are deliberately
different formulations of the same mathematics: pure-Python loops, logistic
closed forms, the online (blockwise) recurrence, and a torch/numpy library
softmax.
"""
from __future__ import annotations

import math

import numpy as np

from exact_softmax_attention_fattn_gb300.inputs import bf16_bits_to_f32


def to_f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def visible(i: int, j: int, N: int, causal: bool, klen: int) -> bool:
    return (not causal or j <= i) and j < min(max(klen, 0), N)


def brute_row(q, k, v, b, h, i, scale, causal, key_len=None):
    """Pure-Python loops, math.fsum, for tiny inputs: the definition once more."""
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    N, d = qf.shape[2], qf.shape[3]
    klen = N if key_len is None else int(key_len[b])
    s = [scale * math.fsum(qf[b, h, i, t] * kf[b, h, j, t] for t in range(d)) for j in range(N)]
    vis = [j for j in range(N) if visible(i, j, N, causal, klen)]
    if not vis:
        return [0.0] * d, -math.inf
    m = max(s[j] for j in vis)
    e = {j: math.exp(s[j] - m) for j in vis}
    tot = math.fsum(e.values())
    o = [math.fsum(e[j] / tot * vf[b, h, j, t] for j in vis) for t in range(d)]
    return o, m + math.log(tot)


def online_blocks(s_row: np.ndarray, v: np.ndarray, splits: list[int]):
    """The blockwise online-softmax recurrence of "understand-flashattention",
    section "two-block derivation", steps 1-8, generalised to any number of
    blocks: running max m, normaliser l and unnormalised output, rescaled by
    exp(m_old - m_new) at every new block, normalised at the end.  Masked
    entries are -inf in s_row."""
    bounds = [0] + list(splits) + [len(s_row)]
    m = -math.inf
    l = 0.0
    o = np.zeros(v.shape[1])
    for a, b in zip(bounds[:-1], bounds[1:]):
        sb = s_row[a:b]
        if sb.size == 0:
            continue
        m_blk = np.max(sb)
        m_new = max(m, m_blk)
        if m_new == -math.inf:
            continue  # nothing visible yet: the state stays empty
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        pb = np.exp(sb - m_new)
        l = alpha * l + float(np.sum(pb))
        o = alpha * o + pb @ v[a:b]
        m = m_new
    if l == 0.0:
        return np.zeros(v.shape[1]), -math.inf
    return o / l, m + math.log(l)


def torch_reference(q, k, v, scale, causal, key_len=None):
    """Library restatement: torch fp64 softmax over scale*Q K^T plus an additive
    0/-inf bias, then P V; an all-masked row is set to 0 / -inf afterwards."""
    import torch

    qf = torch.from_numpy(to_f64(q))
    kf = torch.from_numpy(to_f64(k))
    vf = torch.from_numpy(to_f64(v))
    B, H, N, d = qf.shape
    s = torch.matmul(qf, kf.transpose(-1, -2)) * scale
    ii = torch.arange(N).view(N, 1)
    jj = torch.arange(N).view(1, N)
    vis = torch.ones(B, 1, N, N, dtype=torch.bool)
    if causal:
        vis = vis & (jj <= ii)
    if key_len is not None:
        kl = torch.from_numpy(np.asarray(key_len, dtype=np.int64)).clamp(0, N).view(B, 1, 1, 1)
        vis = vis & (jj.view(1, 1, 1, N) < kl)
    bias = torch.zeros(vis.shape, dtype=torch.float64).masked_fill(~vis, -math.inf)
    z = s + bias
    lse = torch.logsumexp(z, dim=-1)
    p = torch.softmax(z, dim=-1)
    empty = ~vis.any(dim=-1)  # [B,1,N]
    p = torch.where(empty.unsqueeze(-1), torch.zeros_like(p), p)
    o = torch.matmul(p, vf)
    lse = torch.where(empty.expand_as(lse), torch.full_like(lse, -math.inf), lse)
    return o.numpy(), lse.numpy()
