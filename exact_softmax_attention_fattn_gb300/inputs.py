"""Seeded synthetic inputs for the attention forward.

This module holds no attention arithmetic: it only draws random numbers and
rounds them to bfloat16.  Both the CPU oracle's tests and the CUDA path's tests
and benchmark take their inputs from here, so the two sides see the same bits.

Generator (portable, bit-reproducible on x86 and Arm, independent of torch's
RNG): SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) evaluated in counter form, 53-bit uniforms, and the
Box-Muller transform (Box and Muller, 1958) for normals.  fp64 -> fp32 -> bf16
with round-to-nearest-even at each step.

Draw order for one workload: Q, K, V, then key_len; each tensor has its own
stream derived from (seed, stream id), so shapes can change without shifting
the other tensors' values.

The workloads mirror the attention shapes the pages work with: per-head
tensors [batch, heads, seq, head_dim] ("PyTorch profiling part 3: attention",
section "Naive attention with in-place causal masking"), causal masks, and a
per-batch key-padding length ("Linear Attention CUDA kernel", key_lengths).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_KEYLEN = 1, 2, 3, 4

_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    """The SplitMix64 output function on uint64 (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x10001 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix64(s * _GOLDEN + _GOLDEN)[0]


def splitmix64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit draws number start .. start+count-1 of one stream."""
    base = _stream_base(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base + idx * _GOLDEN)


def uniform53(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits."""
    z = splitmix64(seed, stream, start, count)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """`count` N(0, sigma^2) draws as float32, by Box-Muller on pairs of uniforms."""
    out = np.empty(count, dtype=np.float32)
    pairs = (count + 1) // 2
    for p0 in range(0, pairs, _CHUNK):
        n = min(_CHUNK, pairs - p0)
        u = uniform53(seed, stream, 2 * p0, 2 * n)
        u1 = 1.0 - u[0::2]  # (0, 1]: log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1)) * sigma
        th = (2.0 * math.pi) * u2
        z = np.empty(2 * n, dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(count, lo + 2 * n)
        out[lo:hi] = z[: hi - lo].astype(np.float32)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, nearest-even, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention forward problem: shapes, mask and input distribution."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    qk_sigma: float = 1.0
    v_sigma: float = 1.0
    key_len_range: tuple[int, int] | None = None  # inclusive [lo, hi], per batch
    scale: float | None = None  # None: 1/sqrt(d)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass
class Inputs:
    """bf16 bit patterns [B, H, N, d] (uint16) and optional key_len [B] (int32)."""

    w: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    key_len: np.ndarray | None


def make_inputs(w: Workload) -> Inputs:
    shape = (w.B, w.H, w.N, w.d)
    count = w.B * w.H * w.N * w.d
    q = f32_to_bf16_bits(normal(w.seed, STREAM_Q, count, w.qk_sigma)).reshape(shape)
    k = f32_to_bf16_bits(normal(w.seed, STREAM_K, count, w.qk_sigma)).reshape(shape)
    v = f32_to_bf16_bits(normal(w.seed, STREAM_V, count, w.v_sigma)).reshape(shape)
    key_len = None
    if w.key_len_range is not None:
        lo, hi = w.key_len_range
        z = splitmix64(w.seed, STREAM_KEYLEN, 0, w.B)
        key_len = (lo + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int32)
    return Inputs(w, q, k, v, key_len)


# The five workloads the attention forward is measured and checked on; a
# long causal sequence with few heads (fewer blocks of 256 query rows, 128,
# than a GB300 has SMs, 152: the shape split-KV is for); the headline shape
# at two other head dims.
WORKLOADS: dict[str, Workload] = {
    "b1h1n128d64": Workload("b1h1n128d64", 1, 1, 128, 64, False, 0),
    "b1h1n128d64_causal": Workload("b1h1n128d64_causal", 1, 1, 128, 64, True, 0),
    "b4h8n1024d64_causal": Workload("b4h8n1024d64_causal", 4, 8, 1024, 64, True, 1),
    "b2h16n4096d128_causal": Workload("b2h16n4096d128_causal", 2, 16, 4096, 128, True, 2),
    "b1h32n16384d128_causal": Workload("b1h32n16384d128_causal", 1, 32, 16384, 128, True, 3),
    "b8h16n2048d128_keylen": Workload(
        "b8h16n2048d128_keylen", 8, 16, 2048, 128, False, 4,
        qk_sigma=2.0, key_len_range=(1024, 2048),
    ),
    "b1h2n16384d128_causal": Workload("b1h2n16384d128_causal", 1, 2, 16384, 128, True, 5),
    # the headline shape at head dims outside {64, 128}: 96 (the 128-column
    # kernel with zero columns) and 256 (the one-query-tile kernel)
    "b2h16n4096d96_causal": Workload("b2h16n4096d96_causal", 2, 16, 4096, 96, True, 6),
    "b2h16n4096d256_causal": Workload("b2h16n4096d256_causal", 2, 16, 4096, 256, True, 7),
}

HEADLINE = "b2h16n4096d128_causal"


@dataclasses.dataclass(frozen=True)
class LinearWorkload:
    """A causal linear attention problem: Q, K [B, H, N, E] and V [B, H, N, M],
    float32 N(0, 1), optional per-batch key lengths uniform in key_len_range."""

    name: str
    B: int
    H: int
    N: int
    E: int
    M: int
    seed: int
    key_len_range: tuple[int, int] | None = None


@dataclasses.dataclass
class LinearInputs:
    w: LinearWorkload
    q: np.ndarray  # float32 [B, H, N, E]
    k: np.ndarray  # float32 [B, H, N, E]
    v: np.ndarray  # float32 [B, H, N, M]
    key_len: np.ndarray | None


def make_linear_inputs(w: LinearWorkload) -> LinearInputs:
    qk = w.B * w.H * w.N * w.E
    q = normal(w.seed, STREAM_Q, qk).reshape(w.B, w.H, w.N, w.E)
    k = normal(w.seed, STREAM_K, qk).reshape(w.B, w.H, w.N, w.E)
    v = normal(w.seed, STREAM_V, w.B * w.H * w.N * w.M).reshape(w.B, w.H, w.N, w.M)
    key_len = None
    if w.key_len_range is not None:
        lo, hi = w.key_len_range
        z = splitmix64(w.seed, STREAM_KEYLEN, 0, w.B)
        key_len = (lo + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int32)
    return LinearInputs(w, q, k, v, key_len)


# Causal linear attention (the second workload): a language-model head shape
# at the feature size the page's kernels dispatch on (E = M = 64).
LINEAR_WORKLOADS: dict[str, LinearWorkload] = {
    "lin_b2h16n4096e64": LinearWorkload("lin_b2h16n4096e64", 2, 16, 4096, 64, 64, 8),
    "lin_b8h8n2048e64_keylen": LinearWorkload("lin_b8h8n2048e64_keylen", 8, 8, 2048, 64, 64, 9,
                                              key_len_range=(1024, 2048)),
}


def linear_flops(w: LinearWorkload) -> float:
    """Algorithmic FLOPs of the causal linear attention forward, the page's
    recurrence: per row, the state update k v^T and the read q^T S (2 E M
    multiply-adds), and the normaliser's q . s and cumulative key sum (2 E)."""
    return float(w.B * w.H * w.N) * (4.0 * w.E * w.M + 4.0 * w.E)


def algorithmic_bytes(w: Workload, key_len: np.ndarray | None = None) -> float:
    """HBM bytes one forward must move at least: Q read, O written (bf16) and
    LSE written (fp32) for every row, and the K and V rows some query can see
    (all N under the causal mask; the first key_len[b] with key padding)."""
    rows = float(w.B * w.H * w.N)
    kv_rows = rows if key_len is None else float(w.H) * float(np.sum(np.clip(key_len, 0, w.N)))
    return rows * w.d * 2 * 2 + rows * 4 + kv_rows * w.d * 2 * 2


def causal_flops(w: Workload, key_len: np.ndarray | None = None) -> float:
    """Algorithmic FLOPs of one forward: 4*B*H*N^2*d, half of it when causal;
    with key padding, 4*H*N*d*sum(key_len)."""
    if key_len is not None and not w.causal:
        return 4.0 * w.H * w.N * w.d * float(np.sum(np.clip(key_len, 0, w.N)))
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if w.causal else f
