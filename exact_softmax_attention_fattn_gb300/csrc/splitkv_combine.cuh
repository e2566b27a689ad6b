// Split-KV combine, sm_103a.
//
// When the attention kernel splits the key tiles of a query block into
// n_splits near-equal runs (to give every SM work when there are fewer query
// blocks than SMs), split s leaves, for each query row, the normalised
// output O_s = softmax over its keys times V, and its log-sum-exp L_s.  This kernel merges them with the two-block rule of the
// online-softmax derivation ("understand-flashattention": two blocks with
// maxima m1, m2 and sums l1, l2 combine to max m, sum l1 e^(m1-m) + l2 e^(m2-m),
// the outputs weighted the same way), written in terms of L_s = m_s + log l_s:
//     L = log sum_s e^(L_s),   O = sum_s e^(L_s - L) O_s.
// Only the splits whose run meets the key tiles of the row's 128-row query
// tile wrote a partial (each such split holds a visible key for every row of
// the tile); the runs and tile counts are the attention kernel's: the block
// of 256 query rows visits n_blk key tiles (those of its later tile), split
// s takes tiles [s*n_blk/n_splits, (s+1)*n_blk/n_splits), and the row's tile
// visits the first n_t of them.  A row with no visible key gets O = 0 and
// LSE = -inf.
//
// HBM-bound: per row, (splits with a partial) * (D * 4 + 4) bytes read,
// D * 2 + 4 written.
// One thread per 4 columns of a row, so a warp reads whole 512-byte rows
// (D = 128) or two 256-byte rows (D = 64).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace fattn {

constexpr int COMBINE_THREADS = 256;

// Key tiles that query tile `row0` visits (as in the attention kernel).
__device__ __forceinline__ int combine_tiles_of(int row0, int N, int kl, int causal) {
  if (row0 >= N) return 0;
  const int max_lim = causal ? min(kl, row0 + 128) : kl;
  return max_lim > 0 ? (max_lim + 127) / 128 : 0;
}

template <int D>
__global__ void __launch_bounds__(COMBINE_THREADS)
    fattn_splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                 __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                 const int32_t* __restrict__ key_len, int B, int H, int N, int causal,
                                 int n_splits) {
  constexpr int TPR = D / 4;  // threads per row
  constexpr int ROWS = COMBINE_THREADS / TPR;
  const long long n_rows = (long long)B * H * N;
  const long long rg = (long long)blockIdx.x * ROWS + threadIdx.x / TPR;  // row over all heads
  const int c4 = threadIdx.x % TPR;                                       // column group
  if (rg >= n_rows) return;
  const int bh = (int)(rg / N);
  const int row = (int)(rg % N);
  int kl = key_len ? key_len[bh / H] : N;
  kl = kl < 0 ? 0 : (kl > N ? N : kl);
  const int blk0 = row / 256 * 256;
  const int n_blk = max(combine_tiles_of(blk0, N, kl, causal), combine_tiles_of(blk0 + 128, N, kl, causal));
  const int n_t = combine_tiles_of(row / 128 * 128, N, kl, causal);
  uint2* dst = reinterpret_cast<uint2*>(o + rg * D) + c4;
  if (n_t == 0) {
    *dst = make_uint2(0u, 0u);
    if (c4 == 0) lse[rg] = -INFINITY;
    return;
  }
  const long long stride = n_rows;  // between splits, in rows
  float m = -INFINITY;
  // split s holds keys of this row iff its run [s*n_blk/n_splits, ...) starts below n_t
  for (int s = 0; s < n_splits && s * n_blk / n_splits < n_t; ++s)
    if ((s + 1) * n_blk / n_splits > s * n_blk / n_splits) m = fmaxf(m, lse_part[s * stride + rg]);
  float sum = 0.0f, a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  for (int s = 0; s < n_splits && s * n_blk / n_splits < n_t; ++s) {
    if ((s + 1) * n_blk / n_splits == s * n_blk / n_splits) continue;  // an empty run
    const float w = expf(lse_part[s * stride + rg] - m);
    const float4 v = reinterpret_cast<const float4*>(o_part + (s * stride + rg) * D)[c4];
    sum += w;
    a0 = fmaf(w, v.x, a0);
    a1 = fmaf(w, v.y, a1);
    a2 = fmaf(w, v.z, a2);
    a3 = fmaf(w, v.w, a3);
  }
  const float inv = 1.0f / sum;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a0 * inv, a1 * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(a2 * inv, a3 * inv);
  *dst = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  if (c4 == 0) lse[rg] = m + logf(sum);
}

}  // namespace fattn
