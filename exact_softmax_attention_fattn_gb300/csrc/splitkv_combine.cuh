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
// tile wrote a partial; the runs and tile counts are the attention kernel's:
// a block of blk_rows query rows (256 for the two-tile kernel, 128 for the
// head-dim-256 kernel) visits n_blk key tiles of key_tile keys (128, or 64),
// split s takes tiles [s*n_blk/n_splits, (s+1)*n_blk/n_splits), and the
// row's 128-row tile visits the first n_t of them.  (With 128-key tiles every
// such split holds a visible key for every row of the tile; with 64-key
// tiles a split may hold none for some rows, which then carry O = 0 and
// L = -inf and weigh nothing; the first split always holds key 0.)  A row
// with no visible key at all gets O = 0 and LSE = -inf.
//
// HBM-bound: per row, (splits with a partial) * (D * 4 + 4) bytes read,
// D * 2 + 4 written.  Grid (row blocks, heads); D / 16 threads per row, each
// holding 16 columns as 4 float4 loads interleaved with its neighbours' (the
// i-th load of the row's threads covers 128 contiguous bytes), so the
// per-row scalar work (limits, split runs, weights) is shared by few threads.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fattn {

constexpr int COMBINE_THREADS = 256;

// Key tiles of key_tile keys that the 128-row query tile `row0` visits (as
// in the attention kernel).
__device__ __forceinline__ int combine_tiles_of(int row0, int N, int kl, int causal, int key_tile) {
  if (row0 >= N) return 0;
  const int max_lim = causal ? min(kl, row0 + 128) : kl;
  return max_lim > 0 ? (max_lim + key_tile - 1) / key_tile : 0;
}

template <int D>
__global__ void __launch_bounds__(COMBINE_THREADS)
    fattn_splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                                 __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                 const int32_t* __restrict__ key_len, int B, int H, int N, int hd, int causal,
                                 int n_splits, int blk_rows, int key_tile) {
  constexpr int VPT = 4;            // float4 per thread and split
  constexpr int TPR = D / (4 * VPT);  // threads per row (rows of hd <= D columns)
  constexpr int ROWS = COMBINE_THREADS / TPR;
  const int row = blockIdx.x * ROWS + threadIdx.x / TPR;  // grid: (row blocks, heads)
  const int c4 = threadIdx.x % TPR;                       // float4 columns c4 + TPR * i, i < VPT
  if (row >= N) return;
  pdl_wait();  // the partials come from the attention kernel before this one
  const int BH = B * H;
  const size_t stride = (size_t)BH * N;  // rows between two splits' partials
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    int kl = key_len ? __ldg(key_len + bh / H) : N;
    kl = kl < 0 ? 0 : (kl > N ? N : kl);
    const int blk0 = row / blk_rows * blk_rows;
    int n_blk = 0;
    for (int r0 = blk0; r0 < blk0 + blk_rows; r0 += 128) n_blk = max(n_blk, combine_tiles_of(r0, N, kl, causal, key_tile));
    const int n_t = combine_tiles_of(row / 128 * 128, N, kl, causal, key_tile);
    const size_t rg = (size_t)bh * N + row;
    uint2* dst = reinterpret_cast<uint2*>(o + rg * hd) + c4;
    if (n_t == 0) {
#pragma unroll
      for (int i = 0; i < VPT; ++i)
        if (4 * (c4 + TPR * i) < hd) dst[TPR * i] = make_uint2(0u, 0u);
      if (c4 == 0) lse[rg] = -INFINITY;
      continue;
    }
    // one pass over the splits holding keys of this row: split s covers key
    // tiles [j0, j1) = [s*n_blk/n_splits, (s+1)*n_blk/n_splits) and holds
    // keys of the row iff j0 < j1 and j0 < n_t.  The running merge is the
    // two-block rule applied split after split (max m, sum of e^(L_s - m),
    // output weighted alike), rescaled when m grows.
    float m = -INFINITY, sum = 0.0f;
    float4 acc[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int j0 = 0;
#pragma unroll 2
    for (int s = 0; s < n_splits && j0 < n_t; ++s) {
      const int j1 = (s + 1) * n_blk / n_splits;
      if (j1 > j0) {
        const float ls = lse_part[s * stride + rg];
        const float4* src = reinterpret_cast<const float4*>(o_part + (s * stride + rg) * hd) + c4;
        float4 v[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i)
          v[i] = 4 * (c4 + TPR * i) < hd ? src[TPR * i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const float mn = fmaxf(m, ls);
        const float r = expf(m - mn);  // 0 for the first split (m = -inf)
        const float w = expf(ls - mn);
        sum = fmaf(sum, r, w);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          acc[i].x = fmaf(acc[i].x, r, w * v[i].x);
          acc[i].y = fmaf(acc[i].y, r, w * v[i].y);
          acc[i].z = fmaf(acc[i].z, r, w * v[i].z);
          acc[i].w = fmaf(acc[i].w, r, w * v[i].w);
        }
        m = mn;
      }
      j0 = j1;
    }
    const float inv = 1.0f / sum;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
      if (4 * (c4 + TPR * i) < hd)
        dst[TPR * i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    if (c4 == 0) lse[rg] = m + logf(sum);
  }
}

}  // namespace fattn
