// V pre-pass: stores every 128-row tile of V in the type its P V product
// will use.
//
// The attention kernel rounds the probabilities P once, to the operand type
// of the P V tensor-core product, and tcgen05 kind::f16 takes A and B of the
// same type.  fp16 keeps 11 significant bits of P against bf16's 8, which is
// what keeps the bf16 output within the stated error on peaky softmax rows.
// So each tile whose largest |v| lies in [2^-8, 65504] (fp16 then holds every
// element to fp16 precision without overflow) is converted to fp16; any
// other tile (huge or tiny values, inf) keeps its bf16 bits and its P is
// rounded to bf16.  The per-tile choice is written to `mode`.
//
// HBM-bound: one read of V, one write of the same number of bytes.
#pragma once

#include <cstdint>

#include "fattn_kernel.cuh"

namespace fattn {

constexpr int PREPASS_THREADS = 256;
// threads of one block: 8 vectors of 16 bytes per thread at every head-dim bucket
template <int D>
__host__ __device__ constexpr int prepass_threads() { return D > 128 ? 512 : PREPASS_THREADS; }

// FULL: rows are exactly D elements long (hd == D), with the row length a
// compile-time constant; otherwise hd (a multiple of 8, < D).
template <int D, bool FULL>
__global__ void __launch_bounds__(prepass_threads<D>())
    fattn_v_prepass_kernel(const uint4* __restrict__ v, uint4* __restrict__ v16, uint8_t* __restrict__ mode, int N,
                           int hd_arg, int n_tiles, int mode_stride) {
  pdl_launch_dependents();  // the attention kernel may start its set-up now (it waits before reading V)
  const int hd = FULL ? D : hd_arg;
  constexpr int VEC = 8;                                  // bf16 per 16-byte vector
  constexpr int T = prepass_threads<D>();
  constexpr int PER = BN * D / VEC / T;  // vectors per thread (rows of up to D elements)
  const long long tile_id = blockIdx.x;
  const int tile = (int)(tile_id % n_tiles);
  const long long bh = tile_id / n_tiles;
  const int row0 = tile * BN;
  const int rows = min(BN, N - row0);
  const int nvec = rows * hd / VEC;  // rows are hd (a multiple of 8) elements long
  const size_t base = ((size_t)bh * (size_t)N + (size_t)row0) * (size_t)(hd / VEC);

  uint4 buf[PER];
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = threadIdx.x + i * T;
    if (idx < nvec) {
      buf[i] = __ldg(v + base + idx);
      const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mx = fmaxf(mx, fabsf(__uint_as_float(w[k] << 16)));
        mx = fmaxf(mx, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
      }
    }
  }
  __shared__ float warp_max[T / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (threadIdx.x % 32 == 0) warp_max[threadIdx.x / 32] = mx;
  __syncthreads();
  mx = warp_max[0];
#pragma unroll
  for (int i = 1; i < T / 32; ++i) mx = fmaxf(mx, warp_max[i]);
  const bool to_f16 = mx >= 0.00390625f && mx <= 65504.0f;

#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = threadIdx.x + i * T;
    if (idx < nvec) {
      uint4 o = buf[i];
      if (to_f16) {
        o.x = pack_f16x2(__uint_as_float(buf[i].x << 16), __uint_as_float(buf[i].x & 0xFFFF0000u));
        o.y = pack_f16x2(__uint_as_float(buf[i].y << 16), __uint_as_float(buf[i].y & 0xFFFF0000u));
        o.z = pack_f16x2(__uint_as_float(buf[i].z << 16), __uint_as_float(buf[i].z & 0xFFFF0000u));
        o.w = pack_f16x2(__uint_as_float(buf[i].w << 16), __uint_as_float(buf[i].w & 0xFFFF0000u));
      }
      v16[base + idx] = o;
    }
  }
  if (threadIdx.x == 0) mode[bh * mode_stride + tile] = to_f16 ? VMODE_F16 : VMODE_BF16;
}

}  // namespace fattn
