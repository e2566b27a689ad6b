// Causal linear attention forward (the second workload), sm_103a.
//
// What it computes ("Linear Attention CUDA kernel" page: the feature map
// phi(x) = elu(x) + 1, the key-length mask of CausalLinearAttention.forward,
// its causal dot product and its normaliser), per (b, h) and row i:
//     qt_i = phi(q_i),  kt_j = phi(k_j) for j < key_len[b] else 0,
//     out_i = (sum_{j <= i} (qt_i . kt_j) v_j) / (qt_i . sum_{j <= i} kt_j + eps).
// The page's kernels walk the sequence one row at a time keeping the state
// S = sum kt_j v_j^T; here the rows are cut into chunks of LIN_C so that all
// chunks of all heads run at once:
//   1. fattn_linear_state_kernel: per chunk, its share of the state,
//      sum over its rows of kt_j v_j^T (E x M) and of kt_j (E);
//   2. fattn_linear_scan_kernel: per head, the exclusive prefix of those
//      shares over the chunks (the state each chunk starts from), in place;
//   3. fattn_linear_output_kernel: per chunk, the rows' numerators
//      tril(Qt Kt^T) V + Qt S_prefix and denominators
//      rowsum(tril(Qt Kt^T)) + Qt . s_prefix + eps.
// The same sums as the page's recurrence, regrouped (exact up to rounding).
// fp32 throughout, as the page's float kernels, on the CUDA cores: the
// chunk products are small (64 x 64 x E) and the data move is what bounds
// the problem at the feature sizes the page dispatches on.
#pragma once

#include <cstdint>

namespace fattn {

constexpr int LIN_C = 64;  // rows per chunk
constexpr int LIN_THREADS = 256;

struct LinParams {
  const float* q;  // [B*H, N, E]
  const float* k;  // [B*H, N, E]
  const float* v;  // [B*H, N, M]
  float* out;      // [B*H, N, M]
  const int32_t* key_len;  // [B] or nullptr
  float* state;  // [B*H, n_chunks, E*M]: chunk shares, then their exclusive prefix
  float* ksum;   // [B*H, n_chunks, E]: the same for the key sums
  int B, H, N, E, M, n_chunks;
  float eps;
};

__device__ __forceinline__ float lin_phi(float x) { return x > 0.0f ? x + 1.0f : expf(x); }  // elu(x) + 1

__device__ __forceinline__ int lin_key_len(const LinParams& p, int bh) {
  int kl = p.key_len ? p.key_len[bh / p.H] : p.N;
  return kl < 0 ? 0 : (kl > p.N ? p.N : kl);
}

// Shared-memory layout of the output kernel, in floats (every array starts
// on a 16-byte boundary): Qt, Kt [C][E+1] (padded rows), V [C][M], the
// prefix state [E][M] and key sum [E], A = tril(Qt Kt^T) [C][C+1], den [C].
struct LinSmem {
  int qt, kt, v, ps, pks, a, den, total;
  __host__ __device__ LinSmem(int E, int M) {
    auto up4 = [](int x) { return (x + 3) / 4 * 4; };
    qt = 0;
    kt = qt + up4(LIN_C * (E + 1));
    v = kt + up4(LIN_C * (E + 1));
    ps = v + up4(LIN_C * M);
    pks = ps + up4(E * M);
    a = pks + up4(E);
    den = a + up4(LIN_C * (LIN_C + 1));
    total = den + up4(LIN_C);
  }
};

// Loads a chunk's mapped keys (masked rows and rows past N as 0) into
// kt[C][E+1] and its values (rows past N as 0) into vs[C][M].
__device__ __forceinline__ void lin_load_kv(const LinParams& p, int bh, int r0, int kl, float* kt, float* vs) {
  const int E = p.E, M = p.M;
  for (int idx = threadIdx.x; idx < LIN_C * E; idx += LIN_THREADS) {
    const int r = idx / E, e = idx % E, row = r0 + r;
    kt[r * (E + 1) + e] = row < kl ? lin_phi(p.k[((size_t)bh * p.N + row) * E + e]) : 0.0f;
  }
  for (int idx = threadIdx.x; idx < LIN_C * M; idx += LIN_THREADS) {
    const int r = idx / M, m = idx % M, row = r0 + r;
    vs[r * M + m] = row < p.N ? p.v[((size_t)bh * p.N + row) * M + m] : 0.0f;
  }
}

__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_state_kernel(const LinParams p) {
  extern __shared__ float4 lin_smem4[];
  float* sm = reinterpret_cast<float*>(lin_smem4);
  const int E = p.E, M = p.M;
  const int c = (int)(blockIdx.x % (unsigned)p.n_chunks);
  const int bh = (int)(blockIdx.x / (unsigned)p.n_chunks);
  const int r0 = c * LIN_C;
  float* kt = sm;
  float* vs = sm + (LIN_C * (E + 1) + 3) / 4 * 4;
  lin_load_kv(p, bh, r0, lin_key_len(p, bh), kt, vs);
  __syncthreads();
  float* st = p.state + ((size_t)bh * p.n_chunks + c) * (size_t)E * M;
  // four value columns per item: float4 loads of V rows
  const int m4s = M / 4;
  for (int idx = threadIdx.x; idx < E * m4s; idx += LIN_THREADS) {
    const int e = idx / m4s, m4 = idx % m4s;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
    for (int r = 0; r < LIN_C; ++r) {
      const float kv = kt[r * (E + 1) + e];
      const float4 vv = reinterpret_cast<const float4*>(vs + r * M)[m4];
      acc.x = fmaf(kv, vv.x, acc.x);
      acc.y = fmaf(kv, vv.y, acc.y);
      acc.z = fmaf(kv, vv.z, acc.z);
      acc.w = fmaf(kv, vv.w, acc.w);
    }
    reinterpret_cast<float4*>(st + (size_t)e * M)[m4] = acc;
  }
  for (int e = threadIdx.x; e < E; e += LIN_THREADS) {
    float s = 0.0f;
    for (int r = 0; r < LIN_C; ++r) s += kt[r * (E + 1) + e];
    p.ksum[((size_t)bh * p.n_chunks + c) * E + e] = s;
  }
}

// Exclusive prefix over the chunks of one head, in place: one thread per
// element of the state (and of the key sum), walking the chunks in order.
__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_scan_kernel(const LinParams p, int blocks_per_head) {
  const int E = p.E, M = p.M;
  const int bh = (int)(blockIdx.x / (unsigned)blocks_per_head);
  const int idx = (int)(blockIdx.x % (unsigned)blocks_per_head) * LIN_THREADS + threadIdx.x;
  if (idx >= E * M + E) return;
  float* base;
  size_t stride;
  if (idx < E * M) {
    base = p.state + (size_t)bh * p.n_chunks * (size_t)E * M + idx;
    stride = (size_t)E * M;
  } else {
    base = p.ksum + (size_t)bh * p.n_chunks * (size_t)E + (idx - E * M);
    stride = (size_t)E;
  }
  float run = 0.0f;
#pragma unroll 8
  for (int c = 0; c < p.n_chunks; ++c) {
    const float share = base[c * stride];
    base[c * stride] = run;
    run += share;
  }
}

__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_output_kernel(const LinParams p) {
  extern __shared__ float4 lin_smem4[];
  float* sm = reinterpret_cast<float*>(lin_smem4);
  const int E = p.E, M = p.M;
  const LinSmem L(E, M);
  const int c = (int)(blockIdx.x % (unsigned)p.n_chunks);
  const int bh = (int)(blockIdx.x / (unsigned)p.n_chunks);
  const int r0 = c * LIN_C;
  float *qt = sm + L.qt, *kt = sm + L.kt, *vs = sm + L.v, *ps = sm + L.ps, *pks = sm + L.pks, *a = sm + L.a,
        *den = sm + L.den;
  lin_load_kv(p, bh, r0, lin_key_len(p, bh), kt, vs);
  for (int idx = threadIdx.x; idx < LIN_C * E; idx += LIN_THREADS) {
    const int r = idx / E, e = idx % E, row = r0 + r;
    qt[r * (E + 1) + e] = row < p.N ? lin_phi(p.q[((size_t)bh * p.N + row) * E + e]) : 0.0f;
  }
  const float* st = p.state + ((size_t)bh * p.n_chunks + c) * (size_t)E * M;
  for (int idx = threadIdx.x; idx < E * M / 4; idx += LIN_THREADS)
    reinterpret_cast<float4*>(ps)[idx] = reinterpret_cast<const float4*>(st)[idx];
  for (int e = threadIdx.x; e < E; e += LIN_THREADS) pks[e] = p.ksum[((size_t)bh * p.n_chunks + c) * E + e];
  __syncthreads();
  // A = tril(Qt Kt^T): the chunk's own rows j <= i
  for (int idx = threadIdx.x; idx < LIN_C * LIN_C; idx += LIN_THREADS) {
    const int i = idx / LIN_C, j = idx % LIN_C;
    float s = 0.0f;
    if (j <= i) {
#pragma unroll 4
      for (int e = 0; e < E; ++e) s = fmaf(qt[i * (E + 1) + e], kt[j * (E + 1) + e], s);
    }
    a[i * (LIN_C + 1) + j] = s;
  }
  __syncthreads();
  // denominators: the chunk's own keys (row sums of A) and those before it
  for (int i = threadIdx.x; i < LIN_C; i += LIN_THREADS) {
    float d = p.eps;
    for (int j = 0; j <= i; ++j) d += a[i * (LIN_C + 1) + j];
    for (int e = 0; e < E; ++e) d = fmaf(qt[i * (E + 1) + e], pks[e], d);
    den[i] = d;
  }
  __syncthreads();
  // numerators, four value columns per item, divided by the row's denominator
  const int m4s = M / 4;
  for (int idx = threadIdx.x; idx < LIN_C * m4s; idx += LIN_THREADS) {
    const int i = idx / m4s, m4 = idx % m4s, row = r0 + i;
    if (row >= p.N) continue;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j = 0; j <= i; ++j) {
      const float w = a[i * (LIN_C + 1) + j];
      const float4 vv = reinterpret_cast<const float4*>(vs + j * M)[m4];
      acc.x = fmaf(w, vv.x, acc.x);
      acc.y = fmaf(w, vv.y, acc.y);
      acc.z = fmaf(w, vv.z, acc.z);
      acc.w = fmaf(w, vv.w, acc.w);
    }
#pragma unroll 4
    for (int e = 0; e < E; ++e) {
      const float w = qt[i * (E + 1) + e];
      const float4 sv = reinterpret_cast<const float4*>(ps + e * M)[m4];
      acc.x = fmaf(w, sv.x, acc.x);
      acc.y = fmaf(w, sv.y, acc.y);
      acc.z = fmaf(w, sv.z, acc.z);
      acc.w = fmaf(w, sv.w, acc.w);
    }
    const float inv = 1.0f / den[i];
    float* o = p.out + ((size_t)bh * p.N + row) * M + 4 * m4;
    o[0] = acc.x * inv;
    o[1] = acc.y * inv;
    o[2] = acc.z * inv;
    o[3] = acc.w * inv;
  }
}

}  // namespace fattn
