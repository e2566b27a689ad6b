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
//      shares over the chunks (the state each chunk starts from);
//   3. fattn_linear_output_kernel: per chunk, the rows' numerators
//      tril(Qt Kt^T) V + Qt S_prefix and denominators
//      rowsum(tril(Qt Kt^T)) + Qt . s_prefix + eps.
// The same sums as the page's recurrence, regrouped (exact up to rounding).
// The state and output kernels are compiled for feature sizes E = M = 64 as
// constants (every shared-memory offset an immediate) and for any other
// sizes at run time (template arguments 0).
// fp32 throughout, as the page's float kernels, on the CUDA cores: the
// chunk products are small (64 x 64 x E at the feature sizes the page
// dispatches on), and rounding the operands to tf32 for the tensor cores
// would cost more accuracy than the fp32 sums.  The state and output kernels
// are bound by instruction issue (the FFMA products, their shared-memory
// operand loads and the transform of phi), not by HBM.
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
  float* state;   // [B*H, n_chunks, E*M]: each chunk's share of the state
  float* ksum;    // [B*H, n_chunks, E]: each chunk's share of the key sum
  float* pstate;  // [B*H, n_chunks, E*M]: the exclusive prefix of the shares
  float* pksum;   // [B*H, n_chunks, E]
  int B, H, N, E, M, n_chunks;
  float eps;
};

// elu(x) + 1, branch-free: max(x, 0) + 2^(min(x, 0) log2 e) is x + 1 for
// x > 0 (2^0 = 1) and e^x otherwise; the fast exponential's error (a few ulp
// on x <= 0) is far below the fp32 summation error of the sums it feeds.  (A
// select between x + 1 and e^x compiled to a divergent branch per element.)
__device__ __forceinline__ float lin_phi(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fminf(x, 0.0f) * 1.4426950408889634f));
  return fmaxf(x, 0.0f) + e;
}

__device__ __forceinline__ int lin_key_len(const LinParams& p, int bh) {
  int kl = p.key_len ? p.key_len[bh / p.H] : p.N;
  return kl < 0 ? 0 : (kl > p.N ? p.N : kl);
}

// The transposed [E][LIN_C] arrays (phi(Q)^T, phi(K)^T) and A^T [LIN_C][LIN_C]
// are stored unpadded, each row's sixteen float4 groups permuted: group g of
// row e sits in slot g ^ ((e >> 2) & 15).  A warp that writes four rows r of
// eight consecutive e4 (the load below) and a warp that writes A^T rows of
// many (ti, tj) pairs then spread over all 32 banks, while every reader still
// gets whole float4 groups.
__device__ __forceinline__ int lin_slot(int e, int g) { return g ^ ((e >> 2) & 15); }
__device__ __forceinline__ int lin_at(int e, int r) { return e * LIN_C + 4 * lin_slot(e, r >> 2) + (r & 3); }

// Shared-memory layout of the output kernel, in floats (every array starts
// on a 16-byte boundary): phi(Q)^T [E][C]; phi(K)^T [E][C], whose space A^T =
// tril(Qt Kt^T)^T [C][C] takes over once A is formed; X, which holds the
// prefix state [E][M] for the Qt S_prefix products and then V [C][M] for the
// A V products; the prefix key sum [E]; 1 / den for each row [C].
struct LinSmem {
  int qt, kt, at, x, pks, den, total;
  __host__ __device__ LinSmem(int E, int M) {
    auto up4 = [](int x) { return (x + 3) / 4 * 4; };
    auto mx = [](int a, int b) { return a > b ? a : b; };
    qt = 0;
    kt = at = qt + E * LIN_C;
    x = kt + mx(E, LIN_C) * LIN_C;
    pks = x + up4(mx(E, LIN_C) * M);
    den = pks + up4(E);
    total = den + LIN_C;
  }
};

// 16-byte asynchronous copy global -> shared (zero-filled when !valid; `src`
// must still be a valid address), and the wait for all of this thread's.
__device__ __forceinline__ void lin_cp16(void* dst, const void* src, bool valid) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void lin_cp_wait() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// phi(x) of a chunk's rows (masked rows and rows past N as 0), stored
// transposed and permuted: element (e, r) at lin_at(e, r).  Each warp reads
// four rows, eight float4 (128 bytes) of each.  NA arrays at once (phi(Q)
// and phi(K) in the output kernel), each thread keeping 4 * NA loads in
// flight before any is used.
struct LinTSrc {
  const float* src;
  int lim;  // rows at or past lim read as 0
  float* dst;
};
template <int NA>
__device__ __forceinline__ void lin_load_t(const LinTSrc (&a)[NA], int bh, int N, int E, int r0) {
  const int e4s = E / 4;
  const int n = (LIN_C / 4) * ((e4s + 7) / 8) * 32;  // (row quads) x (e4 octets) x lanes
  for (int base = 0; base < n; base += 4 * LIN_THREADS) {
    float4 x[NA][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * LIN_THREADS + threadIdx.x, lane = idx & 31, rest = idx >> 5;
      const int r = 4 * (rest % (LIN_C / 4)) + (lane & 3), e4 = 8 * (rest / (LIN_C / 4)) + (lane >> 2);
      const int row = r0 + r;
#pragma unroll
      for (int t = 0; t < NA; ++t)
        x[t][u] = (idx < n && e4 < e4s && row < a[t].lim)
                      ? reinterpret_cast<const float4*>(a[t].src + ((size_t)bh * N + row) * E)[e4]
                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * LIN_THREADS + threadIdx.x, lane = idx & 31, rest = idx >> 5;
      const int r = 4 * (rest % (LIN_C / 4)) + (lane & 3), e4 = 8 * (rest / (LIN_C / 4)) + (lane >> 2);
      if (idx >= n || e4 >= e4s) continue;
#pragma unroll
      for (int t = 0; t < NA; ++t) {
        const bool live = r0 + r < a[t].lim;
        float* dst = a[t].dst;
        dst[lin_at(4 * e4 + 0, r)] = live ? lin_phi(x[t][u].x) : 0.0f;
        dst[lin_at(4 * e4 + 1, r)] = live ? lin_phi(x[t][u].y) : 0.0f;
        dst[lin_at(4 * e4 + 2, r)] = live ? lin_phi(x[t][u].z) : 0.0f;
        dst[lin_at(4 * e4 + 3, r)] = live ? lin_phi(x[t][u].w) : 0.0f;
      }
    }
  }
}

// dst[0, n_total) <- src[0, n_src) then zeros, as 16-byte asynchronous
// copies (completed by lin_cp_wait).
__device__ __forceinline__ void lin_copy4_async(float4* dst, const float4* src, int n_src, int n_total) {
  for (int idx = threadIdx.x; idx < n_total; idx += LIN_THREADS)
    lin_cp16(dst + idx, idx < n_src ? src + idx : src, idx < n_src);
}

// A chunk's value rows (rows past N as 0), row-major [C][M]: the chunk's rows
// are contiguous in memory.
__device__ __forceinline__ void lin_load_v_async(const LinParams& p, int M, int bh, int r0, float* vs) {
  const int rows = min(LIN_C, p.N - r0);
  lin_copy4_async(reinterpret_cast<float4*>(vs),
                  reinterpret_cast<const float4*>(p.v + ((size_t)bh * p.N + r0) * M), rows * M / 4, LIN_C * M / 4);
}

__device__ __forceinline__ void fma4x4(float (&acc)[4][4], const float4 a, const float4 b) {
  const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(av[u], bv[w], acc[u][w]);
}

// 1. A chunk's share of the state: S_c = phi(K_c)^T V_c (E x M, in 4 x 4
//    register tiles, four rows of the chunk per step: four float4 of phi(K)^T
//    and four of V feed 64 FMAs) and s_c = column sums of phi(K_c).  V is
//    copied asynchronously while phi(K) is loaded, so one memory latency
//    precedes the products.
template <int EC, int MC>
__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_state_kernel(const LinParams p) {
  extern __shared__ float4 lin_smem4[];
  float* sm = reinterpret_cast<float*>(lin_smem4);
  const int E = EC ? EC : p.E, M = MC ? MC : p.M;
  const int c = (int)(blockIdx.x % (unsigned)p.n_chunks);
  const int bh = (int)(blockIdx.x / (unsigned)p.n_chunks);
  const int r0 = c * LIN_C;
  float* kt = sm;                 // [E][C], permuted
  float* vs = sm + E * LIN_C;     // [C][M]
  lin_load_v_async(p, M, bh, r0, vs);  // in flight while phi(K) is formed
  const LinTSrc ks[1] = {{p.k, lin_key_len(p, bh), kt}};
  lin_load_t(ks, bh, p.N, E, r0);
  lin_cp_wait();
  __syncthreads();
  float* st = p.state + ((size_t)bh * p.n_chunks + c) * (size_t)E * M;
  const int e4s = E / 4, m4s = M / 4;
  for (int item = threadIdx.x; item < e4s * m4s; item += LIN_THREADS) {
    const int e4 = item / m4s, m4 = item % m4s;
    const float4* k4 = reinterpret_cast<const float4*>(kt + 4 * e4 * LIN_C);  // rows 4e4.. share one permutation
    float acc[4][4] = {};
#pragma unroll 4
    for (int g = 0; g < LIN_C / 4; ++g) {
      const int sl = lin_slot(4 * e4, g);
      const float4 k0 = k4[sl], k1 = k4[LIN_C / 4 + sl], k2 = k4[LIN_C / 2 + sl], k3 = k4[3 * LIN_C / 4 + sl];
      const float4* v4 = reinterpret_cast<const float4*>(vs + 4 * g * M) + m4;
      fma4x4(acc, make_float4(k0.x, k1.x, k2.x, k3.x), v4[0]);
      fma4x4(acc, make_float4(k0.y, k1.y, k2.y, k3.y), v4[m4s]);
      fma4x4(acc, make_float4(k0.z, k1.z, k2.z, k3.z), v4[2 * m4s]);
      fma4x4(acc, make_float4(k0.w, k1.w, k2.w, k3.w), v4[3 * m4s]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      reinterpret_cast<float4*>(st + (size_t)(4 * e4 + u) * M)[m4] =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
  }
  for (int e = threadIdx.x; e < E; e += LIN_THREADS) {
    float s = 0.0f;
    const float4* row = reinterpret_cast<const float4*>(kt + e * LIN_C);
#pragma unroll 4
    for (int g = 0; g < LIN_C / 4; ++g) {
      const float4 x = row[lin_slot(e, g)];
      s += (x.x + x.y) + (x.z + x.w);
    }
    p.ksum[((size_t)bh * p.n_chunks + c) * E + e] = s;
  }
}

// 2. Exclusive prefix over the chunks of one head: one thread per element of
//    the state (and of the key sum), walking the chunks in order.  Shares and
//    prefixes are separate arrays, so the loads run ahead of the stores.
__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_scan_kernel(const LinParams p, int blocks_per_head) {
  const int E = p.E, M = p.M;
  const int bh = (int)(blockIdx.x / (unsigned)blocks_per_head);
  const int idx = (int)(blockIdx.x % (unsigned)blocks_per_head) * LIN_THREADS + threadIdx.x;
  if (idx >= E * M + E) return;
  const float* __restrict__ in;
  float* __restrict__ out;
  size_t stride;
  if (idx < E * M) {
    in = p.state + (size_t)bh * p.n_chunks * (size_t)E * M + idx;
    out = p.pstate + (size_t)bh * p.n_chunks * (size_t)E * M + idx;
    stride = (size_t)E * M;
  } else {
    in = p.ksum + (size_t)bh * p.n_chunks * (size_t)E + (idx - E * M);
    out = p.pksum + (size_t)bh * p.n_chunks * (size_t)E + (idx - E * M);
    stride = (size_t)E;
  }
  float run = 0.0f;
  int c = 0;
  for (; c + 16 <= p.n_chunks; c += 16) {  // sixteen loads in flight
    float sh[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) sh[u] = __ldg(in + (size_t)(c + u) * stride);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      out[(size_t)(c + u) * stride] = run;
      run += sh[u];
    }
  }
  for (; c < p.n_chunks; ++c) {
    const float share = __ldg(in + (size_t)c * stride);
    out[(size_t)c * stride] = run;
    run += share;
  }
}

// 3. A chunk's outputs: numerators Qt S_prefix + tril(Qt Kt^T) V and
//    denominators rowsum(tril(Qt Kt^T)) + Qt . s_prefix + eps, all products
//    in 4 x 4 register tiles fed by float4 shared-memory loads.  The prefix
//    state and V take turns in one buffer (48.5 KB of shared memory at
//    E = M = 64, four CTAs per SM).
template <int EC, int MC>
__global__ void __launch_bounds__(LIN_THREADS) fattn_linear_output_kernel(const LinParams p) {
  extern __shared__ float4 lin_smem4[];
  float* sm = reinterpret_cast<float*>(lin_smem4);
  const int E = EC ? EC : p.E, M = MC ? MC : p.M;
  const LinSmem L(E, M);
  const int c = (int)(blockIdx.x % (unsigned)p.n_chunks);
  const int bh = (int)(blockIdx.x / (unsigned)p.n_chunks);
  const int r0 = c * LIN_C;
  float *qt = sm + L.qt, *kt = sm + L.kt, *at = sm + L.at, *xs = sm + L.x, *pks = sm + L.pks, *den = sm + L.den;
  const float* st = p.pstate + ((size_t)bh * p.n_chunks + c) * (size_t)E * M;
  lin_copy4_async(reinterpret_cast<float4*>(xs), reinterpret_cast<const float4*>(st), E * M / 4, E * M / 4);
  for (int e = threadIdx.x; e < E; e += LIN_THREADS) pks[e] = p.pksum[((size_t)bh * p.n_chunks + c) * E + e];
  {
    const LinTSrc qk[2] = {{p.q, p.N, qt}, {p.k, lin_key_len(p, bh), kt}};
    lin_load_t(qk, bh, p.N, E, r0);
  }
  lin_cp_wait();
  __syncthreads();
  // A = tril(Qt Kt^T): only its 136 4 x 4 tiles on or below the diagonal,
  // one per thread (tile t -> row ti, column tj <= ti); then, once every
  // thread is done with phi(K)^T, stored transposed (A^T row j = column j of
  // A) over it
  {
    constexpr int NT = LIN_C / 4, N_TRI = NT * (NT + 1) / 2;
    static_assert(N_TRI <= LIN_THREADS, "one tile per thread");
    int ti = 0, tj = threadIdx.x;
    while (tj > ti) tj -= ++ti;  // tj - ti(ti+1)/2 after the loop
    float acc[4][4] = {};
    if (threadIdx.x < N_TRI) {
      // rows 4g..4g+3 of phi(Q)^T and phi(K)^T share one permutation
#pragma unroll 4
      for (int g = 0; g < E / 4; ++g) {
        const float4* q4 = reinterpret_cast<const float4*>(qt + 4 * g * LIN_C) + lin_slot(4 * g, ti);
        const float4* k4 = reinterpret_cast<const float4*>(kt + 4 * g * LIN_C) + lin_slot(4 * g, tj);
#pragma unroll
        for (int u = 0; u < 4; ++u) fma4x4(acc, q4[u * (LIN_C / 4)], k4[u * (LIN_C / 4)]);
      }
    }
    __syncthreads();
    if (threadIdx.x < N_TRI) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int j = 4 * tj + w;
        float4 col;
        col.x = j <= 4 * ti + 0 ? acc[0][w] : 0.0f;
        col.y = j <= 4 * ti + 1 ? acc[1][w] : 0.0f;
        col.z = j <= 4 * ti + 2 ? acc[2][w] : 0.0f;
        col.w = j <= 4 * ti + 3 ? acc[3][w] : 0.0f;
        reinterpret_cast<float4*>(at + j * LIN_C)[lin_slot(j, ti)] = col;
      }
    }
  }
  __syncthreads();
  // denominators: the chunk's own keys (row sums of A: A^T rows j <= i, in
  // quads whose tile was stored; its entries above the diagonal are zero) and
  // those before it (qt_i . s_prefix); four adjacent lanes per row, lane
  // `part` taking A^T row quads 4 part .. 4 part + 3 and a quarter of the
  // feature quads
  {
    static_assert(LIN_THREADS == 4 * LIN_C, "four threads per row");
    const int i = threadIdx.x / 4, part = threadIdx.x % 4;
    float d = 0.0f;
#pragma unroll
    for (int k = 0; k < LIN_C / 16; ++k) {
      const int jq = (LIN_C / 16) * part + k;
      if (jq > (i >> 2)) break;
      const float* a = at + 4 * jq * LIN_C + 4 * lin_slot(4 * jq, i >> 2) + (i & 3);
      d += (a[0] + a[LIN_C]) + (a[2 * LIN_C] + a[3 * LIN_C]);
    }
    const int G = E / 4;
    for (int g = part * G / 4; g < (part + 1) * G / 4; ++g) {
      const float* q = qt + 4 * g * LIN_C + 4 * lin_slot(4 * g, i >> 2) + (i & 3);
      const float4 s4 = reinterpret_cast<const float4*>(pks)[g];
      d = fmaf(q[0], s4.x, d);
      d = fmaf(q[LIN_C], s4.y, d);
      d = fmaf(q[2 * LIN_C], s4.z, d);
      d = fmaf(q[3 * LIN_C], s4.w, d);
    }
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    if (part == 0) den[i] = 1.0f / (d + p.eps);  // kept as its reciprocal
  }
  // numerators in 4 x 4 tiles (rows 4ti.., value columns 4tc..), at most
  // two per thread (M <= 128): Qt S_prefix first, then, with V over the
  // prefix state, tril(Qt Kt^T) V; times 1 / den
  constexpr int MAX_ITEMS = (LIN_C / 4) * (128 / 4) / LIN_THREADS;
  const int m4s = M / 4, n_items = (LIN_C / 4) * m4s;
  float acc[MAX_ITEMS][4][4] = {};
#pragma unroll
  for (int s = 0; s < MAX_ITEMS; ++s) {
    const int item = threadIdx.x + s * LIN_THREADS;
    if (item < n_items) {
      const int ti = item / m4s, tc = item % m4s;
#pragma unroll 4
      for (int g = 0; g < E / 4; ++g) {
        const float4* q4 = reinterpret_cast<const float4*>(qt + 4 * g * LIN_C) + lin_slot(4 * g, ti);
        const float4* s4 = reinterpret_cast<const float4*>(xs + 4 * g * M) + tc;
#pragma unroll
        for (int u = 0; u < 4; ++u) fma4x4(acc[s], q4[u * (LIN_C / 4)], s4[u * m4s]);
      }
    }
  }
  __syncthreads();
  lin_load_v_async(p, M, bh, r0, xs);
  lin_cp_wait();
  __syncthreads();
#pragma unroll
  for (int s = 0; s < MAX_ITEMS; ++s) {
    const int item = threadIdx.x + s * LIN_THREADS;
    if (item < n_items) {
      const int ti = item / m4s, tc = item % m4s;
      for (int jq = 0; jq <= ti; ++jq) {  // A is zero past the tile's last row
        const float4* a4 = reinterpret_cast<const float4*>(at + 4 * jq * LIN_C) + lin_slot(4 * jq, ti);
        const float4* v4 = reinterpret_cast<const float4*>(xs + 4 * jq * M) + tc;
#pragma unroll
        for (int u = 0; u < 4; ++u) fma4x4(acc[s], a4[u * (LIN_C / 4)], v4[u * m4s]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = r0 + 4 * ti + u;
        if (row >= p.N) continue;
        const float inv = den[4 * ti + u];
        reinterpret_cast<float4*>(p.out + ((size_t)bh * p.N + row) * M)[tc] =
            make_float4(acc[s][u][0] * inv, acc[s][u][1] * inv, acc[s][u][2] * inv, acc[s][u][3] * inv);
      }
    }
  }
}

}  // namespace fattn
