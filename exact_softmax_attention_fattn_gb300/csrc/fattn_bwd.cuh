// Exact softmax attention backward, sm_103a.
//
// What it computes ("understand-flashattention", section "Attention forward
// and backward formulas", backward pass steps 1-5, with P recomputed from the
// saved logsumexp as in "recomputing P needs logsumexp"):
//     P  = exp(S - LSE) with S = scale * Q K^T, masked entries 0
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D) with D_i = sum_k dP_ik P_ik,
//     dQ = scale * dS K,  dK = scale * dS^T Q.
// D_i is computed as rowsum(dO_i * O_i), which equals sum_k dP_ik P_ik because
// O_i = sum_k P_ik V_k.
//
// How (GB300):
//   * fattn_bwd_prep_kernel: D per row and -LSE * log2(e), both written to
//     buffers whose rows are padded to a multiple of 128, so every per-tile
//     copy of them is a 512-byte, 16-byte-aligned bulk copy for any N.
//   * fattn_bwd_dkdv_kernel: one CTA per (batch*head, 128-key tile j).  K_j
//     and V_j stay in shared memory; Q_i, dO_i, LSE_i, D_i stream through a
//     two-stage ring over the query tiles i that see tile j.  Per tile:
//     S^T = K_j Q_i^T and dP^T = V_j dO_i^T in tensor memory (lanes = keys);
//     eight warps in two groups (one thread per key in each; group g takes
//     the 64 query columns [64g, 64g + 64)) form P^T = 2^(S^T c - LSE2) and
//     dS^T = P^T (dP^T - D), each group storing its half as bf16 over the
//     first 32 of its own 64 fp32 columns, and the MMA issuer accumulates dV += P^T dO and
//     dK += dS^T Q in tensor memory (P^T, dS^T as the A operand from TMEM;
//     dO, Q as MN-major B).  TMEM: S^T, dP^T, dV, dK = 4 x 128 columns.
//   * fattn_bwd_dq_kernel: one CTA per (batch*head, 128-query tile i).  Q_i and
//     dO_i stay; K_j, V_j stream over the key tiles i sees.  S = Q_i K_j^T,
//     dP = dO_i V_j^T, then two groups of four warps (one thread per query
//     row in each, group g on the key columns [64g, 64g + 64)) form dS (bf16,
//     over S) and dQ += dS K_j accumulates in tensor memory.  Every
//     elementwise quantity has per-row or per-column constants only (LSE, D),
//     so the column split needs no exchange between the groups.
//   Splitting dQ from dK/dV costs two extra GEMMs per tile pair but needs no
//   atomics: tensor memory cannot hold S, dP, dV, dK and a dQ accumulator at
//   d = 128.  Every wait is bounded as in the forward kernel.
#pragma once

#include "fattn_kernel.cuh"

namespace fattn {

// warps 0-7 elementwise (two groups of four: group g takes the tile columns
// [64g, 64g + 64) of the same TMEM lanes), 8 TMA producer, 9 MMA issuer
constexpr int BWD_THREADS = 320;
constexpr int BWD_ELEM_WARPS = 8;
constexpr int BWD_PRODUCER_WARP = 8;
constexpr int BWD_MMA_WARP = 9;
constexpr int BWD_STAGES = 2;
constexpr int PREP_THREADS = 256;

struct BwdParams {
  const float* nlse2;   // [B*H, N_pad]: -LSE * log2(e) (+inf for an empty row; padding rows 0)
  const float* delta;   // [B*H, N_pad]: rowsum(dO * O) (padding rows 0)
  __nv_bfloat16* dq;
  float* dq_acc;        // fused backward only: [B*H, N_pad, 128] fp32 sums of dS K (zeroed before it)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* key_len;  // [B] or nullptr
  int* err;                // int[4]
  int B, H, N, N_pad;
  int hd;            // head dim of the tensors (a multiple of 8, <= D); columns past it are read as zeros
  float scale;       // softmax scale (natural units)
  float scale_log2;  // scale * log2(e)
  int causal;
  int n_tiles;  // ceil(N / 128)
  unsigned long long wait_limit_ns;
};

// ------------------------------------------------------------------ prep
// One row per D/8 threads (16-byte loads of O and dO; a row has hd <= D
// elements); rows past N (padding) get D = 0 and -LSE2 = 0.
// FULL: hd == D, the row length a compile-time constant.
template <int D, bool FULL>
__global__ void __launch_bounds__(PREP_THREADS)
    fattn_bwd_prep_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout, const float* __restrict__ lse,
                          float* __restrict__ nlse2, float* __restrict__ delta, int N, int N_pad, int hd_arg,
                          long long n_rows) {
  pdl_launch_dependents();  // the next kernel may start its set-up now (it waits before reading LSE2 and D)
  const int hd = FULL ? D : hd_arg;
  constexpr int TPR = D / 8;  // threads per row
  const long long r = ((long long)blockIdx.x * PREP_THREADS + threadIdx.x) / TPR;
  const int part = threadIdx.x % TPR;
  float acc = 0.0f;
  const long long bh = r / N_pad;
  const int i = (int)(r % N_pad);
  const bool live = r < n_rows && i < N;
  if (live && 8 * part < hd) {
    const size_t at = ((size_t)bh * (size_t)N + (size_t)i) * (size_t)(hd / 8) + (size_t)part;
    const uint4 a = __ldg(o + at), g = __ldg(dout + at);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      acc = fmaf(__uint_as_float(aw[x] << 16), __uint_as_float(gw[x] << 16), acc);
      acc = fmaf(__uint_as_float(aw[x] & 0xFFFF0000u), __uint_as_float(gw[x] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (r < n_rows && part == 0) {
    delta[r] = live ? acc : 0.0f;
    nlse2[r] = live ? lse[(size_t)bh * (size_t)N + (size_t)i] * -1.4426950408889634f : 0.0f;
  }
}

// ------------------------------------------------------------------ shared layout
// Both main kernels: two stationary 128-row tiles, a BWD_STAGES ring of two
// tiles each, and (dK/dV kernel) 512 bytes of -LSE2 + 512 of D per stage.
template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head-dim bucket 64 or 128");
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE_BYTES = 128u * D * 2u;
  static constexpr uint32_t FIX0_OFF = 0;                // K_j (dK/dV) or Q_i (dQ)
  static constexpr uint32_t FIX1_OFF = TILE_BYTES;       // V_j (dK/dV) or dO_i (dQ)
  static constexpr uint32_t RING_OFF = 2 * TILE_BYTES;   // per stage: two tiles
  static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr uint32_t ROWS_OFF = RING_OFF + BWD_STAGES * STAGE_BYTES;  // per stage: -LSE2[128], D[128]
  static constexpr uint32_t BAR_OFF = ROWS_OFF + BWD_STAGES * 1024u;
  // barrier ids
  static constexpr int B_FIX_FULL = 0;
  static constexpr int B_ST_FULL = 1;                    // [BWD_STAGES]
  static constexpr int B_ST_EMPTY = 1 + BWD_STAGES;      // [BWD_STAGES]
  static constexpr int B_S_FULL = 1 + 2 * BWD_STAGES;
  static constexpr int B_DP_FULL = B_S_FULL + 1;
  static constexpr int B_OPS_READY = B_S_FULL + 2;       // P^T stored (dK/dV kernel) or dS stored (dQ kernel)
  static constexpr int B_ACC_FULL = B_S_FULL + 3;
  static constexpr int B_DRAIN = B_S_FULL + 4;
  static constexpr int B_DS_READY = B_S_FULL + 5;        // dS^T stored (dK/dV kernel)
  static constexpr int NUM_BARS = B_DS_READY + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tmem base (4 B) + abort flag (4 B)
  // + slack for 1024-byte alignment; at least 120 KB so that only one CTA fits
  // an SM (each allocates all 512 TMEM columns)
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16 + 1024;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 120u * 1024u ? SMEM_USED : 120u * 1024u;
};
constexpr uint32_t BWD_TMEM_COLS = 512;
constexpr uint32_t BT_S = 0, BT_DP = 128, BT_ACC0 = 256;  // TMEM columns; accumulators from 256

// f(integral_constant<int, I>) for I = 0 .. N-1 over the MMAs of one GEMM
// (K steps of 16): descriptor offsets are compile-time immediates.
template <int D>
struct BwdMma {
  using C = BwdCfg<D>;
  static constexpr uint32_t IDESC_KMAJOR = idesc_f16kind(128, 128, true, false);  // both operands K-major
  static constexpr uint32_t IDESC_ACC = idesc_f16kind(128, D, true, true);        // B MN-major, N = D

  // D(128 x 128) = A(128 x D) B(128 x D)^T, both K-major tiles in shared
  // memory: D/16 MMAs behind one elect (64-column panels PANEL_BYTES apart).
  __device__ __forceinline__ static void ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
    mma_ss_batch<D / 16>(d_tmem, a_desc, b_desc, IDESC_KMAJOR, 0u);
  }
  // D(128 x D) (+)= A(128 x 128, bf16 in TMEM) B(128 x D, MN-major tile in shared memory).
  // A is packed by the two elementwise groups into TMEM columns [0, 32) (its
  // columns 0-63) and [64, 96) (its columns 64-127); eight MMAs of 16 rows
  // (two 1024-byte row groups of B) behind one elect.
  __device__ __forceinline__ static void ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    mma_ts_batch8_halves(d_tmem, a_tmem, b_desc, IDESC_ACC, accumulate);
  }
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// The elementwise group g's share of an accumulator's row: the 64-column
// blocks hcol = g, g + 2, ... (all of them at D = 128: one each; at D = 64
// group 0 stores the only block).
template <int D>
__device__ __forceinline__ void store_acc_part(uint32_t t_addr, float mul, __nv_bfloat16* out, size_t row_flat,
                                               bool row_ok, int hd, int g) {
  uint4* dst = reinterpret_cast<uint4*>(out + row_flat * hd);
#pragma unroll
  for (int hcol = 0; hcol < D / 64; ++hcol) {
    if (hcol % 2 != g) continue;
    uint32_t av[64];
    tmem_ld64(t_addr + 64u * hcol, av);
    tmem_ld_wait(av);
    if (row_ok) {
#pragma unroll
      for (int x = 0; x < 8; ++x)
        if (64 * hcol + 8 * x < hd)
          dst[8 * hcol + x] = make_uint4(
              pack_bf16x2(__uint_as_float(av[8 * x]) * mul, __uint_as_float(av[8 * x + 1]) * mul),
              pack_bf16x2(__uint_as_float(av[8 * x + 2]) * mul, __uint_as_float(av[8 * x + 3]) * mul),
              pack_bf16x2(__uint_as_float(av[8 * x + 4]) * mul, __uint_as_float(av[8 * x + 5]) * mul),
              pack_bf16x2(__uint_as_float(av[8 * x + 6]) * mul, __uint_as_float(av[8 * x + 7]) * mul));
    }
  }
}

template <int D>
__device__ __forceinline__ void store_zero_part(__nv_bfloat16* out, size_t row_flat, bool row_ok, int hd, int g) {
  if (!row_ok) return;
  uint4* dst = reinterpret_cast<uint4*>(out + row_flat * hd);
#pragma unroll
  for (int x = 0; x < D / 8; ++x)
    if ((x / 8) % 2 == g && 8 * x < hd) dst[x] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ int clamp_kl(const BwdParams& p, int b) {
  int kl = p.key_len ? p.key_len[b] : p.N;
  return kl < 0 ? 0 : (kl > p.N ? p.N : kl);
}

// ------------------------------------------------------------------ dK, dV
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fattn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                          const BwdParams p) {
  using C = BwdCfg<D>;
  using M = BwdMma<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  // unit: heaviest first (under causal the first key tiles see the most queries)
  const int BH = p.B * p.H;
  const int jt = (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.H;
  const int kl = clamp_kl(p, b);
  const int key0 = jt * 128;
  const int i_first = p.causal ? jt : 0;
  const int n_q = key0 < kl ? p.n_tiles - i_first : 0;  // query tiles that see this key tile

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_FIX_FULL), 1);
    for (int s = 0; s < BWD_STAGES; ++s) {
      mbar_init(bar(C::B_ST_FULL + s), 1);
      mbar_init(bar(C::B_ST_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    mbar_init(bar(C::B_OPS_READY), 32 * BWD_ELEM_WARPS);
    mbar_init(bar(C::B_DS_READY), 32 * BWD_ELEM_WARPS);
    mbar_init(bar(C::B_ACC_FULL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BWD_PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == BWD_MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, BWD_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};
  const int u = (int)blockIdx.x;
  pdl_launch_dependents();

  if (n_q > 0 && warp == BWD_PRODUCER_WARP) {
    if (lane == 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      mbar_arrive_expect_tx(bar(C::B_FIX_FULL), 2 * C::TILE_BYTES);
#pragma unroll
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_3d(base + C::FIX0_OFF + pn * PANEL_BYTES, &tmap_k, bar(C::B_FIX_FULL), 64 * pn, key0, bh);
        tma_load_3d(base + C::FIX1_OFF + pn * PANEL_BYTES, &tmap_v, bar(C::B_FIX_FULL), 64 * pn, key0, bh);
      }
      pdl_wait();  // LSE2 and D come from the prep kernel
      int issued = 0;
      for (int n = 0; ok && n < n_q; ++n) {
        const int s = n % BWD_STAGES;
        ok = wait_bar(waiter, bar(C::B_ST_EMPTY + s), ((n / BWD_STAGES) & 1) ^ 1, C::B_ST_EMPTY + s, u);
        if (!ok) break;
        const int q0 = (i_first + n) * 128;
        const uint32_t full = bar(C::B_ST_FULL + s);
        mbar_arrive_expect_tx(full, 2 * C::TILE_BYTES + 1024u);
        const uint32_t st = base + C::RING_OFF + (uint32_t)s * C::STAGE_BYTES;
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn) {
          tma_load_3d(st + pn * PANEL_BYTES, &tmap_q, full, 64 * pn, q0, bh);
          tma_load_3d(st + C::TILE_BYTES + pn * PANEL_BYTES, &tmap_do, full, 64 * pn, q0, bh);
        }
        const size_t row = (size_t)bh * (size_t)p.N_pad + (size_t)q0;
        bulk_load(base + C::ROWS_OFF + (uint32_t)s * 1024u, p.nlse2 + row, 512u, full);
        bulk_load(base + C::ROWS_OFF + (uint32_t)s * 1024u + 512u, p.delta + row, 512u, full);
        issued = n + 1;
      }
      // drain: the last copies may never have been consumed after an abort
      drain_wait(bar(C::B_FIX_FULL), 0, 20000000ull);
      for (int n = issued > BWD_STAGES ? issued - BWD_STAGES : 0; n < issued; ++n)
        drain_wait(bar(C::B_ST_FULL + n % BWD_STAGES), (n / BWD_STAGES) & 1, 20000000ull);
    }
  } else if (n_q > 0 && warp == BWD_MMA_WARP) {
    // Per query tile n the order is S(n), dP(n), dV(n), S(n+1), dK(n), dP(n+1):
    // dV waits only for P^T, dK for dS^T, and the next tile's S^T is computed
    // while the elementwise warps form dS^T, so that the exponentials of tile
    // n+1 overlap dK(n) and dP(n+1).  S(n+1) may overwrite P^T(n) once dV(n)
    // has been issued (the tensor pipe runs in order); dP(n+1) overwrites
    // dS^T(n) after dK(n).
    waiter.role = ROLE_MMA;
    bool ok = wait_bar(waiter, bar(C::B_FIX_FULL), 0, C::B_FIX_FULL, u);
    ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    const uint64_t k_desc = smem_desc(base + C::FIX0_OFF, 16, 1024);
    const uint64_t v_desc = smem_desc(base + C::FIX1_OFF, 16, 1024);
    auto stage_addr = [&](int n) { return base + C::RING_OFF + (uint32_t)(n % BWD_STAGES) * C::STAGE_BYTES; };
    auto wait_stage = [&](int n) {
      const int s = n % BWD_STAGES;
      ok = ok && wait_bar(waiter, bar(C::B_ST_FULL + s), (n / BWD_STAGES) & 1, C::B_ST_FULL + s, u);
      ok = __all_sync(0xffffffffu, ok);
    };
    auto issue_s = [&](int n) {  // S^T = K Q^T
      M::ss(tmem + BT_S, k_desc, smem_desc(stage_addr(n), 16, 1024));
      mma_commit_w(bar(C::B_S_FULL));
    };
    auto issue_dp = [&](int n) {  // dP^T = V dO^T
      M::ss(tmem + BT_DP, v_desc, smem_desc(stage_addr(n) + C::TILE_BYTES, 16, 1024));
      mma_commit_w(bar(C::B_DP_FULL));
    };
    wait_stage(0);
    if (ok) {
      issued_any = true;
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int n = 0; ok && n < n_q; ++n) {
      const uint32_t st = stage_addr(n);
      const uint32_t acc = n > 0 ? 1u : 0u;
      ok = wait_bar(waiter, bar(C::B_OPS_READY), n & 1, C::B_OPS_READY, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      M::ts(tmem + BT_ACC0, tmem + BT_S, smem_desc(st + C::TILE_BYTES, PANEL_BYTES, 1024), acc);  // dV += P^T dO
      if (n + 1 < n_q) {
        wait_stage(n + 1);
        if (!ok) break;
        tc_fence_after();
        issue_s(n + 1);
      }
      ok = wait_bar(waiter, bar(C::B_DS_READY), n & 1, C::B_DS_READY, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      M::ts(tmem + BT_ACC0 + D, tmem + BT_DP, smem_desc(st, PANEL_BYTES, 1024), acc);  // dK += dS^T Q
      mma_commit_w(bar(C::B_ST_EMPTY + n % BWD_STAGES));
      if (n + 1 < n_q) issue_dp(n + 1);
    }
    if (ok) mma_commit_w(bar(C::B_ACC_FULL));
    if (issued_any) {
      mma_commit_w(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
    }
  } else if (warp < BWD_ELEM_WARPS) {
    // every CTA waits here, even one with no query tile, so that this grid
    // ends after the kernels it depends on
    pdl_wait();
    waiter.role = ROLE_SOFTMAX;
    const int g = warp / 4;             // column group: tile columns [64g, 64g + 64)
    const int quarter = warp % 4;       // TMEM lane quarter
    const int r = quarter * 32 + lane;  // key row within the tile = TMEM lane
    const int key = key0 + r;
    const bool key_vis = key < kl;
    const size_t row_flat = (size_t)bh * (size_t)p.N + (size_t)key;
    const bool row_ok = key < p.N;
    if (n_q == 0) {
      store_zero_part<D>(p.dv, row_flat, row_ok, p.hd, g);
      store_zero_part<D>(p.dk, row_flat, row_ok, p.hd, g);
    } else {
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      // this group's 64 columns of S^T and dP^T; P^T and dS^T are packed over
      // the first 32 of them (the other group's columns are never touched)
      const uint32_t s_addr = tmem + lane_off + BT_S + 64u * (uint32_t)g;
      const uint32_t dp_addr = tmem + lane_off + BT_DP + 64u * (uint32_t)g;
      const float c = p.scale_log2;
      bool ok = true;
      for (int n = 0; ok && n < n_q; ++n) {
        const int s = n % BWD_STAGES;
        const int q0 = (i_first + n) * 128;
        ok = wait_bar(waiter, bar(C::B_ST_FULL + s), (n / BWD_STAGES) & 1, C::B_ST_FULL + s, u);
        if (ok) ok = wait_bar(waiter, bar(C::B_S_FULL), n & 1, C::B_S_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float4* nlse4 = reinterpret_cast<const float4*>(base_ptr + C::ROWS_OFF + (uint32_t)s * 1024u) + 16 * g;
        const float4* del4 = nlse4 + 32;
        const uint64_t c2 = f2_pack(c, c);
        // visible columns: query q0 + col sees this key iff the key is inside
        // key_len and (causal) key <= query; rows past N read as zero and
        // contribute nothing (their dO and Q are zero)
        const int min_q = p.causal ? key - q0 : 0;  // columns < min_q are masked
        const bool any_mask = !key_vis || min_q > 64 * g;
        // phase 1: P^T (kept in fp32 for dS^T), released for dV as soon as it is stored
        float pr[64];
        {
          uint32_t sh[64];
          tmem_ld64(s_addr, sh);
          tmem_ld_wait(sh);
          uint32_t pk[32];
          // a separate copy of the loop for tiles with masked columns, so
          // that the others carry no per-element selects
          auto p_loop = [&](auto masked_c) {
            constexpr bool MASKED = decltype(masked_c)::value;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              // exponent arguments S c - LSE2, two columns per f32x2 FMA
              const float4 l4 = nlse4[q4];
              float x[4];
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[4 * q4]), __uint_as_float(sh[4 * q4 + 1])), c2,
                               f2_pack(l4.x, l4.y)),
                        x[0], x[1]);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[4 * q4 + 2]), __uint_as_float(sh[4 * q4 + 3])), c2,
                               f2_pack(l4.z, l4.w)),
                        x[2], x[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int col = 64 * g + 4 * q4 + e;
                float pe = ex2(x[e]);
                if constexpr (MASKED) pe = (key_vis && col >= min_q) ? pe : 0.0f;
                pr[4 * q4 + e] = pe;
              }
              pk[2 * q4] = pack_bf16x2(pr[4 * q4], pr[4 * q4 + 1]);
              pk[2 * q4 + 1] = pack_bf16x2(pr[4 * q4 + 2], pr[4 * q4 + 3]);
            }
          };
          if (any_mask)
            p_loop(std::true_type{});
          else
            p_loop(std::false_type{});
          tmem_st32(s_addr, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_OPS_READY));
        // phase 2: dS^T = P^T (dP^T - D)
        ok = wait_bar(waiter, bar(C::B_DP_FULL), n & 1, C::B_DP_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dh[64];
          tmem_ld64(dp_addr, dh);
          tmem_ld_wait(dh);
          uint32_t dk2[32];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 d4 = del4[q4];
            // dS = P (dP - D) on pairs of columns (f32x2: the same two
            // roundings as the scalar form, half the instructions)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int q = 4 * q4 + 2 * h;
              const uint64_t dd = h ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
              const uint64_t ds = f2_mul(f2_pack(pr[q], pr[q + 1]),
                                         f2_sub(f2_pack(__uint_as_float(dh[q]), __uint_as_float(dh[q + 1])), dd));
              float lo, hi;
              f2_unpack(ds, lo, hi);
              dk2[2 * q4 + h] = pack_bf16x2(lo, hi);
            }
          }
          tmem_st32(dp_addr, dk2);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DS_READY));
      }
      if (ok) {
        ok = wait_bar(waiter, bar(C::B_ACC_FULL), 0, C::B_ACC_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        store_acc_part<D>(tmem + lane_off + BT_ACC0, 1.0f, p.dv, row_flat, row_ok, p.hd, g);
        store_acc_part<D>(tmem + lane_off + BT_ACC0 + D, p.scale, p.dk, row_flat, row_ok, p.hd, g);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == BWD_MMA_WARP) tmem_dealloc(tmem, BWD_TMEM_COLS);
}

// ------------------------------------------------------------------ dQ
// Q_i and dO_i stay; K_j streams through a 3-slot ring and V_j through a
// 2-slot ring.  S is double-buffered in tensor memory (S_j in buffer j % 2):
// per key tile the issuer runs dQ(j), dP(j+1), S(j+2), so S of the next tile
// is long done when its exponentials start, and the K tile of S(j+2) was
// loaded while tile j was in flight (its slot freed by dQ(j-1)).
template <int D>
struct BwdDqCfg {
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE_BYTES = 128u * D * 2u;
  static constexpr int K_SLOTS = 3, V_SLOTS = 2;
  static constexpr uint32_t Q_OFF = 0, DO_OFF = TILE_BYTES;
  static constexpr uint32_t K_OFF = 2 * TILE_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + K_SLOTS * TILE_BYTES;
  static constexpr uint32_t BAR_OFF = V_OFF + V_SLOTS * TILE_BYTES;
  static constexpr int B_FIX_FULL = 0;
  static constexpr int B_K_FULL = 1;                     // [K_SLOTS]
  static constexpr int B_K_EMPTY = B_K_FULL + K_SLOTS;   // [K_SLOTS]
  static constexpr int B_V_FULL = B_K_EMPTY + K_SLOTS;   // [V_SLOTS]
  static constexpr int B_V_EMPTY = B_V_FULL + V_SLOTS;   // [V_SLOTS]
  // one S barrier per tensor-memory S buffer: S(0) and S(1) are issued back
  // to back, so a shared barrier could complete both phases before the
  // elementwise warps first look at it, and a parity wait would then miss
  static constexpr int B_S_FULL = B_V_EMPTY + V_SLOTS;  // [2]
  static constexpr int B_DP_FULL = B_S_FULL + 2;
  static constexpr int B_DS_READY = B_S_FULL + 3;
  static constexpr int B_ACC_FULL = B_S_FULL + 4;
  static constexpr int B_DRAIN = B_S_FULL + 5;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16 + 1024;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 120u * 1024u ? SMEM_USED : 120u * 1024u;
  static_assert(SMEM_USED <= 232448u, "shared memory");
};
constexpr uint32_t BQ_S0 = 0, BQ_DP = 256, BQ_DQ = 384;  // TMEM columns: S buffers at 0 and 128

template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fattn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                        const BwdParams p) {
  using C = BwdDqCfg<D>;
  using M = BwdMma<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  // unit: heaviest first (under causal the last query tiles see the most keys)
  const int BH = p.B * p.H;
  const int it_rev = (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.H;
  const int kl = clamp_kl(p, b);
  const int it = p.causal ? p.n_tiles - 1 - it_rev : it_rev;
  const int q0 = it * 128;
  const int kl_tiles = (kl + 127) / 128;
  const int n_k = p.causal ? min(it + 1, kl_tiles) : kl_tiles;  // key tiles this query tile sees

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_FIX_FULL), 1);
    for (int s = 0; s < C::K_SLOTS; ++s) {
      mbar_init(bar(C::B_K_FULL + s), 1);
      mbar_init(bar(C::B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::V_SLOTS; ++s) {
      mbar_init(bar(C::B_V_FULL + s), 1);
      mbar_init(bar(C::B_V_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_S_FULL + 1), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    mbar_init(bar(C::B_DS_READY), 32 * BWD_ELEM_WARPS);
    mbar_init(bar(C::B_ACC_FULL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BWD_PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == BWD_MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, BWD_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};
  const int u = (int)blockIdx.x;

  if (n_k > 0 && warp == BWD_PRODUCER_WARP) {
    if (lane == 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      mbar_arrive_expect_tx(bar(C::B_FIX_FULL), 2 * C::TILE_BYTES);
#pragma unroll
      for (int pn = 0; pn < C::PANELS; ++pn) {
        tma_load_3d(base + C::Q_OFF + pn * PANEL_BYTES, &tmap_q, bar(C::B_FIX_FULL), 64 * pn, q0, bh);
        tma_load_3d(base + C::DO_OFF + pn * PANEL_BYTES, &tmap_do, bar(C::B_FIX_FULL), 64 * pn, q0, bh);
      }
      int issued = 0;
      for (int n = 0; ok && n < n_k; ++n) {
        const int ks = n % C::K_SLOTS, vs = n % C::V_SLOTS;
        ok = wait_bar(waiter, bar(C::B_K_EMPTY + ks), ((n / C::K_SLOTS) & 1) ^ 1, C::B_K_EMPTY + ks, u);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_K_FULL + ks), C::TILE_BYTES);
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_3d(base + C::K_OFF + (uint32_t)ks * C::TILE_BYTES + pn * PANEL_BYTES, &tmap_k, bar(C::B_K_FULL + ks),
                      64 * pn, n * 128, bh);
        ok = wait_bar(waiter, bar(C::B_V_EMPTY + vs), ((n / C::V_SLOTS) & 1) ^ 1, C::B_V_EMPTY + vs, u);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_V_FULL + vs), C::TILE_BYTES);
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_3d(base + C::V_OFF + (uint32_t)vs * C::TILE_BYTES + pn * PANEL_BYTES, &tmap_v, bar(C::B_V_FULL + vs),
                      64 * pn, n * 128, bh);
        issued = n + 1;
      }
      drain_wait(bar(C::B_FIX_FULL), 0, 20000000ull);
      for (int n = issued > C::V_SLOTS ? issued - C::V_SLOTS : 0; n < issued; ++n)
        drain_wait(bar(C::B_V_FULL + n % C::V_SLOTS), (n / C::V_SLOTS) & 1, 20000000ull);
      for (int n = issued > C::K_SLOTS ? issued - C::K_SLOTS : 0; n < issued; ++n)
        drain_wait(bar(C::B_K_FULL + n % C::K_SLOTS), (n / C::K_SLOTS) & 1, 20000000ull);
    }
  } else if (n_k > 0 && warp == BWD_MMA_WARP) {
    waiter.role = ROLE_MMA;
    bool ok = wait_bar(waiter, bar(C::B_FIX_FULL), 0, C::B_FIX_FULL, u);
    ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    const uint64_t q_desc = smem_desc(base + C::Q_OFF, 16, 1024);
    const uint64_t do_desc = smem_desc(base + C::DO_OFF, 16, 1024);
    auto k_addr = [&](int n) { return base + C::K_OFF + (uint32_t)(n % C::K_SLOTS) * C::TILE_BYTES; };
    auto v_addr = [&](int n) { return base + C::V_OFF + (uint32_t)(n % C::V_SLOTS) * C::TILE_BYTES; };
    auto wait_k = [&](int n) {
      const int s = n % C::K_SLOTS;
      ok = ok && wait_bar(waiter, bar(C::B_K_FULL + s), (n / C::K_SLOTS) & 1, C::B_K_FULL + s, u);
      ok = __all_sync(0xffffffffu, ok);
    };
    auto wait_v = [&](int n) {
      const int s = n % C::V_SLOTS;
      ok = ok && wait_bar(waiter, bar(C::B_V_FULL + s), (n / C::V_SLOTS) & 1, C::B_V_FULL + s, u);
      ok = __all_sync(0xffffffffu, ok);
    };
    auto issue_s = [&](int n) {  // S_n = Q K_n^T into buffer n % 2
      tc_fence_after();
      M::ss(tmem + BQ_S0 + 128u * (uint32_t)(n & 1), q_desc, smem_desc(k_addr(n), 16, 1024));
      mma_commit_w(bar(C::B_S_FULL + (n & 1)));
    };
    auto issue_dp = [&](int n) {  // dP_n = dO V_n^T; V_n is then free
      tc_fence_after();
      M::ss(tmem + BQ_DP, do_desc, smem_desc(v_addr(n), 16, 1024));
      mma_commit_w(bar(C::B_DP_FULL));
      mma_commit_w(bar(C::B_V_EMPTY + n % C::V_SLOTS));
    };
    if (ok) {
      issued_any = true;
      wait_k(0);
      if (ok) issue_s(0);
      wait_v(0);
      if (ok) issue_dp(0);
      if (n_k > 1) {
        wait_k(1);
        if (ok) issue_s(1);
      }
    }
    for (int n = 0; ok && n < n_k; ++n) {
      ok = wait_bar(waiter, bar(C::B_DS_READY), n & 1, C::B_DS_READY, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // dP_n+1 first: the elementwise warps have read dP_n, and the next
      // tile's dS waits on nothing else (its exponentials run meanwhile)
      if (n + 1 < n_k) {
        wait_v(n + 1);
        if (!ok) break;
        issue_dp(n + 1);
      }
      // dQ += dS_n K_n (dS over the first 64 columns of S buffer n % 2); K_n is then free
      M::ts(tmem + BQ_DQ, tmem + BQ_S0 + 128u * (uint32_t)(n & 1), smem_desc(k_addr(n), PANEL_BYTES, 1024),
            n > 0 ? 1u : 0u);
      mma_commit_w(bar(C::B_K_EMPTY + n % C::K_SLOTS));
      if (n + 2 < n_k) {
        wait_k(n + 2);
        if (!ok) break;
        issue_s(n + 2);
      }
    }
    if (ok) mma_commit_w(bar(C::B_ACC_FULL));
    if (issued_any) {
      mma_commit_w(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
    }
  } else if (warp < BWD_ELEM_WARPS) {
    pdl_wait();  // LSE2 and D come from the prep kernel (every CTA waits, as above)
    waiter.role = ROLE_SOFTMAX;
    const int g = warp / 4;             // column group: tile columns (keys) [64g, 64g + 64)
    const int quarter = warp % 4;       // TMEM lane quarter
    const int r = quarter * 32 + lane;  // query row within the tile = TMEM lane
    const int query = q0 + r;
    const size_t row_flat = (size_t)bh * (size_t)p.N + (size_t)query;
    const bool row_ok = query < p.N;
    if (n_k == 0) {
      store_zero_part<D>(p.dq, row_flat, row_ok, p.hd, g);
    } else {
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t dp_addr = tmem + lane_off + BQ_DP + 64u * (uint32_t)g;
      const float c = p.scale_log2;
      const size_t prow = (size_t)bh * (size_t)p.N_pad + (size_t)query;
      const float nlse2 = p.nlse2[prow];
      const float drow = p.delta[prow];
      // keys [0, lim) are visible to this row
      const int lim = p.causal ? min(kl, query + 1) : kl;
      bool ok = true;
      for (int n = 0; ok && n < n_k; ++n) {
        // this group's 64 columns of S_n; dS is packed over the first 32 of them
        const uint32_t s_addr = tmem + lane_off + BQ_S0 + 128u * (uint32_t)(n & 1) + 64u * (uint32_t)g;
        ok = wait_bar(waiter, bar(C::B_S_FULL + (n & 1)), (n >> 1) & 1, C::B_S_FULL + (n & 1), u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int vis_n = lim - n * 128 - 64 * g;  // this group's columns [0, vis_n) visible
        const bool masked = vis_n < 64;
        // phase 1 (while dP is computed): P in fp32 registers
        float pr[64];
        {
          uint32_t sh[64];
          tmem_ld64(s_addr, sh);
          tmem_ld_wait(sh);
          // a separate copy of the loop for masked tiles (no per-element
          // selects on the others)
          // exponent arguments S c - LSE2 two columns per f32x2 FMA
          const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(nlse2, nlse2);
          auto p_loop = [&](auto masked_c) {
            constexpr bool MASKED = decltype(masked_c)::value;
#pragma unroll
            for (int q = 0; q < 64; q += 2) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[q]), __uint_as_float(sh[q + 1])), c2, nl2), x0, x1);
              float p0 = ex2(x0), p1 = ex2(x1);
              if constexpr (MASKED) {
                p0 = q < vis_n ? p0 : 0.0f;
                p1 = q + 1 < vis_n ? p1 : 0.0f;
              }
              pr[q] = p0;
              pr[q + 1] = p1;
            }
          };
          if (masked)
            p_loop(std::true_type{});
          else
            p_loop(std::false_type{});
        }
        // phase 2: dS = P (dP - D), stored as bf16 over this group's first 32 columns of S
        ok = wait_bar(waiter, bar(C::B_DP_FULL), n & 1, C::B_DP_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dh[64];
          tmem_ld64(dp_addr, dh);
          tmem_ld_wait(dh);
          uint32_t pk[32];
          const uint64_t d2 = f2_pack(drow, drow);
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            // dS = P (dP - D), two columns per f32x2 op
            const uint64_t ds = f2_mul(f2_pack(pr[2 * q], pr[2 * q + 1]),
                                       f2_sub(f2_pack(__uint_as_float(dh[2 * q]), __uint_as_float(dh[2 * q + 1])), d2));
            float lo, hi;
            f2_unpack(ds, lo, hi);
            pk[q] = pack_bf16x2(lo, hi);
          }
          tmem_st32(s_addr, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DS_READY));
      }
      if (ok) {
        ok = wait_bar(waiter, bar(C::B_ACC_FULL), 0, C::B_ACC_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        store_acc_part<D>(tmem + lane_off + BQ_DQ, p.scale, p.dq, row_flat, row_ok, p.hd, g);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == BWD_MMA_WARP) tmem_dealloc(tmem, BWD_TMEM_COLS);
}

}  // namespace fattn
