// Exact softmax attention backward in one pass over the tile pairs, sm_103a,
// head dims 72..128 (the 128-column bucket).
//
// What it computes: the same gradients as fattn_bwd.cuh ("understand-
// flashattention", section "Attention forward and backward formulas",
// backward pass steps 1-5, P recomputed from the saved logsumexp):
//     dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K,
//     dS = P * (dP - D),  dP = dO V^T,  D_i = rowsum(dO_i * O_i).
//
// How (GB300): one CTA per (batch*head, 128-key tile j), as the dK/dV kernel
// of fattn_bwd.cuh, but the query tiles that see tile j stream through in
// steps of 64 rows, so that tensor memory holds, besides the dV and dK
// accumulators (2 x 128 columns), S^T and dP^T of one step (64 columns
// each) and two buffers of dQ_i^T = K_j^T dS_ij^T (64 columns each):
//     S^T = K_j Q_i^T, dP^T = V_j dO_i^T          (M = 128 keys, N = 64)
//     dV += P^T dO_i, dK += dS^T Q_i               (A = P^T, dS^T from TMEM)
//     dQ_i^T = K_j^T dS^T                          (M = 128 = d, N = 64 queries;
//                                                    A = K_j read MN-major,
//                                                    B = dS^T from shared memory)
// The elementwise warps store dS^T twice: packed bf16 over dP^T (the A
// operand of dK) and into a shared-memory tile (the B operand of dQ^T, 128
// keys x 64 queries, queries contiguous, 128-byte swizzle).  Each dQ_i^T is
// read back from tensor memory by the elementwise warps one step later and
// added into an fp32 dQ buffer with red.global.add: a warp's lanes are 32
// consecutive head-dim columns of one query row, 128 contiguous bytes per
// instruction; a last kernel scales that buffer by `scale` into bf16 dQ.  So
// five GEMMs run per tile pair instead of the seven of the two-kernel form;
// the price is the fp32 reductions (each query row receives one 512-byte row
// per key tile it sees, in an order that varies from run to run, so dQ is
// not bit-reproducible) and the zeroing and conversion of the dQ buffer.
//
// Measured on the b2h16n4096d128 causal backward: this kernel 336 us against
// 206 + 147 us for the two-kernel form; the whole call 389 us against 378 us.
// What holds it back is the N = 64 of S^T, dP^T and dQ^T: with both operands
// in shared memory, a 128 x 64 x 16 MMA reads 6 KB in the 32 tensor cycles it
// takes, 1.5x the shared-memory bandwidth, so those three GEMMs run at about
// two thirds of the tensor rate (tensor pipe 44 % active in ncu).  Variants
// measured slower: eight elementwise warps (346 us), the dQ^T block staged in
// shared memory and added by the tensor-copy engine (370 us) or with 16-byte
// vector reductions (403 us), dQ^T read back between P^T and dS^T (379 us).
// The library runs it only when FATTN_BWD_FUSED=1 is set in the environment.
//
// Every wait is bounded as in the forward kernel.
#pragma once

#include "fattn_bwd.cuh"

namespace fattn {

constexpr int FB_BQ = 64;      // query rows per step
constexpr int FB_STAGES = 3;   // Q / dO / row-constant ring
constexpr int FB_D = 128;
// warps 0-15 elementwise (four groups of four: group g takes the step's
// query columns [16g, 16g + 16) of the same TMEM lanes), 16 TMA producer,
// 17 MMA issuer
constexpr int FB_GROUPS = 4;
constexpr int FB_CW = FB_BQ / FB_GROUPS;  // query columns per group
constexpr int FB_ELEM_WARPS = 4 * FB_GROUPS;
constexpr int FB_PRODUCER_WARP = FB_ELEM_WARPS;
constexpr int FB_MMA_WARP = FB_ELEM_WARPS + 1;
constexpr int FB_THREADS = 32 * (FB_ELEM_WARPS + 2);

struct FusedCfg {
  static constexpr int D = FB_D;
  static constexpr uint32_t KV_TILE = 128u * D * 2u;        // K_j or V_j: 128 rows, two 64-column panels
  static constexpr uint32_t KV_PANEL = 128u * 128u;         // 16 KB
  static constexpr uint32_t Q_TILE = FB_BQ * D * 2u;        // Q_i or dO_i: 64 rows
  static constexpr uint32_t Q_PANEL = FB_BQ * 128u;         // 8 KB
  static constexpr uint32_t K_OFF = 0;
  static constexpr uint32_t V_OFF = KV_TILE;
  static constexpr uint32_t RING_OFF = 2 * KV_TILE;         // per stage: Q_i then dO_i
  static constexpr uint32_t STAGE_BYTES = 2 * Q_TILE;
  static constexpr uint32_t DS_OFF = RING_OFF + FB_STAGES * STAGE_BYTES;  // [2] dS^T tiles
  static constexpr uint32_t DS_BYTES = 128u * FB_BQ * 2u;   // 128 keys x 64 queries bf16
  static constexpr uint32_t ROWS_OFF = DS_OFF + 2 * DS_BYTES;             // per stage: -LSE2[64], D[64]
  static constexpr uint32_t ROWS_BYTES = 2u * FB_BQ * 4u;
  static constexpr uint32_t BAR_OFF = ROWS_OFF + FB_STAGES * ROWS_BYTES;
  // barrier ids
  static constexpr int B_FIX_FULL = 0;
  static constexpr int B_ST_FULL = 1;                       // [FB_STAGES]
  static constexpr int B_ST_EMPTY = 1 + FB_STAGES;          // [FB_STAGES]
  static constexpr int B_S_FULL = 1 + 2 * FB_STAGES;
  static constexpr int B_DP_FULL = B_S_FULL + 1;
  static constexpr int B_P_READY = B_S_FULL + 2;            // P^T stored (elementwise arrivals)
  static constexpr int B_DS_READY = B_S_FULL + 3;           // dS^T stored in TMEM and shared memory
  static constexpr int B_DQ_FULL = B_S_FULL + 4;            // [2] dQ^T buffer complete
  static constexpr int B_DQ_EMPTY = B_S_FULL + 6;           // [2] dQ^T buffer read back
  static constexpr int B_ACC_FULL = B_S_FULL + 8;
  static constexpr int B_DRAIN = B_S_FULL + 9;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16 + 1024;   // + slack for 1024-byte alignment
  static constexpr uint32_t SMEM_BYTES = SMEM_USED;
  static_assert(SMEM_USED <= 232448u, "shared memory");
  static_assert(DS_OFF % 1024 == 0 && ROWS_OFF % 16 == 0, "operand tiles on 1 KB, row copies on 16 B");
};
// TMEM columns
constexpr uint32_t FT_S = 0, FT_DP = 64, FT_DQ = 128, FT_DV = 256, FT_DK = 384;

// Instruction descriptor for kind::f16 with either operand MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_ab(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                  // D format f32
         | (1u << 7) | (1u << 10)                   // A, B bf16
         | ((a_mn_major ? 1u : 0u) << 15)
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
// 8 registers per thread -> 8 consecutive 32-bit TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct FusedMma {
  using C = FusedCfg;
  static constexpr uint32_t IDESC_ST = idesc_f16_ab(128, FB_BQ, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_ACC = idesc_f16_ab(128, FB_D, false, true);    // dV, dK: B MN-major
  static constexpr uint32_t IDESC_DQ = idesc_f16_ab(128, FB_BQ, true, true);     // dQ^T: A and B MN-major

  // D(128 x 64) = A(128 x 128) B(64 x 128)^T: A a 128-row tile, B a 64-row
  // tile, both K-major with 64-column panels (16 KB and 8 KB apart).
  __device__ __forceinline__ static void st(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
    static_for<FB_D / 16>([&](auto kc) {
      constexpr int kk = decltype(kc)::value;
      constexpr uint32_t aoff = ((kk / 4) * C::KV_PANEL + (kk % 4) * 32u) >> 4;
      constexpr uint32_t boff = ((kk / 4) * C::Q_PANEL + (kk % 4) * 32u) >> 4;
      mma_ss_w_off2<aoff, boff>(d_tmem, a_desc, b_desc, IDESC_ST, kk > 0 ? 1u : 0u);
    });
  }
  // D(128 x 128) (+)= A(128 x 64 queries, bf16 in TMEM) B(64 queries x 128, MN-major).
  // Group g packs its 16 query columns over the first 8 of its 16 TMEM
  // columns (16g .. 16g+7), so the 16 queries of K step kk sit at column 16 kk.
  __device__ __forceinline__ static void ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    static_for<FB_BQ / 16>([&](auto kc) {
      constexpr int kk = decltype(kc)::value;
      constexpr uint32_t boff = (kk * 2048u) >> 4;  // 16 rows = two 1024-byte row groups
      constexpr uint32_t acol = 16u * kk;
      mma_ts_w_off<boff, acol>(d_tmem, a_tmem, b_desc, IDESC_ACC, kk > 0 ? 1u : accumulate);
    });
  }
  // D(128 x 64) = A(128 = d x 128 keys, MN-major: the K_j tile) B(128 keys x 64 queries, MN-major).
  __device__ __forceinline__ static void dq(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
    static_for<8>([&](auto kc) {
      constexpr int kk = decltype(kc)::value;
      constexpr uint32_t off = (kk * 2048u) >> 4;  // 16 keys = 16 rows of 128 bytes in both operands
      mma_ss_w_off<off>(d_tmem, a_desc, b_desc, IDESC_DQ, kk > 0 ? 1u : 0u);
    });
  }
};

__global__ void __launch_bounds__(FB_THREADS, 1)
    fattn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                           const BwdParams p) {
  using C = FusedCfg;
  using M = FusedMma;
  constexpr int D = FB_D;
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
  const int n64 = (p.N + FB_BQ - 1) / FB_BQ;
  const int i_first = p.causal ? 2 * jt : 0;                // 64-row query tiles from here see tile j
  const int n_q = key0 < kl ? n64 - i_first : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_FIX_FULL), 1);
    for (int s = 0; s < FB_STAGES; ++s) {
      mbar_init(bar(C::B_ST_FULL + s), 1);
      mbar_init(bar(C::B_ST_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    mbar_init(bar(C::B_P_READY), 32 * FB_ELEM_WARPS);
    mbar_init(bar(C::B_DS_READY), 32 * FB_ELEM_WARPS);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_DQ_FULL + s), 1);
      mbar_init(bar(C::B_DQ_EMPTY + s), 32 * FB_ELEM_WARPS);
    }
    mbar_init(bar(C::B_ACC_FULL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == FB_PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == FB_MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, BWD_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};
  const int u = (int)blockIdx.x;

  if (n_q > 0 && warp == FB_PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      mbar_arrive_expect_tx(bar(C::B_FIX_FULL), 2 * C::KV_TILE);
#pragma unroll
      for (int pn = 0; pn < D / 64; ++pn) {
        tma_load_3d(base + C::K_OFF + pn * C::KV_PANEL, &tmap_k, bar(C::B_FIX_FULL), 64 * pn, key0, bh);
        tma_load_3d(base + C::V_OFF + pn * C::KV_PANEL, &tmap_v, bar(C::B_FIX_FULL), 64 * pn, key0, bh);
      }
      int issued = 0;
      for (int n = 0; ok && n < n_q; ++n) {
        const int s = n % FB_STAGES;
        ok = wait_bar(waiter, bar(C::B_ST_EMPTY + s), ((n / FB_STAGES) & 1) ^ 1, C::B_ST_EMPTY + s, u);
        if (!ok) break;
        const int q0 = (i_first + n) * FB_BQ;
        const uint32_t full = bar(C::B_ST_FULL + s);
        mbar_arrive_expect_tx(full, 2 * C::Q_TILE + C::ROWS_BYTES);
        const uint32_t st = base + C::RING_OFF + (uint32_t)s * C::STAGE_BYTES;
#pragma unroll
        for (int pn = 0; pn < D / 64; ++pn) {
          tma_load_3d(st + pn * C::Q_PANEL, &tmap_q, full, 64 * pn, q0, bh);
          tma_load_3d(st + C::Q_TILE + pn * C::Q_PANEL, &tmap_do, full, 64 * pn, q0, bh);
        }
        const size_t row = (size_t)bh * (size_t)p.N_pad + (size_t)q0;
        const uint32_t rows = base + C::ROWS_OFF + (uint32_t)s * C::ROWS_BYTES;
        bulk_load(rows, p.nlse2 + row, FB_BQ * 4u, full);
        bulk_load(rows + FB_BQ * 4u, p.delta + row, FB_BQ * 4u, full);
        issued = n + 1;
      }
      // drain: the last copies may never have been consumed after an abort
      drain_wait(bar(C::B_FIX_FULL), 0, 20000000ull);
      for (int n = issued > FB_STAGES ? issued - FB_STAGES : 0; n < issued; ++n)
        drain_wait(bar(C::B_ST_FULL + n % FB_STAGES), (n / FB_STAGES) & 1, 20000000ull);
    }
  } else if (n_q > 0 && warp == FB_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Per step n: dV(n), S(n+1), dK(n), dQ^T(n), dP(n+1).  S(n+1) may
    // overwrite P^T(n) once dV(n) is issued and dP(n+1) dS^T(n) once dK(n)
    // is (the tensor pipe runs in order); dQ^T(n) reads dS^T(n) from shared
    // memory into buffer n % 2, which the elementwise warps have read back
    // (step n - 2) before it is reused.
    waiter.role = ROLE_MMA;
    bool ok = wait_bar(waiter, bar(C::B_FIX_FULL), 0, C::B_FIX_FULL, u);
    ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    const uint64_t k_desc = smem_desc(base + C::K_OFF, 16, 1024);
    const uint64_t v_desc = smem_desc(base + C::V_OFF, 16, 1024);
    const uint64_t kt_desc = smem_desc(base + C::K_OFF, C::KV_PANEL, 1024);  // K_j read MN-major (M = d)
    auto stage_addr = [&](int n) { return base + C::RING_OFF + (uint32_t)(n % FB_STAGES) * C::STAGE_BYTES; };
    auto wait_stage = [&](int n) {
      const int s = n % FB_STAGES;
      ok = ok && wait_bar(waiter, bar(C::B_ST_FULL + s), (n / FB_STAGES) & 1, C::B_ST_FULL + s, u);
      ok = __all_sync(0xffffffffu, ok);
    };
    auto issue_s = [&](int n) {  // S^T = K Q^T
      M::st(tmem + FT_S, k_desc, smem_desc(stage_addr(n), 16, 1024));
      mma_commit_w(bar(C::B_S_FULL));
    };
    auto issue_dp = [&](int n) {  // dP^T = V dO^T
      M::st(tmem + FT_DP, v_desc, smem_desc(stage_addr(n) + C::Q_TILE, 16, 1024));
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
      ok = wait_bar(waiter, bar(C::B_P_READY), n & 1, C::B_P_READY, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      M::ts(tmem + FT_DV, tmem + FT_S, smem_desc(st + C::Q_TILE, C::Q_PANEL, 1024), acc);  // dV += P^T dO
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
      M::ts(tmem + FT_DK, tmem + FT_DP, smem_desc(st, C::Q_PANEL, 1024), acc);  // dK += dS^T Q
      mma_commit_w(bar(C::B_ST_EMPTY + n % FB_STAGES));
      const int bq = n & 1;
      if (n >= 2) {
        ok = wait_bar(waiter, bar(C::B_DQ_EMPTY + bq), ((n >> 1) - 1) & 1, C::B_DQ_EMPTY + bq, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      M::dq(tmem + FT_DQ + 64u * (uint32_t)bq, kt_desc,
            smem_desc(base + C::DS_OFF + (uint32_t)bq * C::DS_BYTES, C::DS_BYTES, 1024));  // dQ^T = K^T dS^T
      mma_commit_w(bar(C::B_DQ_FULL + bq));
      if (n + 1 < n_q) issue_dp(n + 1);
    }
    if (ok) mma_commit_w(bar(C::B_ACC_FULL));
    if (issued_any) {
      mma_commit_w(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
    }
  } else if (warp < FB_ELEM_WARPS) {
    // ------------------------------------------------------------ elementwise
    waiter.role = ROLE_SOFTMAX;
    const int g = warp / 4;             // column group: the step's query columns [16g, 16g + 16)
    const int quarter = warp % 4;       // TMEM lane quarter
    const int r = quarter * 32 + lane;  // key row within the tile (= head-dim row of dQ^T)
    const int key = key0 + r;
    const bool key_vis = key < kl;
    const size_t row_flat = (size_t)bh * (size_t)p.N + (size_t)key;
    const bool row_ok = key < p.N;
    // group g's share of a dK or dV row: columns [32g, 32g + 32)
    auto store_row_part = [&](__nv_bfloat16* out, const uint32_t (&av)[32], float mul) {
      if (!row_ok) return;
      uint4* dst = reinterpret_cast<uint4*>(out + row_flat * p.hd + 32 * g);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        if (32 * g + 8 * x < p.hd)
          dst[x] = make_uint4(pack_bf16x2(__uint_as_float(av[8 * x]) * mul, __uint_as_float(av[8 * x + 1]) * mul),
                              pack_bf16x2(__uint_as_float(av[8 * x + 2]) * mul, __uint_as_float(av[8 * x + 3]) * mul),
                              pack_bf16x2(__uint_as_float(av[8 * x + 4]) * mul, __uint_as_float(av[8 * x + 5]) * mul),
                              pack_bf16x2(__uint_as_float(av[8 * x + 6]) * mul, __uint_as_float(av[8 * x + 7]) * mul));
    };
    if (n_q == 0) {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
      store_row_part(p.dv, z, 1.0f);
      store_row_part(p.dk, z, 1.0f);
    } else {
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t s_addr = tmem + lane_off + FT_S + (uint32_t)(FB_CW * g);
      const uint32_t dp_addr = tmem + lane_off + FT_DP + (uint32_t)(FB_CW * g);
      const float c = p.scale_log2;
      // this thread's row of a dS^T tile: key r, 128-byte swizzle over
      // 16-byte chunks (chunk ^ (row % 8)), the group's chunks 4g .. 4g+3
      const uint32_t ds_row = (uint32_t)(r / 8) * 1024u + (uint32_t)(r % 8) * 128u;
      // dQ^T of step m (buffer m % 2) back to the fp32 dQ buffer: this
      // thread holds head-dim column r of the group's 32 query rows
      auto read_dq = [&](int m) -> bool {
        const int bq = m & 1;
        bool good = wait_bar(waiter, bar(C::B_DQ_FULL + bq), (m >> 1) & 1, C::B_DQ_FULL + bq, u);
        good = __all_sync(0xffffffffu, good);
        if (!good) return false;
        tc_fence_after();
        uint32_t qv[FB_CW];
        tmem_ld16(tmem + lane_off + FT_DQ + 64u * (uint32_t)bq + (uint32_t)(FB_CW * g), qv);
        tmem_ld_wait(qv);
        tc_fence_before();
        mbar_arrive(bar(C::B_DQ_EMPTY + bq));
        const int q0 = (i_first + m) * FB_BQ + FB_CW * g;  // first query row of this group
        float* dst = p.dq_acc + ((size_t)bh * (size_t)p.N_pad + (size_t)q0) * D + r;
#pragma unroll
        for (int i = 0; i < FB_CW; ++i) red_add_f32(dst + (size_t)i * D, __uint_as_float(qv[i]));
        return true;
      };
      bool ok = true;
      for (int n = 0; ok && n < n_q; ++n) {
        const int s = n % FB_STAGES;
        const int q0 = (i_first + n) * FB_BQ;
        ok = wait_bar(waiter, bar(C::B_ST_FULL + s), (n / FB_STAGES) & 1, C::B_ST_FULL + s, u);
        if (ok) ok = wait_bar(waiter, bar(C::B_S_FULL), n & 1, C::B_S_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float4* nlse4 =
            reinterpret_cast<const float4*>(base_ptr + C::ROWS_OFF + (uint32_t)s * C::ROWS_BYTES) + (FB_CW / 4) * g;
        const float4* del4 = nlse4 + FB_BQ / 4;
        // visible columns: query q0 + col sees this key iff the key is inside
        // key_len and (causal) key <= query; rows past N read as zero and
        // contribute nothing (their dO and Q are zero)
        const int min_q = p.causal ? key - q0 : 0;  // columns < min_q are masked
        const bool any_mask = !key_vis || min_q > FB_CW * g;
        // phase 1: P^T (kept in fp32 for dS^T), released for dV as soon as it is stored
        float pr[FB_CW];
        {
          uint32_t sh[FB_CW];
          tmem_ld16(s_addr, sh);
          tmem_ld_wait(sh);
          uint32_t pk[FB_CW / 2];
          auto p_loop = [&](auto masked_c) {
            constexpr bool MASKED = decltype(masked_c)::value;
#pragma unroll
            for (int q4 = 0; q4 < FB_CW / 4; ++q4) {
              // exponent arguments S c - LSE2 (-LSE2 per column), two per f32x2 FMA
              const float4 l4 = nlse4[q4];
              const uint64_t c2 = f2_pack(c, c);
              float x[4];
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[4 * q4]), __uint_as_float(sh[4 * q4 + 1])), c2,
                               f2_pack(l4.x, l4.y)),
                        x[0], x[1]);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[4 * q4 + 2]), __uint_as_float(sh[4 * q4 + 3])), c2,
                               f2_pack(l4.z, l4.w)),
                        x[2], x[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int col = FB_CW * g + 4 * q4 + e;
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
          tmem_st8(s_addr, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_P_READY));
        // phase 2: dS^T = P^T (dP^T - D), into tensor memory (for dK) and
        // into the step's shared-memory tile (for dQ^T)
        ok = wait_bar(waiter, bar(C::B_DP_FULL), n & 1, C::B_DP_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dh[FB_CW];
          tmem_ld16(dp_addr, dh);
          tmem_ld_wait(dh);
          uint32_t dk2[FB_CW / 2];
#pragma unroll
          for (int q4 = 0; q4 < FB_CW / 4; ++q4) {
            const float4 d4 = del4[q4];
            // two columns per f32x2 op (the same roundings as the scalar form)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = 4 * q4 + 2 * h;
              const uint64_t dd = h ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
              const uint64_t ds = f2_mul(f2_pack(pr[i], pr[i + 1]),
                                         f2_sub(f2_pack(__uint_as_float(dh[i]), __uint_as_float(dh[i + 1])), dd));
              float lo, hi;
              f2_unpack(ds, lo, hi);
              dk2[2 * q4 + h] = pack_bf16x2(lo, hi);
            }
          }
          tmem_st8(dp_addr, dk2);
          uint8_t* ds_tile = base_ptr + C::DS_OFF + (uint32_t)(n & 1) * C::DS_BYTES + ds_row;
#pragma unroll
          for (int i = 0; i < FB_CW / 8; ++i) {
            const uint32_t chunk = (uint32_t)(((FB_CW / 8) * g + i) ^ (r % 8));
            *reinterpret_cast<uint4*>(ds_tile + 16u * chunk) =
                make_uint4(dk2[4 * i], dk2[4 * i + 1], dk2[4 * i + 2], dk2[4 * i + 3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_cta();  // the dS^T tile is read by the tensor core (async proxy)
        tc_fence_before();
        mbar_arrive(bar(C::B_DS_READY));
        // the previous step's dQ^T, complete by now (issued once its dS^T was
        // handed over); reading it here, off the dS chain, measured faster
        // than between P^T and dS^T
        if (n > 0) ok = read_dq(n - 1);
      }
      if (ok) ok = read_dq(n_q - 1);
      if (ok) {
        ok = wait_bar(waiter, bar(C::B_ACC_FULL), 0, C::B_ACC_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        uint32_t av[32];
        tmem_ld32(tmem + lane_off + FT_DV + 32u * (uint32_t)g, av);
        tmem_ld_wait(av);
        store_row_part(p.dv, av, 1.0f);
        tmem_ld32(tmem + lane_off + FT_DK + 32u * (uint32_t)g, av);
        tmem_ld_wait(av);
        store_row_part(p.dk, av, p.scale);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == FB_MMA_WARP) tmem_dealloc(tmem, BWD_TMEM_COLS);
}

// dQ = scale * the fp32 buffer (rows padded to N_pad, 128 columns) -> bf16
// [B*H, N, hd]; one thread per 8 columns.
__global__ void __launch_bounds__(256)
    fattn_bwd_dq_finalize_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq, int N, int N_pad, int hd,
                                 float scale, long long n_vec) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;  // over BH * N * hd / 8
  if (i >= n_vec) return;
  const int per_row = hd / 8;
  const long long row = i / per_row;  // bh * N + r
  const int c8 = (int)(i % per_row);
  const long long bh = row / N;
  const long long r = row % N;
  const float4* src = acc + ((bh * N_pad + r) * FB_D + 8 * c8) / 4;
  const float4 a = src[0], b = src[1];
  dq[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                     pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
}

}  // namespace fattn
