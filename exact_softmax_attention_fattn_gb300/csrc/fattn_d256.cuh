// Exact softmax attention forward for head dims 136..256, sm_103a.
//
// Same result as the main kernel (fattn_kernel.cuh: "understand-flashattention"
// forward formulas and two-block online-softmax derivation, scale-then-mask
// order of "PyTorch profiling part 3: attention"), with a layout that fits a
// 256-column head dim: tensor memory cannot hold S and O for two query tiles
// at once (2 x (128 + 256) > 512 columns), so a CTA owns one 128-row query
// tile, and K/V tiles are 64 keys deep so that Q (64 KB) and two-slot K and V
// rings (4 x 32 KB) fit in shared memory.
//
//   * one CTA per (batch*head, 128-row query tile), in groups of heads whose
//     K and V fit in L2 together, heaviest tiles of a group first under
//     causal; 192 threads: warps 0-3 form the softmax group (one query row
//     per thread, a TMEM lane each), warp 4 is the TMA producer, warp 5
//     issues tcgen05.mma;
//   * tensor memory: S double-buffered over key tiles (S_j in columns
//     64*(j%2) .. +64, P_j packed over the first 32 of them), O in columns
//     256..511;
//   * issue order: S_0, S_1, then per key tile j: P_j V_j into O (once the
//     softmax group has released P_j), S_j+2.  The softmax of tile j+1 runs
//     while the tensor core computes P_j V_j and S_j+2;
//   * a rescale of O (skipped while the running max has grown by less than
//     2^8, as in the main kernel) first waits for the previous P V product,
//     which the issuer signals after every tile; P is otherwise released
//     without waiting for it;
//   * head dims below 256 (multiples of 8) are read with zero columns past d
//     by the tensor maps and stored d columns wide;
//   * every wait is bounded; on time-out the kernel records the error word,
//     drains its own copies and MMAs, frees tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fattn_kernel.cuh"

namespace fattn {

constexpr int D256 = 256;
constexpr int D256_BN = 64;  // keys per K/V tile
constexpr int D256_THREADS = 192;
constexpr int D256_PRODUCER_WARP = 4;
constexpr int D256_MMA_WARP = 5;
constexpr uint32_t D256_TMEM_S = 0;    // S_j at column 64 * (j % 2)
constexpr uint32_t D256_TMEM_O = 256;  // O: 256 columns

struct D256Cfg {
  static constexpr uint32_t Q_PANEL = 128u * 128u;            // 128 rows x 64 columns of bf16
  static constexpr uint32_t KV_PANEL = 64u * 128u;            // 64 rows x 64 columns
  static constexpr uint32_t Q_BYTES = 4u * Q_PANEL;           // 64 KB
  static constexpr uint32_t KV_BYTES = 4u * KV_PANEL;         // 32 KB
  static constexpr int SLOTS = 2;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + SLOTS * KV_BYTES;
  static constexpr uint32_t BAR_OFF = V_OFF + SLOTS * KV_BYTES;
  static constexpr int B_Q_FULL = 0;
  static constexpr int B_K_FULL = 1;                 // [SLOTS]
  static constexpr int B_K_EMPTY = B_K_FULL + SLOTS;  // [SLOTS]
  static constexpr int B_V_FULL = B_K_EMPTY + SLOTS;  // [SLOTS]
  static constexpr int B_V_EMPTY = B_V_FULL + SLOTS;  // [SLOTS]
  static constexpr int B_S_FULL = B_V_EMPTY + SLOTS;  // [2]: one per S buffer
  // softmax group released P_j (128 arrivals), one per S buffer: the group
  // may release P_j+1 before the issuer has looked at P_j's barrier
  static constexpr int B_P_FULL = B_S_FULL + 2;       // [2]
  static constexpr int B_PV_DONE = B_P_FULL + 2;      // P_j V_j completed
  static constexpr int B_O_FULL = B_PV_DONE + 1;      // the last P V completed (once)
  static constexpr int B_DRAIN = B_O_FULL + 1;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 232448u, "shared memory");
};

// SPLIT: p.n_splits > 1 CTAs per query tile, split s taking the run
// [s*n/n_splits, (s+1)*n/n_splits) of the n key tiles the query tile visits
// and writing its normalised partial output and log-sum-exp in fp32 for the
// combine kernel (a row with no visible key in the run: O = 0, -inf).
template <bool FULL, bool SPLIT>
__global__ void __launch_bounds__(D256_THREADS, 1)
    fattn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  using C = D256Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int hd = FULL ? D256 : p.hd;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  // the unit: (bh, query tile).  CTAs run in groups of head_group heads (the
  // last group may be smaller); within a group the latest query tiles (the
  // heaviest under causal) of all its heads come first.
  const int BH = p.B * p.H;
  const int n_qt = (p.N + BM - 1) / BM;
  const int u = (int)blockIdx.x;
  const int ns = SPLIT ? p.n_splits : 1;
  const int split = SPLIT ? u % ns : 0;
  const int ub = SPLIT ? u / ns : u;  // the query tile's unit (the splits of one tile are neighbours)
  const int per_group = p.head_group * n_qt;
  const int g0 = (ub / per_group) * p.head_group;
  const int gsz = min(p.head_group, BH - g0);
  const int rem = ub % per_group;
  const int bh = g0 + rem % gsz;
  const int it_rev = rem / gsz;
  const int it = p.causal ? n_qt - 1 - it_rev : it_rev;
  const int row0 = it * BM;
  int kl = p.key_len ? p.key_len[bh / p.H] : p.N;
  kl = kl < 0 ? 0 : (kl > p.N ? p.N : kl);
  const int max_lim = p.causal ? min(kl, row0 + BM) : kl;
  const int min_lim = p.causal ? min(kl, row0 + 1) : kl;
  const int n_all = max_lim > 0 ? (max_lim + D256_BN - 1) / D256_BN : 0;  // key tiles the query tile visits
  const int j0 = split * n_all / ns;                                      // this CTA's run of them:
  const int n = (split + 1) * n_all / ns - j0;                            // tiles j0 .. j0 + n - 1

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q_FULL), 1);
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(bar(C::B_K_FULL + s), 1);
      mbar_init(bar(C::B_K_EMPTY + s), 1);
      mbar_init(bar(C::B_V_FULL + s), 1);
      mbar_init(bar(C::B_V_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_S_FULL + 1), 1);
    mbar_init(bar(C::B_P_FULL), BM);
    mbar_init(bar(C::B_P_FULL + 1), BM);
    mbar_init(bar(C::B_PV_DONE), 1);
    mbar_init(bar(C::B_O_FULL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == D256_PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == D256_MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  if constexpr (SPLIT) pdl_launch_dependents();  // the combine kernel may launch now (it waits before reading)
  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};

  if (warp == D256_PRODUCER_WARP) {
    if (lane == 0 && n > 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      mbar_arrive_expect_tx(bar(C::B_Q_FULL), C::Q_BYTES);
#pragma unroll
      for (int pn = 0; pn < 4; ++pn)
        tma_load_3d(base + C::Q_OFF + pn * C::Q_PANEL, &tmap_q, bar(C::B_Q_FULL), 64 * pn, row0, bh);
      int kk = 0, vv = 0;  // K and V tiles issued
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % C::SLOTS;
        const uint32_t ph = ((uint32_t)(j / C::SLOTS) & 1u) ^ 1u;
        ok = wait_bar(waiter, bar(C::B_K_EMPTY + s), ph, C::B_K_EMPTY + s, u);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_K_FULL + s), C::KV_BYTES);
#pragma unroll
        for (int pn = 0; pn < 4; ++pn)
          tma_load_3d(base + C::K_OFF + s * C::KV_BYTES + pn * C::KV_PANEL, &tmap_k, bar(C::B_K_FULL + s), 64 * pn,
                      (j0 + j) * D256_BN, bh);
        ++kk;
        ok = wait_bar(waiter, bar(C::B_V_EMPTY + s), ph, C::B_V_EMPTY + s, u);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_V_FULL + s), C::KV_BYTES);
#pragma unroll
        for (int pn = 0; pn < 4; ++pn)
          tma_load_3d(base + C::V_OFF + s * C::KV_BYTES + pn * C::KV_PANEL, &tmap_v, bar(C::B_V_FULL + s), 64 * pn,
                      (j0 + j) * D256_BN, bh);
        ++vv;
      }
      // drain: copies that may still be in flight after an abort
      drain_wait(bar(C::B_Q_FULL), 0, 20000000ull);
      for (int j = kk > C::SLOTS ? kk - C::SLOTS : 0; j < kk; ++j)
        drain_wait(bar(C::B_K_FULL + j % C::SLOTS), (uint32_t)(j / C::SLOTS) & 1u, 20000000ull);
      for (int j = vv > C::SLOTS ? vv - C::SLOTS : 0; j < vv; ++j)
        drain_wait(bar(C::B_V_FULL + j % C::SLOTS), (uint32_t)(j / C::SLOTS) & 1u, 20000000ull);
    }
  } else if (warp == D256_MMA_WARP) {
    if (n > 0) {
      waiter.role = ROLE_MMA;
      constexpr uint32_t IDESC_S = idesc_f16kind(BM, D256_BN, true, false);       // Q, K bf16, K-major
      constexpr uint32_t IDESC_PV_F16 = idesc_f16kind(BM, D256, false, true);    // P, V fp16; V MN-major
      constexpr uint32_t IDESC_PV_BF16 = idesc_f16kind(BM, D256, true, true);    // P, V bf16
      const uint64_t q_desc = smem_desc(base + C::Q_OFF, 16, 1024);
      const uint64_t k_desc0 = smem_desc(base + C::K_OFF, 16, 1024);
      const uint64_t v_desc0 = smem_desc(base + C::V_OFF, C::KV_PANEL, 1024);
      const uint8_t* modes = p.v_mode + (size_t)bh * p.mode_stride;
      bool ok = true;
      auto wait_k = [&](int j) {
        const int s = j % C::SLOTS;
        ok = ok && wait_bar(waiter, bar(C::B_K_FULL + s), (uint32_t)(j / C::SLOTS) & 1u, C::B_K_FULL + s, u);
        ok = __all_sync(0xffffffffu, ok);
      };
      // S_j = Q K_j^T into buffer j % 2; then K_j's slot is free
      auto issue_s = [&](int j) {
        const uint64_t kd = k_desc0 + (uint64_t)(((uint32_t)(j % C::SLOTS) * C::KV_BYTES) >> 4);
        const uint32_t dt = tmem + D256_TMEM_S + 64u * (uint32_t)(j & 1);
        tc_fence_after();
        // 16 MMAs of K = 16 behind one elect (Q panels 16 KB, K panels 8 KB apart)
        static_assert(D256 == 256 && C::Q_PANEL == 16384u && C::KV_PANEL == 8192u, "panel strides of the batch");
        mma_ss_batch16_a128_b64(dt, q_desc, kd, IDESC_S, 0u);
        mma_commit_w(bar(C::B_S_FULL + (j & 1)));
        mma_commit_w(bar(C::B_K_EMPTY + j % C::SLOTS));
      };
      ok = wait_bar(waiter, bar(C::B_Q_FULL), 0, C::B_Q_FULL, u);
      ok = __all_sync(0xffffffffu, ok);
      bool issued_any = false;
      if (ok) {
        wait_k(0);
        if (ok) {
          issued_any = true;
          issue_s(0);
        }
      }
      if (ok && n > 1) {
        wait_k(1);
        if (ok) issue_s(1);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % C::SLOTS;
        const uint32_t idesc_pv =
            __ldg(modes + ((j0 + j) * D256_BN) / BN) == VMODE_F16 ? IDESC_PV_F16 : IDESC_PV_BF16;
        ok = wait_bar(waiter, bar(C::B_P_FULL + (j & 1)), (uint32_t)(j >> 1) & 1u, C::B_P_FULL + (j & 1), u);
        if (ok) ok = wait_bar(waiter, bar(C::B_V_FULL + s), (uint32_t)(j / C::SLOTS) & 1u, C::B_V_FULL + s, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // O (+)= P_j V_j: P_j packed over the first 32 columns of its S buffer
        const uint64_t vd = v_desc0 + (uint64_t)(((uint32_t)s * C::KV_BYTES) >> 4);
        const uint32_t at = tmem + D256_TMEM_S + 64u * (uint32_t)(j & 1);
        // 4 MMAs of 16 keys behind one elect (16 keys = 8 TMEM columns of P and
        // two 1024-byte row groups of V)
        static_assert(D256_BN == 64, "the P V batch issues 4 MMAs of 16 keys");
        mma_ts_batch4(tmem + D256_TMEM_O, at, vd, idesc_pv, j > 0 ? 1u : 0u);
        mma_commit_w(bar(C::B_PV_DONE));
        mma_commit_w(bar(C::B_V_EMPTY + s));
        if (j + 2 < n) {
          wait_k(j + 2);
          if (!ok) break;
          issue_s(j + 2);
        }
      }
      if (ok) mma_commit_w(bar(C::B_O_FULL));
      if (issued_any) {
        mma_commit_w(bar(C::B_DRAIN));
        drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
      }
    }
  } else if (warp < 4) {
    waiter.role = ROLE_SOFTMAX;
    const int row_in_tile = warp * 32 + lane;
    const int row = row0 + row_in_tile;
    const bool row_ok = row < p.N;
    const size_t row_flat = (size_t)bh * (size_t)p.N + (size_t)row;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + D256_TMEM_O;
    const float c = p.scale_log2;
    if (n == 0) {
      // no visible key: O = 0, LSE = -inf (an empty split run writes
      // nothing: the combine reads only the runs that hold key tiles)
      if (!SPLIT && row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + row_flat * hd);
        for (int i = 0; i < hd / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        p.lse[row_flat] = -INFINITY;
      }
    } else {
      const int lim = p.causal ? min(kl, row + 1) : kl;  // keys [0, lim) are visible
      const uint8_t* modes = p.v_mode + (size_t)bh * p.mode_stride;
      float m_ref = -INFINITY, l = 0.0f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t s_addr = tmem + lane_off + D256_TMEM_S + 64u * (uint32_t)(j & 1);
        const int vmode = __ldg(modes + ((j0 + j) * D256_BN) / BN);
        ok = wait_bar(waiter, bar(C::B_S_FULL + (j & 1)), (uint32_t)(j >> 1) & 1u, C::B_S_FULL + (j & 1), u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const bool masked_tile = (j0 + j + 1) * D256_BN > min_lim;
        const int vis_n = lim - (j0 + j) * D256_BN;  // columns [0, vis_n) visible
        // S row of this tile; its max from the TMEM load's max reduction when
        // no column is masked, else over the visible columns (tree order)
        float sr[64];
        float mx;
        if (!masked_tile) {
          tmem_ld64_max(s_addr, sr, mx);
          tmem_ld_wait(sr, mx);
        } else {
          {
            uint32_t r32[64];
            tmem_ld64(s_addr, r32);
            tmem_ld_wait(r32);
#pragma unroll
            for (int i = 0; i < 64; ++i) sr[i] = i < vis_n ? __uint_as_float(r32[i]) : -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmax3(sr[i], sr[i + 8], sr[i + 16]);
#pragma unroll
          for (int i = 24; i < 64; i += 16) {
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], sr[i + k], i + 8 + k < 64 ? sr[i + 8 + k] : -INFINITY);
          }
          mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        }
        const float m_new = fmaxf(m_ref, mx);
        float alpha = 1.0f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = m_new;  // the first tile: O is overwritten by its P V
        } else if ((m_new - m_ref) * c > RESCALE_LOG2_THRESHOLD) {
          alpha = ex2((m_ref - m_new) * c);
          m_ref = m_new;
          rescale = true;
        }
        // (a split run can hold rows with no visible key yet: m stays -inf
        // and every p of theirs is masked to 0)
        const float mc = m_ref == -INFINITY ? 0.0f : m_ref * c;
        // p = 2^(s*c - m*c) (packed f32x2 FMA, then ex2), masked entries
        // exactly 0; l from the unrounded p in four packed partial sums; P
        // rounded to the V tile's operand type
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nmc2 = f2_pack(-mc, -mc);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[32];
        // one copy of the loop per (mask, operand type), so that the common
        // case (no mask, fp16) carries no per-element selects
        auto exp_loop = [&](auto masked_c, auto f16_c) {
          constexpr bool MASKED = decltype(masked_c)::value, F16 = decltype(f16_c)::value;
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sr[2 * q], sr[2 * q + 1]), c2, nmc2), x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if constexpr (MASKED) {
              p0 = 2 * q < vis_n ? p0 : 0.0f;
              p1 = 2 * q + 1 < vis_n ? p1 : 0.0f;
            }
            acc[q % 4] = f2_add(acc[q % 4], f2_pack(p0, p1));
            pk[q] = F16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
        };
        const bool f16 = vmode == VMODE_F16;
        if (masked_tile) {
          if (f16)
            exp_loop(std::true_type{}, std::true_type{});
          else
            exp_loop(std::true_type{}, std::false_type{});
        } else {
          if (f16)
            exp_loop(std::false_type{}, std::true_type{});
          else
            exp_loop(std::false_type{}, std::false_type{});
        }
        float a0, a1, a2, a3, a4, a5, a6, a7;
        f2_unpack(acc[0], a0, a1);
        f2_unpack(acc[1], a2, a3);
        f2_unpack(acc[2], a4, a5);
        f2_unpack(acc[3], a6, a7);
        const float rs = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
        l = l * alpha + rs;
        if (__any_sync(0xffffffffu, rescale)) {
          // O must not change under the previous P V product: wait for it.
          // Waited only here and in the epilogue: when tile j's S has landed,
          // P_j-2 V_j-2 has completed (S_j was issued after it) and P_j V_j
          // cannot start before this P is released, so the barrier is at
          // phase j-1 or j and the parity of phase j-1 names it exactly.
          if (j > 0) {
            ok = wait_bar(waiter, bar(C::B_PV_DONE), (uint32_t)(j - 1) & 1u, C::B_PV_DONE, u);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll 1
          for (int cc = 0; cc < D256 / 32; ++cc) {
            uint32_t r32[32];
            tmem_ld32(o_addr + 32u * cc, r32);
            tmem_ld_wait(r32);
#pragma unroll
            for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(__uint_as_float(r32[i]) * alpha);
            tmem_st32(o_addr + 32u * cc, r32);
          }
        }
        tmem_st32(s_addr, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_P_FULL + (j & 1)));
      }
      if (ok) {
        // epilogue: the last P V product (its own barrier: P V products may
        // still be two deep here), then O / l -> bf16, LSE = m*scale + ln(l)
        ok = wait_bar(waiter, bar(C::B_O_FULL), 0, C::B_O_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok && SPLIT) {
        // this run's O / l and log-sum-exp in fp32, for the combine kernel
        // (O = 0 and -inf for a row with no visible key in the run)
        tc_fence_after();
        const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
        const size_t orow = (size_t)split * (size_t)BH * (size_t)p.N + row_flat;
        float4* dstf = reinterpret_cast<float4*>(p.o_part + orow * hd);
#pragma unroll 1
        for (int hcol = 0; hcol < D256 / 64; ++hcol) {
          uint32_t ov[64];
          tmem_ld64(o_addr + 64u * hcol, ov);
          tmem_ld_wait(ov);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (64 * hcol + 4 * i < hd)
                dstf[16 * hcol + i] =
                    make_float4(__uint_as_float(ov[4 * i]) * inv_l, __uint_as_float(ov[4 * i + 1]) * inv_l,
                                __uint_as_float(ov[4 * i + 2]) * inv_l, __uint_as_float(ov[4 * i + 3]) * inv_l);
          }
        }
        if (row_ok) p.lse_part[orow] = l > 0.0f ? (m_ref * c + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      } else if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        uint4* dst = reinterpret_cast<uint4*>(p.o + row_flat * hd);
#pragma unroll 1
        for (int hcol = 0; hcol < D256 / 64; ++hcol) {
          uint32_t ov[64];
          tmem_ld64(o_addr + 64u * hcol, ov);
          tmem_ld_wait(ov);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (64 * hcol + 8 * i < hd)
                dst[8 * hcol + i] = make_uint4(
                    pack_bf16x2(__uint_as_float(ov[8 * i]) * inv_l, __uint_as_float(ov[8 * i + 1]) * inv_l),
                    pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv_l, __uint_as_float(ov[8 * i + 3]) * inv_l),
                    pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv_l, __uint_as_float(ov[8 * i + 5]) * inv_l),
                    pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv_l, __uint_as_float(ov[8 * i + 7]) * inv_l));
          }
        }
        if (row_ok) p.lse[row_flat] = (m_ref * c + __log2f(l)) * 0.69314718055994531f;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == D256_MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace fattn
