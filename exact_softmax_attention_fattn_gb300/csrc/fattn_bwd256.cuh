// Exact softmax attention backward for head dims 136..256, sm_103a.
//
// Same result as fattn_bwd.cuh ("understand-flashattention", section
// "Attention forward and backward formulas", backward pass steps 1-5, with P
// recomputed from the saved logsumexp):
//     P = exp(S - LSE),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//     dQ = scale * dS K,  dK = scale * dS^T Q,   D_i = rowsum(dO_i * O_i).
//
// Why a layout of its own: tensor memory has 512 columns; S (128), dP (128)
// and one 256-column accumulator fill it, so a 256-column head dim cannot
// keep dV and dK (nor dK and dQ) in tensor memory together.  The gradient is
// computed in three passes, one accumulator each:
//   * dV pass, one CTA per (batch*head, 128-key tile): S^T = K Q_i^T, P^T,
//     dV += P^T dO_i over the query tiles i that see the key tile;
//   * dK pass, one CTA per key tile: S^T, dP^T = V dO_i^T, dS^T,
//     dK += dS^T Q_i;
//   * dQ pass, one CTA per 128-query tile: S = Q K_j^T, dP = dO V_j^T, dS,
//     dQ += dS K_j over the key tiles j the query tile sees.
// Every operand moves as 128-column halves (128 rows x 128 columns of bf16,
// two 128-byte-swizzled panels): the CTA's own tiles stay resident (two
// halves in the dV pass, four in the others), the streamed tile's pair of
// halves sits in buffer A and the other streamed operand passes through half
// buffers X: two in the dV pass (both halves of dO in flight at once, 192 KB
// of shared memory), one in the others (half a then half b, 224 KB).
// The 256-column products are two N = 128 products, one per output half; the
// 256-deep contractions S and dP are two K = 128 batches accumulated.
// Roles as in fattn_bwd.cuh: warps 0-7 elementwise (group g = warp / 4 takes
// tile columns [64g, 64g + 64) of lane quarter warp % 4), warp 8 the TMA
// producer (one lane), warp 9 the MMA issuer.  Every wait is bounded.
#pragma once

#include "fattn_bwd.cuh"
#include "fattn_d256.cuh"

namespace fattn {

enum : int { BP_DV = 0, BP_DK = 1, BP_DQ = 2 };

template <int PASS>
struct Bwd256Cfg {
  static constexpr uint32_t HALF = 2u * PANEL_BYTES;   // 128 rows x 128 columns of bf16
  static constexpr int N_RES = PASS == BP_DV ? 2 : 4;  // resident halves
  static constexpr uint32_t RES_OFF = 0;
  static constexpr uint32_t A_OFF = N_RES * HALF;       // the streamed tile's two halves
  static constexpr uint32_t X_OFF = A_OFF + 2u * HALF;  // the other streamed operand, one half at a time
  // the dV pass has room for both halves of dO (one buffer each); the others
  // pass their two halves through one buffer
  static constexpr int N_X = PASS == BP_DV ? 2 : 1;
  static constexpr uint32_t BAR_OFF = X_OFF + N_X * HALF;
  static constexpr int B_RES_FULL = 0;
  static constexpr int B_A_FULL = 1;
  static constexpr int B_A_EMPTY = 2;
  static constexpr int B_X_FULL = 3;
  static constexpr int B_X_EMPTY = 4;
  static constexpr int B_S_FULL = 5;
  static constexpr int B_DP_FULL = 6;
  static constexpr int B_OPS = 7;  // P^T (dV pass) or dS / dS^T stored by the elementwise warps
  static constexpr int B_ACC_FULL = 8;
  static constexpr int B_DRAIN = 9;
  static constexpr int B_X1_FULL = 10;   // dV pass: the second half's buffer
  static constexpr int B_X1_EMPTY = 11;
  static constexpr int NUM_BARS = 12;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tmem base (4 B) + abort flag (4 B)
  // + slack for 1024-byte alignment; at least 120 KB so that one CTA holds an SM
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16 + 1024;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 120u * 1024u ? SMEM_USED : 120u * 1024u;
  static_assert(SMEM_BYTES <= 232448u, "shared memory");
};

template <int PASS>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fattn_bwd256_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                        const BwdParams p) {
  using C = Bwd256Cfg<PASS>;
  constexpr bool KEYS = PASS != BP_DQ;  // the CTA owns a key tile (dV, dK) or a query tile (dQ)
  constexpr uint32_t IDESC_SS = idesc_f16kind(128, 128, true, false);  // both operands K-major
  constexpr uint32_t IDESC_TS = idesc_f16kind(128, 128, true, true);   // B MN-major
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  // the CTA's own tile (rows r0 .. r0 + 127) and the streamed tiles
  // first .. first + count - 1, heaviest CTAs first under causal (the first
  // key tiles see the most queries, the last query tiles the most keys)
  const int BH = p.B * p.H;
  const int bh = (int)(blockIdx.x % BH);
  const int t_rev = (int)(blockIdx.x / BH);
  const int t_own = (KEYS || !p.causal) ? t_rev : p.n_tiles - 1 - t_rev;
  const int r0 = t_own * 128;
  const int kl = clamp_kl(p, bh / p.H);
  int first, count;
  if constexpr (KEYS) {
    first = p.causal ? t_own : 0;
    count = r0 < kl ? p.n_tiles - first : 0;
  } else {
    const int max_lim = p.causal ? min(kl, r0 + 128) : kl;
    first = 0;
    count = max_lim > 0 ? (max_lim + 127) / 128 : 0;
  }
  const int u = (int)blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_RES_FULL), 1);
    mbar_init(bar(C::B_A_FULL), 1);
    mbar_init(bar(C::B_A_EMPTY), 1);
    mbar_init(bar(C::B_X_FULL), 1);
    mbar_init(bar(C::B_X_EMPTY), 1);
    mbar_init(bar(C::B_X1_FULL), 1);
    mbar_init(bar(C::B_X1_EMPTY), 1);
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    mbar_init(bar(C::B_OPS), 32 * BWD_ELEM_WARPS);
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
  pdl_launch_dependents();

  if (count > 0 && warp == BWD_PRODUCER_WARP) {
    if (lane == 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      // half h (columns [128h, 128h + 128)) of the 128 rows from `row`
      auto load_half = [&](uint32_t dst, const CUtensorMap* map, int h, int row, uint32_t full) {
        tma_load_3d(dst, map, full, 128 * h, row, bh);
        tma_load_3d(dst + PANEL_BYTES, map, full, 128 * h + 64, row, bh);
      };
      // resident: K (and V), or Q and dO
      mbar_arrive_expect_tx(bar(C::B_RES_FULL), (uint32_t)C::N_RES * C::HALF);
      for (int h = 0; h < 2; ++h)
        load_half(base + C::RES_OFF + (uint32_t)h * C::HALF, KEYS ? &tmap_k : &tmap_q, h, r0, bar(C::B_RES_FULL));
      if constexpr (C::N_RES == 4)
        for (int h = 0; h < 2; ++h)
          load_half(base + C::RES_OFF + (uint32_t)(2 + h) * C::HALF, KEYS ? &tmap_v : &tmap_do, h, r0,
                    bar(C::B_RES_FULL));
      // streamed: the pair (Q, or K) into A, then the other operand (dO, or
      // V) one half at a time through X
      const CUtensorMap* map_a = KEYS ? &tmap_q : &tmap_k;
      const CUtensorMap* map_x = PASS == BP_DQ ? &tmap_v : &tmap_do;
      int issued_a = 0, issued_x = 0;
      for (int n = 0; ok && n < count; ++n) {
        const int rs = (first + n) * 128;
        ok = wait_bar(waiter, bar(C::B_A_EMPTY), (uint32_t)(n & 1) ^ 1u, C::B_A_EMPTY, u);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_A_FULL), 2u * C::HALF);
        for (int h = 0; h < 2; ++h) load_half(base + C::A_OFF + (uint32_t)h * C::HALF, map_a, h, rs, bar(C::B_A_FULL));
        issued_a = n + 1;
        for (int h = 0; ok && h < 2; ++h) {
          if constexpr (C::N_X == 2) {
            // half h in buffer h, its phases counted per tile
            const int full = h ? C::B_X1_FULL : C::B_X_FULL, empty = h ? C::B_X1_EMPTY : C::B_X_EMPTY;
            ok = wait_bar(waiter, bar(empty), (uint32_t)(n & 1) ^ 1u, empty, u);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(full), C::HALF);
            load_half(base + C::X_OFF + (uint32_t)h * C::HALF, map_x, h, rs, bar(full));
            issued_x = n + 1;
          } else {
            const int x = 2 * n + h;
            ok = wait_bar(waiter, bar(C::B_X_EMPTY), (uint32_t)(x & 1) ^ 1u, C::B_X_EMPTY, u);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(C::B_X_FULL), C::HALF);
            load_half(base + C::X_OFF, map_x, h, rs, bar(C::B_X_FULL));
            issued_x = x + 1;
          }
        }
      }
      // drain: copies that may still be in flight after an abort
      drain_wait(bar(C::B_RES_FULL), 0, 20000000ull);
      if (issued_a) drain_wait(bar(C::B_A_FULL), (uint32_t)(issued_a - 1) & 1u, 20000000ull);
      if (issued_x) drain_wait(bar(C::B_X_FULL), (uint32_t)(issued_x - 1) & 1u, 20000000ull);
      if (C::N_X == 2 && issued_x) drain_wait(bar(C::B_X1_FULL), (uint32_t)(issued_x - 1) & 1u, 20000000ull);
    }
  } else if (count > 0 && warp == BWD_MMA_WARP) {
    // Per streamed tile n: S (two K = 128 batches), then (dK, dQ passes) dP
    // the same way over X's two halves; once the elementwise warps have
    // stored P^T (dV) or dS: the two N = 128 halves of the accumulator.  The
    // next tile's S is issued after that, so it overwrites S only once P^T
    // was consumed (the tensor pipe runs in order) and the elementwise warps
    // have read S and dP.
    waiter.role = ROLE_MMA;
    bool ok = wait_bar(waiter, bar(C::B_RES_FULL), 0, C::B_RES_FULL, u);
    ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    auto kdesc = [&](uint32_t off) { return smem_desc(base + off, 16, 1024); };          // K-major half
    auto ndesc = [&](uint32_t off) { return smem_desc(base + off, PANEL_BYTES, 1024); };  // MN-major half
    for (int n = 0; ok && n < count; ++n) {
      ok = wait_bar(waiter, bar(C::B_A_FULL), (uint32_t)n & 1u, C::B_A_FULL, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      issued_any = true;
      // S^T = K Q^T (dV, dK) or S = Q K^T (dQ): resident halves x A's halves
      mma_ss_batch<8>(tmem + BT_S, kdesc(C::RES_OFF), kdesc(C::A_OFF), IDESC_SS, 0u);
      mma_ss_batch<8>(tmem + BT_S, kdesc(C::RES_OFF + C::HALF), kdesc(C::A_OFF + C::HALF), IDESC_SS, 1u);
      mma_commit_w(bar(C::B_S_FULL));
      if constexpr (PASS == BP_DV) {
        mma_commit_w(bar(C::B_A_EMPTY));  // Q is not needed again
      } else {
        // dP^T = V dO^T (dK) or dP = dO V^T (dQ): resident halves 2, 3 x X
        for (int h = 0; ok && h < 2; ++h) {
          const int x = 2 * n + h;
          ok = wait_bar(waiter, bar(C::B_X_FULL), (uint32_t)x & 1u, C::B_X_FULL, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          mma_ss_batch<8>(tmem + BT_DP, kdesc(C::RES_OFF + (uint32_t)(2 + h) * C::HALF), kdesc(C::X_OFF), IDESC_SS,
                          (uint32_t)h);
          mma_commit_w(bar(C::B_X_EMPTY));
        }
        if (!ok) break;
        mma_commit_w(bar(C::B_DP_FULL));
      }
      ok = wait_bar(waiter, bar(C::B_OPS), (uint32_t)n & 1u, C::B_OPS, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = n > 0 ? 1u : 0u;
      if constexpr (PASS == BP_DV) {
        // dV half h += P^T dO half h (P^T packed over S's columns; dO half h
        // in buffer h)
        for (int h = 0; ok && h < 2; ++h) {
          const int full = h ? C::B_X1_FULL : C::B_X_FULL, empty = h ? C::B_X1_EMPTY : C::B_X_EMPTY;
          ok = wait_bar(waiter, bar(full), (uint32_t)n & 1u, full, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          mma_ts_batch8_halves(tmem + BT_ACC0 + 128u * (uint32_t)h, tmem + BT_S,
                               ndesc(C::X_OFF + (uint32_t)h * C::HALF), IDESC_TS, acc);
          mma_commit_w(bar(empty));
        }
      } else {
        // dK half h += dS^T Q half h, or dQ half h += dS K half h (dS packed
        // over dP's columns; Q or K still in A)
        for (int h = 0; h < 2; ++h)
          mma_ts_batch8_halves(tmem + BT_ACC0 + 128u * (uint32_t)h, tmem + BT_DP,
                               ndesc(C::A_OFF + (uint32_t)h * C::HALF), IDESC_TS, acc);
        mma_commit_w(bar(C::B_A_EMPTY));
      }
    }
    if (ok) mma_commit_w(bar(C::B_ACC_FULL));
    if (issued_any) {
      mma_commit_w(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
    }
  } else if (warp < BWD_ELEM_WARPS) {
    // LSE2 and D come from the prep kernel; only these warps read them, and
    // every CTA waits here so that this grid ends after the ones before it
    pdl_wait();
    waiter.role = ROLE_SOFTMAX;
    const int g = warp / 4;             // column group: tile columns [64g, 64g + 64)
    const int quarter = warp % 4;       // TMEM lane quarter
    const int r = quarter * 32 + lane;  // row within the CTA's own tile = TMEM lane
    const int own = r0 + r;             // the key (dV, dK) or query (dQ) of this lane
    const bool row_ok = own < p.N;
    const size_t row_flat = (size_t)bh * (size_t)p.N + (size_t)own;
    __nv_bfloat16* out = PASS == BP_DV ? p.dv : (PASS == BP_DK ? p.dk : p.dq);
    const float out_mul = PASS == BP_DV ? 1.0f : p.scale;
    if (count == 0) {
      store_zero_part<D256>(out, row_flat, row_ok, p.hd, g);
    } else {
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      // this group's 64 columns of S (S^T) and dP (dP^T); P^T, dS^T or dS are
      // packed over the first 32 of them
      const uint32_t s_addr = tmem + lane_off + BT_S + 64u * (uint32_t)g;
      const uint32_t dp_addr = tmem + lane_off + BT_DP + 64u * (uint32_t)g;
      const float c = p.scale_log2;
      const size_t rows_bh = (size_t)bh * (size_t)p.N_pad;
      // dQ pass: LSE and D are constants of the lane's query row (rows past N
      // are padding, 0)
      const float nlse2_row = KEYS ? 0.0f : __ldg(p.nlse2 + rows_bh + own);
      const float delta_row = KEYS ? 0.0f : __ldg(p.delta + rows_bh + own);
      bool ok = true;
      for (int n = 0; ok && n < count; ++n) {
        const int rs = (first + n) * 128;  // first row of the streamed tile
        const int c0 = rs + 64 * g;        // key or query index of this group's column 0
        ok = wait_bar(waiter, bar(C::B_S_FULL), (uint32_t)n & 1u, C::B_S_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // visibility: key < key_len and (causal) key <= query.  dV, dK: the
        // lane is a key and the columns are queries c0 + i (rows past N read
        // as zero and contribute nothing: their dO and Q are zero); dQ: the
        // lane is a query and the columns are keys c0 + i.
        int first_vis, end_vis;  // columns [first_vis, end_vis) visible
        if constexpr (KEYS) {
          first_vis = own < kl ? (p.causal ? max(0, own - c0) : 0) : 64;
          end_vis = 64;
        } else {
          first_vis = 0;
          end_vis = min(64, max(0, (p.causal ? min(kl, own + 1) : kl) - c0));
        }
        const bool any_mask = first_vis > 0 || end_vis < 64;
        const float4* nlse4 = reinterpret_cast<const float4*>(p.nlse2 + rows_bh + c0);
        float pr[64];
        {
          uint32_t sh[64];
          tmem_ld64(s_addr, sh);
          tmem_ld_wait(sh);
          // a separate copy of the loop for tiles with masked columns, so
          // that the others carry no per-element selects
          auto p_loop = [&](auto masked_c) {
            constexpr bool MASKED = decltype(masked_c)::value;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              // exponent arguments S c - LSE2, two per f32x2 FMA: -LSE2 per
              // column (dV, dK passes) or per row (dQ pass)
              const uint64_t c2 = f2_pack(c, c);
              uint64_t nl[2];
              if constexpr (KEYS) {
                const float4 l4 = __ldg(nlse4 + q4);
                nl[0] = f2_pack(l4.x, l4.y);
                nl[1] = f2_pack(l4.z, l4.w);
              } else {
                nl[0] = nl[1] = f2_pack(nlse2_row, nlse2_row);
              }
              float x[4];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int i = 4 * q4 + 2 * h;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[i]), __uint_as_float(sh[i + 1])), c2, nl[h]), x[2 * h],
                          x[2 * h + 1]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * q4 + e;
                float pe = ex2(x[e]);
                if constexpr (MASKED) pe = (i >= first_vis && i < end_vis) ? pe : 0.0f;
                pr[i] = pe;
              }
            }
          };
          if (any_mask)
            p_loop(std::true_type{});
          else
            p_loop(std::false_type{});
        }
        if constexpr (PASS == BP_DV) {
          uint32_t pk[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) pk[q] = pack_bf16x2(pr[2 * q], pr[2 * q + 1]);
          tmem_st32(s_addr, pk);
        } else {
          // dS = P (dP - D): D per column (dK pass) or per row (dQ pass)
          ok = wait_bar(waiter, bar(C::B_DP_FULL), (uint32_t)n & 1u, C::B_DP_FULL, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          uint32_t dh[64];
          tmem_ld64(dp_addr, dh);
          tmem_ld_wait(dh);
          const float4* del4 = reinterpret_cast<const float4*>(p.delta + rows_bh + c0);
          uint32_t pk[32];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            float dv[4];
            if constexpr (KEYS) {
              const float4 d4 = __ldg(del4 + q4);
              dv[0] = d4.x, dv[1] = d4.y, dv[2] = d4.z, dv[3] = d4.w;
            } else {
              dv[0] = dv[1] = dv[2] = dv[3] = delta_row;
            }
            // two columns per f32x2 op (the same roundings as the scalar form)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = 4 * q4 + 2 * h;
              const uint64_t ds = f2_mul(f2_pack(pr[i], pr[i + 1]),
                                         f2_sub(f2_pack(__uint_as_float(dh[i]), __uint_as_float(dh[i + 1])),
                                                f2_pack(dv[2 * h], dv[2 * h + 1])));
              float lo, hi;
              f2_unpack(ds, lo, hi);
              pk[2 * q4 + h] = pack_bf16x2(lo, hi);
            }
          }
          tmem_st32(dp_addr, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_OPS));
      }
      if (ok) {
        ok = wait_bar(waiter, bar(C::B_ACC_FULL), 0, C::B_ACC_FULL, u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        store_acc_part<D256>(tmem + lane_off + BT_ACC0, out_mul, out, row_flat, row_ok, p.hd, g);
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
