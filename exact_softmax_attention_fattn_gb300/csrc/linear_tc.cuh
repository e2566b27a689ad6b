// Causal linear attention on the tensor cores, sm_103a (feature sizes E, M up
// to 64; larger sizes run the CUDA-core kernels of linear_attn.cuh).
//
// What it computes is the page's ("Linear Attention CUDA kernel":
// CausalLinearAttention.forward with elu + 1 features, the key-length mask,
// its causal dot product and normaliser), per (b, h) and row i:
//     qt_i = phi(q_i),  kt_j = phi(k_j) for j < key_len[b] else 0,
//     out_i = (sum_{j <= i} (qt_i . kt_j) v_j) / (qt_i . sum_{j <= i} kt_j + eps).
//
// The same sums, regrouped over tiles of 128 rows.  With S_t = sum of kt_j
// v_j^T and z_t = sum of kt_j over the rows before tile t (the page's running
// state at the tile's start), a tile's rows get
//     num = Qt S_t + tril(Qt Kt^T) V,   den = Qt z_t + rowsum(tril(Qt Kt^T)) + eps,
// and S_t+1 = S_t + Kt^T V.  A head's rows are cut into parts of whole tiles,
// one CTA per (head, part), each walking its tiles in order with S kept on
// chip; a part starts from the sum of the earlier parts' totals, which a
// first launch of the same kernel (STATE: the totals only) writes.
//
// fp32 in and out, as the page's float kernels.  Every product runs on
// tcgen05 (kind::f16) in three bf16 terms: each fp32 operand x is split into
// hi = bf16(x) and lo = bf16(x - hi) (16 significant bits together), and
// a b = a_hi b_hi + a_hi b_lo + a_lo b_hi, accumulated in fp32 in tensor
// memory; the dropped a_lo b_lo and the splits' own rounding are about 2^-17
// of |a b|.  The row sums of tril(Qt Kt^T) and the dot products Qt z, which
// take one value per row, are formed in fp32 on the CUDA cores.
//
// Roles (576 threads, one CTA per SM):
//   * warp 16 (one lane): TMA producer, fp32 tiles of Q, K, V (128 rows x 64
//     columns, zero past N and past the feature size) into a two-stage ring;
//   * warps 8-15: transform, in place in each stage: phi of Q and K (zero
//     past E, and K zero past the key length), the bf16 hi/lo split of Q, K
//     and V into 128-byte-swizzled operand tiles, and the key sums z;
//   * warp 17: issues tcgen05.mma; S = Qt Kt^T (tensor memory), num = Qt S_t
//     + A V, and S_t+1 = S_t + Kt^T V accumulated in tensor memory, where
//     Kt^T V is one M = 128 product of the stacked [Kt_hi | Kt_lo] (MN-major
//     A) with [V_hi | V_lo] (MN-major B): its four 64 x 64 quadrants are
//     hi.hi, hi.lo, lo.hi and lo.lo;
//   * warps 0-7, one row (tensor-memory lane) per thread and two warps per
//     lane quarter, each on half of the columns: A = tril(S) split into bf16
//     hi/lo back into tensor memory, the row's denominator, the output, and
//     after each tile the state S_t+1 (sum of the quadrants) split into the
//     shared-memory operand of the next tile's Qt S_t+1.
// The two groups of eight warps each meet at hardware named barriers that
// also AND the members' wait results, so a time-out is seen by the whole
// group at once.  Every other wait is bounded; on time-out the kernel records
// the error word, drains its own copies and MMAs, frees tensor memory and
// returns.
#pragma once

#include <cstdint>

#include "fattn_kernel.cuh"
#include "linear_attn.cuh"

namespace fattn {

constexpr int LTC_T = 128;  // rows per tile
constexpr int LTC_F = 64;   // feature columns of every operand tile (E, M <= 64, zero-padded)
constexpr int LTC_THREADS = 576;
constexpr int LTC_ROW_THREADS = 256;    // warps 0-7
constexpr int LTC_XF_THREADS = 256;     // warps 8-15
constexpr int LTC_PRODUCER_WARP = 16;
constexpr int LTC_MMA_WARP = 17;
constexpr int LTC_BAR_XF = 1;   // named barrier of the transform warps
constexpr int LTC_BAR_ROW = 2;  // named barrier of the row warps
constexpr uint32_t LTC_TMEM_S = 0;    // S = Qt Kt^T (128 columns), then A_hi / A_lo over it
constexpr uint32_t LTC_TMEM_NUM = 128;  // num (64 columns)
constexpr uint32_t LTC_TMEM_ST = 256;   // the running state, four quadrants (128 columns)

struct LtcParams {
  float* out;              // [B*H, N, M]
  const int32_t* key_len;  // [B] or nullptr
  float* tot;              // [B*H, n_parts, tot_stride]: each part's sum of kt v^T ([E][M]) then of kt ([E])
  int* err;                // int[4]
  int B, H, N, E, M;
  int n_parts, tiles_per_part, tot_stride;
  float eps;
  unsigned long long wait_limit_ns;
};

struct LtcCfg {
  static constexpr uint32_t TILE = LTC_T * LTC_F * 4;   // one fp32 tile; also its bf16 hi + lo tiles
  // A stage's bf16 operand tiles: per group of 8 rows, the hi atom (8 rows
  // x 128 bytes, 128-byte swizzle) then the lo atom, so that a group's hi
  // and lo atoms take exactly the 2048 bytes of its 8 fp32 rows.
  static constexpr uint32_t GROUP = 2048;               // stride between 8-row groups
  static constexpr uint32_t LO = 1024;                  // lo atom after the hi atom
  static constexpr uint32_t Q_OFF = 0, K_OFF = TILE, V_OFF = 2 * TILE;
  static constexpr uint32_t STAGE = 3 * TILE;
  static constexpr uint32_t PST_OFF = 2 * STAGE;        // state operand: hi [64 x 64] bf16, then lo
  static constexpr uint32_t PST_BYTES = LTC_F * 128;
  static constexpr uint32_t XCH_OFF = PST_OFF + 2 * PST_BYTES;  // fp32 [64][64]: lo-rows' quadrant sums
  static constexpr uint32_t Z_OFF = XCH_OFF + LTC_F * LTC_F * 4;  // z [64], z at each stage's tile start [2][64]
  static constexpr uint32_t RSQ_OFF = Z_OFF + 3 * LTC_F * 4;      // per row and column half: row sum + Qt . z
  static constexpr uint32_t BAR_OFF = RSQ_OFF + 2 * LTC_T * 4;
  static constexpr int B_FULL = 0;       // [2] TMA -> transform
  static constexpr int B_OPREADY = 2;    // [2] transform -> MMA (transform-warp arrivals)
  static constexpr int B_EMPTY = 4;      // [2] MMA -> producer
  static constexpr int B_S_FULL = 6;     // Qt Kt^T landed
  static constexpr int B_A_FULL = 7;     // A written (row-warp arrivals)
  static constexpr int B_NUM_FULL = 8;   // num complete
  static constexpr int B_NUM_EMPTY = 9;  // num read (row-warp arrivals)
  static constexpr int B_ST_DONE = 10;   // state update complete
  static constexpr int B_PST_READY = 11; // state operand written (row-warp arrivals)
  static constexpr int B_DRAIN = 12;
  static constexpr int NUM_BARS = 13;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tmem base, abort flag
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
  static_assert(SMEM_BYTES <= 232448u, "shared memory");
};

// Generic-proxy shared-memory writes made visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte chunk c (columns 8c .. 8c+7) of row r in a
// 128-byte-swizzled bf16 tile of 64 columns (chunk c XOR r % 8), with
// `group` bytes between groups of 8 rows.
__device__ __forceinline__ uint32_t ltc_swz16(int r, int c, uint32_t group = 1024u) {
  return (uint32_t)(r >> 3) * group + (uint32_t)(r & 7) * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}
// The same for the 8-byte half (columns 4*c4 .. 4*c4+3) of a chunk.
__device__ __forceinline__ uint32_t ltc_swz8(int r, int c4, uint32_t group = 1024u) {
  return ltc_swz16(r, c4 >> 1, group) + ((uint32_t)(c4 & 1) << 3);
}

// Splits two floats into packed bf16 pairs hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void ltc_split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  lo = pack_bf16x2(x0 - bf16lo_as_f32(hi), x1 - bf16hi_as_f32(hi));
}

// Instruction descriptor for kind::f16 with both operands bf16 and either
// operand K-major (false) or MN-major (true).
__host__ __device__ constexpr uint32_t ltc_idesc(int M, int N, bool a_mn_major, bool b_mn_major) {
  return idesc_f16kind(M, N, true, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// Barrier of one group of eight warps (named barrier `id`, 256 threads) that
// also ANDs every member's `ok`: all members get the same answer, so they
// leave a loop together after a time-out.
__device__ __forceinline__ bool ltc_group_and(int id, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(id)
      : "memory");
  return r != 0;
}

// STATE: only the part totals (sum of kt v^T and of kt over the part's rows),
// written to p.tot[bh, part]; grid B*H x (n_parts - 1).  Otherwise the
// outputs; grid B*H x n_parts.
template <bool STATE>
__global__ void __launch_bounds__(LTC_THREADS, 1)
    fattn_linear_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const LtcParams p) {
  using C = LtcCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);
  float* zmaster = reinterpret_cast<float*>(base_ptr + C::Z_OFF);
  float* zsnap = zmaster + LTC_F;  // [2][64]
  float* xch = reinterpret_cast<float*>(base_ptr + C::XCH_OFF);
  float* rsq = reinterpret_cast<float*>(base_ptr + C::RSQ_OFF);  // [2][128]

  const int parts_run = STATE ? p.n_parts - 1 : p.n_parts;
  const int bh = (int)(blockIdx.x / (unsigned)parts_run);
  const int part = (int)(blockIdx.x % (unsigned)parts_run);
  const int unit = (int)blockIdx.x;
  const int row0 = part * p.tiles_per_part * LTC_T;  // first row of the part
  const int row_end = min(p.N, row0 + p.tiles_per_part * LTC_T);
  const int nt = row_end > row0 ? (row_end - row0 + LTC_T - 1) / LTC_T : 0;
  int klim = p.key_len ? p.key_len[bh / p.H] : p.N;
  klim = klim < 0 ? 0 : (klim > p.N ? p.N : klim);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_OPREADY + s), LTC_XF_THREADS);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_A_FULL), LTC_ROW_THREADS);
    mbar_init(bar(C::B_NUM_FULL), 1);
    mbar_init(bar(C::B_NUM_EMPTY), LTC_ROW_THREADS);
    mbar_init(bar(C::B_ST_DONE), 1);
    mbar_init(bar(C::B_PST_READY), LTC_ROW_THREADS);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == LTC_PRODUCER_WARP && lane == 0) {
    if (!STATE) prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == LTC_MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};
  const size_t tot_head = (size_t)bh * p.n_parts * (size_t)p.tot_stride;

  if (warp == LTC_PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nt > 0) {
      waiter.role = ROLE_PRODUCER;
      bool ok = true;
      int issued = 0;
      for (int t = 0; ok && t < nt; ++t) {
        const int s = t & 1;
        ok = wait_bar(waiter, bar(C::B_EMPTY + s), (uint32_t)((t >> 1) & 1) ^ 1u, C::B_EMPTY + s, unit);
        if (!ok) break;
        const uint32_t full = bar(C::B_FULL + s);
        mbar_arrive_expect_tx(full, (STATE ? 2u : 3u) * C::TILE);
        const uint32_t st = base + (uint32_t)s * C::STAGE;
        const int row = row0 + t * LTC_T;
        if (!STATE) tma_load_3d(st + C::Q_OFF, &tmap_q, full, 0, row, bh);
        tma_load_3d(st + C::K_OFF, &tmap_k, full, 0, row, bh);
        tma_load_3d(st + C::V_OFF, &tmap_v, full, 0, row, bh);
        ++issued;
      }
      // drain: copies that may still be in flight after an abort
      for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t)
        drain_wait(bar(C::B_FULL + (t & 1)), (uint32_t)((t >> 1) & 1), 20000000ull);
    }
  } else if (warp == LTC_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (nt > 0) {
      waiter.role = ROLE_MMA;
      constexpr uint32_t IDESC_S = ltc_idesc(128, 128, false, false);   // Qt, Kt: both K-major
      constexpr uint32_t IDESC_N64 = ltc_idesc(128, 64, false, true);   // Qt or A (tmem) x MN-major B
      constexpr uint32_t IDESC_ST = ltc_idesc(128, 128, true, true);    // [Kt_hi | Kt_lo]^T [V_hi | V_lo]
      const uint32_t t_s = tmem + LTC_TMEM_S, t_num = tmem + LTC_TMEM_NUM, t_st = tmem + LTC_TMEM_ST;
      const uint64_t pst_h = smem_desc(base + C::PST_OFF, 16, 1024);
      const uint64_t pst_l = smem_desc(base + C::PST_OFF + C::PST_BYTES, 16, 1024);
      bool ok = true;
      bool issued_any = false;
      auto wait_w = [&](int id, uint32_t parity) {
        ok = ok && wait_bar(waiter, bar(id), parity, id, unit);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) tc_fence_after();
      };
      // operand descriptors of stage s
      struct StageDesc {
        uint64_t qh, ql, kh, kl, vh, vl, kt_stack;
      };
      auto stage_desc = [&](int s) {
        const uint32_t st = base + (uint32_t)s * C::STAGE;
        StageDesc d;
        d.qh = smem_desc(st + C::Q_OFF, 16, C::GROUP);
        d.ql = smem_desc(st + C::Q_OFF + C::LO, 16, C::GROUP);
        d.kh = smem_desc(st + C::K_OFF, 16, C::GROUP);
        d.kl = smem_desc(st + C::K_OFF + C::LO, 16, C::GROUP);
        d.vh = smem_desc(st + C::V_OFF, C::LO, C::GROUP);            // N panels: V_hi, V_lo
        d.vl = smem_desc(st + C::V_OFF + C::LO, C::LO, C::GROUP);
        d.kt_stack = smem_desc(st + C::K_OFF, C::LO, C::GROUP);      // M panels: Kt_hi, Kt_lo
        return d;
      };
      // S = Qt Kt^T in three terms; K = 64 features in steps of 16 (32 bytes)
      auto issue_s = [&](const StageDesc& d) {
        auto s_term = [&](uint64_t a, uint64_t b, bool first) {
          static_for<LTC_F / 16>([&](auto kc) {
            constexpr int k = decltype(kc)::value;
            mma_ss_w_off<(uint32_t)(k * 2)>(t_s, a, b, IDESC_S, (first && k == 0) ? 0u : 1u);
          });
        };
        s_term(d.qh, d.kh, true);
        s_term(d.qh, d.kl, false);
        s_term(d.ql, d.kh, false);
        mma_commit_w(bar(C::B_S_FULL));
      };
      // S_t+1 = S_t + [Kt_hi | Kt_lo]^T [V_hi | V_lo]: K = 128 rows in steps of
      // 16 (two 8-row groups, 4096 bytes)
      auto issue_state = [&](const StageDesc& d, uint32_t acc0) {
        static_for<LTC_T / 16>([&](auto kc) {
          constexpr int k = decltype(kc)::value;
          mma_ss_w_off<(uint32_t)(k * 256)>(t_st, d.kt_stack, d.vh, IDESC_ST, k == 0 ? acc0 : 1u);
        });
      };
      if (!STATE) {
        // Order per tile t: A V (once A is formed), Qt S_t (once the row warps
        // have refreshed the state operand, which they do while A V runs), the
        // state update, the stage's release, then S of tile t+1; S of tile 0
        // first.
        wait_w(C::B_OPREADY + 0, 0u);
        if (ok) {
          issued_any = true;
          issue_s(stage_desc(0));
        }
        for (int t = 0; ok && t < nt; ++t) {
          const int s = t & 1;
          const StageDesc d = stage_desc(s);
          wait_w(C::B_A_FULL, (uint32_t)(t & 1));
          if (t > 0) wait_w(C::B_NUM_EMPTY, (uint32_t)((t - 1) & 1));
          if (!ok) break;
          // num = A V: A from tensor memory, each group of 32 keys in 32
          // columns: its hi words in the first 16, its lo words in the last 16
          auto av_term = [&](uint32_t a_off, uint64_t b, bool first) {
            static_for<LTC_T / 16>([&](auto kc) {
              constexpr int k = decltype(kc)::value;
              constexpr uint32_t acol = 32u * (uint32_t)(k / 2) + 8u * (uint32_t)(k & 1);
              mma_ts_w_off<(uint32_t)(k * 256), acol>(t_num, t_s + a_off, b, IDESC_N64,
                                                       (first && k == 0) ? 0u : 1u);
            });
          };
          av_term(0u, d.vh, true);
          av_term(0u, d.vl, false);
          av_term(16u, d.vh, false);
          // num += Qt S_t: the state operand of this tile
          wait_w(C::B_PST_READY, (uint32_t)(t & 1));
          if (!ok) break;
          auto qs_term = [&](uint64_t a, uint64_t b) {
            static_for<LTC_F / 16>([&](auto kc) {
              constexpr int k = decltype(kc)::value;
              // A K-major: 32 bytes per step; B MN-major: 16 rows = 2048 bytes per step
              mma_ss_w_off2<(uint32_t)(k * 2), (uint32_t)(k * 128)>(t_num, a, b, IDESC_N64, 1u);
            });
          };
          qs_term(d.qh, pst_h);
          qs_term(d.qh, pst_l);
          qs_term(d.ql, pst_h);
          mma_commit_w(bar(C::B_NUM_FULL));
          issue_state(d, 1u);  // the accumulator holds the part's starting state
          mma_commit_w(bar(C::B_ST_DONE));
          mma_commit_w(bar(C::B_EMPTY + s));  // the stage's last reader: its next tile may load
          if (t + 1 < nt) {
            // S of the next tile overwrites A in tensor memory after A V (in issue order)
            wait_w(C::B_OPREADY + (s ^ 1), (uint32_t)(((t + 1) >> 1) & 1));
            if (!ok) break;
            issue_s(stage_desc(s ^ 1));
          }
        }
      } else {
        for (int t = 0; ok && t < nt; ++t) {
          const int s = t & 1;
          wait_w(C::B_OPREADY + s, (uint32_t)((t >> 1) & 1));
          if (!ok) break;
          issued_any = true;
          issue_state(stage_desc(s), t > 0 ? 1u : 0u);
          mma_commit_w(bar(C::B_EMPTY + s));
        }
      }
      if (STATE && ok) mma_commit_w(bar(C::B_ST_DONE));
      if (issued_any) {
        mma_commit_w(bar(C::B_DRAIN));
        drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ transform
    waiter.role = ROLE_SOFTMAX;
    const int tt = threadIdx.x - LTC_ROW_THREADS;  // 0..255
    bool ok = true;
    // z at the part's start: the earlier parts' key sums
    if (tt < LTC_F) {
      float z0 = 0.0f;
      if (!STATE && tt < p.E)
        for (int pp = 0; pp < part; ++pp) z0 += p.tot[tot_head + (size_t)pp * p.tot_stride + (size_t)p.E * p.M + tt];
      zmaster[tt] = z0;
    }
    ok = ltc_group_and(LTC_BAR_XF, ok);
    // One fp32 tile of 128 x 64, converted in place: warp w takes the 8-row
    // groups w and w + 8, lane l the float4 number 32k + l of each (row 2k +
    // l/16 of the group, columns 4*(l%16) ...).  A group's fp32 rows and its
    // bf16 hi / lo atoms are the same 2048 bytes, so the warp reads both of
    // its groups, meets at __syncwarp, and writes them.  kind: 0 = Q (phi),
    // 1 = K (phi, key mask, key sums), 2 = V.
    const int xw = tt >> 5;
    auto convert = [&](uint32_t buf, int kind, int grow0) {
      uint8_t* tile = base_ptr + (buf - base);
      float4 x[2][4];
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          x[gi][k] = reinterpret_cast<const float4*>(tile + (uint32_t)(xw + 8 * gi) * C::GROUP)[32 * k + lane];
      __syncwarp();
      const int c4 = lane & 15;
      const int nfeat = kind == 2 ? p.M : p.E;
      float cs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = 8 * (xw + 8 * gi) + 2 * k + (lane >> 4);
          float v[4] = {x[gi][k].x, x[gi][k].y, x[gi][k].z, x[gi][k].w};
          if (kind != 2) {
            const bool row_live = kind == 0 || grow0 + r < klim;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const bool live = row_live && 4 * c4 + i < nfeat;
              v[i] = live ? lin_phi(v[i]) : 0.0f;
              cs[i] += v[i];
            }
          }
          uint32_t h01, l01, h23, l23;
          ltc_split2(v[0], v[1], h01, l01);
          ltc_split2(v[2], v[3], h23, l23);
          const uint32_t off = ltc_swz8(r, c4, C::GROUP);
          *reinterpret_cast<uint2*>(tile + off) = make_uint2(h01, h23);
          *reinterpret_cast<uint2*>(tile + C::LO + off) = make_uint2(l01, l23);
        }
      if (kind == 1) {
        // key sums of this tile: lanes l and l ^ 16 hold the same columns
#pragma unroll
        for (int i = 0; i < 4; ++i) cs[i] += __shfl_xor_sync(0xffffffffu, cs[i], 16);
        if (lane < 16) {
#pragma unroll
          for (int i = 0; i < 4; ++i) atomicAdd(zmaster + 4 * c4 + i, cs[i]);
        }
      }
    };
    for (int t = 0; ok && t < nt; ++t) {
      const int s = t & 1;
      // (a group barrier: every transform warp has finished the previous
      // tile, its key-sum atomics included)
      ok = ltc_group_and(LTC_BAR_XF,
                         wait_bar(waiter, bar(C::B_FULL + s), (uint32_t)((t >> 1) & 1), C::B_FULL + s, unit));
      if (!ok) break;
      const uint32_t st = base + (uint32_t)s * C::STAGE;
      const int grow0 = row0 + t * LTC_T;
      if (!STATE) {
        // z before this tile's keys, copied before any of them is added
        if (tt < LTC_F) zsnap[s * LTC_F + tt] = zmaster[tt];
        ltc_group_and(LTC_BAR_XF, true);
        convert(st + C::Q_OFF, 0, grow0);
      }
      convert(st + C::K_OFF, 1, grow0);
      convert(st + C::V_OFF, 2, grow0);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_OPREADY + s));
    }
    if (STATE && ok) {
      // the part's key sum, once every tile's atomics are in
      ok = ltc_group_and(LTC_BAR_XF, ok);
      if (ok && tt < p.E) p.tot[tot_head + (size_t)part * p.tot_stride + (size_t)p.E * p.M + tt] = zmaster[tt];
    }
  } else {
    // ------------------------------------------------------------ row warps
    waiter.role = ROLE_SOFTMAX;
    const int quarter = warp & 3;   // TMEM lane quarter
    const int ch = warp >> 2;       // column half of this warp
    const int row = quarter * 32 + lane;  // TMEM lane: tile row, or state row (lo rows at 64..127)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + LTC_TMEM_S;
    const uint32_t t_num = tmem + lane_off + LTC_TMEM_NUM;
    const uint32_t t_st = tmem + lane_off + LTC_TMEM_ST;
    bool ok = true;
    auto wait_w = [&](int id, uint32_t parity) {
      ok = ok && wait_bar(waiter, bar(id), parity, id, unit);
      ok = ltc_group_and(LTC_BAR_ROW, ok);
      if (ok) tc_fence_after();
      return ok;
    };
    // 32 columns (this warp's half) of state row `row` (< 64) into the
    // shared-memory operand tiles: hi and lo, 128-byte-swizzled rows of 64 bf16
    auto write_state_operand = [&](const float (&sh)[32]) {
      uint8_t* ph = base_ptr + C::PST_OFF;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ltc_split2(sh[8 * c + 2 * i], sh[8 * c + 2 * i + 1], h[i], l[i]);
        const uint32_t off = ltc_swz16(row, 4 * ch + c);
        *reinterpret_cast<uint4*>(ph + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(ph + C::PST_BYTES + off) = make_uint4(l[0], l[1], l[2], l[3]);
      }
    };
    // this warp's 32 columns of the state after the last update: lanes e and
    // 64 + e hold the quadrant sums of row e (hi.hi + hi.lo and lo.hi +
    // lo.lo); lanes 64.. pass theirs through `xch`, lanes 0..63 return the
    // total in sh
    auto read_state = [&](float (&sh)[32]) {
      {
        uint32_t a[32];
        tmem_ld32(t_st + 32u * ch, a);
        tmem_ld_wait(a);
#pragma unroll
        for (int i = 0; i < 32; ++i) sh[i] = __uint_as_float(a[i]);
      }
      {
        uint32_t b[32];
        tmem_ld32(t_st + 64u + 32u * ch, b);
        tmem_ld_wait(b);
#pragma unroll
        for (int i = 0; i < 32; ++i) sh[i] += __uint_as_float(b[i]);
      }
      // chunk c of exchange row e sits at position c ^ (e % 16): a warp's 32
      // rows then spread one chunk index over all banks
      const int xr = row & (LTC_F - 1);
      if (row >= LTC_F) {
        float4* dst = reinterpret_cast<float4*>(xch + xr * LTC_F);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[(8 * ch + c) ^ (xr & 15)] = make_float4(sh[4 * c], sh[4 * c + 1], sh[4 * c + 2], sh[4 * c + 3]);
      }
      if (!ltc_group_and(LTC_BAR_ROW, true)) return false;
      if (row < LTC_F) {
        const float4* srcx = reinterpret_cast<const float4*>(xch + xr * LTC_F);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = srcx[(8 * ch + c) ^ (xr & 15)];
          sh[4 * c] += v.x;
          sh[4 * c + 1] += v.y;
          sh[4 * c + 2] += v.z;
          sh[4 * c + 3] += v.w;
        }
      }
      return true;
    };

    if (!STATE && nt > 0) {
      // the state at the part's start (the earlier parts' totals) into the
      // state accumulator (hi.hi quadrant; the others zero) and its operand
      float sh[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) sh[i] = 0.0f;
      if (row < p.E)
        for (int pp = 0; pp < part; ++pp) {
          const float* tp = p.tot + tot_head + (size_t)pp * p.tot_stride + (size_t)row * p.M;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * ch + i < p.M) sh[i] += tp[32 * ch + i];
        }
      {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = row < LTC_F ? __float_as_uint(sh[i]) : 0u;
        tmem_st32(t_st + 32u * ch, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
        tmem_st32(t_st + 64u + 32u * ch, w);
      }
      if (row < LTC_F) write_state_operand(sh);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PST_READY));
    }

    for (int t = 0; !STATE && ok && t < nt; ++t) {
      const int s = t & 1;
      const int grow = row0 + t * LTC_T + row;
      // (a) A = tril(S) split into hi / lo, the row sum, and Qt . z, over this
      // warp's half of the keys and of the features.  The stage's operand
      // barrier (complete once S has landed) is waited on as well, as the
      // acquire for this warp's own reads of the transform's Qt tiles and z.
      if (!wait_w(C::B_S_FULL, (uint32_t)(t & 1))) break;
      if (!wait_w(C::B_OPREADY + s, (uint32_t)((t >> 1) & 1))) break;
      float part_sum = 0.0f;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        // keys 32gg .. 32gg+31 (gg = 2ch + g): read from columns 32gg ..
        // 32gg+31, then replaced in place by their packed hi words (the
        // group's first 16 columns) and lo words (its last 16)
        const uint32_t col = 64u * ch + 32u * g;
        uint32_t sv[32];
        tmem_ld32(t_s + col, sv);
        tmem_ld_wait(sv);
        uint32_t wh[16], wl[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int j = (int)col + 2 * q;
          const float a0 = j <= row ? __uint_as_float(sv[2 * q]) : 0.0f;
          const float a1 = j + 1 <= row ? __uint_as_float(sv[2 * q + 1]) : 0.0f;
          part_sum += a0 + a1;
          ltc_split2(a0, a1, wh[q], wl[q]);
        }
        tmem_st16(t_s + col, wh);
        tmem_st16(t_s + col + 16u, wl);
      }
      {
        const uint8_t* qt = base_ptr + (uint32_t)s * C::STAGE + C::Q_OFF;
        const float* zs = zsnap + s * LTC_F;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int cc = 4 * ch + c;  // features 8cc .. 8cc+7
          const uint32_t off = ltc_swz16(row, cc, C::GROUP);
          const uint4 h4 = *reinterpret_cast<const uint4*>(qt + off);
          const uint4 l4 = *reinterpret_cast<const uint4*>(qt + C::LO + off);
          const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w}, lw[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            part_sum += (bf16lo_as_f32(hw[i]) + bf16lo_as_f32(lw[i])) * zs[8 * cc + 2 * i];
            part_sum += (bf16hi_as_f32(hw[i]) + bf16hi_as_f32(lw[i])) * zs[8 * cc + 2 * i + 1];
          }
        }
      }
      rsq[ch * LTC_T + row] = part_sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_A_FULL));
      // (b) the state this tile's Qt S_t needs: S_t = S_t-1 + Kt^T V of tile
      // t-1, refreshed while A V of this tile runs on the tensor cores
      if (t > 0) {
        if (!wait_w(C::B_ST_DONE, (uint32_t)((t - 1) & 1))) break;
        float sh[32];
        if (!(ok = read_state(sh))) break;
        if (row < LTC_F) write_state_operand(sh);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_PST_READY));
      }
      // (c) this warp's half of the output row (the group barrier in the wait
      // also makes both halves' row sums visible)
      if (!wait_w(C::B_NUM_FULL, (uint32_t)(t & 1))) break;
      {
        const float inv = 1.0f / (rsq[row] + rsq[LTC_T + row] + p.eps);
        uint32_t nv[32];
        tmem_ld32(t_num + 32u * ch, nv);
        tmem_ld_wait(nv);
        tc_fence_before();
        mbar_arrive(bar(C::B_NUM_EMPTY));
        if (grow < row_end) {
          float4* dst = reinterpret_cast<float4*>(p.out + ((size_t)bh * p.N + (size_t)grow) * p.M + 32 * ch);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (32 * ch + 4 * c < p.M)
              dst[c] = make_float4(__uint_as_float(nv[4 * c]) * inv, __uint_as_float(nv[4 * c + 1]) * inv,
                                   __uint_as_float(nv[4 * c + 2]) * inv, __uint_as_float(nv[4 * c + 3]) * inv);
        }
      }
    }
    if (STATE && nt > 0) {
      // the part's total: the state accumulated over all of its tiles
      if (wait_w(C::B_ST_DONE, 0u)) {
        float sh[32];
        if (read_state(sh) && row < p.E) {
          float* tp = p.tot + tot_head + (size_t)part * p.tot_stride + (size_t)row * p.M + 32 * ch;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * ch + i < p.M) tp[i] = sh[i];
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == LTC_MMA_WARP) tmem_dealloc(tmem, 512);
}

}  // namespace fattn
