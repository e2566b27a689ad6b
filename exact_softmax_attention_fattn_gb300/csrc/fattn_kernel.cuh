// Exact softmax attention forward, sm_103a: one fused, persistent kernel.
//
// What it computes ("understand-flashattention": forward-pass formulas,
// numerically stable softmax, two-block online-softmax derivation, logsumexp
// derivation; scale-then-mask order of "PyTorch profiling part 3: attention",
// section "Naive attention"):
//     O = softmax(mask(scale * Q K^T)) V,   LSE = rowwise log-sum-exp of the
//     masked, scaled scores (natural log); an all-masked row gives O = 0 and
//     LSE = -inf ("The safe softmax" section of the same profiling page).
//
// How (GB300 design, not the pages' Ampere blocking):
//   * work unit = (batch*head, block of 2 x 128 query rows, K/V split); CTAs
//     are persistent and walk the units with a static stride, heaviest
//     (latest, for causal) query blocks first.  With one split a unit covers
//     all of its key tiles and writes O and LSE.  With several (split-KV, for
//     grids with fewer units than SMs) the n key tiles a query block visits
//     are cut into n_splits near-equal runs (split s: tiles
//     [s*n/n_splits, (s+1)*n/n_splits)), and each writes its normalised
//     partial output and log-sum-exp in fp32, which the combine kernel merges
//     with the two-block rule of the same derivation;
//   * warp 8 (one lane) is the TMA producer: Q tiles into two fixed buffers,
//     K and V tiles into a STAGES-deep ring, all 128-byte swizzled panels of
//     64 columns;
//   * warp 9 issues tcgen05.mma (the whole warp runs the loop, one elected
//     lane issues): S_t = Q_t K_j^T (both operands in shared memory) and
//     O_t += P_t V_j (P from tensor memory, V from shared memory), completion
//     signalled with tcgen05.commit on mbarriers.  The two
//     query tiles ping-pong: while one softmax group works on S_0, the tensor
//     core runs the other tile's PV and S;
//   * warps 0-3 and 4-7 are one softmax group per query tile, one thread per
//     query row: the online-softmax step of the two-block derivation (running
//     max m, normaliser l, rescaling of the unnormalised output by
//     2^(m_old - m_new)), exponentials in base 2 with the scale folded in, P
//     written back to tensor memory in the operand type of its V tile (fp16,
//     or bf16 for a V tile outside fp16's range; see v_prepass.cuh), then the
//     final O / l and LSE.
//     The rescale of O is skipped while the running max has grown by less
//     than 2^8 since the last rescale: O and l keep a common, slightly stale
//     reference, so the final O / l is unchanged (exact up to rounding).
//   * every wait is bounded; on time-out the kernel records an error word,
//     drains its own copies and MMAs, frees tensor memory and returns;
//   * launched as a programmatic dependent of the V pre-pass, the
//     producer loads Q and K before griddepcontrol.wait and V after it, and
//     the other roles wait before reading the V tile modes.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace fattn {

constexpr int BM = 128;  // query rows per Q tile (TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int QT = 2;    // Q tiles per work unit
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;     // warps 10 and 11 complete the third warpgroup and idle
constexpr int NUM_THREADS = 384;
// Register split (setmaxnreg): the block launches with LAUNCH_REGS per thread
// (ptxas' cap for 384 threads, one SM); the two softmax warpgroups grow to
// SOFTMAX_REGS and the producer/MMA warpgroup shrinks to OTHER_REGS.  The
// split uses exactly the launch allocation: 256*192 + 128*120 = 384*168.
constexpr int LAUNCH_REGS = 168;
constexpr int SOFTMAX_REGS = 192;
constexpr int OTHER_REGS = 120;
static_assert(256 * SOFTMAX_REGS + 128 * OTHER_REGS <= NUM_THREADS * LAUNCH_REGS, "register split exceeds launch");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S0 = 0;    // S_t at column 128*t, P_t packed into its first 64 columns
constexpr uint32_t TMEM_O0 = 256;  // O_t at column 256 + 128*t
constexpr float RESCALE_LOG2_THRESHOLD = 8.0f;
constexpr uint32_t PANEL_BYTES = 128 * 128;  // 128 rows x 128 bytes (64 bf16 columns)

// Storage type of one 128-row V tile in the pre-converted V buffer.
enum : int { VMODE_F16 = 0, VMODE_BF16 = 1 };

// Error word layout (int[4]): [0] status (0 ok, 4 timed out), [1] role,
// [2] barrier id, [3] work unit.
enum : int { ERR_TIMEOUT = 4 };
enum : int { ROLE_SOFTMAX = 1, ROLE_PRODUCER = 2, ROLE_MMA = 3 };

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* key_len;  // [B] or nullptr
  const uint8_t* v_mode;   // [B*H, mode_stride]: storage type of each V tile (VMODE_*)
  int* err;                // int[4]
  int B, H, N;
  int hd;            // head dim of the tensors (a multiple of 8, <= D): rows are hd elements long;
                     // the kernel computes D columns, the tensor maps read the rest as zeros
  float scale;       // softmax scale (natural units), >= 0
  float scale_log2;  // scale * log2(e)
  int causal;
  int o_v8;       // O is 32-byte aligned and hd a multiple of 16: rows of O take 32-byte stores
  int n_qblocks;  // ceil(N / 256)
  int n_units;    // B * H * n_qblocks * n_splits
  const uint16_t* sched;  // nullptr: snake order; else [rounds, G]: CTA c's place in round r's units
  int n_splits;    // K/V splits per query block (1: no split, O and LSE written directly)
  int head_group;  // one-query-tile kernel (head dims above 128): heads per group of its CTA order
  float* o_part;   // n_splits > 1: [n_splits, B*H, N, D] fp32 O / l of each split
  float* lse_part; // n_splits > 1: [n_splits, B*H, N] fp32 log-sum-exp of each split
  int n_kv_tiles; // ceil(N / 128)
  int mode_stride; // n_kv_tiles rounded up to 8: modes are read 8 at a time
  unsigned long long wait_limit_ns;
};

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head-dim bucket 64 or 128");
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE_BYTES = BM * D * 2;  // one Q, K or V tile (BN == BM)
  static constexpr int STAGES = D == 128 ? 5 : 8;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t RING_OFF = QT * TILE_BYTES;
  static constexpr uint32_t BAR_OFF = RING_OFF + STAGES * TILE_BYTES;
  // barrier ids
  static constexpr int B_Q_FULL = 0;                     // [2]
  static constexpr int B_Q_EMPTY = 2;                    // [2]
  static constexpr int B_S_FULL = 4;                     // [2]
  static constexpr int B_P_FULL = 6;                     // [2]
  static constexpr int B_O_FULL = 8;                     // [2]
  static constexpr int B_O_EMPTY = 10;                   // [2]
  static constexpr int B_DRAIN = 12;                     // [1]
  // K/V tiles are loaded in groups, one per MMA step (see the producer);
  // group k uses barrier pair k % KV_GROUPS.  At most STAGES groups hold ring
  // slots at a time, so a pair is never re-armed before its last use ended.
  static constexpr int KV_GROUPS = 2 * STAGES;
  static_assert(KV_GROUPS <= 32, "group sizes are kept in one 32-bit mask");
  static constexpr int B_KV_FULL = 13;                   // [KV_GROUPS]
  static constexpr int B_KV_EMPTY = 13 + KV_GROUPS;      // [KV_GROUPS]
  static constexpr int NUM_BARS = 13 + 2 * KV_GROUPS;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tmem base (4 B) + abort flag (4 B)
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
};

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start address,
// leading- and stride-dimension byte offsets (all >> 4), descriptor version 1,
// layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16: D fp32; A and B both bf16 or both
// f16; shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool ab_bf16, bool b_mn_major) {
  return (1u << 4)                          // D format f32
         | ((ab_bf16 ? 1u : 0u) << 7)      // A format: 0 f16, 1 bf16
         | ((ab_bf16 ? 1u : 0u) << 10)     // B format: same as A
         | (0u << 15)                       // A K-major
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ work units
struct Unit {
  int bh, b, r0;
  int split, j0;           // K/V split and its first key tile
  int n0, n1;              // K/V tiles Q tile 0 / 1 visits in this split (0: nothing to do)
  int min_lim0, min_lim1;  // smallest per-row key limit in each tile
  int kl;                  // effective key length of this batch entry
  int nkv;                 // max(n0, n1)
  bool valid0, valid1;     // tile has at least one row < N
  __device__ __forceinline__ int n(int t) const { return t ? n1 : n0; }
  __device__ __forceinline__ int min_lim(int t) const { return t ? min_lim1 : min_lim0; }
  __device__ __forceinline__ bool valid(int t) const { return t ? valid1 : valid0; }
};

// Unit u = ((round * n_splits) + split) * B*H + bh: the query block of a round
// is n_qblocks - 1 - round (latest, the heaviest under causal, first).

// Key tiles that query tile `row0` visits over the whole key range, with
// key length kl (clamped): every one of them holds a visible key for every
// row of the tile.
__device__ __forceinline__ int tile_kv_count(const Params& p, int row0, int kl) {
  if (row0 >= p.N) return 0;
  const int max_lim = p.causal ? min(kl, row0 + BM) : kl;
  return max_lim > 0 ? (max_lim + BN - 1) / BN : 0;
}


template <bool SPLIT>
__device__ __forceinline__ Unit decode_unit(const Params& p, int u, int kl_raw) {
  Unit w;
  const int BH = p.B * p.H;
  const int ns = SPLIT ? p.n_splits : 1;
  const int round = u / (BH * ns);
  w.split = SPLIT ? (u / BH) % ns : 0;
  w.bh = u % BH;
  w.b = w.bh / p.H;
  const int qb = p.n_qblocks - 1 - round;  // latest (heaviest under causal) blocks first
  w.r0 = qb * (QT * BM);
  const int kl = kl_raw < 0 ? 0 : (kl_raw > p.N ? p.N : kl_raw);
  w.kl = kl;
  int n_all[QT], ml[QT];
  bool vv[QT];
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    const int row0 = w.r0 + t * BM;
    vv[t] = row0 < p.N;
    n_all[t] = tile_kv_count(p, row0, kl);  // tiles of the whole key range
    ml[t] = p.causal ? min(kl, row0 + 1) : kl;
  }
  int nn[QT];
  if constexpr (SPLIT) {
    // this split's run of the block's key tiles: [j0, j1)
    const int n_blk = max(n_all[0], n_all[1]);
    w.j0 = w.split * n_blk / ns;
    const int j1 = (w.split + 1) * n_blk / ns;
#pragma unroll
    for (int t = 0; t < QT; ++t) nn[t] = max(min(n_all[t], j1) - w.j0, 0);
  } else {
    w.j0 = 0;
#pragma unroll
    for (int t = 0; t < QT; ++t) nn[t] = n_all[t];
  }
  w.n0 = nn[0];
  w.n1 = nn[1];
  w.min_lim0 = ml[0];
  w.min_lim1 = ml[1];
  w.valid0 = vv[0];
  w.valid1 = vv[1];
  w.nkv = max(w.n0, w.n1);
  return w;
}

// Persistent schedule: CTA c takes, in round r, unit r*G + c (r even) or
// r*G + G-1-c (r odd).  Units are ordered heaviest first, so the snake pairs
// heavy and light units on each CTA.
// A host-built table may replace the snake: it deals each round's units
// (the same set, so the same K/V working set per round) to the CTAs so that
// their totals come out more even.
__device__ __forceinline__ int unit_of(const Params& p, int r, int c, int G) {
  if (p.sched) return r * G + (int)__ldg(p.sched + (r * G + c));
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// The units of one CTA in schedule order, read one unit ahead: the next
// unit's key length and first V-tile storage mode are requested once
// the current unit is under way (at its second tile), so no role waits on a
// global load at a unit boundary, where the epilogue's output stores occupy
// the memory pipeline.
struct UnitIter {
  bool modes = true;       // read the V storage modes (not in the producer)
  int r, u, kl_raw;        // current unit (u < 0: done)
  int mode0;               // storage mode of its first V tile
  int r_next, u_next;      // the one after it
  int kl_next, mode_next;
  int next_bh;             // its batch*head, for the loads below
  int fetch_at;            // tile index at which the loads are issued (runtime value)

  __device__ __forceinline__ static int round_from(const Params& p, int r, int cta, int G) {
    while (r * G < p.n_units && unit_of(p, r, cta, G) >= p.n_units) ++r;
    return r * G < p.n_units ? r : -1;
  }
  // the two loads for the next unit; cheap enough to sit inside the tile loop
  __device__ __forceinline__ void load_next(const Params& p) {
    if (u_next < 0) return;
    kl_next = p.key_len ? __ldg(p.key_len + next_bh / p.H) : p.N;
    if (modes) mode_next = __ldg(p.v_mode + (size_t)next_bh * p.mode_stride);  // (split units read theirs at the unit start)
  }
  __device__ __forceinline__ void locate_next(const Params& p, int cta, int G) {
    r_next = r < 0 ? -1 : round_from(p, r + 1, cta, G);
    u_next = r_next < 0 ? -1 : unit_of(p, r_next, cta, G);
    next_bh = u_next < 0 ? 0 : u_next % (p.B * p.H);
    fetch_at = 1;
  }
  __device__ __forceinline__ void begin(const Params& p, int cta, int G) {
    r = round_from(p, 0, cta, G);
    u = r < 0 ? -1 : unit_of(p, r, cta, G);
    if (u >= 0) {
      const int bh = u % (p.B * p.H);
      kl_raw = p.key_len ? __ldg(p.key_len + bh / p.H) : p.N;
      if (modes) mode0 = __ldg(p.v_mode + (size_t)bh * p.mode_stride);
    }
    locate_next(p, cta, G);
    load_next(p);
    fetch_at = -1;  // already requested
  }
  // call once per tile with its index; issues the next unit's loads at tile `fetch_at`
  __device__ __forceinline__ void at_tile(const Params& p, int j) {
    if (j == fetch_at) {
      load_next(p);
      fetch_at = -1;
    }
  }
  __device__ __forceinline__ void advance(const Params& p, int cta, int G) {
    if (fetch_at >= 0) load_next(p);  // the unit ended before its request point
    r = r_next;
    u = u_next;
    kl_raw = kl_next;
    mode0 = mode_next;
    locate_next(p, cta, G);
  }
};

// ------------------------------------------------------------------ bounded wait
struct Waiter {
  volatile int* abort_flag;  // shared memory
  int* err;
  unsigned long long limit_ns;
  int role;
};

// Returns false (and raises the CTA's abort flag) if the wait gave up.  The
// thread is suspended in hardware between checks (try_wait with a time hint),
// so waiting warps take no issue slots from the warps that compute.
__device__ __forceinline__ bool wait_slow(const Waiter& w, uint32_t bar, uint32_t parity, int bar_id, int unit) {
  const uint64_t t0 = globaltimer_ns();
  const uint32_t hint = w.limit_ns < 1000000ull ? (uint32_t)w.limit_ns : 1000000u;
  while (true) {
    if (mbar_try_wait_hint(bar, parity, hint)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort_flag = 1;
      if (atomicCAS(w.err, 0, ERR_TIMEOUT) == 0) {
        w.err[1] = w.role;
        w.err[2] = bar_id;
        w.err[3] = unit;
      }
      __threadfence();
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(const Waiter& w, uint32_t bar, uint32_t parity, int bar_id, int unit) {
  if (mbar_test_wait(bar, parity)) return true;
  return wait_slow(w, bar, parity, bar_id, unit);
}

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
  }
}

template <int T>
using TileC = std::integral_constant<int, T>;

// f(integral_constant<int, I>) for I = 0 .. N-1, unrolled at compile time.
template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<N, I + 1>(f);
  }
}


// ------------------------------------------------------------------ the kernel
// SPLIT: the split-KV instantiation (p.n_splits > 1: partial outputs in fp32
// for the combine kernel); without it the kernel writes O and LSE itself.
// FULL: the head dim is D (rows of the output a compile-time length);
// otherwise p.hd < D.
template <int D, bool SPLIT, bool FULL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fattn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  using C = Cfg<D>;
  const int hd = FULL ? D : p.hd;  // output row length
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  auto bar = [&](int id) -> uint32_t { return base + C::BAR_OFF + 8u * (uint32_t)id; };
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(base_ptr + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int t = 0; t < QT; ++t) {
      mbar_init(bar(C::B_Q_FULL + t), 1);
      mbar_init(bar(C::B_Q_EMPTY + t), 1);
      mbar_init(bar(C::B_S_FULL + t), 1);
      mbar_init(bar(C::B_P_FULL + t), BM);
      mbar_init(bar(C::B_O_FULL + t), 1);
      mbar_init(bar(C::B_O_EMPTY + t), BM);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    for (int s = 0; s < C::KV_GROUPS; ++s) {
      mbar_init(bar(C::B_KV_FULL + s), 1);
      mbar_init(bar(C::B_KV_EMPTY + s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(base + C::MISC_OFF, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  if constexpr (SPLIT) pdl_launch_dependents();  // the combine kernel may launch now (it waits before reading)

  Waiter waiter{abort_flag, p.err, p.wait_limit_ns, 0};

  if (warp >= 8) {
  regs_shrink<OTHER_REGS>();
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      waiter.role = ROLE_PRODUCER;
      uint32_t g = 0;                 // K/V tiles issued so far (ring position)
      uint32_t q_use0 = 0, q_use1 = 0;  // Q tiles issued so far, per buffer
      bool ok = true;
      auto load_q = [&](auto tc, const Unit& w, int u, uint32_t& q_use) {
        constexpr int t = decltype(tc)::value;
        if (!ok || w.n(t) == 0) return;
        ok = wait_bar(waiter, bar(C::B_Q_EMPTY + t), (q_use & 1u) ^ 1u, C::B_Q_EMPTY + t, u);
        if (!ok) return;
        mbar_arrive_expect_tx(bar(C::B_Q_FULL + t), C::TILE_BYTES);
        const uint32_t dst = base + C::Q_OFF + (uint32_t)t * C::TILE_BYTES;
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_3d(dst + pn * PANEL_BYTES, &tmap_q, bar(C::B_Q_FULL + t), 64 * pn, w.r0 + t * BM, w.bh);
        ++q_use;
      };
      // K and V tiles go into a STAGES-deep ring of tile slots (ring position
      // g -> slot g % STAGES), in groups read by one MMA step: a unit's first
      // K tile alone, then (V_j, K_j+1) for each step j, the last step's V
      // tile alone.  A group completes one full barrier (one transaction count
      // for all its tiles) and is released by one commit, so the MMA issuer
      // waits and commits once per step.  A slot is written again once the
      // group holding its previous tile has been released; groups are
      // released in order, so the positions released so far are counted.
      uint32_t gk = 0;        // groups armed
      uint32_t gr = 0;        // groups seen released
      uint32_t released = 0;  // ring positions of released groups
      uint32_t two = 0;       // bit k % 32: group k holds two tiles
      auto make_room = [&](uint32_t pos, uint32_t groups_armed, int u) {
        while (ok && (released + C::STAGES <= pos || groups_armed >= gr + C::KV_GROUPS)) {
          const int id = C::B_KV_EMPTY + (int)(gr % C::KV_GROUPS);
          ok = wait_bar(waiter, bar(id), (gr / C::KV_GROUPS) & 1u, id, u);
          released += 1u + ((two >> (gr % 32u)) & 1u);
          ++gr;
        }
      };
      auto load_kv = [&](const CUtensorMap* map, int j, int bh, uint32_t full) {
        const uint32_t dst = base + C::RING_OFF + (g % C::STAGES) * C::TILE_BYTES;
#pragma unroll
        for (int pn = 0; pn < C::PANELS; ++pn) tma_load_3d(dst + pn * PANEL_BYTES, map, full, 64 * pn, j * BN, bh);
        ++g;
      };
      UnitIter it;
      it.modes = false;
      bool v_ready = false;  // the V copy (the pre-pass's output) waited for
      it.begin(p, cta, G);
      for (; ok && it.u >= 0; it.advance(p, cta, G)) {
        const int u = it.u;
        const Unit w = decode_unit<SPLIT>(p, u, it.kl_raw);
        it.at_tile(p, it.fetch_at);
        load_q(TileC<0>{}, w, u, q_use0);
        load_q(TileC<1>{}, w, u, q_use1);
        // group of step j: V_j (j >= 0) and K_j+1 (j+1 < nkv); j = -1 is K_0.
        // A unit with no key tile loads nothing (the MMA issuer skips it too).
        for (int j = -1; ok && w.nkv > 0 && j < w.nkv; ++j) {
          const bool has_v = j >= 0, has_k = j + 1 < w.nkv;
          const uint32_t ntiles = (has_v ? 1u : 0u) + (has_k ? 1u : 0u);
          make_room(g, gk, u);
          if (!ok) break;
          const uint32_t full = bar(C::B_KV_FULL + (int)(gk % C::KV_GROUPS));
          mbar_arrive_expect_tx(full, ntiles * C::TILE_BYTES);
          const uint32_t bit = 1u << (gk % 32u);
          two = ntiles == 2u ? (two | bit) : (two & ~bit);
          ++gk;
          if (has_v && !v_ready) {
            pdl_wait();
            v_ready = true;
          }
          if (has_v) load_kv(&tmap_v, w.j0 + j, w.bh, full);
          if (has_k) {
            make_room(g, gk - 1u, u);
            if (!ok) break;
            load_kv(&tmap_k, w.j0 + j + 1, w.bh, full);
          }
        }
      }
      // Drain: wait (bounded) for every group that may still have copies in
      // flight -- after an abort anywhere in the CTA they may never have been
      // consumed.  A barrier pair is re-armed only after its previous group
      // was released, so the last KV_GROUPS groups are the ones still tracked;
      // in a normal run every phase below has already completed.
      const uint32_t first = gk > (uint32_t)C::KV_GROUPS ? gk - C::KV_GROUPS : 0u;
      for (uint32_t k = first; k < gk; ++k)
        drain_wait(bar(C::B_KV_FULL + (int)(k % C::KV_GROUPS)), (k / C::KV_GROUPS) & 1u, 20000000ull);
      if (q_use0) drain_wait(bar(C::B_Q_FULL + 0), (q_use0 - 1) & 1u, 20000000ull);
      if (q_use1) drain_wait(bar(C::B_Q_FULL + 1), (q_use1 - 1) & 1u, 20000000ull);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop so that descriptors and addresses are
    // warp-uniform; elect.sync inside each MMA / commit picks the one lane
    // that issues it.  Every wait result is made warp-uniform.
    {
      waiter.role = ROLE_MMA;
      constexpr uint32_t IDESC_S = idesc_f16kind(BM, BN, true, false);      // Q, K bf16
      constexpr uint32_t IDESC_PV_F16 = idesc_f16kind(BM, D, false, true);  // P, V f16; V MN-major
      constexpr uint32_t IDESC_PV_BF16 = idesc_f16kind(BM, D, true, true);  // P, V bf16; V MN-major
      uint32_t g = 0;   // ring position consumed
      uint32_t gm = 0;  // K/V groups consumed
      uint32_t q_use[QT] = {0, 0};
      uint32_t units_done[QT] = {0, 0};
      uint32_t pv_cnt[QT] = {0, 0};
      bool ok = true;
      bool issued_any = false;

      // Descriptors: built once per operand tile, then advanced along K by adding
      // the byte offset >> 4 to the start-address field (no carry: smem < 256 KB).
      const uint64_t q_desc0 = smem_desc(base + C::Q_OFF, 16, 1024);
      const uint64_t ring_kdesc0 = smem_desc(base + C::RING_OFF, 16, 1024);
      const uint64_t ring_vdesc0 = smem_desc(base + C::RING_OFF, PANEL_BYTES, 1024);

      // S_t = Q_t K^T from the K tile in `slot` (D/16 MMAs behind one elect).
      auto issue_s = [&](auto tc, uint32_t slot) {
        constexpr int t = decltype(tc)::value;
        const uint64_t qd = q_desc0 + (uint64_t)((t * C::TILE_BYTES) >> 4);
        const uint64_t kd = ring_kdesc0 + (uint64_t)((slot * C::TILE_BYTES) >> 4);
        const uint32_t dt = tmem + TMEM_S0 + 128u * t;
        mma_ss_batch<D / 16>(dt, qd, kd, IDESC_S, 0u);
      };
      // O_t (+)= P_t V over the tile's 128 keys: P in tensor memory, V (keys x
      // D, D contiguous) in `slot`; eight MMAs behind one elect.
      static_assert(BN == 128, "the P V batch issues 8 MMAs of 16 keys");
      auto issue_pv = [&](auto tc, uint32_t slot, uint32_t accumulate, uint32_t idesc_pv) {
        constexpr int t = decltype(tc)::value;
        const uint64_t vd = ring_vdesc0 + (uint64_t)((slot * C::TILE_BYTES) >> 4);
        mma_ts_batch8(tmem + TMEM_O0 + 128u * t, tmem + TMEM_S0 + 128u * t, vd, idesc_pv, accumulate);
      };

      pdl_wait();  // the V storage modes come from the pre-pass
      UnitIter it;
      it.begin(p, cta, G);
      for (; ok && it.u >= 0; it.advance(p, cta, G)) {
        const int u = it.u;
        const Unit w = decode_unit<SPLIT>(p, u, it.kl_raw);
        if (w.nkv == 0) continue;  // (advance requests the next unit)
        auto kslot = [&](int j) { return (g + 2u * j) % C::STAGES; };
        auto vslot = [&](int j) { return (g + 2u * j + 1u) % C::STAGES; };

        // K/V group gm: one full barrier for the tiles of one step
        // (no vote after the waits of the step loop: every lane tests the same
        // barrier word in the same instruction, so the result is warp-uniform)
        auto kv_wait = [&]() {
          const int id = C::B_KV_FULL + (int)(gm % C::KV_GROUPS);
          ok = wait_bar(waiter, bar(id), (gm / C::KV_GROUPS) & 1u, id, u);
        };
        auto kv_release = [&]() {
          mma_commit_w(bar(C::B_KV_EMPTY + (int)(gm % C::KV_GROUPS)));
          ++gm;
        };

        // prologue: S_t,0 for each tile with work
        kv_wait();
        issued_any = true;  // before any MMA, so an abort mid-prologue still drains
        auto prologue = [&](auto tc) {
          constexpr int t = decltype(tc)::value;
          if (!ok || w.n(t) == 0) return;
          ok = wait_bar(waiter, bar(C::B_Q_FULL + t), q_use[t] & 1u, C::B_Q_FULL + t, u);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) return;
          ++q_use[t];
          tc_fence_after();
          issue_s(tc, kslot(0));
          mma_commit_w(bar(C::B_S_FULL + t));
          if (w.n(t) == 1) mma_commit_w(bar(C::B_Q_EMPTY + t));
        };
        prologue(TileC<0>{});
        prologue(TileC<1>{});
        if (!ok) break;
        kv_release();

        const uint8_t* modes = p.v_mode + (size_t)w.bh * p.mode_stride + w.j0;
        int vmode_next = SPLIT ? (int)__ldg(modes) : it.mode0;  // a split's first V tile is read here
        for (int j = 0; ok && j < w.nkv; ++j) {
          const uint32_t idesc_pv = vmode_next == VMODE_F16 ? IDESC_PV_F16 : IDESC_PV_BF16;
          if (j + 1 < w.nkv) vmode_next = __ldg(modes + j + 1);  // fetched a tile ahead
          it.at_tile(p, j);
          // V_j and K_j+1 (almost always resident already), before waiting on P
          kv_wait();
          // O_t += P_t V_j, then S_t,j+1 = Q_t K_j+1^T (tile 1's MMAs run while tile 0's softmax works)
          auto step = [&](auto tc) {
            constexpr int t = decltype(tc)::value;
            if (!ok || j >= w.n(t)) return;
            if (j == 0) {
              ok = wait_bar(waiter, bar(C::B_O_EMPTY + t), (units_done[t] & 1u) ^ 1u, C::B_O_EMPTY + t, u);
          ok = __all_sync(0xffffffffu, ok);
              if (!ok) return;
            }
            ok = wait_bar(waiter, bar(C::B_P_FULL + t), pv_cnt[t] & 1u, C::B_P_FULL + t, u);
            if (!ok) return;
            ++pv_cnt[t];
            tc_fence_after();
            issue_pv(tc, vslot(j), j > 0 ? 1u : 0u, idesc_pv);
            if (j == w.n(t) - 1) mma_commit_w(bar(C::B_O_FULL + t));
            if (j + 1 < w.n(t)) {
              issue_s(tc, kslot(j + 1));
              mma_commit_w(bar(C::B_S_FULL + t));
              if (j + 1 == w.n(t) - 1) mma_commit_w(bar(C::B_Q_EMPTY + t));
            }
          };
          step(TileC<0>{});
          step(TileC<1>{});
          if (!ok) break;
          kv_release();
        }
        g += 2u * (uint32_t)w.nkv;
        if (w.n0 > 0) ++units_done[0];
        if (w.n1 > 0) ++units_done[1];
      }
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      if (issued_any) {
        mma_commit_w(bar(C::B_DRAIN));
        drain_wait(bar(C::B_DRAIN), 0, 50000000ull);
      }
    }
  }
  } else {
    regs_grow<SOFTMAX_REGS>();
    // ------------------------------------------------------------ softmax groups
    waiter.role = ROLE_SOFTMAX;
    const int t = warp / 4;                  // query tile of this group
    const int quarter = warp % 4;            // TMEM lane quarter
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + TMEM_S0 + 128u * t;
    const uint32_t o_addr = tmem + lane_off + TMEM_O0 + 128u * t;
    const uint32_t bar_s_full = bar(C::B_S_FULL + t);
    const uint32_t bar_p_full = bar(C::B_P_FULL + t);
    const uint32_t bar_o_full = bar(C::B_O_FULL + t);
    const uint32_t bar_o_empty = bar(C::B_O_EMPTY + t);
    const float c = p.scale_log2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;

    pdl_wait();  // the V storage modes come from the pre-pass
    UnitIter it;
    it.begin(p, cta, G);
    for (; ok && it.u >= 0; it.advance(p, cta, G)) {
      const int u = it.u;
      const Unit w = decode_unit<SPLIT>(p, u, it.kl_raw);
      if (!w.valid(t)) continue;
      const int n_t = w.n(t);
      const int min_lim = w.min_lim(t);
      const int row = w.r0 + t * BM + row_in_tile;
      const bool row_ok = row < p.N;
      const size_t row_flat = (size_t)w.bh * (size_t)p.N + (size_t)row;
      if (n_t == 0) {
        // split-KV: this split holds none of the tile's keys (the combine
        // kernel reads only the splits that do)
        if constexpr (SPLIT) continue;
        // no visible key at all: O = 0, LSE = -inf
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + row_flat * hd);
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            if (8 * i < hd) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[row_flat] = -INFINITY;
        }
        continue;
      }
      // keys [0, lim) are visible; both limits are taken relative to the
      // split's first key, so the tile loop below counts from 0
      const int lim = (p.causal ? min(w.kl, row + 1) : w.kl) - w.j0 * BN;
      const int min_lim_s = min_lim - w.j0 * BN;
      float m_ref = -INFINITY;
      float l = 0.0f;
      const uint8_t* modes = p.v_mode + (size_t)w.bh * p.mode_stride + w.j0;
      int vmode_next = it.mode0;

      for (int j = 0; j < n_t; ++j) {
        int vmode;
        if constexpr (SPLIT) {
          // storage type of V_j, needed only once P is formed (the load's
          // latency hides behind the S wait and the exponentials)
          vmode = __ldg(modes + j);
        } else {
          vmode = vmode_next;
          if (j + 1 < n_t) vmode_next = __ldg(modes + j + 1);  // fetched a tile ahead
        }
        it.at_tile(p, j);
        ok = wait_bar(waiter, bar_s_full, s_cnt & 1u, C::B_S_FULL + t, u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();

        const bool masked_tile = (j + 1) * BN > min_lim_s;
        const int vis_n = lim - j * BN;  // columns [0, vis_n) visible
        // row max: from the TMEM load's max reduction on tiles without a mask;
        // with a mask, in registers over the visible columns only
        float mx;
        if (!masked_tile) {
          float m0, m1;
          {
            float sr[64];
            tmem_ld64_max(s_addr, sr, m0);
            tmem_ld_wait(sr, m0);
          }
          {
            float sr[64];
            tmem_ld64_max(s_addr + 64u, sr, m1);
            tmem_ld_wait(sr, m1);
          }
          mx = fmaxf(m0, m1);
        } else {
          float s[BN];
          {
            uint32_t r32[BN];
            tmem_ld128(s_addr, r32);
            tmem_ld_wait(r32);
#pragma unroll
            for (int i = 0; i < BN; ++i) s[i] = i < vis_n ? __uint_as_float(r32[i]) : -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(s[i], s[i + 8], s[i + 16]);
#pragma unroll
          for (int i = 24; i < BN; i += 16) {
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], s[i + k], i + 8 + k < BN ? s[i + 8 + k] : -INFINITY);
          }
          mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        }
        const float m_new = fmaxf(m_ref, mx);
        float alpha = 1.0f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = m_new;  // first visible scores: O is overwritten by this tile's PV
        } else if ((m_new - m_ref) * c > RESCALE_LOG2_THRESHOLD) {
          alpha = ex2((m_ref - m_new) * c);
          m_ref = m_new;
          rescale = true;
        }
        const float mc = (m_ref == -INFINITY) ? 0.0f : m_ref * c;

        // correction first: rescale this row of O (PV of the previous tile has
        // completed, since S of this tile was issued after it and has completed)
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r32[32];
            tmem_ld32(o_addr + 32u * cc, r32);
            tmem_ld_wait(r32);
#pragma unroll
            for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(__uint_as_float(r32[i]) * alpha);
            tmem_st32(o_addr + 32u * cc, r32);
          }
        }

        // p = 2^(s*c - m*c): kept in fp32 for l, rounded for PV to fp16 (11
        // significant bits), the type of the V tile in the usual case.  Where
        // the V tile is stored in bf16, the packed P is rewritten as bf16 after
        // both halves are stored (a short, rarely run pass; p <= 1, so fp16
        // cannot overflow, and values under 2^-24 of the row max drop to zero).
        // Masked entries are exactly zero.
        // The row is done in two halves of 64 keys, each reloaded from tensor
        // memory, so that S and P of only one half are held in registers.
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nmc2 = f2_pack(-mc, -mc);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // MASKED: the limit tile of the row (keys at or past vis_n are zero);
        // a separate copy of the loop, so that tiles without a mask carry no
        // per-element selects
        auto half_row = [&](int h, auto masked_c) {
          constexpr bool MASKED = decltype(masked_c)::value;
          // S of this half row again (cheap to reload; keeps registers free)
          uint32_t sh[64];
          tmem_ld64(s_addr + 64u * h, sh);
          tmem_ld_wait(sh);
          uint32_t pk[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int i = 64 * h + 2 * q;
            float x0, x1, p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sh[2 * q]), __uint_as_float(sh[2 * q + 1])), c2, nmc2), x0, x1);
            p0 = ex2(x0);
            p1 = ex2(x1);
            if constexpr (MASKED) {
              p0 = i < vis_n ? p0 : 0.0f;
              p1 = i + 1 < vis_n ? p1 : 0.0f;
            }
            acc[q % 4] = f2_add(acc[q % 4], f2_pack(p0, p1));
            pk[q] = pack_f16x2(p0, p1);
          }
          tmem_st32(s_addr + 32u * h, pk);
        };
        // (the two halves share one copy of the loop body: a smaller hot
        // loop, measured faster than the unrolled pair)
        if (masked_tile) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) half_row(h, std::true_type{});
        } else {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) half_row(h, std::false_type{});
        }
        if (vmode != VMODE_F16) {
          tmem_st_wait();  // the fp16 P must be in tensor memory before it is read back
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
            tmem_ld32(s_addr + 32u * h, pk);
            tmem_ld_wait(pk);
#pragma unroll
            for (int q = 0; q < 32; ++q) pk[q] = f16x2_to_bf16x2(pk[q]);
            tmem_st32(s_addr + 32u * h, pk);
          }
        }
        float a0, a1, a2, a3, a4, a5, a6, a7;
        f2_unpack(acc[0], a0, a1);
        f2_unpack(acc[1], a2, a3);
        f2_unpack(acc[2], a4, a5);
        f2_unpack(acc[3], a6, a7);
        const float rs = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
        l = l * alpha + rs;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_full);
      }
      if (!ok) break;

      // epilogue: O / l -> bf16, LSE = m*scale + ln(l)
      ok = wait_bar(waiter, bar_o_full, o_cnt & 1u, C::B_O_FULL + t, u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
      if constexpr (SPLIT) {
        // this split's O / l and log-sum-exp in fp32, for the combine kernel;
        // O is handed back to the MMA issuer once both halves are in registers
        const size_t orow = (size_t)w.split * (size_t)(p.B * p.H) * (size_t)p.N + row_flat;
#pragma unroll
        for (int hcol = 0; hcol < D / 64; ++hcol) {
          uint32_t ov[64];
          tmem_ld64(o_addr + 64u * hcol, ov);
          tmem_ld_wait(ov);
          if (hcol == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(bar_o_empty);
          }
          if (row_ok) {
            // 32-byte stores (the partials are the library's own scratch, rows
            // of hd fp32: 32-byte aligned for every head dim)
            float* dstf = p.o_part + orow * hd + 64 * hcol;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (64 * hcol + 8 * i < hd)
                st_global_v8(dstf + 8 * i, __float_as_uint(__uint_as_float(ov[8 * i]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 1]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 2]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 3]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 4]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 5]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 6]) * inv_l),
                             __float_as_uint(__uint_as_float(ov[8 * i + 7]) * inv_l));
          }
        }
        if (row_ok) p.lse_part[orow] = (m_ref * c + __log2f(l)) * 0.69314718055994531f;  // l > 0 here
      } else {
        // read O 64 columns at a time, pack to bf16 and store each half; O is
        // handed back to the MMA issuer once both halves are in registers
        uint4* dst = reinterpret_cast<uint4*>(p.o + row_flat * hd);
#pragma unroll
        for (int hcol = 0; hcol < D / 64; ++hcol) {
          uint32_t ov[64];
          tmem_ld64(o_addr + 64u * hcol, ov);
          tmem_ld_wait(ov);
          uint32_t ob[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ob[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
          if (hcol == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(bar_o_empty);
          }
          if (row_ok) {
            if (p.o_v8) {
              // 32-byte stores: whole sectors of the row (measured 0.4 % faster
              // on the b2h16n4096d128 causal call, 2 % with key padding)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (64 * hcol + 16 * i < hd)
                  st_global_v8(dst + 8 * hcol + 2 * i, ob[8 * i], ob[8 * i + 1], ob[8 * i + 2], ob[8 * i + 3],
                               ob[8 * i + 4], ob[8 * i + 5], ob[8 * i + 6], ob[8 * i + 7]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (64 * hcol + 8 * i < hd)
                  dst[8 * hcol + i] = make_uint4(ob[4 * i], ob[4 * i + 1], ob[4 * i + 2], ob[4 * i + 3]);
            }
          }
        }
        if (row_ok) {
          const float lse = (l > 0.0f) ? (m_ref * c + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          p.lse[row_flat] = lse;
        }
      }
    }
  }

  __syncwarp();  // the producer and MMA warps ran their roles on one lane
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace fattn
