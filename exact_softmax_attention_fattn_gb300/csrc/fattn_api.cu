// C ABI of libfattn: argument validation, TMA tensor-map encoding and the
// launch of the sm_103a attention kernel.  See include/fattn.h for the
// contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/fattn.h"
#include "fattn_bwd.cuh"
#include "fattn_bwd256.cuh"
#include "fattn_bwd_fused.cuh"
#include "fattn_d256.cuh"
#include "fattn_kernel.cuh"
#include "linear_attn.cuh"
#include "linear_tc.cuh"
#include "splitkv_combine.cuh"
#include "v_prepass.cuh"

namespace {

// Launches `kernel` as a programmatic dependent of the kernel before it on
// `stream`: its CTAs may start (set-up, loads of inputs the caller owns) as
// the earlier grid's CTAs retire; each reads what that grid wrote only after
// griddepcontrol.wait, and every CTA of it waits there before it exits.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int* err = nullptr;             // int[4] device workspace
  cudaMemPool_t pool = nullptr;   // private stream-ordered pool for per-call scratch
  cudaStream_t copy_in = nullptr;   // host-buffer entry point: host -> device copies
  cudaStream_t copy_out = nullptr;  // and device -> host copies
  // The host-buffer entry point's events, made once and reused from call to
  // call (a wait enqueued on an event refers to the record before it, so a
  // later call may record the event again); its calls on one device enqueue
  // one at a time under host_mu.
  std::mutex host_mu;
  std::vector<cudaEvent_t> host_events;
  // Unit schedules of recent causal shapes (see round_schedule); a null
  // table means the snake order is as good.
  struct Sched {
    int BH, N, G;
    std::vector<uint16_t> host;
    uint16_t* dev;
  };
  std::mutex sched_mu;
  std::vector<Sched> scheds;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Events the calling thread asked to have recorded around the dominant
// kernel of its calls (fattn_set_kernel_events); null: none.
thread_local cudaEvent_t t_kernel_start = nullptr;
thread_local cudaEvent_t t_kernel_stop = nullptr;
void mark_kernel_start(cudaStream_t s) {
  if (t_kernel_start) cudaEventRecord(t_kernel_start, s);
}
void mark_kernel_stop(cudaStream_t s) {
  if (t_kernel_stop) cudaEventRecord(t_kernel_stop, s);
}
EncodeTiledFn g_encode = nullptr;

// Limit of every bounded wait inside the kernel: 2 s unless FATTN_WAIT_LIMIT_MS
// or (finer, taking precedence) FATTN_WAIT_LIMIT_US is set; read once (the
// static's initialisation is thread-safe).
unsigned long long wait_limit_ns() {
  static const unsigned long long limit = [] {
    unsigned long long ns = 2000ull * 1000000ull;
    if (const char* e = std::getenv("FATTN_WAIT_LIMIT_MS")) {
      long long v = std::atoll(e);
      if (v > 0) ns = (unsigned long long)v * 1000000ull;
    }
    if (const char* e = std::getenv("FATTN_WAIT_LIMIT_US")) {
      long long v = std::atoll(e);
      if (v > 0) ns = (unsigned long long)v * 1000ull;
    }
    return ns;
  }();
  return limit;
}

// Sets the kernel's shared-memory limit and checks that it was compiled with
// the register count its setmaxnreg split assumes (a split larger than the
// launch allocation would never be granted).
template <int D, bool SPLIT, bool FULL>
int configure_fwd_kernel() {
  cudaError_t e = cudaFuncSetAttribute(fattn::fattn_fwd_kernel<D, SPLIT, FULL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fattn::Cfg<D>::SMEM_BYTES);
  if (e != cudaSuccess) return FATTN_ERR_CUDA;
  cudaFuncAttributes a;
  if (cudaFuncGetAttributes(&a, fattn::fattn_fwd_kernel<D, SPLIT, FULL>) != cudaSuccess) return FATTN_ERR_CUDA;
  if (a.numRegs != fattn::LAUNCH_REGS) return FATTN_ERR_UNSUPPORTED;
  return FATTN_OK;
}

// The three passes of the 256-column backward.
int configure_bwd256_kernels() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  return cudaFuncSetAttribute(fattn::fattn_bwd256_kernel<fattn::BP_DV>, attr,
                              (int)fattn::Bwd256Cfg<fattn::BP_DV>::SMEM_BYTES) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_bwd256_kernel<fattn::BP_DK>, attr,
                                      (int)fattn::Bwd256Cfg<fattn::BP_DK>::SMEM_BYTES) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_bwd256_kernel<fattn::BP_DQ>, attr,
                                      (int)fattn::Bwd256Cfg<fattn::BP_DQ>::SMEM_BYTES) == cudaSuccess
             ? FATTN_OK
             : FATTN_ERR_CUDA;
}

template <bool FULL>
int configure_d256_kernel() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const int bytes = (int)fattn::D256Cfg::SMEM_BYTES;
  return cudaFuncSetAttribute(fattn::fattn_fwd_d256_kernel<FULL, false>, attr, bytes) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_fwd_d256_kernel<FULL, true>, attr, bytes) == cudaSuccess
             ? FATTN_OK
             : FATTN_ERR_CUDA;
}

// The linear-attention kernels' shared memory, at the largest feature sizes.
int configure_linear_kernels() {
  const fattn::LinSmem L(128, 128);
  const int state_bytes = (128 * fattn::LIN_C + fattn::LIN_C * 128) * 4;
  const fattn::LinSmem L64(64, 64);
  const int state64 = (64 * fattn::LIN_C + fattn::LIN_C * 64) * 4;
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const int tc_bytes = (int)fattn::LtcCfg::SMEM_BYTES;
  return cudaFuncSetAttribute(fattn::fattn_linear_tc_kernel<true>, attr, tc_bytes) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_linear_tc_kernel<false>, attr, tc_bytes) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_linear_state_kernel<0, 0>, attr, state_bytes) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_linear_output_kernel<0, 0>, attr, L.total * 4) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_linear_state_kernel<64, 64>, attr, state64) == cudaSuccess &&
                 cudaFuncSetAttribute(fattn::fattn_linear_output_kernel<64, 64>, attr, L64.total * 4) == cudaSuccess
             ? FATTN_OK
             : FATTN_ERR_CUDA;
}

template <int D>
int configure_kernel() {
  int rc = configure_fwd_kernel<D, false, true>();
  if (rc == FATTN_OK) rc = configure_fwd_kernel<D, true, true>();
  if (rc == FATTN_OK) rc = configure_fwd_kernel<D, false, false>();
  if (rc == FATTN_OK) rc = configure_fwd_kernel<D, true, false>();
  if (rc != FATTN_OK) return rc;
  if (cudaFuncSetAttribute(fattn::fattn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fattn::BwdCfg<D>::SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(fattn::fattn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fattn::BwdDqCfg<D>::SMEM_BYTES) != cudaSuccess)
    return FATTN_ERR_CUDA;
  return FATTN_OK;
}

// A pool that keeps its memory (release threshold = max) so the per-call
// scratch is recycled in stream order instead of returned to the driver.
int make_pool(int dev, cudaMemPool_t* pool) {
  cudaMemPoolProps props = {};
  props.allocType = cudaMemAllocationTypePinned;
  props.handleTypes = cudaMemHandleTypeNone;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t made = nullptr;
  if (cudaMemPoolCreate(&made, &props) != cudaSuccess) return FATTN_ERR_CUDA;
  uint64_t keep = UINT64_MAX;
  if (cudaMemPoolSetAttribute(made, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
    cudaMemPoolDestroy(made);
    return FATTN_ERR_CUDA;
  }
  *pool = made;  // set only once the pool is complete
  return FATTN_OK;
}

// Per-device set-up, once: SM count, kernel attributes, the error word.  A
// set-up that failed part of the way is resumed by the next call: resources
// already made are kept, not made again.
int device_state(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  int rc = FATTN_OK;
  if (!s.ready) {
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FATTN_ERR_CUDA;
    rc = configure_kernel<64>();
    if (rc == FATTN_OK) rc = configure_kernel<128>();
    if (rc == FATTN_OK) rc = configure_d256_kernel<true>();
    if (rc == FATTN_OK) rc = configure_d256_kernel<false>();
    if (rc == FATTN_OK) rc = configure_bwd256_kernels();
    if (rc == FATTN_OK && cudaFuncSetAttribute(fattn::fattn_bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)fattn::FusedCfg::SMEM_BYTES) != cudaSuccess)
      rc = FATTN_ERR_CUDA;
    if (rc == FATTN_OK) rc = configure_linear_kernels();
    if (rc != FATTN_OK) return rc;
    if (!s.pool && make_pool(dev, &s.pool) != FATTN_OK) return FATTN_ERR_CUDA;
    if (!s.err && cudaMalloc(&s.err, 4 * sizeof(int)) != cudaSuccess) {
      s.err = nullptr;
      return FATTN_ERR_CUDA;
    }
    if (!s.copy_in && cudaStreamCreateWithFlags(&s.copy_in, cudaStreamNonBlocking) != cudaSuccess) {
      s.copy_in = nullptr;
      return FATTN_ERR_CUDA;
    }
    if (!s.copy_out && cudaStreamCreateWithFlags(&s.copy_out, cudaStreamNonBlocking) != cudaSuccess) {
      s.copy_out = nullptr;
      return FATTN_ERR_CUDA;
    }
    if (cudaMemset(s.err, 0, 4 * sizeof(int)) != cudaSuccess) return FATTN_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return FATTN_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return FATTN_OK;
}

bool is_device_pointer(const void* ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Tensor maps already encoded, keyed by everything a map is made from
// (address, shape, element type, box): a map depends on nothing else, so a
// hit is exactly the map that encoding again would give, even when the
// memory behind the address was freed and reallocated meanwhile.  Encoding
// is host work repeated on every call of a training or serving loop, where
// the same buffers come back call after call.
struct MapKey {
  const void* ptr;
  int BH, N, d;
  int type;
  unsigned box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && BH == o.BH && N == o.N && d == o.d && type == o.type && box_rows == o.box_rows;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_maps_used = 0, g_maps_next = 0;
std::atomic<long long> g_map_hits{0}, g_map_misses{0};

bool map_lookup(const MapKey& key, CUtensorMap* map) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_maps_used; ++i)
    if (g_maps[i].key == key) {
      *map = g_maps[i].map;
      return true;
    }
  return false;
}

void map_insert(const MapKey& key, const CUtensorMap& map) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_maps_used; ++i)
    if (g_maps[i].key == key) return;  // another thread got there first
  g_maps[g_maps_next] = MapEntry{key, map};
  g_maps_next = (g_maps_next + 1) % kMapCache;
  if (g_maps_used < kMapCache) ++g_maps_used;
}

// [B*H, N, d] 16-bit elements viewed as a 3-D tensor: x = head dim (innermost),
// y = row, z = batch*head.  Boxes of 64 x box_rows x 1 with 128-byte swizzle;
// rows past N and columns past d (head dims below the kernel's column count)
// read as zero.
int encode_map(CUtensorMap* map, const void* ptr, int BH, int N, int d, CUtensorMapDataType type,
               unsigned box_rows = 128u) {
  const MapKey key{ptr, BH, N, d, (int)type, box_rows};
  if (map_lookup(key, map)) {
    g_map_hits.fetch_add(1, std::memory_order_relaxed);
    return FATTN_OK;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2ull, (cuuint64_t)N * (cuuint64_t)d * 2ull};
  cuuint32_t box[3] = {64u, box_rows, 1u};
  cuuint32_t elem[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, type, 3, const_cast<void*>(ptr), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FATTN_ERR_CUDA;
  g_map_misses.fetch_add(1, std::memory_order_relaxed);
  map_insert(key, *map);
  return FATTN_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }


// [B*H, N, F] fp32 viewed as a 3-D tensor {F, N, B*H}, boxes of 64 x 128 x 1
// without swizzle (rows of 256 bytes in shared memory); columns past F and
// rows past N read as zero.
int encode_map_f32(CUtensorMap* map, const void* ptr, int BH, int N, int F) {
  const MapKey key{ptr, BH, N, F, (int)CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (unsigned)fattn::LTC_T};
  if (map_lookup(key, map)) {
    g_map_hits.fetch_add(1, std::memory_order_relaxed);
    return FATTN_OK;
  }
  cuuint64_t dims[3] = {(cuuint64_t)F, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)F * 4ull, (cuuint64_t)N * (cuuint64_t)F * 4ull};
  cuuint32_t box[3] = {(cuuint32_t)fattn::LTC_F, (cuuint32_t)fattn::LTC_T, 1u};
  cuuint32_t elem[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FATTN_ERR_CUDA;
  g_map_misses.fetch_add(1, std::memory_order_relaxed);
  map_insert(key, *map);
  return FATTN_OK;
}

// Head dims the kernels run: multiples of 8 (rows of 16-byte vectors, TMA
// strides in 16-byte units), computed in the 64-, 128- or 256-column kernel
// with the columns past d read as zeros by the tensor maps.  The forward and
// the backward run up to 256.
bool head_dim_supported(int d, int max_d = 256) { return d >= 8 && d <= max_d && d % 8 == 0; }

// Scratch of one call: V in its per-tile storage type, then one mode byte per
// tile, each head's row of modes padded to a multiple of 8 bytes; with
// split-KV, then the fp32 partial outputs and log-sum-exps of every split.
size_t scratch_bytes(int BH, int N, int D, int n_tiles, int n_splits = 1) {
  size_t b = round_up((size_t)BH * (size_t)N * (size_t)D * 2u, 256) +
             round_up((size_t)BH * round_up((size_t)n_tiles, 8), 256);
  if (n_splits > 1)
    b += round_up((size_t)n_splits * BH * (size_t)N * (size_t)D * 4u, 256) +
         round_up((size_t)n_splits * BH * (size_t)N * 4u, 256);
  return b;
}

// ------------------------------------------------------------------ split-KV plan
// Per work unit with work, a fixed cost (Q load, first S, epilogue) and, for
// a split launch, the combine pass, both in K/V steps of the attention kernel;
// set from GB300 timings of the low-occupancy shapes.
constexpr double kUnitOverheadSteps = 10.0;
constexpr double kCombineSteps = 6.0;
constexpr int kMaxSplits = 16;

// Makespan estimate, in K/V steps, of the kernel's static snake schedule for
// one split count (key padding unknown on the host: all N keys assumed).
// Split s of a block with n key tiles takes [s*n/splits, (s+1)*n/splits).
double split_cost(int B, int H, int N, int causal, int num_sms, int splits) {
  const long long BH = (long long)B * H;
  const int nqb = (N + fattn::QT * fattn::BM - 1) / (fattn::QT * fattn::BM);
  const long long units = BH * nqb * splits;
  const int G = (int)std::min<long long>(units, num_sms);
  std::vector<double> load((size_t)G, 0.0);
  for (long long u = 0; u < units; ++u) {
    const long long r = u / G, i = u % G;
    const int c = (int)((r & 1) ? G - 1 - i : i);
    const int round = (int)(u / (BH * splits));
    const int sp = (int)((u / BH) % splits);
    const int r0 = (nqb - 1 - round) * fattn::QT * fattn::BM;
    int n_blk = 0;
    for (int t = 0; t < fattn::QT; ++t) {
      const int row0 = r0 + t * fattn::BM;
      if (row0 >= N) continue;
      const int max_lim = causal ? std::min(N, row0 + fattn::BM) : N;
      n_blk = std::max(n_blk, (max_lim + fattn::BN - 1) / fattn::BN);
    }
    const int n = (sp + 1) * n_blk / splits - sp * n_blk / splits;
    if (n > 0) load[(size_t)c] += n + kUnitOverheadSteps;
  }
  return *std::max_element(load.begin(), load.end()) + (splits > 1 ? kCombineSteps : 0.0);
}

// The searched plans of recent shapes: the search simulates the schedule for
// every candidate, too slow to repeat on each call of a hot loop.
struct PlanEntry {
  int B, H, N, causal, num_sms, splits;
};
constexpr int kPlanCache = 64;
std::mutex g_plan_mu;
PlanEntry g_plans[kPlanCache];
int g_plans_used = 0, g_plans_next = 0;

// K/V splits per query block.  requested > 0: that many, at most one per key
// tile; 0: the cheapest by split_cost, searched only when the query blocks
// alone leave SMs idle.
int plan_splits(int B, int H, int N, int causal, int num_sms, int requested) {
  const int n_kv = (N + fattn::BN - 1) / fattn::BN;
  const long long units = (long long)B * H * ((N + fattn::QT * fattn::BM - 1) / (fattn::QT * fattn::BM));
  if (requested > 0) return std::min(requested, n_kv);
  if (units >= num_sms || n_kv < 2) return 1;
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (int i = 0; i < g_plans_used; ++i) {
      const PlanEntry& e = g_plans[i];
      if (e.B == B && e.H == H && e.N == N && e.causal == causal && e.num_sms == num_sms) return e.splits;
    }
  }
  int best = 1;
  {
    double best_cost = split_cost(B, H, N, causal, num_sms, 1);
    for (int sp = 2; sp <= std::min(n_kv, kMaxSplits); ++sp) {
      const double cst = split_cost(B, H, N, causal, num_sms, sp);
      if (cst < best_cost) {
        best_cost = cst;
        best = sp;
      }
    }
  }
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plans[g_plans_next] = PlanEntry{B, H, N, causal, num_sms, best};
  g_plans_next = (g_plans_next + 1) % kPlanCache;
  if (g_plans_used < kPlanCache) ++g_plans_used;
  return best;
}

// K/V splits per query tile of the head-dim-256 kernel (one CTA per 128-row
// query tile and split, 64-key tiles).  requested > 0: that many, at most one
// per key tile; 0: when the query tiles alone leave SMs idle, enough splits
// to give every SM a CTA, keeping at least two key tiles per split.
int plan_splits_d256(int B, int H, int N, int num_sms, int requested) {
  const long long n_kv = (N + fattn::D256_BN - 1) / fattn::D256_BN;
  const long long tiles = (long long)B * H * ((N + fattn::BM - 1) / fattn::BM);
  if (requested > 0) return (int)std::min<long long>(requested, std::max<long long>(1, n_kv));
  if (tiles >= num_sms || n_kv < 4) return 1;
  return (int)std::max<long long>(1, std::min<long long>({num_sms / tiles, n_kv / 2, (long long)kMaxSplits}));
}

// Enqueues the V pre-pass, the attention kernel and, with split-KV, the
// combine kernel; `scratch` must hold scratch_bytes(..., p.n_splits).
template <int D>
int enqueue(const void* q, const void* k, const void* v, fattn::Params p, void* scratch, int grid,
            cudaStream_t stream) {
  const int BH = p.B * p.H;
  uint8_t* v16 = reinterpret_cast<uint8_t*>(scratch);
  uint8_t* modes = v16 + round_up((size_t)BH * (size_t)p.N * (size_t)p.hd * 2u, 256);
  p.v_mode = modes;
  if (p.n_splits > 1) {
    uint8_t* part = modes + round_up((size_t)BH * round_up((size_t)p.n_kv_tiles, 8), 256);
    p.o_part = reinterpret_cast<float*>(part);
    p.lse_part =
        reinterpret_cast<float*>(part + round_up((size_t)p.n_splits * BH * (size_t)p.N * (size_t)p.hd * 4u, 256));
  }
  CUtensorMap mq, mk, mv;
  if (encode_map(&mq, q, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mk, k, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mv, v16, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) != FATTN_OK)
    return FATTN_ERR_CUDA;
  const long long prepass_blocks = (long long)BH * p.n_kv_tiles;
  if (p.hd == D)
    fattn::fattn_v_prepass_kernel<D, true><<<(unsigned)prepass_blocks, fattn::PREPASS_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(v16), modes, p.N, p.hd, p.n_kv_tiles,
        p.mode_stride);
  else
    fattn::fattn_v_prepass_kernel<D, false><<<(unsigned)prepass_blocks, fattn::PREPASS_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(v16), modes, p.N, p.hd, p.n_kv_tiles,
        p.mode_stride);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  constexpr uint32_t smem = fattn::Cfg<D>::SMEM_BYTES;
  constexpr int nt = fattn::NUM_THREADS;
  const bool full = p.hd == D;
  mark_kernel_start(stream);
  {
    // The attention kernel is launched as a programmatic dependent of the
    // pre-pass: its CTAs start on the SMs the pre-pass leaves free and run
    // their set-up, Q/K loads and first S products while it finishes; every
    // read of the V copy or the tile modes comes after griddepcontrol.wait.
    // (Measured 1.6 % faster on the b2h16n4096d128 causal call, and more on
    // grids smaller than the GPU.)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)nt);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (p.n_splits > 1 && full)
      e = cudaLaunchKernelEx(&cfg, fattn::fattn_fwd_kernel<D, true, true>, mq, mk, mv, p);
    else if (p.n_splits > 1)
      e = cudaLaunchKernelEx(&cfg, fattn::fattn_fwd_kernel<D, true, false>, mq, mk, mv, p);
    else if (full)
      e = cudaLaunchKernelEx(&cfg, fattn::fattn_fwd_kernel<D, false, true>, mq, mk, mv, p);
    else
      e = cudaLaunchKernelEx(&cfg, fattn::fattn_fwd_kernel<D, false, false>, mq, mk, mv, p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return FATTN_ERR_CUDA;
    }
  }
  mark_kernel_stop(stream);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  if (p.n_splits > 1) {
    constexpr int rows_per_block = fattn::COMBINE_THREADS / (D / 16);
    const dim3 cgrid((unsigned)((p.N + rows_per_block - 1) / rows_per_block), (unsigned)(BH < 65535 ? BH : 65535));
    // a programmatic dependent of the attention kernel: its launch overlaps
    // the attention kernel's last CTAs, and it reads the partials only after
    // griddepcontrol.wait
    if (launch_dependent(fattn::fattn_splitkv_combine_kernel<D>, cgrid, fattn::COMBINE_THREADS, 0, stream,
                         (const float*)p.o_part, (const float*)p.lse_part, p.o, p.lse, p.key_len, p.B, p.H, p.N,
                         p.hd, p.causal, p.n_splits, fattn::QT * fattn::BM, fattn::BN) != cudaSuccess) {
      cudaGetLastError();
      return FATTN_ERR_CUDA;
    }
  }
  return FATTN_OK;
}

// Head dims 136..256: V pre-pass, the one-query-tile kernel and, with
// split-KV (p.n_splits > 1), the combine kernel; `scratch` must hold
// scratch_bytes(..., p.n_splits).
int enqueue_d256(const void* q, const void* k, const void* v, fattn::Params p, void* scratch, cudaStream_t stream) {
  const int BH = p.B * p.H;
  uint8_t* v16 = reinterpret_cast<uint8_t*>(scratch);
  uint8_t* modes = v16 + round_up((size_t)BH * (size_t)p.N * (size_t)p.hd * 2u, 256);
  p.v_mode = modes;
  if (p.n_splits > 1) {
    uint8_t* part = modes + round_up((size_t)BH * round_up((size_t)p.n_kv_tiles, 8), 256);
    p.o_part = reinterpret_cast<float*>(part);
    p.lse_part =
        reinterpret_cast<float*>(part + round_up((size_t)p.n_splits * BH * (size_t)p.N * (size_t)p.hd * 4u, 256));
  }
  CUtensorMap mq, mk, mv;
  if (encode_map(&mq, q, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 128u) != FATTN_OK ||
      encode_map(&mk, k, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (unsigned)fattn::D256_BN) != FATTN_OK ||
      encode_map(&mv, v16, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (unsigned)fattn::D256_BN) != FATTN_OK)
    return FATTN_ERR_CUDA;
  const long long prepass_blocks = (long long)BH * p.n_kv_tiles;
  const bool full = p.hd == fattn::D256;
  if (full)
    fattn::fattn_v_prepass_kernel<256, true><<<(unsigned)prepass_blocks, fattn::prepass_threads<256>(), 0, stream>>>(
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(v16), modes, p.N, p.hd, p.n_kv_tiles,
        p.mode_stride);
  else
    fattn::fattn_v_prepass_kernel<256, false><<<(unsigned)prepass_blocks, fattn::prepass_threads<256>(), 0, stream>>>(
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(v16), modes, p.N, p.hd, p.n_kv_tiles,
        p.mode_stride);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  const long long ctas = (long long)BH * ((p.N + fattn::BM - 1) / fattn::BM) * p.n_splits;
  if (ctas > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  // heads per group of the CTA order: the K and V of a group's heads (read by
  // every CTA of the head) should stay in L2 while the group runs, ~48 MB
  const double kv_head = 4.0 * (double)p.N * (double)p.hd;
  p.head_group = (int)std::max(1.0, std::min((double)BH, (48.0 * 1024 * 1024) / kv_head));
  constexpr uint32_t smem = fattn::D256Cfg::SMEM_BYTES;
  const bool split = p.n_splits > 1;
  mark_kernel_start(stream);
  if (full && split)
    fattn::fattn_fwd_d256_kernel<true, true><<<(unsigned)ctas, fattn::D256_THREADS, smem, stream>>>(mq, mk, mv, p);
  else if (full)
    fattn::fattn_fwd_d256_kernel<true, false><<<(unsigned)ctas, fattn::D256_THREADS, smem, stream>>>(mq, mk, mv, p);
  else if (split)
    fattn::fattn_fwd_d256_kernel<false, true><<<(unsigned)ctas, fattn::D256_THREADS, smem, stream>>>(mq, mk, mv, p);
  else
    fattn::fattn_fwd_d256_kernel<false, false><<<(unsigned)ctas, fattn::D256_THREADS, smem, stream>>>(mq, mk, mv, p);
  mark_kernel_stop(stream);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  if (split) {
    constexpr int rows_per_block = fattn::COMBINE_THREADS / (fattn::D256 / 16);
    const dim3 cgrid((unsigned)((p.N + rows_per_block - 1) / rows_per_block), (unsigned)(BH < 65535 ? BH : 65535));
    if (launch_dependent(fattn::fattn_splitkv_combine_kernel<fattn::D256>, cgrid, fattn::COMBINE_THREADS, 0, stream,
                         (const float*)p.o_part, (const float*)p.lse_part, p.o, p.lse, p.key_len, p.B, p.H, p.N,
                         p.hd, p.causal, p.n_splits, fattn::BM, fattn::D256_BN) != cudaSuccess) {
      cudaGetLastError();
      return FATTN_ERR_CUDA;
    }
  }
  return FATTN_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace

extern "C" FATTN_API int fattn_version(void) { return 100; }

extern "C" FATTN_API int fattn_tensor_map_stats(long long* hits, long long* misses) {
  if (hits) *hits = g_map_hits.load(std::memory_order_relaxed);
  if (misses) *misses = g_map_misses.load(std::memory_order_relaxed);
  return FATTN_OK;
}

extern "C" FATTN_API const char* fattn_status_string(int status) {
  switch (status) {
    case FATTN_OK: return "ok";
    case FATTN_ERR_INVALID_ARG: return "invalid argument";
    case FATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case FATTN_ERR_CUDA: return "CUDA error";
    case FATTN_ERR_TIMEOUT: return "kernel wait timed out";
    default: return "unknown status";
  }
}

namespace {

// ------------------------------------------------------------------------
// Unit schedule of the persistent forward kernel for causal attention.
//
// The kernel deals its units (batch*head, block of 256 query rows), heaviest
// first, to G CTAs in rounds of G; the snake (CTA c takes unit c of even
// rounds, G-1-c of odd ones) pairs heavy and light units but leaves the
// CTAs' totals uneven when the rounds are not whole (on B2 H16 N4096: 512
// units for 152 CTAs, 123 against a mean of 118 tile steps).  This deals
// each round's units (the same set as the snake's, so the same K/V working
// set in each round; the first round, whose CTAs start together, as the
// snake) so that the totals come out even: the cost of a unit is the tiles
// its two query tiles visit plus two for its prologue and epilogue, and a
// deterministic annealing of swaps within a round minimises the squared
// excess of each CTA's total over the mean.  An empty result: the snake is
// as good.
std::vector<uint16_t> build_round_schedule(int BH, int N, int nqb, int G) {
  const long long units = (long long)BH * nqb;
  const int R = (int)((units + G - 1) / G);
  if (R < 2 || G > 65535) return {};
  auto weight = [&](long long u) -> int {
    if (u >= units) return 0;
    const int qb = nqb - 1 - (int)(u / BH);
    int w = 2;
    for (int tq = 0; tq < fattn::QT; ++tq) {
      const int row0 = (qb * fattn::QT + tq) * fattn::BM;
      if (row0 < N) w += (std::min(N, row0 + fattn::BM) + fattn::BN - 1) / fattn::BN;
    }
    return w;
  };
  std::vector<uint16_t> pos((size_t)R * G);
  std::vector<int> w((size_t)R * G), load((size_t)G, 0);
  long long total = 0;
  for (int r = 0; r < R; ++r)
    for (int c = 0; c < G; ++c) {
      const int slot = (r & 1) ? G - 1 - c : c;
      pos[(size_t)r * G + c] = (uint16_t)slot;
      w[(size_t)r * G + slot] = weight((long long)r * G + slot);
      load[(size_t)c] += w[(size_t)r * G + slot];
      total += w[(size_t)r * G + slot];
    }
  const int snake_max = *std::max_element(load.begin(), load.end());
  const int target = (int)(total / G);
  auto excess = [&](int x) { const long long e = std::max(0, x - target); return e * e; };
  uint64_t rng = 0x9E3779B97F4A7C15ull;
  auto next = [&]() {
    rng ^= rng << 13;
    rng ^= rng >> 7;
    rng ^= rng << 17;
    return rng;
  };
  std::vector<uint16_t> best = pos;
  int best_max = snake_max;
  double temp = 4.0;
  const int iters = 400000;
  const double cool = std::pow(0.05 / temp, 1.0 / iters);
  for (int it = 0; it < iters; ++it, temp *= cool) {
    const int r = 1 + (int)(next() % (uint64_t)(R - 1));
    const int c1 = (int)(next() % (uint64_t)G), c2 = (int)(next() % (uint64_t)G);
    if (c1 == c2) continue;
    uint16_t& p1 = pos[(size_t)r * G + c1];
    uint16_t& p2 = pos[(size_t)r * G + c2];
    const int d = w[(size_t)r * G + p1] - w[(size_t)r * G + p2];
    if (d == 0) continue;
    const int n1 = load[(size_t)c1] - d, n2 = load[(size_t)c2] + d;
    const long long delta = excess(n1) + excess(n2) - excess(load[(size_t)c1]) - excess(load[(size_t)c2]);
    const double u01 = (double)(next() >> 11) * (1.0 / 9007199254740992.0);
    if (delta > 0 && u01 >= std::exp(-(double)delta / temp)) continue;
    std::swap(p1, p2);
    load[(size_t)c1] = n1;
    load[(size_t)c2] = n2;
    if (delta < 0 && std::max(n1, n2) < best_max) {
      const int m = *std::max_element(load.begin(), load.end());
      if (m < best_max) {
        best_max = m;
        best = pos;
      }
    }
  }
  if (best_max >= snake_max) return {};
  return best;
}

// The device copy of the schedule for (BH, N, G), built and uploaded on
// first use (not while `s` is being captured into a graph); nullptr: the
// snake order.
const uint16_t* round_schedule(DeviceState* ds, int BH, int N, int nqb, int G, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(ds->sched_mu);
  for (const auto& e : ds->scheds)
    if (e.BH == BH && e.N == N && e.G == G) return e.dev;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  if (ds->scheds.size() >= 64) return nullptr;
  DeviceState::Sched e{BH, N, G, build_round_schedule(BH, N, nqb, G), nullptr};
  if (!e.host.empty()) {
    void* dev = nullptr;
    if (cudaMalloc(&dev, e.host.size() * sizeof(uint16_t)) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (cudaMemcpy(dev, e.host.data(), e.host.size() * sizeof(uint16_t), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(dev);
      return nullptr;
    }
    e.dev = reinterpret_cast<uint16_t*>(dev);
  }
  ds->scheds.push_back(std::move(e));
  return ds->scheds.back().dev;
}

// check_pointers = false: the caller owns the buffers (the host-buffer entry
// point's chunks inside its pool allocation) and has validated the rest.
int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, const int32_t* key_len, int splits_requested, void* stream,
               bool check_pointers = true) {
  // ---- synchronous argument checks: nothing is enqueued on failure
  if (B < 0 || H < 0 || N < 0 || splits_requested < 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.0f) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!head_dim_supported(d)) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFll || N > 0x7FFFFFFF - 512) return FATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (key_len && !aligned(key_len, 4)))
    return FATTN_ERR_INVALID_ARG;
  if (check_pointers &&
      (!is_device_pointer(q) || !is_device_pointer(k) || !is_device_pointer(v) || !is_device_pointer(o) ||
       !is_device_pointer(lse) || (key_len && !is_device_pointer(key_len))))
    return FATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  DeviceState* ds = nullptr;
  int rc = device_state(dev, &ds);
  if (rc != FATTN_OK) return rc;

  fattn::Params p;
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.o_v8 = (aligned(o, 32) && d % 16 == 0) ? 1 : 0;  // rows of O take 32-byte stores
  p.lse = lse;
  p.key_len = key_len;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.hd = d;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.causal = causal ? 1 : 0;
  p.n_qblocks = (N + fattn::QT * fattn::BM - 1) / (fattn::QT * fattn::BM);
  p.n_kv_tiles = (N + fattn::BN - 1) / fattn::BN;
  p.n_splits = d > 128 ? plan_splits_d256(B, H, N, ds->num_sms, splits_requested)
                       : plan_splits(B, H, N, p.causal, ds->num_sms, splits_requested);
  const long long units = (long long)B * H * p.n_qblocks * p.n_splits;
  if (units > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  p.n_units = (int)units;
  p.o_part = nullptr;
  p.head_group = 1;
  p.lse_part = nullptr;
  p.mode_stride = (p.n_kv_tiles + 7) / 8 * 8;
  if ((long long)B * H * p.mode_stride > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  p.v_mode = nullptr;
  p.wait_limit_ns = wait_limit_ns();
  const int grid = (int)(units < ds->num_sms ? units : ds->num_sms);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // causal, all keys, whole blocks: a schedule that evens out the CTAs' totals
  p.sched = (p.causal && !key_len && p.n_splits == 1 && d <= 128 && units > grid)
                ? round_schedule(ds, B * H, N, p.n_qblocks, grid, s)
                : nullptr;

  void* scratch = nullptr;
  if (cudaMallocFromPoolAsync(&scratch, scratch_bytes(B * H, N, d, p.n_kv_tiles, p.n_splits), ds->pool, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  rc = d <= 64    ? enqueue<64>(q, k, v, p, scratch, grid, s)
       : d <= 128 ? enqueue<128>(q, k, v, p, scratch, grid, s)
                  : enqueue_d256(q, k, v, p, scratch, s);
  if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  return rc;
}

}  // namespace

extern "C" FATTN_API int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                         int d, float scale, int causal, const int32_t* key_len, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, scale, causal, key_len, 0, stream);
}

extern "C" FATTN_API int fattn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                           int H, int N, int d, float scale, int causal, const int32_t* key_len,
                                           int n_splits, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, scale, causal, key_len, n_splits, stream);
}

// ------------------------------------------------------------------------
// fattn_fwd_host: the forward on host buffers.  The problem is cut into a few
// chunks (ranges of whole batch entries, or of heads within one entry, so
// that each chunk has one key-length pointer); chunk i's inputs are copied
// in on one stream while chunk i-1 computes on the caller's stream and chunk
// i-2's outputs are copied out on a third.
namespace {

struct HostChunk {
  int b0, nb;  // batch entries [b0, b0 + nb)
  int h0, nh;  // heads [h0, h0 + nh) of each
};

// `target` chunks of about equal size (fewer when B*H is smaller).
std::vector<HostChunk> host_chunks_even(int B, int H, int target);

std::vector<HostChunk> host_chunks(int B, int H, long long bytes, double flops_per_head) {
  const int target = bytes < (16ll << 20) ? 1 : 8;  // small problems: one chunk
  std::vector<HostChunk> c = host_chunks_even(B, H, target);
  // The last chunk's kernels and output copies run after every input has
  // landed.  Where that chunk's kernels are long (over ~60 GFLOP, some 50 us),
  // halve it twice (into 1/2, 1/4, 1/4 of its heads or batch entries) so that
  // this tail is short; below that the extra copies cost more than they save
  // (measured: B1 H32 N16384 causal 2476 -> 2400 us, B2 H16 N4096 causal
  // 724 -> 743 us with the split).
  const double last_flops = c.empty() ? 0.0 : flops_per_head * c.back().nb * c.back().nh;
  for (int k = 0; k < 2 && target > 1 && !c.empty() && last_flops > 60e9; ++k) {
    HostChunk last = c.back();
    if (last.nb >= 2) {
      const int keep = last.nb - last.nb / 2;
      c.back().nb = keep;
      c.push_back({last.b0 + keep, last.nb - keep, 0, H});
    } else if (last.nh >= 2) {
      const int keep = last.nh - last.nh / 2;
      c.back().nh = keep;
      c.push_back({last.b0, 1, last.h0 + keep, last.nh - keep});
    }
  }
  return c;
}

std::vector<HostChunk> host_chunks_even(int B, int H, int target) {
  std::vector<HostChunk> c;
  if (B >= target) {
    for (int i = 0; i < target; ++i) {
      const int b0 = (int)((long long)B * i / target), b1 = (int)((long long)B * (i + 1) / target);
      if (b1 > b0) c.push_back({b0, b1 - b0, 0, H});
    }
  } else {
    const int per_b = std::min(H, (target + B - 1) / B);
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < per_b; ++i) {
        const int h0 = (int)((long long)H * i / per_b), h1 = (int)((long long)H * (i + 1) / per_b);
        if (h1 > h0) c.push_back({b, 1, h0, h1 - h0});
      }
  }
  return c;
}

}  // namespace

extern "C" FATTN_API int fattn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                        int H, int N, int d, float scale, int causal, const int32_t* key_len,
                                        void* stream) {
  if (B < 0 || H < 0 || N < 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.0f) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!head_dim_supported(d)) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFll || N > 0x7FFFFFFF - 512) return FATTN_ERR_INVALID_ARG;
  if (is_device_pointer(q) || is_device_pointer(k) || is_device_pointer(v) || is_device_pointer(o) ||
      is_device_pointer(lse) || (key_len && is_device_pointer(key_len)))
    return FATTN_ERR_INVALID_ARG;  // host buffers only (fattn_fwd takes device ones)

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  DeviceState* ds = nullptr;
  int rc = device_state(dev, &ds);
  if (rc != FATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const size_t n_elem = (size_t)B * H * (size_t)N * (size_t)d;
  const size_t t16 = round_up(n_elem * 2u, 256), t_lse = round_up((size_t)B * H * (size_t)N * 4u, 256);
  void* buf = nullptr;
  if (cudaMallocFromPoolAsync(&buf, 4 * t16 + t_lse + round_up((size_t)B * 4u, 256), ds->pool, s) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  uint8_t* base = reinterpret_cast<uint8_t*>(buf);
  uint16_t* qd = reinterpret_cast<uint16_t*>(base);
  uint16_t* kd = reinterpret_cast<uint16_t*>(base + t16);
  uint16_t* vd = reinterpret_cast<uint16_t*>(base + 2 * t16);
  uint16_t* od = reinterpret_cast<uint16_t*>(base + 3 * t16);
  float* lsed = reinterpret_cast<float*>(base + 4 * t16);
  int32_t* kld = reinterpret_cast<int32_t*>(base + 4 * t16 + t_lse);

  // causal: half the score matrix (about)
  const double flops_per_head = (causal ? 2.0 : 4.0) * (double)N * (double)N * (double)d;
  const std::vector<HostChunk> chunks = host_chunks(B, H, (long long)(n_elem * 2u), flops_per_head);
  const int nc = (int)chunks.size();
  std::lock_guard<std::mutex> host_lock(ds->host_mu);
  while ((int)ds->host_events.size() < 2 * nc + 2) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      rc = FATTN_ERR_CUDA;
      break;
    }
    ds->host_events.push_back(e);
  }
  const std::vector<cudaEvent_t>& ev = ds->host_events;
  cudaEvent_t ev_alloc = rc == FATTN_OK ? ev[2 * nc] : nullptr, ev_done = rc == FATTN_OK ? ev[2 * nc + 1] : nullptr;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (rc == FATTN_OK && !(ok(cudaEventRecord(ev_alloc, s)) && ok(cudaStreamWaitEvent(ds->copy_in, ev_alloc, 0))))
    rc = FATTN_ERR_CUDA;
  if (rc == FATTN_OK && key_len &&
      !ok(cudaMemcpyAsync(kld, key_len, (size_t)B * 4u, cudaMemcpyHostToDevice, ds->copy_in)))
    rc = FATTN_ERR_CUDA;
  const uint16_t* qh = reinterpret_cast<const uint16_t*>(q);
  const uint16_t* kh = reinterpret_cast<const uint16_t*>(k);
  const uint16_t* vh = reinterpret_cast<const uint16_t*>(v);
  uint16_t* oh = reinterpret_cast<uint16_t*>(o);
  auto rows_of = [&](const HostChunk& c) { return (size_t)c.nb * c.nh * (size_t)N; };
  auto row0_of = [&](const HostChunk& c) { return ((size_t)c.b0 * H + c.h0) * (size_t)N; };
  // inputs, chunk by chunk
  for (int i = 0; rc == FATTN_OK && i < nc; ++i) {
    const size_t e0 = row0_of(chunks[i]) * d, ne = rows_of(chunks[i]) * d;
    if (!(ok(cudaMemcpyAsync(qd + e0, qh + e0, ne * 2u, cudaMemcpyHostToDevice, ds->copy_in)) &&
          ok(cudaMemcpyAsync(kd + e0, kh + e0, ne * 2u, cudaMemcpyHostToDevice, ds->copy_in)) &&
          ok(cudaMemcpyAsync(vd + e0, vh + e0, ne * 2u, cudaMemcpyHostToDevice, ds->copy_in)) &&
          ok(cudaEventRecord(ev[i], ds->copy_in))))
      rc = FATTN_ERR_CUDA;
  }
  // compute each chunk once its inputs are in, then copy its outputs out
  for (int i = 0; rc == FATTN_OK && i < nc; ++i) {
    const HostChunk& c = chunks[i];
    const size_t r0 = row0_of(c), nr = rows_of(c);
    if (!ok(cudaStreamWaitEvent(s, ev[i], 0))) {
      rc = FATTN_ERR_CUDA;
      break;
    }
    rc = fwd_common(qd + r0 * d, kd + r0 * d, vd + r0 * d, od + r0 * d, lsed + r0, c.nb, c.nh, N, d, scale, causal,
                    key_len ? kld + c.b0 : nullptr, 0, stream, false);
    if (rc != FATTN_OK) break;
    if (!(ok(cudaEventRecord(ev[nc + i], s)) && ok(cudaStreamWaitEvent(ds->copy_out, ev[nc + i], 0)) &&
          ok(cudaMemcpyAsync(oh + r0 * d, od + r0 * d, nr * d * 2u, cudaMemcpyDeviceToHost, ds->copy_out)) &&
          ok(cudaMemcpyAsync(lse + r0, lsed + r0, nr * 4u, cudaMemcpyDeviceToHost, ds->copy_out))))
      rc = FATTN_ERR_CUDA;
  }
  // join both copy streams back into the caller's stream, then release the buffers there
  cudaEvent_t ev_in_done = ev_alloc;  // reused: the allocation event has been consumed
  bool joined = ev_in_done && ok(cudaEventRecord(ev_in_done, ds->copy_in)) &&
                ok(cudaStreamWaitEvent(s, ev_in_done, 0)) && ok(cudaEventRecord(ev_done, ds->copy_out)) &&
                ok(cudaStreamWaitEvent(s, ev_done, 0));
  if (!joined) {
    // cannot order the release after the copies: wait for them here instead
    cudaStreamSynchronize(ds->copy_in);
    cudaStreamSynchronize(ds->copy_out);
    if (rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  }
  if (cudaFreeAsync(buf, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  return rc;
}

// ------------------------------------------------------------------------
// fattn_linear_fwd: causal linear attention (the second workload).
extern "C" FATTN_API int fattn_linear_fwd(const float* q, const float* k, const float* v, float* out, int B, int H,
                                          int N, int E, int M, const int32_t* key_len, float eps, void* stream) {
  if (B < 0 || H < 0 || N < 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.0f) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FATTN_OK;
  if (!q || !k || !v || !out) return FATTN_ERR_INVALID_ARG;
  if (E < 4 || E > 128 || E % 4 || M < 4 || M > 128 || M % 4) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFll || N > 0x7FFFFFFF - fattn::LIN_C) return FATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      (key_len && !aligned(key_len, 4)))
    return FATTN_ERR_INVALID_ARG;
  if (!is_device_pointer(q) || !is_device_pointer(k) || !is_device_pointer(v) || !is_device_pointer(out) ||
      (key_len && !is_device_pointer(key_len)))
    return FATTN_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  const int n_chunks = (N + fattn::LIN_C - 1) / fattn::LIN_C;
  const int blocks_per_head = (E * M + E + fattn::LIN_THREADS - 1) / fattn::LIN_THREADS;
  if (BH * n_chunks > 0x7FFFFFFFll || BH * blocks_per_head > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  DeviceState* ds = nullptr;
  int rc = device_state(dev, &ds);
  if (rc != FATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (E <= fattn::LTC_F && M <= fattn::LTC_F) {
    // tensor cores: parts of whole 128-row tiles, about one CTA per SM in all
    const int n_tiles = (N + fattn::LTC_T - 1) / fattn::LTC_T;
    int n_parts = (int)std::max(1ll, std::min<long long>(n_tiles, ds->num_sms / std::max(1ll, BH)));
    const int tpp = (n_tiles + n_parts - 1) / n_parts;
    n_parts = (n_tiles + tpp - 1) / tpp;
    if (BH * n_parts > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
    fattn::LtcParams lp;
    lp.out = out;
    lp.key_len = key_len;
    lp.tot = nullptr;
    lp.err = ds->err;
    lp.B = B;
    lp.H = H;
    lp.N = N;
    lp.E = E;
    lp.M = M;
    lp.n_parts = n_parts;
    lp.tiles_per_part = tpp;
    lp.tot_stride = (int)round_up((size_t)(E * M + E), 4);
    lp.eps = eps;
    lp.wait_limit_ns = wait_limit_ns();
    CUtensorMap mq, mk, mv;
    if (encode_map_f32(&mq, q, (int)BH, N, E) != FATTN_OK || encode_map_f32(&mk, k, (int)BH, N, E) != FATTN_OK ||
        encode_map_f32(&mv, v, (int)BH, N, M) != FATTN_OK)
      return FATTN_ERR_CUDA;
    void* tot = nullptr;
    if (n_parts > 1) {
      // each part's totals, written by the state launch and read by the output launch
      if (cudaMallocFromPoolAsync(&tot, (size_t)BH * n_parts * (size_t)lp.tot_stride * 4u, ds->pool, s) !=
          cudaSuccess) {
        cudaGetLastError();
        return FATTN_ERR_CUDA;
      }
      lp.tot = reinterpret_cast<float*>(tot);
      fattn::fattn_linear_tc_kernel<true>
          <<<(unsigned)(BH * (n_parts - 1)), fattn::LTC_THREADS, fattn::LtcCfg::SMEM_BYTES, s>>>(mq, mk, mv, lp);
    }
    mark_kernel_start(s);
    fattn::fattn_linear_tc_kernel<false>
        <<<(unsigned)(BH * n_parts), fattn::LTC_THREADS, fattn::LtcCfg::SMEM_BYTES, s>>>(mq, mk, mv, lp);
    mark_kernel_stop(s);
    if (cudaGetLastError() != cudaSuccess) rc = FATTN_ERR_CUDA;
    if (tot && cudaFreeAsync(tot, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
    return rc;
  }
  const size_t state_floats = (size_t)BH * n_chunks * (size_t)E * M;
  const size_t ksum_floats = (size_t)BH * n_chunks * (size_t)E;
  void* scratch = nullptr;
  const size_t t_state = round_up(state_floats * 4u, 256), t_ksum = round_up(ksum_floats * 4u, 256);
  if (cudaMallocFromPoolAsync(&scratch, 2 * (t_state + t_ksum), ds->pool, s) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  fattn::LinParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.key_len = key_len;
  uint8_t* sb = reinterpret_cast<uint8_t*>(scratch);
  p.state = reinterpret_cast<float*>(sb);
  p.ksum = reinterpret_cast<float*>(sb + t_state);
  p.pstate = reinterpret_cast<float*>(sb + t_state + t_ksum);
  p.pksum = reinterpret_cast<float*>(sb + 2 * t_state + t_ksum);
  p.B = B;
  p.H = H;
  p.N = N;
  p.E = E;
  p.M = M;
  p.n_chunks = n_chunks;
  p.eps = eps;
  const int state_smem = (E * fattn::LIN_C + fattn::LIN_C * M) * 4;
  const int out_smem = fattn::LinSmem(E, M).total * 4;
  const bool f64 = E == 64 && M == 64;  // the sizes compiled as constants
  if (f64)
    fattn::fattn_linear_state_kernel<64, 64><<<(unsigned)(BH * n_chunks), fattn::LIN_THREADS, state_smem, s>>>(p);
  else
    fattn::fattn_linear_state_kernel<0, 0><<<(unsigned)(BH * n_chunks), fattn::LIN_THREADS, state_smem, s>>>(p);
  fattn::fattn_linear_scan_kernel<<<(unsigned)(BH * blocks_per_head), fattn::LIN_THREADS, 0, s>>>(p,
                                                                                                   blocks_per_head);
  mark_kernel_start(s);
  if (f64)
    fattn::fattn_linear_output_kernel<64, 64><<<(unsigned)(BH * n_chunks), fattn::LIN_THREADS, out_smem, s>>>(p);
  else
    fattn::fattn_linear_output_kernel<0, 0><<<(unsigned)(BH * n_chunks), fattn::LIN_THREADS, out_smem, s>>>(p);
  mark_kernel_stop(s);
  if (cudaGetLastError() != cudaSuccess) rc = FATTN_ERR_CUDA;
  if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  return rc;
}

extern "C" FATTN_API int fattn_set_kernel_events(void* start, void* stop) {
  t_kernel_start = reinterpret_cast<cudaEvent_t>(start);
  t_kernel_stop = reinterpret_cast<cudaEvent_t>(stop);
  return FATTN_OK;
}

extern "C" FATTN_API int fattn_splitkv_plan(int B, int H, int N, int causal, int num_sms, int n_splits) {
  if (B <= 0 || H <= 0 || N <= 0 || num_sms <= 0 || n_splits < 0) return 0;
  return plan_splits(B, H, N, causal ? 1 : 0, num_sms, n_splits);
}

extern "C" FATTN_API long long fattn_unit_schedule(int B, int H, int N, int num_ctas, int* table,
                                                   long long capacity) {
  if (B <= 0 || H <= 0 || N <= 0 || num_ctas <= 0) return 0;
  if ((long long)B * H > 0x7FFFFFFFll) return 0;
  const int nqb = (N + fattn::QT * fattn::BM - 1) / (fattn::QT * fattn::BM);
  const long long units = (long long)B * H * nqb;
  if (units > 0x7FFFFFFFll) return 0;
  const int G = (int)std::min<long long>(units, num_ctas);
  const std::vector<uint16_t> pos = build_round_schedule(B * H, N, nqb, G);
  if (pos.empty()) return 0;
  const long long n = (long long)pos.size();
  if (!table) return n;
  if (capacity < n) return -1;
  for (long long i = 0; i < n; ++i) table[i] = (int)((i / G) * G + pos[(size_t)i]);
  return n;
}

// ------------------------------------------------------------------------
// fattn_bwd: gradients dQ, dK, dV from dO, the forward's O and LSE.
namespace {

template <int D>
int enqueue_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                fattn::BwdParams p, float* rows, cudaStream_t stream) {
  const int BH = p.B * p.H;
  const long long n_rows = (long long)BH * p.N_pad;
  float* nlse2 = rows;
  float* delta = rows + n_rows;
  p.nlse2 = nlse2;
  p.delta = delta;
  const long long prep_threads = n_rows * (D / 8);
  const unsigned prep_blocks = (unsigned)((prep_threads + fattn::PREP_THREADS - 1) / fattn::PREP_THREADS);
  if (p.hd == D)
    fattn::fattn_bwd_prep_kernel<D, true><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, nlse2, delta, p.N, p.N_pad, p.hd,
        n_rows);
  else
    fattn::fattn_bwd_prep_kernel<D, false><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, nlse2, delta, p.N, p.N_pad, p.hd,
        n_rows);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo;
  if (encode_map(&mq, q, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mk, k, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mv, v, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mdo, dout, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK)
    return FATTN_ERR_CUDA;
  const unsigned grid = (unsigned)((long long)BH * p.n_tiles);
  // The two kernels read only the call's inputs and the prep kernel's rows,
  // so each starts as a programmatic dependent of the one before it.
  mark_kernel_start(stream);
  cudaError_t e = launch_dependent(fattn::fattn_bwd_dkdv_kernel<D>, grid, fattn::BWD_THREADS,
                                   fattn::BwdCfg<D>::SMEM_BYTES, stream, mq, mk, mv, mdo, p);
  mark_kernel_stop(stream);
  if (e == cudaSuccess)
    e = launch_dependent(fattn::fattn_bwd_dq_kernel<D>, grid, fattn::BWD_THREADS, fattn::BwdDqCfg<D>::SMEM_BYTES,
                         stream, mq, mk, mv, mdo, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  return FATTN_OK;
}

// Head dims 72..128 in one pass (fattn_bwd_fused.cuh): the prep kernel, the
// zeroing of the fp32 dQ buffer `dq_acc` ([B*H, N_pad, 128]), the fused
// kernel and the conversion of dQ to bf16.
int enqueue_bwd_fused(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                      fattn::BwdParams p, float* rows, float* dq_acc, cudaStream_t stream) {
  constexpr int D = fattn::FB_D;
  const int BH = p.B * p.H;
  const long long n_rows = (long long)BH * p.N_pad;
  p.nlse2 = rows;
  p.delta = rows + n_rows;
  p.dq_acc = dq_acc;
  const long long prep_threads = n_rows * (D / 8);
  const unsigned prep_blocks = (unsigned)((prep_threads + fattn::PREP_THREADS - 1) / fattn::PREP_THREADS);
  if (p.hd == D)
    fattn::fattn_bwd_prep_kernel<D, true><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, rows, rows + n_rows, p.N,
        p.N_pad, p.hd, n_rows);
  else
    fattn::fattn_bwd_prep_kernel<D, false><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, rows, rows + n_rows, p.N,
        p.N_pad, p.hd, n_rows);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaMemsetAsync(dq_acc, 0, (size_t)n_rows * D * sizeof(float), stream) != cudaSuccess) return FATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo;
  if (encode_map(&mq, q, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, fattn::FB_BQ) != FATTN_OK ||
      encode_map(&mk, k, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mv, v, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mdo, dout, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, fattn::FB_BQ) != FATTN_OK)
    return FATTN_ERR_CUDA;
  const unsigned grid = (unsigned)((long long)BH * p.n_tiles);
  mark_kernel_start(stream);
  fattn::fattn_bwd_fused_kernel<<<grid, fattn::FB_THREADS, fattn::FusedCfg::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, p);
  mark_kernel_stop(stream);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  const long long n_vec = (long long)BH * p.N * (p.hd / 8);
  fattn::fattn_bwd_dq_finalize_kernel<<<(unsigned)((n_vec + 255) / 256), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(p.dq), p.N, p.N_pad, p.hd, p.scale, n_vec);
  return cudaGetLastError() == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

bool fused_bwd_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FATTN_BWD_FUSED");
    return e && e[0] == '1';
  }();
  return on;
}

// Head dims 136..256: the prep kernel, then the dV, dK and dQ passes of the
// 256-column backward (fattn_bwd256.cuh).
int enqueue_bwd256(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   fattn::BwdParams p, float* rows, cudaStream_t stream) {
  const int BH = p.B * p.H;
  const long long n_rows = (long long)BH * p.N_pad;
  float* nlse2 = rows;
  float* delta = rows + n_rows;
  p.nlse2 = nlse2;
  p.delta = delta;
  constexpr int D = fattn::D256;
  const long long prep_threads = n_rows * (D / 8);
  const unsigned prep_blocks = (unsigned)((prep_threads + fattn::PREP_THREADS - 1) / fattn::PREP_THREADS);
  if (p.hd == D)
    fattn::fattn_bwd_prep_kernel<D, true><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, nlse2, delta, p.N, p.N_pad, p.hd,
        n_rows);
  else
    fattn::fattn_bwd_prep_kernel<D, false><<<prep_blocks, fattn::PREP_THREADS, 0, stream>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dout), lse, nlse2, delta, p.N, p.N_pad, p.hd,
        n_rows);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo;
  if (encode_map(&mq, q, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mk, k, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mv, v, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK ||
      encode_map(&mdo, dout, BH, p.N, p.hd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != FATTN_OK)
    return FATTN_ERR_CUDA;
  const unsigned grid = (unsigned)((long long)BH * p.n_tiles);
  // The passes read only the call's inputs and the prep kernel's rows, so
  // each starts as a programmatic dependent of the one before it.
  cudaError_t e = launch_dependent(fattn::fattn_bwd256_kernel<fattn::BP_DV>, grid, fattn::BWD_THREADS,
                                   fattn::Bwd256Cfg<fattn::BP_DV>::SMEM_BYTES, stream, mq, mk, mv, mdo, p);
  if (e == cudaSuccess) {
    mark_kernel_start(stream);
    e = launch_dependent(fattn::fattn_bwd256_kernel<fattn::BP_DK>, grid, fattn::BWD_THREADS,
                         fattn::Bwd256Cfg<fattn::BP_DK>::SMEM_BYTES, stream, mq, mk, mv, mdo, p);
    mark_kernel_stop(stream);
  }
  if (e == cudaSuccess)
    e = launch_dependent(fattn::fattn_bwd256_kernel<fattn::BP_DQ>, grid, fattn::BWD_THREADS,
                         fattn::Bwd256Cfg<fattn::BP_DQ>::SMEM_BYTES, stream, mq, mk, mv, mdo, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  return FATTN_OK;
}

}  // namespace

extern "C" FATTN_API int fattn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                   float scale, int causal, const int32_t* key_len, void* stream) {
  // ---- synchronous argument checks: nothing is enqueued on failure
  if (B < 0 || H < 0 || N < 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.0f) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (!head_dim_supported(d)) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFll || N > 0x7FFFFFFF - 512) return FATTN_ERR_INVALID_ARG;
  const void* ptrs16[8] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* ptr : ptrs16)
    if (!aligned(ptr, 16) || !is_device_pointer(ptr)) return FATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !is_device_pointer(lse)) return FATTN_ERR_INVALID_ARG;
  if (key_len && (!aligned(key_len, 4) || !is_device_pointer(key_len))) return FATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  DeviceState* ds = nullptr;
  int rc = device_state(dev, &ds);
  if (rc != FATTN_OK) return rc;

  fattn::BwdParams p;
  p.dq = reinterpret_cast<__nv_bfloat16*>(dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  p.key_len = key_len;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.N = N;
  p.n_tiles = (N + 127) / 128;
  p.N_pad = p.n_tiles * 128;
  p.hd = d;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.causal = causal ? 1 : 0;
  p.wait_limit_ns = wait_limit_ns();
  p.nlse2 = nullptr;
  p.delta = nullptr;
  p.dq_acc = nullptr;
  if ((long long)B * H * p.n_tiles > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* rows = nullptr;
  const size_t row_bytes = 2u * (size_t)B * (size_t)H * (size_t)p.N_pad * sizeof(float);
  if (cudaMallocFromPoolAsync(&rows, row_bytes, ds->pool, s) != cudaSuccess) {
    cudaGetLastError();
    return FATTN_ERR_CUDA;
  }
  float* rf = reinterpret_cast<float*>(rows);
  if (d > 64 && d <= 128 && fused_bwd_enabled()) {
    void* acc = nullptr;
    if (cudaMallocFromPoolAsync(&acc, (size_t)B * H * (size_t)p.N_pad * fattn::FB_D * sizeof(float), ds->pool, s) !=
        cudaSuccess) {
      cudaGetLastError();
      cudaFreeAsync(rows, s);
      return FATTN_ERR_CUDA;
    }
    rc = enqueue_bwd_fused(q, k, v, o, dout, lse, p, rf, reinterpret_cast<float*>(acc), s);
    if (cudaFreeAsync(acc, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  } else {
    rc = d <= 64    ? enqueue_bwd<64>(q, k, v, o, dout, lse, p, rf, s)
         : d <= 128 ? enqueue_bwd<128>(q, k, v, o, dout, lse, p, rf, s)
                    : enqueue_bwd256(q, k, v, o, dout, lse, p, rf, s);
  }
  if (cudaFreeAsync(rows, s) != cudaSuccess && rc == FATTN_OK) rc = FATTN_ERR_CUDA;
  return rc;
}

// ------------------------------------------------------------------------
// fattn_fwd_noalloc: the same forward for callers that cannot allocate
// device memory.  Its scratch (the V copy in the P V operand type, the
// per-tile storage modes and a 16-byte error word) lives in one static
// device array, fixed at build time, instead of a pool allocation.
namespace {

constexpr size_t kNoAllocScratch = FATTN_NOALLOC_SCRATCH_BYTES;  // V copy + tile modes
constexpr size_t kNoAllocErrWord = 256;                          // error word after them

}  // namespace

// Device scratch of the no-allocation entry point.  In host code this name is
// only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratch + kNoAllocErrWord];

namespace {

struct NoAllocState {
  bool ready = false;
  int num_sms = 0;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mu;
NoAllocState g_noalloc[kMaxDevices];

// Per-device set-up with `dev` current: kernel attributes, SM count, the
// tensor-map encoder and the scratch symbol's device address.  Allocates nothing.
int noalloc_state(int dev, NoAllocState** out) {
  if (dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocState& s = g_noalloc[dev];
  if (!s.ready) {
    {
      std::lock_guard<std::mutex> enc_lock(g_mu);
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
          return FATTN_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FATTN_ERR_CUDA;
    int rc = configure_kernel<64>();
    if (rc == FATTN_OK) rc = configure_kernel<128>();
    if (rc == FATTN_OK) rc = configure_d256_kernel<true>();
    if (rc == FATTN_OK) rc = configure_d256_kernel<false>();
    if (rc != FATTN_OK) return rc;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return FATTN_ERR_CUDA;
    }
    s.scratch = reinterpret_cast<uint8_t*>(ptr);
    s.ready = true;
  }
  *out = &s;
  return FATTN_OK;
}

}  // namespace

extern "C" FATTN_API int fattn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                           int H, int N, int d, float scale, int causal, const int32_t* key_len,
                                           void* stream) {
  if (B < 0 || H < 0 || N < 0) return FATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.0f) return FATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FATTN_OK;
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!head_dim_supported(d)) return FATTN_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFll || N > 0x7FFFFFFF - 512) return FATTN_ERR_INVALID_ARG;
  const int n_kv_tiles = (N + fattn::BN - 1) / fattn::BN;
  if ((long long)B * H * ((n_kv_tiles + 7) / 8 * 8) > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  // the static scratch bounds the problem size
  if (scratch_bytes(B * H, N, d, n_kv_tiles) > kNoAllocScratch) return FATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (key_len && !aligned(key_len, 4)))
    return FATTN_ERR_INVALID_ARG;
  if (!is_device_pointer(q) || !is_device_pointer(k) || !is_device_pointer(v) || !is_device_pointer(o) ||
      !is_device_pointer(lse) || (key_len && !is_device_pointer(key_len)))
    return FATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  NoAllocState* ns = nullptr;
  int rc = noalloc_state(dev, &ns);
  if (rc != FATTN_OK) return rc;

  fattn::Params p;
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.o_v8 = (aligned(o, 32) && d % 16 == 0) ? 1 : 0;  // rows of O take 32-byte stores
  p.lse = lse;
  p.key_len = key_len;
  p.err = reinterpret_cast<int*>(ns->scratch + kNoAllocScratch);
  p.B = B;
  p.H = H;
  p.N = N;
  p.hd = d;
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.causal = causal ? 1 : 0;
  p.n_qblocks = (N + fattn::QT * fattn::BM - 1) / (fattn::QT * fattn::BM);
  const long long units = (long long)B * H * p.n_qblocks;
  if (units > 0x7FFFFFFFll) return FATTN_ERR_INVALID_ARG;
  p.n_units = (int)units;
  p.sched = nullptr;  // the snake order: nothing to build or upload during a capture
  p.n_splits = 1;  // no split-KV here: its partials would not fit a fixed array
  p.o_part = nullptr;
  p.head_group = 1;
  p.lse_part = nullptr;
  p.n_kv_tiles = n_kv_tiles;
  p.mode_stride = (n_kv_tiles + 7) / 8 * 8;
  p.v_mode = nullptr;
  p.wait_limit_ns = wait_limit_ns();
  const int grid = (int)(units < ns->num_sms ? units : ns->num_sms);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The V copy and the tile modes are fully rewritten by this call.  The error
  // word is zero at load and cleared by fattn_last_error when it reports a
  // time-out, so it is not cleared here: a time-out stays readable until then.
  return d <= 64    ? enqueue<64>(q, k, v, p, ns->scratch, grid, s)
         : d <= 128 ? enqueue<128>(q, k, v, p, ns->scratch, grid, s)
                    : enqueue_d256(q, k, v, p, ns->scratch, s);
}

// ------------------------------------------------------------------------
// fattn_last_error: the error words of both kinds of entry point on the
// current device -- the pool-backed calls' word and the no-alloc array's --
// read only where that kind has been set up, so it allocates nothing.
extern "C" FATTN_API int fattn_last_error(void* stream, int* detail) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FATTN_ERR_CUDA;
  int* words[2] = {nullptr, nullptr};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[dev].ready) words[0] = g_dev[dev].err;
  }
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc[dev].ready) words[1] = reinterpret_cast<int*>(g_noalloc[dev].scratch + kNoAllocScratch);
  }
  int first[4] = {0, 0, 0, 0};
  for (int* word : words) {
    if (!word) continue;
    int h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, word, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return FATTN_ERR_CUDA;
    if (h[0] == 0) continue;
    if (cudaMemset(word, 0, sizeof h) != cudaSuccess) return FATTN_ERR_CUDA;
    if (first[0] == 0)
      for (int i = 0; i < 4; ++i) first[i] = h[i];
  }
  if (detail)
    for (int i = 0; i < 4; ++i) detail[i] = first[i];
  return first[0] != 0 ? FATTN_ERR_TIMEOUT : FATTN_OK;
}
