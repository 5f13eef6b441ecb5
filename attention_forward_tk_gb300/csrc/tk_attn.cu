// tk_attn.cu -- host side of the attention forward library: argument checks,
// TMA tensor-map encoding, persistent-grid sizing and the C ABI declared in
// include/tk_attn.h.  The device work is in tk_attn_fwd.cuh (attention),
// tk_attn_combine.cuh (key-range merge) and tk_gemm.cuh (bf16 GEMM).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <array>
#include <atomic>
#include <memory>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "tk_attn.h"
#include "tk_attn_combine.cuh"
#include "tk_attn_bwd.cuh"
#include "tk_attn_fwd.cuh"
#include "tk_based.cuh"
#include "tk_based_linear.cuh"
#include "tk_gemm.cuh"

namespace tkattn {
namespace {

// Device error word: kernels record a bounded wait that ran out here.
__device__ int g_dev_error;

// Scratch of the no-allocation split-over-keys entry point: the per-range
// partial O (fp32) and LSE.  Every device that loads the library holds it
// until the process exits.  Host code must not take its name for a device
// address: the address comes from cudaGetSymbolAddress at per-device set-up.
constexpr size_t kStaticScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  std::once_flag once;
  int status = TK_ATTN_ERR_ARCH;
  int num_sms = 0;
  int *err_word = nullptr;  // address of g_dev_error on this device
  void *static_scratch = nullptr;  // address of g_splitkv_scratch on this device
  int gemm_pairs = 0;  // CTA pairs of tk_gemm_kernel that fit on the device at once
  // tk_based_linear_kernel's register split (setmaxnreg) assumes 72
  // registers a thread at launch; a build that gives it another count
  // disables that entry point alone
  bool based_linear_ok = false;
};

DeviceState g_dev[kMaxDevices];
std::atomic<int> g_test_drop_load{0};
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

template <int D, bool kCausal, bool kSplit = false, bool kHalf = false>
int configure_kernel() {
  auto kern = tk_attn_fwd_kernel<D, kCausal, kSplit, kHalf>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FwdCfg<D>::kSmemAlloc) != cudaSuccess)
    return TK_ATTN_ERR_LAUNCH;
  // The register split between warpgroups (setmaxnreg) assumes the kernel is
  // launched with exactly 128 registers per thread; refuse anything else.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return TK_ATTN_ERR_LAUNCH;
  if (fa.numRegs != 128) return TK_ATTN_ERR_LAUNCH;
  return TK_ATTN_OK;
}

template <int D, bool kCausal>
int configure_bwd() {
  if (cudaFuncSetAttribute(tk_attn_bwd_dkdv_kernel<D, kCausal>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<D>::kSmemAlloc) != cudaSuccess ||
      cudaFuncSetAttribute(tk_attn_bwd_dq_kernel<D, kCausal>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           BwdCfg<D>::kDqSmemAlloc) != cudaSuccess)
    return TK_ATTN_ERR_LAUNCH;
  return TK_ATTN_OK;
}

// Per-device set-up, once, with that device current.
void init_device(int dev, DeviceState &ds) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    ds.status = TK_ATTN_ERR_ARCH;
    return;
  }
  if (major != 10 || minor != 3) {  // the kernels are built for sm_103a only
    ds.status = TK_ATTN_ERR_ARCH;
    return;
  }
  int st = configure_kernel<64, false>();
  if (!st) st = configure_kernel<64, true>();
  if (!st) st = configure_kernel<128, false>();
  if (!st) st = configure_kernel<128, true>();
  if (!st) st = configure_kernel<64, false, true>();
  if (!st) st = configure_kernel<128, false, true>();
  if (!st) st = configure_kernel<64, true, true>();
  if (!st) st = configure_kernel<128, true, true>();
  // launches of at most 128 queries
  if (!st) st = configure_kernel<64, false, false, true>();
  if (!st) st = configure_kernel<64, true, false, true>();
  if (!st) st = configure_kernel<128, false, false, true>();
  if (!st) st = configure_kernel<128, true, false, true>();
  if (!st) st = configure_kernel<64, false, true, true>();
  if (!st) st = configure_kernel<64, true, true, true>();
  if (!st) st = configure_kernel<128, false, true, true>();
  if (!st) st = configure_kernel<128, true, true, true>();
  if (!st && (cudaFuncSetAttribute(tk_based_fwd_kernel<false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   BasedCfg::kSmemAlloc) != cudaSuccess ||
              cudaFuncSetAttribute(tk_based_fwd_kernel<true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   BasedCfg::kSmemAlloc) != cudaSuccess ||
              cudaFuncSetAttribute(tk_based_linear_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   BasedLinCfg::kSmemAlloc) != cudaSuccess))
    st = TK_ATTN_ERR_LAUNCH;
  if (!st) {
    cudaFuncAttributes fa;
    ds.based_linear_ok =
        cudaFuncGetAttributes(&fa, tk_based_linear_kernel) == cudaSuccess && fa.numRegs == 72;
  }
  if (!st) st = configure_bwd<64, false>();
  if (!st) st = configure_bwd<64, true>();
  if (!st) st = configure_bwd<128, false>();
  if (!st) st = configure_bwd<128, true>();
  if (!st && cudaFuncSetAttribute(tk_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  GemmCfg::kSmemAlloc) != cudaSuccess)
    st = TK_ATTN_ERR_LAUNCH;
  if (!st) {
    // Pairs live on the two SMs of a TPC; ask how many fit at once rather
    // than assume every SM has a partner.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ds.num_sms, 1, 1);
    cfg.blockDim = dim3(GemmCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = GemmCfg::kSmemAlloc;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tk_gemm_kernel, &cfg) != cudaSuccess ||
        clusters <= 0) {
      cudaGetLastError();
      clusters = ds.num_sms / 2;
    }
    ds.gemm_pairs = clusters;
  }
  if (!st && cudaGetSymbolAddress(reinterpret_cast<void **>(&ds.err_word), g_dev_error) !=
                 cudaSuccess)
    st = TK_ATTN_ERR_LAUNCH;
  if (!st && cudaMemset(ds.err_word, 0, sizeof(int)) != cudaSuccess) st = TK_ATTN_ERR_LAUNCH;
  if (!st && cudaGetSymbolAddress(&ds.static_scratch, g_splitkv_scratch) != cudaSuccess)
    st = TK_ATTN_ERR_LAUNCH;
  if (!st && cudaDeviceSynchronize() != cudaSuccess) st = TK_ATTN_ERR_LAUNCH;
  ds.status = st;
}

DeviceState *current_device(int *status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = TK_ATTN_ERR_ARCH;
    return nullptr;
  }
  DeviceState &ds = g_dev[dev];
  std::call_once(ds.once, init_device, dev, std::ref(ds));
  *status = ds.status;
  return ds.status == TK_ATTN_OK ? &ds : nullptr;
}

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// [BH, N, D] bf16 viewed as a 3-D tensor (d fastest); boxes of 64 columns x
// 128 rows x 1 slice with the 128-byte swizzle the MMA descriptors expect.
// Rows past N read as zero, which is what ragged tiles need.
bool make_map(CUtensorMap *map, const void *ptr, int BH, int N, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, K] bf16 row-major as a 2-D tensor (k fastest); boxes of 64 columns
// x box_rows rows, 128-byte swizzle.  Rows past `rows` and columns past K
// read as zero, so ragged tiles add nothing to the sums.
bool make_map_2d(CUtensorMap *map, const void *ptr, int rows, int K, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, N, 16] bf16 feature rows (32 bytes each) as a 3-D tensor map: boxes of
// 16 columns x 128 rows x 1 slice with the 32-byte swizzle; rows past N read
// as zero.
bool make_map_feat(CUtensorMap *map, const void *ptr, int BH, int N) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {16, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {32, (cuuint64_t)N * 32};
  cuuint32_t box[3] = {16, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
  return a < b + nb && b < a + na;
}

// Causal unit lists (see SchedTable): every unit, in the unit order, goes to
// the CTA with the fewest K/V steps so far (ties: lowest index), costing
// n0 + n1 + 1 steps (both Q tiles' steps plus one for the unit's start-up).
void build_sched(const FwdParams &p, int grid, SchedTable *tab) {
  tab->n = 0;
  if (p.num_units > kSchedCap || grid > kSchedMaxGrid) return;  // stride order
  typedef std::pair<long long, int> Load;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int b = 0; b < grid; ++b) heap.push(Load(0, b));
  std::vector<int> owner(p.num_units), count(grid, 0);
  for (int u = 0; u < p.num_units; ++u) {
    int bh, mb;
    unit_coords(p, true, u, bh, mb);
    const Load top = heap.top();
    heap.pop();
    owner[u] = top.second;
    ++count[top.second];
    heap.push(Load(top.first + kv_tiles(p, true, mb, 0) + kv_tiles(p, true, mb, 1) + 1,
                   top.second));
  }
  tab->off[0] = 0;
  for (int b = 0; b < grid; ++b) tab->off[b + 1] = (uint16_t)(tab->off[b] + count[b]);
  std::vector<int> pos(tab->off, tab->off + grid);
  for (int u = 0; u < p.num_units; ++u) tab->units[pos[owner[u]]++] = (uint16_t)u;
  tab->n = p.num_units;
}

// Unit lists depend only on the shape; the last few are kept.
struct SchedKey {
  int BH, N, Nk, q_off, head_group, grid;
  bool operator==(const SchedKey &o) const {
    return BH == o.BH && N == o.N && Nk == o.Nk && q_off == o.q_off &&
           head_group == o.head_group && grid == o.grid;
  }
};
std::mutex g_sched_mu;
std::vector<std::pair<SchedKey, std::shared_ptr<SchedTable>>> g_sched_cache;

std::shared_ptr<SchedTable> sched_for(const FwdParams &p, int grid) {
  const SchedKey key{p.BH, p.N, p.Nk, p.q_off, p.head_group, grid};
  std::lock_guard<std::mutex> lock(g_sched_mu);
  for (auto &e : g_sched_cache)
    if (e.first == key) return e.second;
  auto tab = std::make_shared<SchedTable>();
  build_sched(p, grid, tab.get());
  if (g_sched_cache.size() >= 8) g_sched_cache.erase(g_sched_cache.begin());
  g_sched_cache.emplace_back(key, tab);
  return tab;
}

template <int D, bool kCausal, bool kSplit, bool kHalf>
cudaError_t launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   const FwdParams &p, int grid, cudaStream_t stream) {
  SchedFor<kCausal> tab;
  std::shared_ptr<SchedTable> keep;
  if constexpr (kCausal && !kSplit) {
    keep = sched_for(p, grid);
    tab = *keep;
  } else if constexpr (kCausal) {
    tab.n = 0;  // causal key ranges run in stride order
  }
  tk_attn_fwd_kernel<D, kCausal, kSplit, kHalf>
      <<<grid, FwdCfg<D>::kThreads, FwdCfg<D>::kSmemAlloc, stream>>>(tq, tk, tv, p, tab);
  return cudaGetLastError();
}

// The kernel variant for a head dim, mask and query count: with at most 128
// queries (p.N <= 128) every unit's second Q tile is empty, and the kHalf
// variant gives tile 0 the decoupled S and P.
template <bool kSplit>
cudaError_t launch_fwd(int D, bool causal, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdParams &p, int grid, cudaStream_t s) {
  const bool half = p.N <= 128;
  if (D == 64) {
    if (causal)
      return half ? launch<64, true, kSplit, true>(tq, tk, tv, p, grid, s)
                  : launch<64, true, kSplit, false>(tq, tk, tv, p, grid, s);
    return half ? launch<64, false, kSplit, true>(tq, tk, tv, p, grid, s)
                : launch<64, false, kSplit, false>(tq, tk, tv, p, grid, s);
  }
  if (causal)
    return half ? launch<128, true, kSplit, true>(tq, tk, tv, p, grid, s)
                : launch<128, true, kSplit, false>(tq, tk, tv, p, grid, s);
  return half ? launch<128, false, kSplit, true>(tq, tk, tv, p, grid, s)
              : launch<128, false, kSplit, false>(tq, tk, tv, p, grid, s);
}

}  // namespace
}  // namespace tkattn

using namespace tkattn;

extern "C" int tk_attn_check_args(const void *q, const void *k, const void *v, const void *o,
                                  const float *lse, int B, int H, int N, int D, float scale,
                                  int causal) {
  (void)causal;
  if (!q || !k || !v || !o || !lse) return TK_ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return TK_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TK_ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TK_ATTN_ERR_UNSUPPORTED;
  const uintptr_t pq = (uintptr_t)q, pk = (uintptr_t)k, pv = (uintptr_t)v, po = (uintptr_t)o,
                  pl = (uintptr_t)lse;
  if ((pq | pk | pv | po | pl) & 15u) return TK_ATTN_ERR_UNSUPPORTED;
  // sizes: B*H slices and the unit count must fit an int; tensor bytes must
  // fit the tensor map's 40-bit stride range.
  const long long BH = (long long)B * H;
  const long long units = BH * ((N + 255LL) / 256);
  if (BH > 0x7fffffffLL || units > 0x7fffffffLL) return TK_ATTN_ERR_UNSUPPORTED;
  const unsigned long long elems = (unsigned long long)BH * (unsigned long long)N * D;
  const unsigned long long tensor_bytes = elems * 2ull;
  if (tensor_bytes >= (1ull << 40)) return TK_ATTN_ERR_UNSUPPORTED;
  const size_t lse_bytes = (size_t)BH * (size_t)N * 4u;
  // outputs must not overlap each other or any input
  if (overlaps(po, tensor_bytes, pl, lse_bytes)) return TK_ATTN_ERR_INVALID_ARG;
  const uintptr_t ins[3] = {pq, pk, pv};
  for (uintptr_t in : ins)
    if (overlaps(po, tensor_bytes, in, tensor_bytes) || overlaps(pl, lse_bytes, in, tensor_bytes))
      return TK_ATTN_ERR_INVALID_ARG;
  return TK_ATTN_OK;
}

extern "C" int tk_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int N, int D, float scale, int causal,
                           tk_attn_stream_t stream) {
  int st = tk_attn_check_args(q, k, v, o, lse, B, H, N, D, scale, causal);
  if (st) return st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, BH, N, D) || !make_map(&tk, k, BH, N, D) || !make_map(&tv, v, BH, N, D))
    return TK_ATTN_ERR_LAUNCH;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.err = ds->err_word;
  p.BH = BH;
  p.N = N;
  p.Nk = N;
  p.q_off = 0;
  p.units_per_bh = 0;
  p.num_splits = 1;
  p.split_tiles = (N + 127) / 128;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.num_mblocks = (N + 255) / 256;
  p.num_units = BH * p.num_mblocks;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.test_drop_load = g_test_drop_load.load(std::memory_order_relaxed);
  // Causal order: sections of heads whose K and V (4*N*D bytes each head)
  // take about 40 MB together, a third of the L2, so concurrent query blocks
  // of a section reuse K/V from L2 instead of re-reading HBM.  Measured on
  // B8 H16 N8192 and B4 H32 N16384: DRAM reads 1.00-1.02x of Q+K+V, against
  // 1.30x with 64 MB sections, at the same speed.
  {
    const long long per_head = 4LL * N * D;
    long long g = (40LL << 20) / (per_head > 0 ? per_head : 1);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    p.head_group = (int)g;
  }
  const int grid = p.num_units < ds->num_sms ? p.num_units : ds->num_sms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_fwd<false>(D, causal != 0, tq, tk, tv, p, grid, s);
  return e == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

// ---------------------------------------------------------------- split over keys

namespace tkattn {
namespace {

// Ranges for a split over keys: `requested` (> 0), or by default the count
// that minimises the launch's makespan in K/V tile steps, when that beats
// one range by at least 10% (5% with at most 128 queries).  Units = (slice,
// query block) pairs x ranges run in ceil(units / SMs) rounds of one unit
// per SM; a unit of T tiles costs about c = 3 tiles more for its start and
// end, and with more than one range it also writes its rows' fp32 partial O
// (a block of r <= 256 rows: r / 128 tiles' worth of bytes), which the
// combine kernel reads back, spread over all SMs.  At most one range per
// 128-key tile, and no empty range: ranges of T tiles, S = ceil(nkv / T).
// (Measured on GB300, B1 H32 Nq256 Nk32768: 4 ranges 0.144 ms, 9 ranges
// 0.148 ms, the count the model chose before it counted the partial
// results.)
void resolve_splits(int requested, long long units_q, int nkv, int num_sms, int Nq, int *S,
                    int *T) {
  auto fit = [nkv](long long s, int *S_, int *T_) {
    if (s > nkv) s = nkv;
    if (s < 1) s = 1;
    *T_ = (int)((nkv + s - 1) / s);
    *S_ = (nkv + *T_ - 1) / *T_;
  };
  if (requested > 0) {
    fit(requested, S, T);
    return;
  }
  // costs in 1/128 of a tile step
  constexpr long long kUnitCost = 3 * 128;
  const long long rows = Nq < 256 ? Nq : 256;  // query rows a unit holds
  long long best = -1, one = -1;
  for (long long s = 1; s <= nkv && s <= 8LL * num_sms; ++s) {
    int s2, t2;
    fit(s, &s2, &t2);
    if (s2 != s) continue;  // the same ranges as a smaller count
    const long long rounds = (units_q * s2 + num_sms - 1) / num_sms;
    const long long partial = s2 > 1 ? rows : 0;
    const long long combine = s2 > 1 ? s2 * units_q * rows / num_sms : 0;
    const long long cost = rounds * (128LL * t2 + kUnitCost + partial) + combine;
    if (s2 == 1) one = cost;
    if (best < 0 || cost < best) {
      best = cost;
      *S = s2;
      *T = t2;
    }
  }
  // The ranges' fp32 partial results make a round trip through memory and a
  // second kernel: split only for a clearly shorter makespan, >= 10%, or
  // >= 5% with at most 128 queries a slice, whose partial results are small
  // (a decode step: 4 ranges instead of 1 took B8 H32 Nq1 Nk16384 from 0.420
  // to 0.400 ms on GB300).
  const long long pct = Nq <= 128 ? 5 : 10;
  if (best < 0 || 100 * best > (100 - pct) * one) fit(1, S, T);
}

size_t split_workspace(long long BH, int Nq, int D, int S) {
  return S > 1 ? (size_t)S * (size_t)BH * (size_t)Nq * (size_t)(D + 1) * sizeof(float) : 0;
}

int check_splitkv_args(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, int B, int H, int Nq, int Nk, int D, float scale) {
  if (!q || !k || !v || !o || !lse) return TK_ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return TK_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TK_ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TK_ATTN_ERR_UNSUPPORTED;
  const uintptr_t pq = (uintptr_t)q, pk = (uintptr_t)k, pv = (uintptr_t)v, po = (uintptr_t)o,
                  pl = (uintptr_t)lse;
  if ((pq | pk | pv | po | pl) & 15u) return TK_ATTN_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  const long long nkv = (Nk + 127LL) / 128;
  // units (slice x query block x range) and their claims must fit an int
  if (BH > 0x7fffffffLL || BH * ((Nq + 255LL) / 256) * nkv > 0x7fffffffLL)
    return TK_ATTN_ERR_UNSUPPORTED;
  const unsigned long long qbytes = (unsigned long long)BH * Nq * D * 2ull;
  const unsigned long long kbytes = (unsigned long long)BH * Nk * D * 2ull;
  if (qbytes >= (1ull << 40) || kbytes >= (1ull << 40)) return TK_ATTN_ERR_UNSUPPORTED;
  const size_t lbytes = (size_t)BH * (size_t)Nq * 4u;
  if (overlaps(po, qbytes, pl, lbytes) || overlaps(po, qbytes, pq, qbytes) ||
      overlaps(po, qbytes, pk, kbytes) || overlaps(po, qbytes, pv, kbytes) ||
      overlaps(pl, lbytes, pq, qbytes) || overlaps(pl, lbytes, pk, kbytes) ||
      overlaps(pl, lbytes, pv, kbytes))
    return TK_ATTN_ERR_INVALID_ARG;
  return TK_ATTN_OK;
}

}  // namespace
}  // namespace tkattn

extern "C" size_t tk_attn_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int D,
                                                  int num_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (D != 64 && D != 128)) return 0;
  int st;
  DeviceState *ds = current_device(&st);
  if (!ds) return 0;
  const long long BH = (long long)B * H;
  int S, T;
  resolve_splits(num_splits, BH * ((Nq + 255LL) / 256), (Nk + 127) / 128, ds->num_sms, Nq, &S,
                 &T);
  return split_workspace(BH, Nq, D, S);
}

namespace tkattn {
namespace {

// Queries and keys of different lengths (both entry points below).
int fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int Nq, int Nk, int D, float scale, int causal, int num_splits, void *workspace,
           size_t workspace_bytes, cudaStream_t s) {
  int st = check_splitkv_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale);
  if (st) return st;
  if (causal && Nq > Nk) return TK_ATTN_ERR_INVALID_ARG;  // the first queries would see no key
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  const int BH = B * H;
  const int nmb = (Nq + 255) / 256, nkv = (Nk + 127) / 128;
  int S, T;
  resolve_splits(num_splits, (long long)BH * nmb, nkv, ds->num_sms, Nq, &S, &T);
  const size_t need = split_workspace(BH, Nq, D, S);
  FwdParams p;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.err = ds->err_word;
  p.BH = BH;
  p.N = Nq;
  p.Nk = Nk;
  p.q_off = causal ? Nk - Nq : 0;
  p.num_mblocks = nmb;
  p.split_tiles = T;
  p.num_splits = S;
  p.units_per_bh = nmb * S;
  if (causal && S > 1) {
    // Causal: block mb's keys stop at its last row's position, so it has
    // causal_ranges(mb) ranges, the last block the most.
    int total = 0;
    for (int mb = 0; mb < nmb; ++mb) total += causal_ranges(p, mb);
    p.units_per_bh = total;
    S = causal_ranges(p, nmb - 1);
    if (S == 1) {  // every block fits one range: the single-pass kernel
      T = nkv;
      p.split_tiles = T;
    }
  }
  if (S > 1) {
    const uintptr_t pw = (uintptr_t)workspace;
    if (!workspace || (pw & 15u) || workspace_bytes < need) return TK_ATTN_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)BH * Nq * D * 2, kbytes = (size_t)BH * Nk * D * 2;
    if (overlaps(pw, need, (uintptr_t)q, qbytes) || overlaps(pw, need, (uintptr_t)k, kbytes) ||
        overlaps(pw, need, (uintptr_t)v, kbytes) || overlaps(pw, need, (uintptr_t)o, qbytes) ||
        overlaps(pw, need, (uintptr_t)lse, (size_t)BH * Nq * 4))
      return TK_ATTN_ERR_INVALID_ARG;
  }
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, BH, Nq, D) || !make_map(&tk, k, BH, Nk, D) ||
      !make_map(&tv, v, BH, Nk, D))
    return TK_ATTN_ERR_LAUNCH;
  // the layout of the partial results keeps the unmasked range count
  const int S_layout = p.num_splits;
  p.o_part = S > 1 ? static_cast<float *>(workspace) : nullptr;
  p.lse_part = S > 1 ? static_cast<float *>(workspace) + (size_t)S_layout * BH * Nq * D : nullptr;
  p.num_units = S > 1 ? BH * p.units_per_bh : BH * nmb;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.test_drop_load = g_test_drop_load.load(std::memory_order_relaxed);
  {
    const long long per_head = 4LL * Nk * D;  // causal sections of ~40 MB of K/V
    long long g = (40LL << 20) / (per_head > 0 ? per_head : 1);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    p.head_group = causal ? (int)g : 1;
  }
  const int grid = p.num_units < ds->num_sms ? p.num_units : ds->num_sms;
  cudaError_t e;
  if (S == 1) {  // one range: the single-pass kernel writes O and LSE directly
    e = launch_fwd<false>(D, causal != 0, tq, tk, tv, p, grid, s);
  } else {
    e = launch_fwd<true>(D, causal != 0, tq, tk, tv, p, grid, s);
    if (e == cudaSuccess) {
      CombineParams cp;
      cp.S = S_layout;
      cp.rows = (long long)BH * Nq;
      cp.Nq = Nq;
      cp.causal = causal ? 1 : 0;
      cp.q_off = p.q_off;
      cp.split_tiles = T;
      cp.nkv = nkv;
      const unsigned int blocks = (unsigned int)((cp.rows + kCombineWarps - 1) / kCombineWarps);
      if (D == 64)
        tk_attn_combine_kernel<64><<<blocks, kCombineWarps * 32, 0, s>>>(p.o_part, p.lse_part,
                                                                         p.o, p.lse, cp);
      else
        tk_attn_combine_kernel<128><<<blocks, kCombineWarps * 32, 0, s>>>(p.o_part, p.lse_part,
                                                                          p.o, p.lse, cp);
      e = cudaGetLastError();
    }
  }
  return e == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

}  // namespace
}  // namespace tkattn

extern "C" int tk_attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int H, int Nq, int Nk, int D, float scale,
                                   int num_splits, void *workspace, size_t workspace_bytes,
                                   tk_attn_stream_t stream) {
  return fwd_qk(q, k, v, o, lse, B, H, Nq, Nk, D, scale, 0, num_splits, workspace,
                workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int tk_attn_fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int Nq, int Nk, int D, float scale, int causal,
                              int num_splits, void *workspace, size_t workspace_bytes,
                              tk_attn_stream_t stream) {
  return fwd_qk(q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, num_splits, workspace,
                workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int tk_attn_fwd_splitkv_static(const void *q, const void *k, const void *v, void *o,
                                          float *lse, int B, int H, int Nq, int Nk, int D,
                                          float scale, int num_splits,
                                          tk_attn_stream_t stream) {
  int st = check_splitkv_args(q, k, v, o, lse, B, H, Nq, Nk, D, scale);
  if (st) return st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  const long long BH = (long long)B * H;
  int S, T;
  resolve_splits(num_splits, BH * ((Nq + 255LL) / 256), (Nk + 127) / 128, ds->num_sms, Nq, &S,
                 &T);
  if (split_workspace(BH, Nq, D, S) > kStaticScratchBytes) return TK_ATTN_ERR_TOO_LARGE;
  return tk_attn_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, D, scale, num_splits,
                             ds->static_scratch, kStaticScratchBytes, stream);
}

// ---------------------------------------------------------------- backward

namespace tkattn {
namespace {

size_t bwd_workspace(long long BH, int N) {
  const long long npad = (N + 127LL) / 128 * 128;
  return (size_t)(2 * BH * npad) * sizeof(float);
}

// Causal backward unit lists (the device's bwd_unit_at): units in the
// order of causal_section, each to the CTA with the fewest tile steps so far
// (ties: lowest index).  Unit u of rank r within its section runs nt - r
// steps in both gradient kernels (dK/dV: key tile j = r against query tiles
// j..nt-1; dQ: query tile nt-1-r against key tiles 0..nt-1-r), plus one
// for its start.  Against the stride order this takes the makespan of B8
// H16 N8192 from 3.3% to 0.2% above the mean load (in that cost model).
void build_bwd_sched(const BwdParams &p, int grid, SchedTable *tab) {
  tab->n = 0;
  if (p.num_units > kSchedCap || grid > kSchedMaxGrid) return;  // stride order
  typedef std::pair<long long, int> Load;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int b = 0; b < grid; ++b) heap.push(Load(0, b));
  std::vector<int> owner(p.num_units), count(grid, 0);
  const int per_section = p.head_group * p.nt;
  for (int u = 0; u < p.num_units; ++u) {
    const int section = u / per_section;
    const int rr = u - section * per_section;
    const int g = std::min(p.head_group, p.BH - section * p.head_group);
    const int r = rr / g;
    const Load top = heap.top();
    heap.pop();
    owner[u] = top.second;
    ++count[top.second];
    heap.push(Load(top.first + (p.nt - r) + 1, top.second));
  }
  tab->off[0] = 0;
  for (int b = 0; b < grid; ++b) tab->off[b + 1] = (uint16_t)(tab->off[b] + count[b]);
  std::vector<int> pos(tab->off, tab->off + grid);
  for (int u = 0; u < p.num_units; ++u) tab->units[pos[owner[u]]++] = (uint16_t)u;
  tab->n = p.num_units;
}

// The lists depend only on the shape; the last few are kept.
std::mutex g_bwd_sched_mu;
std::vector<std::pair<std::array<int, 4>, std::shared_ptr<SchedTable>>> g_bwd_sched_cache;

std::shared_ptr<SchedTable> bwd_sched_for(const BwdParams &p, int grid) {
  const std::array<int, 4> key{p.BH, p.nt, p.head_group, grid};
  std::lock_guard<std::mutex> lock(g_bwd_sched_mu);
  for (auto &e : g_bwd_sched_cache)
    if (e.first == key) return e.second;
  auto tab = std::make_shared<SchedTable>();
  build_bwd_sched(p, grid, tab.get());
  if (g_bwd_sched_cache.size() >= 8) g_bwd_sched_cache.erase(g_bwd_sched_cache.begin());
  g_bwd_sched_cache.emplace_back(key, tab);
  return tab;
}

template <int D, bool kCausal>
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, BwdParams p, const void *o, const void *dout,
                       const float *lse, float *lse2, float *delta, int num_sms,
                       cudaStream_t s) {
  const long long rows = (long long)p.BH * p.Npad;
  tk_attn_bwd_prep_kernel<D><<<(unsigned)((rows + kPrepWarps - 1) / kPrepWarps),
                               kPrepWarps * 32, 0, s>>>(
      static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse,
      lse2, delta, p.N, p.Npad, rows);
  p.num_units = p.BH * p.nt;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  SchedFor<kCausal> tab;
  std::shared_ptr<SchedTable> keep;
  if constexpr (kCausal) {
    keep = bwd_sched_for(p, grid);
    tab = *keep;
  }
  tk_attn_bwd_dkdv_kernel<D, kCausal>
      <<<grid, BwdCfg<D>::kThreads, BwdCfg<D>::kSmemAlloc, s>>>(tq, tk, tv, tdo, p, tab);
  tk_attn_bwd_dq_kernel<D, kCausal>
      <<<grid, BwdCfg<D>::kDqThreads, BwdCfg<D>::kDqSmemAlloc, s>>>(tq, tk, tv, tdo, p, tab);
  return cudaGetLastError();
}

}  // namespace
}  // namespace tkattn

extern "C" size_t tk_attn_bwd_workspace_bytes(int B, int H, int N, int D) {
  if (B <= 0 || H <= 0 || N <= 0 || (D != 64 && D != 128)) return 0;
  return bwd_workspace((long long)B * H, N);
}

extern "C" int tk_attn_bwd_check_args(const void *q, const void *k, const void *v,
                                      const void *o, const float *lse, const void *dout,
                                      const void *dq, const void *dk, const void *dv, int B,
                                      int H, int N, int D, float scale, const void *workspace,
                                      size_t workspace_bytes) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return TK_ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return TK_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TK_ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TK_ATTN_ERR_UNSUPPORTED;
  const uintptr_t ptrs[10] = {(uintptr_t)q,  (uintptr_t)k,  (uintptr_t)v,  (uintptr_t)o,
                              (uintptr_t)lse, (uintptr_t)dout, (uintptr_t)dq, (uintptr_t)dk,
                              (uintptr_t)dv, (uintptr_t)workspace};
  uintptr_t any = 0;
  for (uintptr_t x : ptrs) any |= x;
  if (any & 15u) return TK_ATTN_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL || BH * ((N + 127LL) / 128) > 0x7fffffffLL) return TK_ATTN_ERR_UNSUPPORTED;
  const unsigned long long tb = (unsigned long long)BH * N * D * 2ull;
  if (tb >= (1ull << 40)) return TK_ATTN_ERR_UNSUPPORTED;
  const size_t need = bwd_workspace(BH, N);
  if (workspace_bytes < need) return TK_ATTN_ERR_INVALID_ARG;
  // the outputs and the workspace overlap nothing else
  const size_t lb = (size_t)BH * N * 4;
  const uintptr_t outs[4] = {(uintptr_t)dq, (uintptr_t)dk, (uintptr_t)dv, (uintptr_t)workspace};
  const size_t out_n[4] = {tb, tb, tb, need};
  const uintptr_t ins[6] = {(uintptr_t)q, (uintptr_t)k, (uintptr_t)v, (uintptr_t)o,
                            (uintptr_t)lse, (uintptr_t)dout};
  const size_t in_n[6] = {tb, tb, tb, tb, lb, tb};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_n[a], ins[b], in_n[b])) return TK_ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return TK_ATTN_ERR_INVALID_ARG;
  }
  return TK_ATTN_OK;
}

extern "C" int tk_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dout, void *dq, void *dk, void *dv,
                           int B, int H, int N, int D, float scale, int causal, void *workspace,
                           size_t workspace_bytes, tk_attn_stream_t stream) {
  int st = tk_attn_bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D, scale,
                                  workspace, workspace_bytes);
  if (st) return st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(&tq, q, BH, N, D) || !make_map(&tk, k, BH, N, D) ||
      !make_map(&tv, v, BH, N, D) || !make_map(&tdo, dout, BH, N, D))
    return TK_ATTN_ERR_LAUNCH;
  BwdParams p;
  p.dq = static_cast<__nv_bfloat16 *>(dq);
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.nt = (N + 127) / 128;
  p.Npad = p.nt * 128;
  float *lse2 = static_cast<float *>(workspace);
  float *delta = lse2 + (size_t)BH * p.Npad;
  p.lse2 = lse2;
  p.delta = delta;
  p.err = ds->err_word;
  p.BH = BH;
  p.N = N;
  p.num_units = 0;
  {  // causal sections: the streamed tiles of a slice (Q and dO, or K and V) take 4*N*D bytes
    long long g = (40LL << 20) / (4LL * N * D);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    p.head_group = (int)g;
  }
  p.scale = scale;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (D == 64)
    e = causal ? launch_bwd<64, true>(tq, tk, tv, tdo, p, o, dout, lse, lse2, delta,
                                      ds->num_sms, s)
               : launch_bwd<64, false>(tq, tk, tv, tdo, p, o, dout, lse, lse2, delta,
                                       ds->num_sms, s);
  else
    e = causal ? launch_bwd<128, true>(tq, tk, tv, tdo, p, o, dout, lse, lse2, delta,
                                       ds->num_sms, s)
               : launch_bwd<128, false>(tq, tk, tv, tdo, p, o, dout, lse, lse2, delta,
                                        ds->num_sms, s);
  return e == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

// ---------------------------------------------------------------- Based

extern "C" int tk_based_check_args(const void *q, const void *k, const void *v, const void *y,
                                   const float *z, int B, int H, int N, int Df, int Dv,
                                   float scale) {
  if (!q || !k || !v || !y || !z) return TK_ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return TK_ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return TK_ATTN_ERR_INVALID_ARG;
  if (Df != BasedCfg::kDf || Dv != BasedCfg::kDv) return TK_ATTN_ERR_UNSUPPORTED;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)y | (uintptr_t)z) & 15u)
    return TK_ATTN_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL || BH * ((N + 127LL) / 128) > 0x7fffffffLL) return TK_ATTN_ERR_UNSUPPORTED;
  const unsigned long long fb = (unsigned long long)BH * N * Df * 2ull;
  const unsigned long long vb = (unsigned long long)BH * N * Dv * 2ull;
  if (vb >= (1ull << 40)) return TK_ATTN_ERR_UNSUPPORTED;
  const size_t zb = (size_t)BH * N * 4;
  const uintptr_t py = (uintptr_t)y, pz = (uintptr_t)z;
  if (overlaps(py, vb, pz, zb) || overlaps(py, vb, (uintptr_t)q, fb) ||
      overlaps(py, vb, (uintptr_t)k, fb) || overlaps(py, vb, (uintptr_t)v, vb) ||
      overlaps(pz, zb, (uintptr_t)q, fb) || overlaps(pz, zb, (uintptr_t)k, fb) ||
      overlaps(pz, zb, (uintptr_t)v, vb))
    return TK_ATTN_ERR_INVALID_ARG;
  return TK_ATTN_OK;
}

extern "C" int tk_based_fwd(const void *q, const void *k, const void *v, void *y, float *z,
                            int B, int H, int N, int Df, int Dv, float scale, int causal,
                            tk_attn_stream_t stream) {
  int st = tk_based_check_args(q, k, v, y, z, B, H, N, Df, Dv, scale);
  if (st) return st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!make_map_feat(&tq, q, BH, N) || !make_map_feat(&tk, k, BH, N) ||
      !make_map(&tv, v, BH, N, Dv))
    return TK_ATTN_ERR_LAUNCH;
  BasedParams p;
  p.y = static_cast<__nv_bfloat16 *>(y);
  p.z = z;
  p.err = ds->err_word;
  p.BH = BH;
  p.N = N;
  p.nt = (N + 127) / 128;
  p.num_units = BH * p.nt;
  p.scale = scale;
  {  // causal sections: K and V of a slice take N * (16 + 64) * 2 bytes; ~64 MB per section
    long long g = (64LL << 20) / ((long long)N * (BasedCfg::kDf + BasedCfg::kDv) * 2);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    p.head_group = (int)g;
  }
  const int grid = p.num_units < ds->num_sms ? p.num_units : ds->num_sms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (causal)
    tk_based_fwd_kernel<true><<<grid, BasedCfg::kThreads, BasedCfg::kSmemAlloc, s>>>(tq, tk, tv, p);
  else
    tk_based_fwd_kernel<false><<<grid, BasedCfg::kThreads, BasedCfg::kSmemAlloc, s>>>(tq, tk, tv,
                                                                                     p);
  return cudaGetLastError() == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

extern "C" int tk_based_fwd_linear(const void *q, const void *k, const void *v, void *y, float *z,
                                   int B, int H, int N, int Df, int Dv, float scale,
                                   tk_attn_stream_t stream) {
  int st = tk_based_check_args(q, k, v, y, z, B, H, N, Df, Dv, scale);
  if (st) return st;
  if (!(scale >= 0.f)) return TK_ATTN_ERR_INVALID_ARG;  // the feature maps take sqrt(scale)
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  if (!ds->based_linear_ok) return TK_ATTN_ERR_LAUNCH;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!make_map_feat(&tq, q, BH, N) || !make_map_feat(&tk, k, BH, N) ||
      !make_map(&tv, v, BH, N, Dv))
    return TK_ATTN_ERR_LAUNCH;
  BasedLinParams p;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k = static_cast<const __nv_bfloat16 *>(k);
  p.y = static_cast<__nv_bfloat16 *>(y);
  p.z = z;
  p.err = ds->err_word;
  p.BH = BH;
  p.N = N;
  p.nc = (N + 127) / 128;
  p.scale = scale;
  p.sqrt_scale = std::sqrt(scale);
  // one CTA per slice, its chunks in order
  const int grid = BH < ds->num_sms ? BH : ds->num_sms;
  tk_based_linear_kernel<<<grid, BasedLinCfg::kThreads, BasedLinCfg::kSmemAlloc,
                           reinterpret_cast<cudaStream_t>(stream)>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

// ---------------------------------------------------------------- GEMM

extern "C" int tk_gemm_bf16_check_args(const void *a, const void *b, const void *c, int M,
                                       int N, int K) {
  if (!a || !b || !c) return TK_ATTN_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return TK_ATTN_ERR_INVALID_ARG;
  if (((uintptr_t)a | (uintptr_t)b | (uintptr_t)c) & 15u) return TK_ATTN_ERR_UNSUPPORTED;
  // row strides of A, B (K * 2 bytes) and C (N * 2 bytes) must be 16-byte multiples
  if ((K & 7) || (N & 7)) return TK_ATTN_ERR_UNSUPPORTED;
  const unsigned long long abytes = (unsigned long long)M * K * 2ull;
  const unsigned long long bbytes = (unsigned long long)N * K * 2ull;
  const unsigned long long cbytes = (unsigned long long)M * N * 2ull;
  if (abytes >= (1ull << 40) || bbytes >= (1ull << 40)) return TK_ATTN_ERR_UNSUPPORTED;
  const long long tiles = ((M + (long long)GemmCfg::kBM - 1) / GemmCfg::kBM) *
                          ((N + (long long)GemmCfg::kBN - 1) / GemmCfg::kBN);
  if (tiles > 0x7fffffffLL) return TK_ATTN_ERR_UNSUPPORTED;
  if (overlaps((uintptr_t)c, cbytes, (uintptr_t)a, abytes) ||
      overlaps((uintptr_t)c, cbytes, (uintptr_t)b, bbytes))
    return TK_ATTN_ERR_INVALID_ARG;
  return TK_ATTN_OK;
}

extern "C" int tk_gemm_bf16(const void *a, const void *b, void *c, int M, int N, int K,
                            tk_attn_stream_t stream) {
  int st = tk_gemm_bf16_check_args(a, b, c, M, N, K);
  if (st) return st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0 || N == 0) return TK_ATTN_OK;  // an empty C: nothing to write
  if (K == 0)                               // empty sums: C = 0
    return cudaMemsetAsync(c, 0, (size_t)M * N * 2, s) == cudaSuccess ? TK_ATTN_OK
                                                                     : TK_ATTN_ERR_LAUNCH;
  CUtensorMap ta, tb;
  if (!make_map_2d(&ta, a, M, K, GemmCfg::kHalf) || !make_map_2d(&tb, b, N, K, GemmCfg::kHalf))
    return TK_ATTN_ERR_LAUNCH;
  GemmParams p;
  p.c = static_cast<__nv_bfloat16 *>(c);
  p.err = ds->err_word;
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + GemmCfg::kBM - 1) / GemmCfg::kBM;
  p.tiles_n = (N + GemmCfg::kBN - 1) / GemmCfg::kBN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.k_blocks = (K + GemmCfg::kBK - 1) / GemmCfg::kBK;
  const int pairs = p.num_tiles < ds->gemm_pairs ? p.num_tiles : ds->gemm_pairs;
  tk_gemm_kernel<<<2 * pairs, GemmCfg::kThreads, GemmCfg::kSmemAlloc, s>>>(ta, tb, p);
  return cudaGetLastError() == cudaSuccess ? TK_ATTN_OK : TK_ATTN_ERR_LAUNCH;
}

extern "C" const char *tk_attn_status_string(int status) {
  switch (status) {
    case TK_ATTN_OK: return "ok";
    case TK_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case TK_ATTN_ERR_UNSUPPORTED: return "unsupported head dim, alignment or size";
    case TK_ATTN_ERR_ARCH: return "no compute-capability 10.3 GPU current";
    case TK_ATTN_ERR_LAUNCH: return "CUDA error while preparing or launching the kernel";
    case TK_ATTN_ERR_DEVICE_TIMEOUT: return "a kernel abandoned a barrier wait";
    case TK_ATTN_ERR_TOO_LARGE:
      return "the split needs more than the 64 MiB static scratch of tk_attn_fwd_splitkv_static "
             "(use fewer key ranges, or tk_attn_fwd_splitkv with a workspace)";
    default: return "unknown status";
  }
}

extern "C" int tk_attn_version(void) { return TK_ATTN_VERSION; }

extern "C" int tk_attn_last_device_error(tk_attn_stream_t stream) {
  int st;
  DeviceState *ds = current_device(&st);
  if (!ds) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, ds->err_word, sizeof(int), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return TK_ATTN_ERR_LAUNCH;
  }
  if (word != 0) {
    if (cudaMemsetAsync(ds->err_word, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return TK_ATTN_ERR_LAUNCH;
    return TK_ATTN_ERR_DEVICE_TIMEOUT;
  }
  return TK_ATTN_OK;
}

extern "C" void tk_attn_debug_drop_load(int enable) {
  g_test_drop_load.store(enable ? 1 : 0, std::memory_order_relaxed);
}
