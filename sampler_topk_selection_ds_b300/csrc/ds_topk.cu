// ds_topk.cu — host side of libds_topk.so: argument validation, launch planning
// and kernel launches behind the C ABI declared in include/ds_topk.h.
//
// The call surface restates deep_select.topk(x, topk, sorted_index, indices_type)
// and its return_value option (deepseek.csdn.net, "DeepSeek 一次开源三个仓库",
// section 三; deepseek-v4-pro.uk (zh-tw), section "DeepSelect：快速且刻意狹義的
// TopK") as one C function over raw device pointers. The pages say the fastest
// algorithm depends on dtype, batch, row length and k (github-research.aiutil.com,
// "deepseek-ai/DeepSelect", section 关键技术亮点); the plan below picks how many
// CTAs share one row from those sizes and the SM count.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "ds_topk.h"
#include "topk_kernel.cuh"
#include "warp_rows_kernel.cuh"
#include "value_order_kernel.cuh"
#include "sampler_kernel.cuh"

namespace {

using ds_topk_dev::kGranuleCap;
using ds_topk_dev::kRadix;
using ds_topk_dev::kThreads;
using ds_topk_dev::Params;

constexpr int kMaxDevices = 64;
constexpr int kMaxCluster = 16;
// Rows at most this long (bytes) are never split: one CTA streams them.
constexpr int64_t kSplitMinRowBytes = 64 * 1024;
// A CTA of a split row gets at least this many bytes of it.
constexpr int64_t kMinSliceBytes = 16 * 1024;
// Dynamic shared memory one CTA may use (B300: 227 KB), shared memory of an SM
// and the part of it the runtime reserves per resident CTA.
constexpr int64_t kSmemLimit = 227 * 1024;
constexpr int64_t kSmemPerSm = 228 * 1024;
constexpr int64_t kSmemPerCtaReserved = 1024;
// Most vectors per thread held in the next-row prefetch buffer.
constexpr int64_t kMaxStageVecs = 16;
// The one-warp-per-row path is taken from this many rows per SM on: a warp needs
// about as long for one row as a CTA needs for several, so the warps of every SM
// must have rows to share. Measured crossover: about 32 rows per SM for rows of
// 32K bf16 elements; shorter rows cross over sooner.
int64_t wr_min_rows_per_sm(int64_t len) {
  int64_t r = len / 1024;
  return r < 4 ? 4 : (r > 32 ? 32 : r);
}

struct Plan {
  ds_topk_plan_t pub;
  Params prm;
  ds_topk_dev::WrParams wprm;
  bool warp_rows;
  int es;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int validate_sizes(int dtype, int64_t batch, int64_t len, int64_t row_stride, int k) {
  if (dtype != DS_TOPK_BF16 && dtype != DS_TOPK_FP32) return DS_TOPK_EINVAL;
  if (batch < 0 || len < 1 || len > INT32_MAX || row_stride < len) return DS_TOPK_EINVAL;
  if (k < 1 || k > DS_TOPK_MAX_K || static_cast<int64_t>(k) > len) return DS_TOPK_EINVAL;
  const int64_t es = dtype == DS_TOPK_BF16 ? 2 : 4;
  if (row_stride > INT64_MAX / es) return DS_TOPK_EINVAL;
  if (batch > 0 && row_stride * es > INT64_MAX / batch) return DS_TOPK_EINVAL;
  return DS_TOPK_OK;
}

// Pure host planning: how the rows map onto CTAs and clusters. x_aligned: x
// starts on a 16-byte boundary (with a row stride of a multiple of 16 bytes,
// then so does every row).
int make_plan(int dtype, int64_t batch, int64_t len, int64_t row_stride, int k, int sm_count,
              int max_cluster, bool stage, bool x_aligned, Plan* out) {
  const int rc = validate_sizes(dtype, batch, len, row_stride, k);
  if (rc != DS_TOPK_OK) return rc;
  if (sm_count < 1) return DS_TOPK_EINVAL;
  const int es = dtype == DS_TOPK_BF16 ? 2 : 4;
  const int vec = 16 / es;
  const int64_t nvec = ceil_div(len, vec);
  const int64_t row_bytes = len * es;
  out->warp_rows = false;

  // Many short rows: one warp per row (candidate indices fit 16 bits, and a
  // warp's candidate buffer of about 2k entries leaves room for 2+ CTAs per SM).
  // Rows need not start on a 16-byte boundary: the kernel reads the 16-byte
  // blocks that overlap each row and masks the elements outside it.
  if (len <= ds_topk_dev::kWrMaxLen && k <= ds_topk_dev::kWrMaxK &&
      batch >= wr_min_rows_per_sm(len) * static_cast<int64_t>(sm_count)) {
    int64_t cap = 2 * static_cast<int64_t>(k) + 256;
    if (cap > static_cast<int64_t>(k) + 512) cap = static_cast<int64_t>(k) + 512;
    cap = (cap + 31) / 32 * 32;
    const int64_t all = (len + 31) / 32 * 32;  // every element fits
    if (cap > all) cap = all;
    // Most warps per SM first (3 CTAs, then 2), then the deepest streaming ring
    // (3 chunks, then 2) that fits.
    int depth = 0;
    int64_t smem = 0;
    for (int ctas = 3; ctas >= 2 && depth == 0; --ctas) {
      for (int d = ds_topk_dev::kWrMaxDepth; d >= 2; --d) {
        const int64_t b = ds_topk_dev::kWrWarps * ds_topk_dev::wr_warp_bytes(es, cap, d);
        if (ctas * (b + kSmemPerCtaReserved) <= kSmemPerSm) {
          depth = d;
          smem = b;
          break;
        }
      }
    }
    if (depth > 0) {
      out->es = es;
      out->warp_rows = true;
      ds_topk_plan_t& pl = out->pub;
      pl.path = DS_TOPK_PATH_WARP_ROWS;
      pl.cluster_size = 1;
      pl.threads_per_cta = ds_topk_dev::kWrThreads;
      pl.vectors_per_granule = 1;
      // persistent: each warp walks rows with a stride of all warps, so the grid
      // may be capped at the largest launchable size
      pl.grid_ctas = ceil_div(batch, ds_topk_dev::kWrWarps);
      if (pl.grid_ctas > INT32_MAX) pl.grid_ctas = INT32_MAX;
      pl.granules_per_cta = cap;
      pl.smem_bytes = static_cast<int32_t>(smem);
      pl.launches = 1;
      ds_topk_dev::WrParams& w = out->wprm;
      w.x = nullptr;
      w.batch = batch;
      w.row_stride_bytes = row_stride * es;
      w.len = static_cast<int32_t>(len);
      w.cap = static_cast<int32_t>(cap);
      w.depth = depth;
      w.k = k;
      w.return_value = 0;
      w.ordered = 1;
      w.out_values = nullptr;
      w.out_indices = nullptr;
      w.idx64 = 0;
      w.flag = nullptr;
      return DS_TOPK_OK;
    }
  }

  // Rows that do not all start on a 16-byte boundary are read as the 16-byte
  // blocks that overlap them: up to one block more than an aligned row, and no
  // next-row prefetch (its copies need aligned rows).
  const bool rows_aligned = x_aligned && (row_stride * es) % 16 == 0;
  const int64_t nvec_cov = rows_aligned ? nvec : ceil_div(len + vec - 1, vec);
  if (!rows_aligned) stage = false;

  int S = 1;
  if (row_bytes > kSplitMinRowBytes && batch < 2 * static_cast<int64_t>(sm_count)) {
    const int64_t want = ceil_div(2 * static_cast<int64_t>(sm_count), batch > 0 ? batch : 1);
    const int64_t by_size = row_bytes / kMinSliceBytes;
    while (S < max_cluster && S * 2 <= want && S * 2 <= by_size) S *= 2;
    if (S < 2 && by_size >= 2 && want >= 2) S = 2;
    if (S > max_cluster) S = max_cluster;
  }
  const int64_t vec_per_cta = ceil_div(nvec_cov, S);
  const int64_t gv = ceil_div(vec_per_cta, kGranuleCap);
  const int64_t g_cap = ceil_div(vec_per_cta, gv);
  const int64_t g_cap_pad = (g_cap + 7) & ~int64_t(7);
  int64_t g_total = 0;
  for (int r = 0; r < S; ++r) {
    int64_t n = nvec_cov - r * vec_per_cta;
    if (n > vec_per_cta) n = vec_per_cta;
    if (n > 0) g_total += ceil_div(n, gv);
  }
  const int64_t grid = batch * S;
  if (grid > INT32_MAX) return DS_TOPK_EINVAL;
  // Per-warp granule lists (warp w owns granules [w*segm, (w+1)*segm) of the slice).
  const int64_t segm = ((ceil_div(g_cap, ds_topk_dev::kWarps) + 31) / 32) * 32;
  const int64_t list_cap = ds_topk_dev::kWarps * segm;
  // Candidate array of a CTA: about k*(1+small)/S candidates per CTA for data
  // without heavy ties; a CTA that overflows it sends the row to the fallback
  // path (selection over the listed granules, re-read from L2).
  int64_t cand_cap = (ceil_div(4 * static_cast<int64_t>(k), S) + 255) / 256 * 256;
  if (cand_cap < 512) cand_cap = 512;
  // The cluster leader gathers every CTA's candidates of the row.
  // (multiples of 4 entries keep every later shared-memory region 16-byte aligned)
  const int64_t gath_cap = S > 1 ? (2 * static_cast<int64_t>(k) + 256 + 3) / 4 * 4 : 0;
  // Next-row prefetch (only useful when a CTA walks several rows): up to 16
  // vectors per thread, copied with cp.async while the current row is selected.
  // The listed vectors that the streaming pass copies for the candidate pass
  // (threshold-guess rows only, i.e. with the prefetch): ~k*(1+small) per CTA.
  int64_t stage_vecs = 0, lvec_cap = 0;
  if (gv == 1) {
    lvec_cap = (ceil_div(2 * static_cast<int64_t>(k), ds_topk_dev::kWarps * S) + 31) / 32 * 32;
    if (lvec_cap < 64) lvec_cap = 64;
    if (lvec_cap > segm) lvec_cap = segm;
  }
  if (stage && gv == 1) {
    stage_vecs = ceil_div(vec_per_cta, kThreads);
    if (stage_vecs > kMaxStageVecs) stage_vecs = kMaxStageVecs;
  }
  auto size = [&]() {
    return ds_topk_dev::smem_bytes(g_cap_pad, list_cap, cand_cap, gath_cap, stage_vecs, lvec_cap);
  };
  int64_t smem = size();
  while (smem > kSmemLimit && stage_vecs > 0) {
    stage_vecs /= 2;
    smem = size();
  }
  while (smem > kSmemLimit && cand_cap > 512) {
    cand_cap /= 2;
    smem = size();
  }
  if (smem > kSmemLimit) return DS_TOPK_EINVAL;

  out->es = es;
  ds_topk_plan_t& pl = out->pub;
  pl.path = S > 1 ? DS_TOPK_PATH_CLUSTER : DS_TOPK_PATH_ROW;
  pl.cluster_size = S;
  pl.threads_per_cta = kThreads;
  pl.vectors_per_granule = static_cast<int32_t>(gv);
  pl.grid_ctas = grid;
  pl.granules_per_cta = g_cap;
  pl.smem_bytes = static_cast<int32_t>(smem);
  pl.launches = batch > 0 ? 1 : 0;

  Params& p = out->prm;
  p.x = nullptr;
  p.batch = batch;
  p.row_stride_bytes = row_stride * es;
  p.len = len;
  p.nvec = nvec_cov;
  p.vec_per_cta = vec_per_cta;
  p.g_total = g_total;
  p.gv = static_cast<int32_t>(gv);
  p.g_cap_pad = static_cast<int32_t>(g_cap_pad);
  p.list_cap = static_cast<int32_t>(list_cap);
  p.cand_cap = static_cast<int32_t>(cand_cap);
  p.gath_cap = static_cast<int32_t>(gath_cap);
  p.stage_vecs = static_cast<int32_t>(stage_vecs);
  p.lvec_cap = static_cast<int32_t>(lvec_cap);
  p.k = k;
  p.return_value = 0;
  p.out_values = nullptr;
  p.out_indices = nullptr;
  p.idx64 = 0;
  p.flag = nullptr;
  return DS_TOPK_OK;
}

// Per-device facts, filled once under a lock.
struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int max_cluster = 8;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

constexpr int kMaxSmem = static_cast<int>(kSmemLimit);

template <int ES, int S, bool GV1>
cudaError_t prepare_kernel() {
  auto* fn = ds_topk_dev::topk_rows_kernel<ES, S, GV1>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e != cudaSuccess) return e;
  if (S > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int ES, bool GV1>
cudaError_t prepare_variant() {
  cudaError_t e;
  if ((e = prepare_kernel<ES, 1, GV1>()) != cudaSuccess) return e;
  if ((e = prepare_kernel<ES, 2, GV1>()) != cudaSuccess) return e;
  if ((e = prepare_kernel<ES, 4, GV1>()) != cudaSuccess) return e;
  if ((e = prepare_kernel<ES, 8, GV1>()) != cudaSuccess) return e;
  return prepare_kernel<ES, 16, GV1>();
}

template <int ES>
cudaError_t prepare_dtype() {
  cudaError_t e = prepare_variant<ES, true>();
  if (e == cudaSuccess) e = prepare_variant<ES, false>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ds_topk_dev::topk_warp_rows_kernel<ES>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  return e;
}

// Largest cluster size (<= 16) that can be resident with the biggest CTA we launch.
template <int ES, bool GV1>
int probe_cluster16() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kMaxSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ds_topk_dev::topk_rows_kernel<ES, 16, GV1>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DS_TOPK_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      return DS_TOPK_ECUDA;
    if (prepare_dtype<2>() != cudaSuccess || prepare_dtype<4>() != cudaSuccess) return DS_TOPK_ECUDA;
    const bool ok16 = probe_cluster16<2, true>() > 0 && probe_cluster16<4, true>() > 0 &&
                      probe_cluster16<2, false>() > 0 && probe_cluster16<4, false>() > 0;
    d.sm_count = sms;
    d.max_cluster = ok16 ? 16 : 8;
    d.ready = true;
  }
  *out = d;
  return DS_TOPK_OK;
}

// How many clusters of S CTAs (S = 1: plain CTAs) of this kernel can be resident
// at once with `smem` bytes of dynamic shared memory each.
template <int ES, int S, bool GV1>
int resident_clusters(int smem, int sm_count) {
  auto* fn = ds_topk_dev::topk_rows_kernel<ES, S, GV1>;
  int n = 0;
  if (S == 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n * sm_count;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int ES, bool GV1>
int resident_variant(int S, int smem, int sm_count) {
  switch (S) {
    case 1: return resident_clusters<ES, 1, GV1>(smem, sm_count);
    case 2: return resident_clusters<ES, 2, GV1>(smem, sm_count);
    case 4: return resident_clusters<ES, 4, GV1>(smem, sm_count);
    case 8: return resident_clusters<ES, 8, GV1>(smem, sm_count);
    default: return resident_clusters<ES, 16, GV1>(smem, sm_count);
  }
}

struct ResidencyEntry {
  int dev, es, S, gv1, smem, clusters;
};
constexpr int kResidencySlots = 64;
ResidencyEntry g_residency[kResidencySlots];
int g_residency_used = 0;

template <int ES>
int resident_warp_rows(int smem, int sm_count) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ds_topk_dev::topk_warp_rows_kernel<ES>,
                                                    ds_topk_dev::kWrThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n * sm_count;
}

// Cached resident_clusters() per (device, dtype, cluster size, variant, shared memory);
// the warp-rows kernel is cached as variant 2.
int resident_cached(int dev, const Plan& pl, int sm_count) {
  const int es = pl.es, S = pl.pub.cluster_size, smem = pl.pub.smem_bytes;
  const int gv1 = pl.warp_rows ? 2 : (pl.prm.gv == 1 ? 1 : 0);
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_residency_used; ++i) {
    const ResidencyEntry& e = g_residency[i];
    if (e.dev == dev && e.es == es && e.S == S && e.gv1 == gv1 && e.smem == smem) return e.clusters;
  }
  int n;
  if (gv1 == 2) n = es == 2 ? resident_warp_rows<2>(smem, sm_count) : resident_warp_rows<4>(smem, sm_count);
  else if (es == 2) n = gv1 ? resident_variant<2, true>(S, smem, sm_count) : resident_variant<2, false>(S, smem, sm_count);
  else n = gv1 ? resident_variant<4, true>(S, smem, sm_count) : resident_variant<4, false>(S, smem, sm_count);
  if (g_residency_used < kResidencySlots) g_residency[g_residency_used++] = {dev, es, S, gv1, smem, n};
  return n;
}

template <int ES, int S, bool GV1>
cudaError_t launch_one(const Plan& pl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.pub.grid_ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.pub.smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  // may start while the previous kernel in the stream finishes (the kernel waits
  // for it with griddepcontrol.wait before touching global memory)
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (S > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = S;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, ds_topk_dev::topk_rows_kernel<ES, S, GV1>, pl.prm);
}

template <int ES, bool GV1>
cudaError_t launch_variant(const Plan& pl, cudaStream_t stream) {
  switch (pl.pub.cluster_size) {
    case 1: return launch_one<ES, 1, GV1>(pl, stream);
    case 2: return launch_one<ES, 2, GV1>(pl, stream);
    case 4: return launch_one<ES, 4, GV1>(pl, stream);
    case 8: return launch_one<ES, 8, GV1>(pl, stream);
    case 16: return launch_one<ES, 16, GV1>(pl, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int ES>
cudaError_t launch_warp_rows(const Plan& pl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.pub.grid_ctas), 1, 1);
  cfg.blockDim = dim3(ds_topk_dev::kWrThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.pub.smem_bytes);
  cfg.stream = stream;
  // Launched without programmatic dependent launch: measured on the decode-shaped
  // call, back-to-back calls ran 1.5 us faster without it (the early-started
  // grid's waiting CTAs cost the previous call more than the launch they hide).
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, ds_topk_dev::topk_warp_rows_kernel<ES>, pl.wprm);
}

template <int ES>
cudaError_t launch_dtype(const Plan& pl, cudaStream_t stream) {
  if (pl.warp_rows) return launch_warp_rows<ES>(pl, stream);
  return pl.prm.gv == 1 ? launch_variant<ES, true>(pl, stream) : launch_variant<ES, false>(pl, stream);
}

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

// The sampler tail's inputs, for a value-order sort that draws the tokens too.
struct SampleTail {
  int32_t* tokens;
  const float* u;
  float inv_temperature;
  float top_p;
};

// Rows per SM from which the value order sorts one row per warp (measured: with
// 4 rows per SM the CTA sort is still as fast, from 8 on the warp sort is faster).
#ifndef DS_TOPK_VO_WARP_ROWS_PER_SM
#define DS_TOPK_VO_WARP_ROWS_PER_SM 8
#endif

template <int E>
cudaError_t launch_vo_warp(cudaLaunchConfig_t cfg, const ds_topk_dev::OrderParams& op, int sm_count) {
  constexpr int warps = ds_topk_dev::kVoWarps;
  const int64_t ctas = (op.batch + warps - 1) / warps;
  const int64_t max_ctas = static_cast<int64_t>(sm_count) * 16;  // rows are walked with a grid stride
  cfg.gridDim = dim3(static_cast<unsigned>(ctas < max_ctas ? ctas : max_ctas), 1, 1);
  cfg.blockDim = dim3(32 * warps, 1, 1);
  cfg.dynamicSmemBytes = 0;
  using namespace ds_topk_dev;
  if (op.idx64)
    return op.return_value ? cudaLaunchKernelEx(&cfg, topk_value_order_warp_kernel<E, true, true>, op)
                           : cudaLaunchKernelEx(&cfg, topk_value_order_warp_kernel<E, true, false>, op);
  return op.return_value ? cudaLaunchKernelEx(&cfg, topk_value_order_warp_kernel<E, false, true>, op)
                         : cudaLaunchKernelEx(&cfg, topk_value_order_warp_kernel<E, false, false>, op);
}

// sorted_index == DS_TOPK_SORT_VALUE: a second kernel on the same stream sorts
// each row's k outputs by value: for many bf16 rows of at most 65536 elements
// and k <= 1024 one warp per row with the sort words in registers, otherwise one
// CTA per row with a bitonic sort in shared memory. Either waits for the
// selection kernel's outputs (griddepcontrol.wait) before reading them; the warp
// sort may start early through programmatic dependent launch.
template <int ES>
cudaError_t launch_value_order(const char* x, int64_t batch, int64_t len, int64_t row_stride_bytes, int k,
                               int return_value, void* out_values, void* out_indices, int idx64,
                               int sm_count, const SampleTail* tail, bool* drawn, cudaStream_t stream) {
  ds_topk_dev::OrderParams op;
  op.x = x;
  op.batch = batch;
  op.row_stride_bytes = row_stride_bytes;
  op.len = len;
  op.k = k;
  int n2 = 64;  // one 64-word block per warp at least
  while (n2 < k) n2 <<= 1;
  op.n2 = n2;
  op.return_value = return_value;
  op.out_values = return_value ? out_values : nullptr;
  op.out_indices = out_indices;
  op.idx64 = idx64;
  op.tokens = nullptr;
  op.u = nullptr;
  op.inv_temperature = 1.f;
  op.top_p = 1.f;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ES == 2 && len <= ds_topk_dev::kVoMaxLen && k <= ds_topk_dev::kVoMaxK &&
      batch >= static_cast<int64_t>(sm_count) * DS_TOPK_VO_WARP_ROWS_PER_SM) {
    // (with programmatic dependent launch: 3 us faster on the decode-shaped call)
    // one warp per row, 32-bit sort words in registers; with fewer rows one CTA
    // per row finishes sooner, its warps sharing each row's sort
    int n32 = 32;
    while (n32 < k) n32 <<= 1;
    switch (n32 / 32) {
      case 1: return launch_vo_warp<1>(cfg, op, sm_count);
      case 2: return launch_vo_warp<2>(cfg, op, sm_count);
      case 4: return launch_vo_warp<4>(cfg, op, sm_count);
      case 8: return launch_vo_warp<8>(cfg, op, sm_count);
      case 16: return launch_vo_warp<16>(cfg, op, sm_count);
      default: return launch_vo_warp<32>(cfg, op, sm_count);
    }
  }
  // The CTA sort is launched plainly: after the cluster selection of the sampler
  // call it measured 4 us faster without programmatic dependent launch. It also
  // draws the sampler tail's tokens when asked to, saving the draw's launch.
  cfg.numAttrs = 0;
  if (tail) {
    op.tokens = tail->tokens;
    op.u = tail->u;
    op.inv_temperature = tail->inv_temperature;
    op.top_p = tail->top_p;
    *drawn = true;
  }
  const int threads = n2 / 2 < 1024 ? n2 / 2 : 1024;  // n2 >= 64: at least one warp
  const int64_t max_grid = static_cast<int64_t>(sm_count) * 16;
  cfg.gridDim = dim3(static_cast<unsigned>(batch < max_grid ? batch : max_grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(n2) * 8;  // <= 32 KB
  return cudaLaunchKernelEx(&cfg, ds_topk_dev::topk_value_order_kernel<ES>, op);
}

// The optional value-order pass after a selection launch; DS_TOPK_OK or DS_TOPK_ECUDA.
int finish_order(int es, int sorted_index, const void* x, int64_t batch, int64_t len, int64_t row_stride,
                 int k, int return_value, void* out_values, void* out_indices, int idx64, int sm_count,
                 const SampleTail* tail, bool* drawn, cudaStream_t stream) {
  if (sorted_index != DS_TOPK_SORT_VALUE) return DS_TOPK_OK;
  const char* xb = static_cast<const char*>(x);
  const cudaError_t e =
      es == 2 ? launch_value_order<2>(xb, batch, len, row_stride * 2, k, return_value, out_values, out_indices,
                                      idx64, sm_count, tail, drawn, stream)
              : launch_value_order<4>(xb, batch, len, row_stride * 4, k, return_value, out_values, out_indices,
                                      idx64, sm_count, tail, drawn, stream);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) {
    cudaGetLastError();
    return DS_TOPK_ECUDA;
  }
  return DS_TOPK_OK;
}

// The TopK call; with a sampler tail (value order only), *drawn tells whether
// the value-order sort drew the tokens too.
int topk_impl(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride, int k,
              int sorted_index, int return_value, int index_type, void* out_values, void* out_indices,
              int32_t* nan_flag, const SampleTail* tail, bool* drawn, cudaStream_t stream) {
  int rc = validate_sizes(dtype, batch, len, row_stride, k);
  if (rc != DS_TOPK_OK) return rc;
  if (sorted_index < DS_TOPK_SORT_NONE || sorted_index > DS_TOPK_SORT_VALUE ||
      (return_value != 0 && return_value != 1) ||
      (index_type != DS_TOPK_INDEX_INT32 && index_type != DS_TOPK_INDEX_INT64))
    return DS_TOPK_EINVAL;
  if (batch == 0) return DS_TOPK_OK;
  if (!x || !out_indices || !nan_flag || (return_value && !out_values)) return DS_TOPK_EINVAL;
  const int es = dtype == DS_TOPK_BF16 ? 2 : 4;
  const int idx64 = index_type == DS_TOPK_INDEX_INT64 ? 1 : 0;
  if (misaligned(x, es) || misaligned(out_indices, idx64 ? 8 : 4) || misaligned(nan_flag, 4) ||
      (return_value && misaligned(out_values, es)))
    return DS_TOPK_EALIGN;
  const bool x_aligned = !misaligned(x, 16);

  DeviceInfo dev;
  rc = device_info(&dev);
  if (rc != DS_TOPK_OK) return rc;
  Plan pl;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  // With the next-row prefetch, if more rows than co-resident clusters (so that a
  // persistent cluster walks several rows); otherwise without it.
  rc = make_plan(dtype, batch, len, row_stride, k, dev.sm_count, dev.max_cluster, false, x_aligned, &pl);
  if (rc != DS_TOPK_OK) return rc;
  if (pl.warp_rows) {
    pl.wprm.x = static_cast<const char*>(x);
    pl.wprm.return_value = return_value;
    pl.wprm.ordered = sorted_index == DS_TOPK_SORT_INDEX ? 1 : 0;
    pl.wprm.out_values = return_value ? out_values : nullptr;
    pl.wprm.out_indices = out_indices;
    pl.wprm.idx64 = idx64;
    pl.wprm.flag = nan_flag;
    const int resident_ctas = resident_cached(dev_id, pl, dev.sm_count);
    if (resident_ctas > 0 && pl.pub.grid_ctas > resident_ctas) pl.pub.grid_ctas = resident_ctas;
    const cudaError_t e = es == 2 ? launch_dtype<2>(pl, stream) : launch_dtype<4>(pl, stream);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) {
      cudaGetLastError();
      return DS_TOPK_ECUDA;
    }
    return finish_order(es, sorted_index, x, batch, len, row_stride, k, return_value, out_values, out_indices,
                        idx64, dev.sm_count, tail, drawn, stream);
  }
  int resident = resident_cached(dev_id, pl, dev.sm_count);
  if (resident > 0 && batch > resident) {
    Plan ps;
    if (make_plan(dtype, batch, len, row_stride, k, dev.sm_count, dev.max_cluster, true, x_aligned, &ps) ==
            DS_TOPK_OK &&
        ps.prm.stage_vecs > 0) {
      const int rs = resident_cached(dev_id, ps, dev.sm_count);
      if (rs > 0 && batch > rs) {
        pl = ps;
        resident = rs;
      }
    }
  }
  pl.prm.x = static_cast<const char*>(x);
  pl.prm.return_value = return_value;
  pl.prm.out_values = return_value ? out_values : nullptr;
  pl.prm.out_indices = out_indices;
  pl.prm.idx64 = idx64;
  pl.prm.flag = nan_flag;
  // Persistent launch: no more clusters than can be resident at once; each one
  // walks the rows with a stride (and reuses its threshold from row to row).
  if (resident > 0 && batch > resident) pl.pub.grid_ctas = static_cast<int64_t>(resident) * pl.pub.cluster_size;

  const cudaError_t e = es == 2 ? launch_dtype<2>(pl, stream) : launch_dtype<4>(pl, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DS_TOPK_ECUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return DS_TOPK_ECUDA;
  return finish_order(es, sorted_index, x, batch, len, row_stride, k, return_value, out_values, out_indices,
                      idx64, dev.sm_count, tail, drawn, stream);
}

}  // namespace

extern "C" int ds_topk_ex(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
                          int k, int sorted_index, int return_value, int index_type, void* out_values,
                          void* out_indices, int32_t* nan_flag, cudaStream_t stream) {
  return topk_impl(x, dtype, batch, len, row_stride, k, sorted_index, return_value, index_type, out_values,
                   out_indices, nan_flag, nullptr, nullptr, stream);
}

extern "C" int ds_topk(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride, int k,
                       int sorted_index, int return_value, void* out_values, int32_t* out_indices,
                       int32_t* nan_flag, cudaStream_t stream) {
  return ds_topk_ex(x, dtype, batch, len, row_stride, k, sorted_index, return_value, DS_TOPK_INDEX_INT32,
                    out_values, out_indices, nan_flag, stream);
}

extern "C" int ds_topk_sample(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
                              int k, float temperature, float top_p, const float* u, void* out_values,
                              int32_t* out_indices, int32_t* out_tokens, int32_t* nan_flag,
                              cudaStream_t stream) {
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !(top_p > 0.f) || !(top_p <= 1.f))
    return DS_TOPK_EINVAL;
  int rc = validate_sizes(dtype, batch, len, row_stride, k);
  if (rc != DS_TOPK_OK) return rc;
  if (batch == 0) return DS_TOPK_OK;
  if (!u || !out_tokens || !out_values) return DS_TOPK_EINVAL;
  if (misaligned(u, 4) || misaligned(out_tokens, 4)) return DS_TOPK_EALIGN;
  // the k survivors in value order, with their values (and the draw, when the
  // value order is one CTA per row)
  const SampleTail tail{out_tokens, u, 1.0f / temperature, top_p};
  bool drawn = false;
  rc = topk_impl(x, dtype, batch, len, row_stride, k, DS_TOPK_SORT_VALUE, 1, DS_TOPK_INDEX_INT32, out_values,
                 out_indices, nan_flag, &tail, &drawn, stream);
  if (rc != DS_TOPK_OK || drawn) return rc;
  DeviceInfo dev;
  rc = device_info(&dev);
  if (rc != DS_TOPK_OK) return rc;
  ds_topk_dev::SampleParams sp;
  sp.batch = batch;
  sp.k = k;
  sp.inv_temperature = 1.0f / temperature;
  sp.top_p = top_p;
  sp.u = u;
  sp.values = out_values;
  sp.indices = out_indices;
  sp.tokens = out_tokens;
  const int64_t max_grid = static_cast<int64_t>(dev.sm_count) * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(batch < max_grid ? batch : max_grid), 1, 1);
  cfg.blockDim = dim3(ds_topk_dev::kSampleThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.numAttrs = 0;  // plain launch: measured faster than a programmatic dependent one
  const cudaError_t e = dtype == DS_TOPK_BF16 ? cudaLaunchKernelEx(&cfg, ds_topk_dev::topk_sample_kernel<2>, sp)
                                              : cudaLaunchKernelEx(&cfg, ds_topk_dev::topk_sample_kernel<4>, sp);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) {
    cudaGetLastError();
    return DS_TOPK_ECUDA;
  }
  return DS_TOPK_OK;
}

extern "C" int ds_topk_plan(int dtype, int64_t batch, int64_t len, int64_t row_stride, int k,
                            int sm_count, ds_topk_plan_t* plan) {
  if (!plan) return DS_TOPK_EINVAL;
  Plan pl;
  const int rc = make_plan(dtype, batch, len, row_stride, k, sm_count, kMaxCluster, false, true, &pl);
  if (rc == DS_TOPK_OK) *plan = pl.pub;
  return rc;
}

extern "C" const char* ds_topk_status_string(int status) {
  switch (status) {
    case DS_TOPK_OK: return "ok";
    case DS_TOPK_EINVAL: return "invalid argument";
    case DS_TOPK_EALIGN: return "misaligned pointer";
    case DS_TOPK_ECUDA: return "CUDA runtime error";
    case DS_TOPK_ETIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" int ds_topk_version(void) { return 100; }
