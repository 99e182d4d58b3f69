// topk_kernel.cuh — device code of the batched row-wise TopK (sm_103a).
//
// One row is handled by one CTA, or by the S CTAs of a thread-block cluster that
// each own a contiguous slice of the row. Per row:
//
//  P1  stream the slice once with 16-byte loads; for every granule (gv
//      consecutive 16-byte vectors) keep the top 16 bits of the order key of its
//      maximum in shared memory (M), and test every element for NaN through a
//      NaN-propagating max.
//  A   threshold: t = the k-th largest granule maximum over the whole row (two
//      8-bit radix levels over M). At least k elements are >= t, so t is a lower
//      bound of the row's k-th largest key; elements below t are never touched
//      again. This plays the role of the pages' threshold filter (raise the
//      threshold to the minimum of K survivors), computed from all granules at
//      once instead of raised along a randomised scan.
//  L   list, in index order, the granules whose maximum reaches t.
//  B   exact k-th key K* among the elements >= t: shared-memory histogram
//      levels over the candidate keys (a 256-key window starting at t, then
//      8-bit digits), summed over the cluster through distributed shared memory
//      where the candidates are spread over the cluster's CTAs.
//  C   ordered compaction: every element with key > K*, plus the lowest-index
//      elements with key == K* until k are taken, written in ascending index
//      order (so sorted_index costs nothing).
//
// When some CTA's candidates overflow its buffer (heavy ties, sorted, ramp or
// few-level rows), B and C run over the listed granules instead, re-read from
// L2, after the listed granules are spread evenly over every warp of the
// cluster (a sorted row lists only its top, which one CTA holds).
//
// A row may start at any element offset: it is read as the 16-byte aligned
// blocks that overlap it (its element i is element i + lead of the first
// block). Blocks wholly inside the row take the fast 16-byte path; the elements
// of the two partial blocks that lie outside the row read as -inf, and a block
// past the row is never read.
//
// Sources: deepseek.csdn.net, "DeepSeek 一次开源三个仓库", section 三 (算子层): the
// selection of each row's top K and its threshold/candidate scheme;
// deepseek-v4-pro.uk (zh-tw), "深入 DeepSeek V4.1 全新開放推論工具包", section
// "DeepSelect：快速且刻意狹義的 TopK": bf16 and fp32 paths, k <= 4096, the
// always-on NaN check (a device flag here, never a trap);
// github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点:
// effective memory bandwidth is the metric, so the row is read from HBM once.
//
// Order key: key(v) = 2^(W-1) + |v| for v >= +0 and 2^(W-1) - |v| for v <= -0,
// on the W-bit pattern's magnitude field (W = 16 for bf16, 32 for fp32). It is
// monotone in the value, maps -0.0 and +0.0 to the same key, and keeps +-inf as
// ordinary extremes; the total order of the pages' reading is (key desc, index
// asc). No floating-point arithmetic touches a value: outputs copy input bits.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>
#include <type_traits>

#include "ds_topk.h"

namespace ds_topk_dev {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;            // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kRadix = 256;              // 8-bit digits
constexpr int kGranuleCap = 8192;        // max granules (entries of M) per CTA
constexpr int kMiscWords = 64;           // small shared scalars (see the misc layout below)

struct Params {
  const char* x;
  int64_t batch;         // rows
  int64_t row_stride_bytes;
  int64_t len;           // elements per row
  int64_t nvec;          // 16-byte vectors per row, ceil(len / VEC)
  int64_t vec_per_cta;   // vectors per CTA slice
  int64_t g_total;       // granules per row, summed over the cluster
  int32_t gv;            // vectors per granule
  int32_t g_cap_pad;     // per-CTA granule-maximum array size (multiple of 8)
  int32_t list_cap;      // per-CTA granule list size (kWarps segments)
  int32_t cand_cap;      // per-CTA candidate capacity (kWarps equal regions)
  int32_t gath_cap;      // leader's gathered-candidate capacity (clusters only)
  int32_t stage_vecs;    // vectors per thread prefetched for the next row (0: none)
  int32_t lvec_cap;      // per-warp copies of listed vectors kept by the streaming pass
  int32_t k;
  int32_t return_value;
  void* out_values;
  void* out_indices;     // int32 or int64 (idx64)
  int32_t idx64;
  int32_t* flag;
};

template <int ES>
struct Traits;
template <>
struct Traits<2> {
  static constexpr int kVec = 8;          // bf16 elements per 16 bytes
  static constexpr int kKeyBits = 16;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;  // two bf16 -inf
};
template <>
struct Traits<4> {
  static constexpr int kVec = 4;
  static constexpr int kKeyBits = 32;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;  // fp32 -inf
};

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Block v of a row read as 16-byte aligned blocks (rowp: the row's first block;
// the row's element i is element i + lead of that sequence; nvr blocks overlap
// the row): elements outside the row read as -inf, and a block past the row is
// not read at all. A block holding any row element is read whole (an aligned
// 16-byte block never crosses a page).
template <int ES>
__device__ __forceinline__ uint4 load_blk(const char* rowp, int64_t v, int lead, int64_t len, int64_t nvr) {
  constexpr int VEC = Traits<ES>::kVec;
  constexpr uint32_t NI = Traits<ES>::kNegInfWord;
  if (v >= nvr) return make_uint4(NI, NI, NI, NI);
  uint4 w = ld_nc_v4(rowp + v * 16);
  const int64_t e0 = v * VEC - lead;  // row index of the block's element 0
  if (e0 >= 0 && e0 + VEC <= len) return w;
  uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    if (e0 + e < 0 || e0 + e >= len) {
      if constexpr (ES == 2) {
        const int sh = (e & 1) * 16;
        ws[e >> 1] = (ws[e >> 1] & ~(0xFFFFu << sh)) | ((NI & 0xFFFFu) << sh);
      } else {
        ws[e] = NI;
      }
    }
  }
  return make_uint4(ws[0], ws[1], ws[2], ws[3]);
}

template <int ES>
__device__ __forceinline__ uint32_t elem_bits(const uint4& w, int e) {
  const uint32_t word = (ES == 2 ? (e >> 1) : e) == 0   ? w.x
                        : (ES == 2 ? (e >> 1) : e) == 1 ? w.y
                        : (ES == 2 ? (e >> 1) : e) == 2 ? w.z
                                                        : w.w;
  if constexpr (ES == 2) return (e & 1) ? (word >> 16) : (word & 0xFFFFu);
  return word;
}

template <int ES>
__device__ __forceinline__ uint32_t key_of(uint32_t bits) {
  if constexpr (ES == 2) {
    const uint32_t mag = bits & 0x7FFFu;
    return (bits & 0x8000u) ? 0x8000u - mag : 0x8000u + mag;
  } else {
    const uint32_t mag = bits & 0x7FFFFFFFu;
    return (bits & 0x80000000u) ? 0x80000000u - mag : 0x80000000u + mag;
  }
}

// Input bits of an order key; -0.0 and +0.0 share a key, so the key of zero
// returns false and the caller reads the bits back from the input.
template <int ES>
__device__ __forceinline__ bool bits_of_key(uint32_t key, uint32_t* bits) {
  constexpr uint32_t kMid = ES == 2 ? 0x8000u : 0x80000000u;
  if (key == kMid) return false;
  *bits = key > kMid ? key - kMid : (kMid | (kMid - key));
  return true;
}

template <int ES>
__device__ __forceinline__ bool is_nan_bits(uint32_t bits) {
  if constexpr (ES == 2) return (bits & 0x7FFFu) > 0x7F80u;
  return (bits & 0x7FFFFFFFu) > 0x7F800000u;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t f32_max_nan(uint32_t a, uint32_t b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
  return __float_as_uint(d);
}

// Running maximum of vectors in "packed" form: bf16x2 lanes for bf16, one f32
// for fp32. NaN propagates, so a NaN anywhere in the granule shows in the result.
template <int ES>
__device__ __forceinline__ uint32_t max_acc(uint32_t acc, const uint4& w) {
  if constexpr (ES == 2) {
    return bf16x2_max_nan(acc, bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w)));
  } else {
    return f32_max_nan(acc, f32_max_nan(f32_max_nan(w.x, w.y), f32_max_nan(w.z, w.w)));
  }
}

// One NaN-propagating max of two packed accumulators.
template <int ES>
__device__ __forceinline__ uint32_t max_packed(uint32_t a, uint32_t b) {
  if constexpr (ES == 2) return bf16x2_max_nan(a, b);
  return f32_max_nan(a, b);
}

template <int ES>
__device__ __forceinline__ uint32_t finish_max(uint32_t acc) {
  if constexpr (ES == 2) {
    const uint32_t m = bf16x2_max_nan(acc, __byte_perm(acc, 0, 0x1032));
    return m & 0xFFFFu;
  } else {
    return acc;
  }
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int round_up32(int n) { return (n + 31) & ~31; }

// Histogram update: plain shared-memory atomic. Contention is low by design:
// every histogram here is either over a 256-key window next to the selection
// boundary (values spread over many bins) or over the few candidates of a row.
__device__ __forceinline__ void hist_add(uint32_t* h, uint32_t digit, bool valid) {
  if (valid) atomicAdd(&h[digit], 1u);
}

// Output index store and load: int32, or int64 when the caller asked for it.
__device__ __forceinline__ void put_index(void* out, int64_t pos, int64_t idx, int32_t idx64) {
  if (idx64) static_cast<int64_t*>(out)[pos] = idx;
  else static_cast<int32_t*>(out)[pos] = static_cast<int32_t>(idx);
}
__device__ __forceinline__ int64_t get_index(const void* out, int64_t pos, int32_t idx64) {
  return idx64 ? static_cast<const int64_t*>(out)[pos] : static_cast<int64_t>(static_cast<const int32_t*>(out)[pos]);
}

// Load a u16 from the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_ld_u16(const uint16_t* local, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  uint16_t v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(ra) : "memory");
  return v;
}

// Load a u32 from the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_ld_u32(const uint32_t* local, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

template <int S>
__device__ __forceinline__ void row_sync() {
  if constexpr (S > 1) {
    cg::this_cluster().sync();
  } else {
    __syncthreads();
  }
}

// Non-blocking reductions into the same shared-memory word of cluster CTA `rank`.
__device__ __forceinline__ void dsmem_red_add_u32(uint32_t* local, uint32_t rank, uint32_t v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_red_max_u32(uint32_t* local, uint32_t rank, uint32_t v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

struct LevelResult {
  uint32_t digit;  // bin holding the need-th largest key
  uint32_t above;  // keys above that bin (including the window's overflow count)
  uint32_t count;  // keys in that bin
  bool found;      // false: fewer than `need` keys in the window and above it
  bool shift;      // true: the need-th largest key lies above the window
};

// Locates the bin d with  over + sum(h[> d]) < need <= over + sum(h[>= d])  in a
// 256-bin histogram h (16-byte aligned) and broadcasts it through bc[0..2].
// Every thread of the CTA calls it; h and over must already be final.
__device__ __forceinline__ LevelResult scan_level(const uint32_t* h, uint32_t over, uint32_t* bc,
                                                  uint32_t need) {
  const int tid = threadIdx.x;
  if (tid < 32 && over < need) {
    const int lane = tid;
    const uint32_t n2 = need - over;
    const uint4 c0 = reinterpret_cast<const uint4*>(h)[lane * 2];
    const uint4 c1 = reinterpret_cast<const uint4*>(h)[lane * 2 + 1];
    const uint32_t c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += c[j];
    uint32_t suf = s;  // sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, o);
      if (lane + o < 32) suf += t;
    }
    if (lane == 0) bc[2] = suf >= n2;  // found
    const uint32_t above_lane = suf - s;
    if (above_lane < n2 && n2 <= suf) {
      uint32_t run = above_lane;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (run + c[j] >= n2) {
          bc[0] = static_cast<uint32_t>(lane * 8 + j);
          bc[1] = run + over;
          bc[3] = c[j];
          break;
        }
        run += c[j];
      }
    }
  }
  __syncthreads();
  LevelResult r;
  r.shift = over >= need;
  r.found = r.shift || bc[2] != 0u;
  r.digit = bc[0];
  r.above = bc[1];
  r.count = bc[3];
  __syncthreads();  // bc may be rewritten by the next level
  return r;
}

// Histogram levels whose counts are summed over the cluster. Clusters of up to
// 4 CTAs: every CTA adds its local counts into every CTA's receive histogram
// (red.shared::cluster, non-blocking), one cluster barrier, local scan. Larger
// clusters, by reduce-scatter: bin b belongs to CTA (b mod S); every CTA adds
// its count of bin b into the owner's receive histogram, one cluster barrier,
// then every CTA reads the 256 sums back from their owners (one
// distributed-shared-memory load per thread) and scans them locally. Receive
// histograms rotate over three buffers (the level counter runs on across rows,
// identically in every CTA of the cluster): the buffer a level clears for the
// next one was last read two levels earlier, before a barrier every CTA has
// passed, and is next written only after the current level's barrier.
struct ClusterLevels {
  uint32_t* hist;  // local kRadix | 3 x received kRadix
  uint32_t* ovw;   // [0] local overflow, [1..3] received overflow (held by CTA 0)
  uint32_t* bc;
  __device__ uint32_t* loc() const { return hist; }
  __device__ uint32_t* rcv(int lvl) const { return hist + kRadix * (1 + lvl % 3); }
  __device__ uint32_t* ov() const { return ovw; }

  // Clears the local histogram and overflow word (callers then add).
  __device__ void begin() const {
    if (threadIdx.x < kRadix) hist[threadIdx.x] = 0;
    if (threadIdx.x == 0) ovw[0] = 0;
    __syncthreads();
  }

  template <int S>
  __device__ LevelResult finish(int lvl, uint32_t need) const {
    __syncthreads();  // local counts complete
    const int tid = threadIdx.x;
    if constexpr (S > 1 && S <= 4) {
      // small clusters: every CTA adds its counts into every CTA's receive
      // histogram (S adds per bin), so no read-back round trip is needed
      if (tid < kRadix) {
        const uint32_t v = hist[tid];
        if (v) {
#pragma unroll
          for (int r = 0; r < S; ++r) dsmem_red_add_u32(rcv(lvl) + tid, static_cast<uint32_t>(r), v);
        }
        rcv(lvl + 1)[tid] = 0;
      }
      if (tid == 0) {
        if (ovw[0]) {
          for (int r = 0; r < S; ++r) dsmem_red_add_u32(ovw + 1 + lvl % 3, static_cast<uint32_t>(r), ovw[0]);
        }
        ovw[1 + (lvl + 1) % 3] = 0;
      }
      cg::this_cluster().sync();
      return scan_level(rcv(lvl), ovw[1 + lvl % 3], bc, need);
    } else if constexpr (S > 4) {
      if (tid < kRadix) {
        const uint32_t v = hist[tid];
        if (v) dsmem_red_add_u32(rcv(lvl) + tid, static_cast<uint32_t>(tid % S), v);
        rcv(lvl + 1)[tid] = 0;
      }
      if (tid == 0) {
        if (ovw[0]) dsmem_red_add_u32(ovw + 1 + lvl % 3, 0u, ovw[0]);
        ovw[1 + (lvl + 1) % 3] = 0;
      }
      cg::this_cluster().sync();
      if (tid < kRadix) hist[tid] = dsmem_ld_u32(rcv(lvl) + tid, static_cast<uint32_t>(tid % S));
      if (tid == 0) ovw[0] = dsmem_ld_u32(ovw + 1 + lvl % 3, 0u);
      __syncthreads();
    }
    return scan_level(hist, ovw[0], bc, need);
  }
};

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(0xFFFFFFFFu, v); }

__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += t;
  }
  return inc - v;
}


// Store a u32 at the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ void dsmem_st_u32(uint32_t* local, uint32_t rank, uint32_t v) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// misc[] layout (u32 words)
constexpr int kBc = 0;        // [0..2]   level result: digit, above, found
constexpr int kXmax = 4;      // [4]      cluster: row's largest granule key (pushed max)
constexpr int kXtot = 5;      // [5]      cluster: listed granules under the guess (pushed sum)
constexpr int kXpreGt = 6;    // [6]      cluster: selected '>' elements of lower ranks (pushed)
constexpr int kXpreEq = 7;    // [7]      cluster: '==' elements of lower ranks (pushed)
constexpr int kOvw = 8;       // [8..11]  overflow words of cluster levels (local + 3 received)
constexpr int kOvl = 12;      // [12]     overflow word of local levels
constexpr int kRdTot = 13;    // [13]     fallback: listed granules of the whole row
constexpr int kRdMax = 14;    // [14]     fallback: most listed granules of one warp
constexpr int kWtot = 16;     // [16..31] per-warp totals (2 x kWarps)
constexpr int kSegBase = 32;  // [32..39] candidate segment start per warp
constexpr int kSegCnt = 40;   // [40..47] candidate segment length per warp
constexpr int kLcnt = 48;     // [48..55] listed granules per warp
constexpr int kPub = 64;      // [64..79] counts published to the cluster (per warp + flags)
constexpr int kAll = 80;      // [80..80+16*kMaxCluster) counts gathered from every CTA
constexpr int kMaxCluster = 16;
constexpr int kMiscTotal = kAll + 16 * kMaxCluster;
constexpr int kHistWords = 5 * kRadix;  // cluster levels: local + 3 received; one local-level histogram

// Shared-memory footprint of one CTA (bytes) for a plan.
// Layout: stage | listed vectors | their candidate masks | list | union(M, candidates) |
// gathered | hist | misc.
// M (granule maxima) is dead once the list is built, before candidates exist.
__host__ __device__ constexpr int64_t union_bytes(int64_t g_cap_pad, int64_t cand_cap) {
  return ((g_cap_pad * 2 > cand_cap * 8 ? g_cap_pad * 2 : cand_cap * 8) + 15) & ~int64_t(15);
}
__host__ __device__ constexpr int64_t smem_bytes(int64_t g_cap_pad, int64_t list_cap,
                                                 int64_t cand_cap, int64_t gath_cap,
                                                 int64_t stage_vecs, int64_t lvec_cap) {
  return stage_vecs * kThreads * 16 + lvec_cap * kWarps * 16 + ((lvec_cap * kWarps + 15) & ~int64_t(15)) +
         ((list_cap * 2 + 15) & ~int64_t(15)) + union_bytes(g_cap_pad, cand_cap) + gath_cap * 8 +
         (kHistWords + kMiscTotal) * 4;
}

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Threshold reuse across rows: a persistent CTA (or cluster) first tries the
// previous row's threshold lowered by this many top-16 key units; the guess is
// kept only if it provably holds for the new row (at least k granule maxima
// reach it) and is not too loose (at most max(2k, k + 1024) of them do).
constexpr uint32_t kGuessMargin = 4;

// The float value whose order key is `key` (so that, for non-NaN v,
// v >= value  <=>  key(v) >= key). Keys at or below key(-inf) map to -inf.
template <int ES>
__device__ __forceinline__ float key_threshold_value(uint32_t key) {
  if constexpr (ES == 2) {
    if (key <= 0x0080u) return __uint_as_float(0xFF800000u);
    const uint32_t raw = key >= 0x8000u ? key - 0x8000u : (0x8000u | (0x8000u - key));
    return __uint_as_float(raw << 16);
  } else {
    if (key <= 0x00800000u) return __uint_as_float(0xFF800000u);
    const uint32_t raw = key >= 0x80000000u ? key - 0x80000000u : (0x80000000u | (0x80000000u - key));
    return __uint_as_float(raw);
  }
}

// fp32 value of a packed maximum's result (bf16 widens exactly).
template <int ES>
__device__ __forceinline__ float max_value(uint32_t raw) {
  if constexpr (ES == 2) return __uint_as_float(raw << 16);
  return __uint_as_float(raw);
}

// Bit e set iff element e of the vector is a candidate: not below the
// threshold value, or NaN (unordered comparison), so a granule whose maximum
// reaches the threshold always contributes at least one candidate. bf16 uses a
// packed compare of both halves (setp.geu.bf16x2: exact for subnormals, the
// first predicate reports the low half, i.e. the even element); tv2 holds the
// threshold's bf16 bits in both halves.
template <int ES>
__device__ __forceinline__ uint32_t cand_mask(const uint4& w, float tval, uint32_t tv2) {
  uint32_t m = 0;
  if constexpr (ES == 2) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r;
      asm("{\n\t.reg .pred lo, hi;\n\t"
          "setp.geu.bf16x2 lo|hi, %1, %2;\n\t"
          "selp.u32 %0, 1, 0, lo;\n\t"
          "@hi or.b32 %0, %0, 2;\n\t}"
          : "=r"(r) : "r"(ws[j]), "r"(tv2));
      m |= r << (2 * j);
    }
  } else {
    (void)tv2;
    m = static_cast<uint32_t>(!(__uint_as_float(w.x) < tval)) |
        static_cast<uint32_t>(!(__uint_as_float(w.y) < tval)) << 1 |
        static_cast<uint32_t>(!(__uint_as_float(w.z) < tval)) << 2 |
        static_cast<uint32_t>(!(__uint_as_float(w.w) < tval)) << 3;
  }
  return m;
}

// Candidate storage: word 0 carries what the order needs, word 1 the index.
// bf16: key in the low half, input bits in the high half; fp32: input bits.
template <int ES>
__device__ __forceinline__ uint32_t cand_pack(uint32_t bits) {
  if constexpr (ES == 2) return key_of<2>(bits) | (bits << 16);
  return bits;
}
template <int ES>
__device__ __forceinline__ uint32_t cand_key(uint32_t w0) {
  if constexpr (ES == 2) return w0 & 0xFFFFu;
  return key_of<4>(w0);
}
template <int ES>
__device__ __forceinline__ uint32_t cand_bits(uint32_t w0) {
  if constexpr (ES == 2) return w0 >> 16;
  return w0;
}

// 8 consecutive u16 granule maxima starting at `base` (a multiple of 8).
__device__ __forceinline__ void load_m8(const uint16_t* M, int base, uint32_t m[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(M + base);
  m[0] = q.x & 0xFFFFu; m[1] = q.x >> 16;
  m[2] = q.y & 0xFFFFu; m[3] = q.y >> 16;
  m[4] = q.z & 0xFFFFu; m[5] = q.z >> 16;
  m[6] = q.w & 0xFFFFu; m[7] = q.w >> 16;
}

// GV1: one 16-byte vector per granule (every slice of at most 8192 vectors);
// the general case (several vectors per granule, very long slices) is a
// separate instantiation so that its code does not weigh on the common one.
template <int ES, int S, bool GV1>
__global__ void __launch_bounds__(kThreads, 2) topk_rows_kernel(const Params p) {
  using T = Traits<ES>;
  constexpr int VEC = T::kVec;
  constexpr int KB = T::kKeyBits;
  constexpr uint32_t kFull = 0xFFFFFFFFu;
  using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;

  // Programmatic dependent launch: a kernel queued behind this one may be
  // scheduled now, and this one touches global memory only once every kernel
  // queued before it has completed (griddepcontrol.wait), so its inputs and
  // outputs are ordered as in a plain stream whatever those kernels do.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  // next-row prefetch: slot (i, thread) holds step i of the thread's P1 vectors
  uint4* stage = reinterpret_cast<uint4*>(smem_raw);                            // stage_vecs*kThreads
  uint4* lvec = stage + p.stage_vecs * kThreads;                                // lvec_cap*kWarps
  uint8_t* lmask = reinterpret_cast<uint8_t*>(lvec + p.lvec_cap * kWarps);      // lvec_cap*kWarps
  uint16_t* list = reinterpret_cast<uint16_t*>(lmask + ((p.lvec_cap * kWarps + 15) & ~15));  // list_cap
  unsigned char* uni = reinterpret_cast<unsigned char*>(list) + ((p.list_cap * 2 + 15) & ~15);
  uint16_t* M = reinterpret_cast<uint16_t*>(uni);                               // g_cap_pad
  uint32_t* cw0 = reinterpret_cast<uint32_t*>(uni);                             // cand_cap
  uint32_t* cw1 = cw0 + p.cand_cap;                                             // cand_cap
  uint32_t* gw0 = reinterpret_cast<uint32_t*>(uni + union_bytes(p.g_cap_pad, p.cand_cap));  // gath_cap
  uint32_t* gw1 = gw0 + p.gath_cap;                                             // gath_cap
  uint32_t* hist = gw1 + p.gath_cap;                                            // kHistWords
  uint32_t* hloc = hist + 4 * kRadix;                                           // local levels
  uint32_t* misc = hist + kHistWords;                                           // kMiscTotal
  uint32_t* bc = misc + kBc;
  uint32_t* wtot = misc + kWtot;
  const ClusterLevels CL{hist, misc + kOvw, bc};

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t lt_mask = lanemask_lt();
  int rank = 0;
  if constexpr (S > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
  const int64_t v0 = rank * p.vec_per_cta;
  const int64_t v1 = min(v0 + p.vec_per_cta, p.nvec);
  const int64_t nv = v1 > v0 ? v1 - v0 : 0;
  const int gv = GV1 ? 1 : p.gv;
  const int G = static_cast<int>((nv + gv - 1) / gv);
  const uint32_t k = static_cast<uint32_t>(p.k);
  const int64_t row_step = gridDim.x / S;
  // Warp w owns the contiguous granule segment [sb, se); its lanes interleave
  // (granule sb + 32 i + lane), so every warp load is 512 contiguous bytes and
  // the warp's list and candidates come out in index order.
  const int segm = round_up32((G + kWarps - 1) / kWarps);
  const int sb = min(warp * segm, G);
  const int se = min(sb + segm, G);
  uint16_t* wlist = list + warp * segm;
  uint4* wvec = lvec + warp * p.lvec_cap;
  uint8_t* wmask = lmask + warp * p.lvec_cap;
  // granules whose vectors all lie inside [0, len) (gv == 1: full vectors)
  const int Gf = gv == 1 ? static_cast<int>(min(v1, max(v0, p.len / VEC)) - v0) : G;

  bool have_guess = false;
  uint32_t t_guess = 0;
  // Steps of the P1 walk whose vectors are prefetched into shared memory with
  // cp.async while the previous row is being selected (each thread copies and
  // later reads only its own slots, so no barrier is needed around them).
  const int nsteps = (se - sb + 31) / 32;
  // (only rows on 16-byte boundaries: the copies are 16-byte cp.async)
  const bool rows_aligned = (reinterpret_cast<uintptr_t>(p.x) % 16 == 0) && (p.row_stride_bytes % 16 == 0);
  const int nstage = (gv == 1 && rows_aligned) ? min(p.stage_vecs, nsteps) : 0;
  auto prefetch = [&](int64_t r) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + r * p.row_stride_bytes) + v0;
    for (int i = 0; i < nstage; ++i) {
      const int g = sb + 32 * i + lane;
      if (g < min(se, Gf)) cp_async_16(stage + i * kThreads + tid, src + g);
    }
    cp_async_commit();
  };
  if (nstage > 0 && blockIdx.x / S < p.batch) prefetch(blockIdx.x / S);
  // receive histograms and cluster-pushed words start cleared in every CTA
  if (tid < kRadix) {
    hist[kRadix + tid] = 0;
    hist[2 * kRadix + tid] = 0;
    hist[3 * kRadix + tid] = 0;
  }
  if (tid < 4) misc[kOvw + tid] = 0;
  if (tid < 4) misc[kXmax + tid] = 0;
  int lvl = 0;  // cluster levels so far (runs across rows; identical in the cluster)
  if constexpr (S > 1) cg::this_cluster().sync();
  else __syncthreads();

#pragma unroll 1
  for (int64_t row = blockIdx.x / S; row < p.batch; row += row_step) {
    // the row as 16-byte aligned blocks: its element i is element i + lead of
    // block 0; blocks [vf0, vf1) lie wholly inside it, nvr blocks overlap it
    // (a row that starts on a 16-byte boundary has lead 0)
    const uintptr_t raddr = reinterpret_cast<uintptr_t>(p.x + row * p.row_stride_bytes);
    const char* rowp = reinterpret_cast<const char*>(raddr & ~static_cast<uintptr_t>(15));
    const uint4* rowv = reinterpret_cast<const uint4*>(rowp);
    const int lead = static_cast<int>((raddr & 15u) / ES);
    const int64_t nvr = (lead + p.len + VEC - 1) / VEC;
    const int gf0 = (lead != 0 && v0 == 0) ? 1 : 0;  // slice blocks [gf0, Gfr) are whole
    const int Gfr = gv == 1 ? static_cast<int>(max(int64_t(0), min(nv, (lead + p.len) / VEC - v0))) : G;
    auto blk = [&](int64_t v) -> uint4 { return load_blk<ES>(rowp, v, lead, p.len, nvr); };
    if (tid == 0) {  // level results start defined even if a NaN row breaks the counts
      bc[0] = 0;
      bc[1] = 0;
      bc[2] = 0;
    }

    // ---- P1: one streaming pass over the slice -----------------------------------
    // guess mode: a granule whose maximum reaches the guessed threshold goes to the
    //             warp's list right away (nothing else is stored);
    // exact mode: every granule's maximum key goes to M.
    // Both modes test every element for NaN through the NaN-propagating maxima.
    uint32_t t16 = 0;
    uint32_t row_max16 = 0xFFFFFFFFu;  // the row's largest top-16 key, when the exact threshold found it
    int lc = 0;  // granules in this warp's list (warp-uniform)
    bool vec_kept = false;  // the list's vectors were copied to wvec by the streaming pass
    bool guess_mode = have_guess;
#pragma unroll 1
    for (int attempt = 0; attempt < 2; ++attempt) {
      uint32_t nan_acc = T::kNegInfWord;
      uint32_t mmax = 0;
      const float tg = key_threshold_value<ES>((KB == 16) ? t_guess : (t_guess << 16));
      lc = 0;
      if (gv == 1) {
        constexpr int U = 8;
        const bool staged = attempt == 0 && nstage > 0;
        if (staged) cp_async_wait_all();
        const bool next = staged && row + row_step < p.batch;
        const uint4* nsrc = reinterpret_cast<const uint4*>(p.x + (row + row_step) * p.row_stride_bytes) + v0;
        for (int i0 = 0; i0 < nsteps; i0 += U) {
          uint4 w[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + u;
            const int g = sb + 32 * i + lane;
            if (g >= gf0 && g < min(se, Gfr)) {
              if (staged && i < nstage) {
                w[u] = stage[i * kThreads + tid];
              } else {
                w[u] = ld_nc_v4(rowv + (v0 + g));
              }
            } else if (g < se) {
              w[u] = blk(v0 + g);  // a block the row only partly covers
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int g = sb + 32 * (i0 + u) + lane;
            const bool ok = g < se;
            const uint32_t acc = ok ? max_acc<ES>(T::kNegInfWord, w[u]) : T::kNegInfWord;
            // the slot's value is in registers and consumed: refill it for the next row
            if (next && i0 + u < nstage && g < min(se, Gf))
              cp_async_16(stage + (i0 + u) * kThreads + tid, nsrc + g);
            nan_acc = max_packed<ES>(nan_acc, acc);
            const uint32_t raw = finish_max<ES>(acc);
            if (guess_mode) {
              const bool pass = ok && !(max_value<ES>(raw) < tg);
              const uint32_t b = __ballot_sync(kFull, pass);
              if (pass) {
                const int pos = lc + __popc(b & lt_mask);
                wlist[pos] = static_cast<uint16_t>(g);
                if (pos < p.lvec_cap) wvec[pos] = w[u];  // the candidate pass reads it back
              }
              lc += __popc(b);
            } else if (ok) {
              const uint32_t mk = key_of<ES>(raw) >> (KB - 16);
              mmax = max(mmax, mk);
              M[g] = static_cast<uint16_t>(mk);
            }
          }
        }
        if (next) cp_async_commit();
      } else {
        for (int i0 = sb; i0 < se; i0 += 32) {
          const int g = i0 + lane;
          const bool ok = g < se;
          uint32_t acc = T::kNegInfWord;
          if (ok) {
            const int64_t vb = v0 + static_cast<int64_t>(g) * gv;
            const int64_t ve = min(vb + gv, v1);
            for (int64_t v = vb; v < ve; ++v) acc = max_acc<ES>(acc, blk(v));
          }
          nan_acc = max_packed<ES>(nan_acc, acc);
          const uint32_t raw = finish_max<ES>(acc);
          if (guess_mode) {
            const bool pass = ok && !(max_value<ES>(raw) < tg);
            const uint32_t b = __ballot_sync(kFull, pass);
            if (pass) wlist[lc + __popc(b & lt_mask)] = static_cast<uint16_t>(g);
            lc += __popc(b);
          } else if (ok) {
            const uint32_t mk = key_of<ES>(raw) >> (KB - 16);
            mmax = max(mmax, mk);
            M[g] = static_cast<uint16_t>(mk);
          }
        }
      }
      mmax = __reduce_max_sync(kFull, mmax);
      if (lane == 0) {
        wtot[warp] = mmax;
        misc[kLcnt + warp] = static_cast<uint32_t>(lc);
      }
      if (__syncthreads_or(is_nan_bits<ES>(finish_max<ES>(nan_acc))) && tid == 0)
        atomicOr(p.flag, DS_TOPK_FLAG_NAN);

      if (guess_mode) {
        // keep the guess only if at least k granule maxima reach it (safety) and
        // not too many do (tightness)
        uint32_t total = 0;
        for (int w = 0; w < kWarps; ++w) total += misc[kLcnt + w];
        if constexpr (S > 1) {
          if (tid < S) dsmem_red_add_u32(misc + kXtot, static_cast<uint32_t>(tid), total);
          cg::this_cluster().sync();
          total = misc[kXtot];
        }
        t16 = t_guess;
        __syncthreads();  // every warp has read the per-warp counts before they change
        if (total >= k && total <= max(2u * k, k + 1024u)) {
          vec_kept = gv == 1;
          break;
        }
        guess_mode = false;  // rerun the pass in exact mode
        continue;
      }

      // ---- A: exact threshold t16 = the k-th largest granule maximum ----------------
      mmax = 0;
      for (int w = 0; w < kWarps; ++w) mmax = max(mmax, wtot[w]);
      t16 = 0;
      if (p.g_total >= static_cast<int64_t>(k)) {
        // histogram over the 256 key values just below the row's largest maximum
        if constexpr (S > 1) {
          if (tid < S) dsmem_red_max_u32(misc + kXmax, static_cast<uint32_t>(tid), mmax);
          cg::this_cluster().sync();
          mmax = misc[kXmax];
        }
        row_max16 = mmax;
        const uint32_t wbase = mmax > 255u ? mmax - 255u : 0u;
        CL.begin();
        for (int b0 = sb; b0 < se; b0 += 256) {  // 8 maxima per lane per step
          const int base = b0 + lane * 8;
          if (base < se) {
            uint32_t m[8];
            load_m8(M, base, m);
#pragma unroll
            for (int e = 0; e < 8; ++e) hist_add(CL.loc(), m[e] - wbase, base + e < se && m[e] >= wbase);
          }
        }
        const LevelResult r = CL.finish<S>(lvl++, k);
        if (r.found) {
          t16 = wbase + r.digit;
        } else {
          // fewer than k maxima within 256 keys of the largest: two 8-bit levels
          CL.begin();
          for (int b0 = sb; b0 < se; b0 += 256) {
            const int base = b0 + lane * 8;
            if (base < se) {
              uint32_t m[8];
              load_m8(M, base, m);
#pragma unroll
              for (int e = 0; e < 8; ++e) hist_add(CL.loc(), m[e] >> 8, base + e < se);
            }
          }
          const LevelResult r1 = CL.finish<S>(lvl++, k);
          CL.begin();
          for (int b0 = sb; b0 < se; b0 += 256) {
            const int base = b0 + lane * 8;
            if (base < se) {
              uint32_t m[8];
              load_m8(M, base, m);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                hist_add(CL.loc(), m[e] & 0xFFu, base + e < se && (m[e] >> 8) == r1.digit);
            }
          }
          const LevelResult r2 = CL.finish<S>(lvl++, k - r1.above);
          t16 = (r1.digit << 8) | r2.digit;
        }
        t_guess = t16 > 0x0080u + kGuessMargin ? t16 - kGuessMargin : 0u;
        have_guess = true;
      }
      // this warp's list: granules whose maximum reaches t16, in index order
      // (8 consecutive maxima per lane per step, lanes in order)
      lc = 0;
      for (int b0 = sb; b0 < se; b0 += 256) {
        const int base = b0 + lane * 8;
        uint32_t mask = 0;
        if (base < se) {
          uint32_t m[8];
          load_m8(M, base, m);
#pragma unroll
          for (int e = 0; e < 8; ++e) mask |= static_cast<uint32_t>(base + e < se && m[e] >= t16) << e;
        }
        const uint32_t c = __popc(mask);
        int excl = 0, tot = 0;
#pragma unroll 1
        for (uint32_t t = 1;; ++t) {  // positions from ballots: counts are mostly 0 or 1
          const uint32_t b = __ballot_sync(kFull, c >= t);
          if (b == 0) break;
          excl += __popc(b & lt_mask);
          tot += __popc(b);
        }
        int pos = lc + excl;
        lc += tot;
        while (mask) {
          const int e = __ffs(mask) - 1;
          mask &= mask - 1;
          wlist[pos++] = static_cast<uint16_t>(base + e);
        }
      }
      __syncwarp();  // the warp's list is read back by other lanes below
      break;
    }

    // ---- D: candidates (key >= t, or NaN) of the listed granules, in index order ----
    // Pass 1 counts each warp's candidates (keeping every listed vector's 8-bit
    // candidate mask); a prefix over the warps then gives each warp its place in
    // the CTA's candidate array, and pass 2 writes them there. Listed vectors are
    // read from the warp's shared copy (kept by the streaming pass, or fetched
    // now from L2); entries beyond its capacity are read from L2 in both passes.
    const uint32_t T_full = (KB == 16) ? t16 : (t16 << 16);
    const float tval = key_threshold_value<ES>(T_full);
    const uint32_t tv2 = (__float_as_uint(tval) >> 16) * 0x00010001u;  // bf16 bits, both halves
    const uint4* slice = rowv + v0;
    const int nvs = static_cast<int>(nv);  // vectors in this slice
    const int nfull = gv == 1 ? Gfr : static_cast<int>(max(int64_t(0), min(nv, (lead + p.len) / VEC - v0)));
    // candidate mask of slice vector v (in a block the row only partly covers,
    // the elements outside the row are cleared)
    auto vmask_of = [&](int v, const uint4& w) -> uint32_t {
      uint32_t m = cand_mask<ES>(w, tval, tv2);
      if (v < gf0 || v >= nfull) {  // only the row's elements of a partly covered block
        const int64_t e0 = (v0 + v) * VEC - lead;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (e0 + e < 0 || e0 + e >= p.len) m &= ~(1u << e);
      }
      return m;
    };
    auto load_slice = [&](int v) -> uint4 {
      return (v >= gf0 && v < nfull) ? ld_nc_v4(slice + v) : blk(v0 + v);
    };
    const int ncache = gv == 1 ? min(lc, p.lvec_cap) : 0;  // list entries held in wvec
    // Every listed granule holds at least one candidate, so a CTA whose listed
    // granules alone exceed the candidate capacity overflows for certain: it
    // skips the counting pass (rows made of a few repeated values list most of
    // their granules).
    if (lane == 0) misc[kLcnt + warp] = static_cast<uint32_t>(lc);
    __syncthreads();
    uint32_t listed = 0;
    for (int w = 0; w < kWarps; ++w) listed += misc[kLcnt + w];
    const bool sure_over = listed > static_cast<uint32_t>(p.cand_cap);
    if (gv == 1 && !vec_kept && !sure_over) {
      for (int j = lane; j < ncache; j += 32) wvec[j] = load_slice(wlist[j]);
      __syncwarp();
    }
    uint32_t wc = 0;
    for (int j = lane; j < (sure_over ? 0 : lc); j += 32) {
      if (gv == 1) {
        const int v = wlist[j];
        const uint32_t m = vmask_of(v, j < ncache ? wvec[j] : load_slice(v));
        if (j < ncache) wmask[j] = static_cast<uint8_t>(m);
        wc += __popc(m);
      } else {
        const int vb = static_cast<int>(wlist[j]) * gv;
        const int ve = min(vb + gv, nvs);
        for (int v = vb; v < ve; ++v) wc += __popc(vmask_of(v, load_slice(v)));
      }
    }
    wc = warp_sum(wc);
    if (lane == 0) wtot[kWarps + warp] = wc;
    __syncthreads();
    uint32_t cbase = 0, ncand = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t t = wtot[kWarps + w];
      if (w < warp) cbase += t;
      ncand += t;
    }
    if (sure_over) ncand = listed;
    const bool cta_over = ncand > static_cast<uint32_t>(p.cand_cap);
    if (!cta_over) {
      // pass 2: write, lanes in index order; positions from ballots (almost every
      // listed granule holds exactly one candidate)
      for (int j0 = 0; j0 < lc; j0 += 32) {
        const int j = j0 + lane;
        int vb = 0, ve = 0;
        uint32_t c = 0, m0 = 0;
        uint4 w0 = make_uint4(0u, 0u, 0u, 0u);
        if (j < lc) {
          if (gv == 1) {
            vb = wlist[j];
            ve = vb + 1;
            if (j < ncache) {
              m0 = wmask[j];
            } else {
              w0 = load_slice(vb);
              m0 = vmask_of(vb, w0);
            }
            c = __popc(m0);
          } else {
            vb = static_cast<int>(wlist[j]) * gv;
            ve = min(vb + gv, nvs);
            for (int v = vb; v < ve; ++v) c += __popc(vmask_of(v, load_slice(v)));
          }
        }
        int excl = 0, tot = 0;
#pragma unroll 1
        for (uint32_t t = 1;; ++t) {
          const uint32_t b = __ballot_sync(kFull, c >= t);
          if (b == 0) break;
          excl += __popc(b & lt_mask);
          tot += __popc(b);
        }
        uint32_t pos = cbase + excl;
        cbase += tot;
        if (c == 0) continue;
        for (int v = vb; v < ve; ++v) {
          uint4 w;
          uint32_t m;
          const bool in_cache = gv == 1 && j < ncache;
          if (gv == 1) {
            w = w0;
            m = m0;
          } else {
            w = load_slice(v);
            m = vmask_of(v, w);
          }
          const uint32_t ibase = static_cast<uint32_t>((v0 + v) * VEC - lead);
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1;
            uint32_t bits;
            if (in_cache) {
              if constexpr (ES == 2) bits = reinterpret_cast<const uint16_t*>(wvec + j)[e];
              else bits = reinterpret_cast<const uint32_t*>(wvec + j)[e];
            } else {
              bits = elem_bits<ES>(w, e);
            }
            cw0[pos] = cand_pack<ES>(bits);
            cw1[pos] = ibase + e;
            ++pos;
          }
        }
      }
    }
    // candidates are contiguous in index order: 8 equal warp segments for B and C
    if (lane == 0) {
      const uint32_t per = (ncand + kWarps - 1) / kWarps;
      const uint32_t b = min(static_cast<uint32_t>(warp) * per, ncand);
      misc[kSegBase + warp] = b;
      misc[kSegCnt + warp] = min(b + per, ncand) - b;
    }
    __syncthreads();

    // ---- cluster: ship every CTA's candidates to the leader (rank 0) --------------
    bool dense = !cta_over;
    bool work_here = true;  // this CTA runs the selection (always, unless a non-leader)
    if constexpr (S > 1) {
      if (tid == 0) {
        misc[kPub] = ncand;
        misc[kPub + 1] = cta_over ? 1u : 0u;
      }
      cg::this_cluster().sync();
      if (tid < 2 * S) misc[kAll + tid] = dsmem_ld_u32(misc + kPub + (tid & 1), static_cast<uint32_t>(tid >> 1));
      __syncthreads();
      uint32_t total = 0, before = 0;
      bool any_over = false;
      for (int r = 0; r < S; ++r) {
        any_over |= misc[kAll + 2 * r + 1] != 0u;
        const uint32_t c = misc[kAll + 2 * r];
        if (r < rank) before += c;
        total += c;
      }
      dense = !any_over && total <= static_cast<uint32_t>(p.gath_cap);
      if (dense) {
        for (uint32_t c = tid; c < ncand; c += kThreads) {
          dsmem_st_u32(gw0 + before + c, 0u, cw0[c]);
          dsmem_st_u32(gw1 + before + c, 0u, cw1[c]);
        }
        cg::this_cluster().sync();  // the leader's gathered array is complete
        work_here = rank == 0;
        if (work_here && lane == 0) {
          const uint32_t per = (total + kWarps - 1) / kWarps;
          const uint32_t b = min(static_cast<uint32_t>(warp) * per, total);
          misc[kSegBase + warp] = b;
          misc[kSegCnt + warp] = min(b + per, total) - b;
        }
        __syncthreads();
      }
    }

    const int64_t out_base = row * static_cast<int64_t>(k);  // this row's first output
    VT* out_val = p.return_value ? reinterpret_cast<VT*>(p.out_values) + row * static_cast<int64_t>(k) : nullptr;

    if (dense && work_here) {
      // ---- B (dense): exact k-th key among the candidates, locally -------------------
      const uint32_t* c0 = (S > 1) ? gw0 : cw0;
      const uint32_t* c1 = (S > 1) ? gw1 : cw1;
      const int sbase = static_cast<int>(misc[kSegBase + warp]);
      const int scnt = static_cast<int>(misc[kSegCnt + warp]);
      uint32_t need = k, kstar = 0, small = 0;
      const uint32_t wbase = t16;
      uint32_t* ovl = misc + kOvl;
      {  // windowed level on the top 16 key bits: the 256 values from t16 up
        if (tid < kRadix) hloc[tid] = 0;
        if (tid == 0) *ovl = 0;
        __syncthreads();
        uint32_t lover = 0;
        for (int c = lane; c < round_up32(scnt); c += 32) {
          const bool okc = c < scnt;
          const uint32_t k16v = cand_key<ES>(okc ? c0[sbase + c] : 0u) >> (KB - 16);
          const bool ok = okc && k16v >= wbase;
          const uint32_t d = k16v - wbase;
          hist_add(hloc, d, ok && d < 256u);
          lover += __popc(__ballot_sync(kFull, ok && d >= 256u));
        }
        if (lane == 0 && lover) atomicAdd(ovl, lover);
        __syncthreads();
        const LevelResult r = scan_level(hloc, *ovl, bc, need);
        if (r.shift && wbase + 256u <= 0xFFFFu) {
          // the k-th key lies above the window: two 8-bit levels over the top 16
          // key bits of the candidates above it
          const uint32_t lo16 = wbase + 256u;
          uint32_t hi8 = 0;
#pragma unroll 1
          for (int lv = 0; lv < 2; ++lv) {
            if (tid < kRadix) hloc[tid] = 0;
            __syncthreads();
            for (int c = lane; c < scnt; c += 32) {
              const uint32_t k16v = cand_key<ES>(c0[sbase + c]) >> (KB - 16);
              const bool ok = k16v >= lo16 && (lv == 0 || (k16v >> 8) == hi8);
              hist_add(hloc, lv == 0 ? (k16v >> 8) : (k16v & 0xFFu), ok);
            }
            __syncthreads();
            const LevelResult rl = scan_level(hloc, 0u, bc, need);
            need -= rl.above;
            if (lv == 0) {
              hi8 = rl.digit;
            } else {
              kstar = ((hi8 << 8) | rl.digit) << (KB - 16);
              small = rl.count;
            }
          }
        } else {
          kstar = (wbase + r.digit) << (KB - 16);
          need -= r.above;
          small = r.count;
        }
      }
      if constexpr (KB == 32) {
        const uint32_t pre16 = kstar >> 16;
        if (small <= 32) {
          // few candidates share K*'s top 16 bits: collect them, then one warp
          // ranks them exactly (the need-th largest of at most 32 keys)
          if (tid == 0) *ovl = 0;
          __syncthreads();
          for (int c = lane; c < scnt; c += 32) {
            const uint32_t key = cand_key<ES>(c0[sbase + c]);
            if ((key >> 16) == pre16) hloc[atomicAdd(ovl, 1u)] = key;
          }
          __syncthreads();
          if (tid < 32) {
            const uint32_t m = *ovl;
            const uint32_t mine = lane < static_cast<int>(m) ? hloc[lane] : 0u;
            uint32_t gt = 0, eq = 0;
            for (uint32_t j = 0; j < m; ++j) {
              const uint32_t other = __shfl_sync(0xFFFFFFFFu, mine, static_cast<int>(j));
              gt += other > mine;
              eq += other == mine;
            }
            if (lane < static_cast<int>(m) && gt < need && need <= gt + eq) {
              bc[0] = mine;  // every lane holding K* writes the same values
              bc[1] = gt;
            }
          }
          __syncthreads();
          kstar = bc[0];
          need -= bc[1];
          __syncthreads();
        } else {
#pragma unroll 1
          for (int j = 0; j < 2; ++j) {  // low 16 bits: two 8-bit levels
            const int shift = 8 - 8 * j;
            if (tid < kRadix) hloc[tid] = 0;
            __syncthreads();
            const uint32_t pre = kstar >> (shift + 8);
            for (int c = lane; c < scnt; c += 32) {
              const uint32_t key = cand_key<ES>(c0[sbase + c]);
              hist_add(hloc, (key >> shift) & 0xFFu, (key >> (shift + 8)) == pre);
            }
            __syncthreads();
            const LevelResult r = scan_level(hloc, 0u, bc, need);
            kstar |= r.digit << shift;
            need -= r.above;
          }
        }
      }
      const uint32_t r_ties = need;  // elements equal to K* that are taken

      // ---- C (dense): ordered compaction -------------------------------------------
      uint32_t c_gt = 0, c_eq = 0;
      for (int c = lane; c < round_up32(scnt); c += 32) {
        const uint32_t key = cand_key<ES>(c < scnt ? c0[sbase + c] : 0u);
        c_gt += __popc(__ballot_sync(kFull, c < scnt && key > kstar));
        c_eq += __popc(__ballot_sync(kFull, c < scnt && key == kstar));
      }
      if (lane == 0) {
        wtot[warp] = c_gt;
        wtot[kWarps + warp] = c_eq;
      }
      __syncthreads();
      uint32_t base_gt = 0, base_eq = 0;
      for (int w = 0; w < warp; ++w) {
        base_gt += wtot[w];
        base_eq += wtot[kWarps + w];
      }
      for (int c = lane; c < round_up32(scnt); c += 32) {
        const bool ok = c < scnt;
        const uint32_t w0 = ok ? c0[sbase + c] : 0u;
        const uint32_t key = cand_key<ES>(w0);
        const uint32_t mg = __ballot_sync(kFull, ok && key > kstar);
        const uint32_t mq = __ballot_sync(kFull, ok && key == kstar);
        const uint32_t bg = base_gt + __popc(mg & lt_mask);
        const uint32_t bq = base_eq + __popc(mq & lt_mask);
        base_gt += __popc(mg);
        base_eq += __popc(mq);
        uint32_t pos = 0xFFFFFFFFu;
        if ((mg >> lane) & 1u) pos = bg + min(bq, r_ties);
        else if (((mq >> lane) & 1u) && bq < r_ties) pos = bg + bq;
        if (pos < k) {
          put_index(p.out_indices, out_base + pos, c1[sbase + c], p.idx64);
          if (out_val) out_val[pos] = static_cast<VT>(cand_bits<ES>(w0));
        }
      }
    } else if (!dense) {
      // ---- fallback: candidates did not fit; select over the listed granules, ------
      // re-read from global memory, with cluster-wide histograms.
      //
      // The listed granules of a row can sit in a few warps of one CTA (a sorted
      // or ramp row lists only the top of the row). So they are first spread
      // evenly over every warp of the cluster: the per-warp list counts of all
      // CTAs give a prefix in (CTA, warp) order, which is index order, and
      // global warp g takes the contiguous share [g T / G, (g + 1) T / G) of the
      // concatenated lists, read from the owners' shared memory into its own
      // (the granule maxima and candidate arrays are dead here).
      const int G = kWarps * S;
      uint32_t* gcnt = misc + kAll;      // [G] listed granules per (CTA, warp)
      uint32_t* gpre = misc + kAll + G;  // [G] their exclusive prefix
      __syncthreads();                   // the published counts in misc[kAll..] are read
      if (tid < G) {
        if constexpr (S > 1) gcnt[tid] = dsmem_ld_u32(misc + kLcnt + tid % kWarps, static_cast<uint32_t>(tid / kWarps));
        else gcnt[tid] = misc[kLcnt + tid];
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[4], sum = 0, most = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = lane * 4 + i;
          c[i] = q < G ? gcnt[q] : 0u;
          sum += c[i];
          most = max(most, c[i]);
        }
        uint32_t run = warp_excl_scan(sum);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = lane * 4 + i;
          if (q < G) gpre[q] = run;
          run += c[i];
        }
        most = __reduce_max_sync(kFull, most);
        if (lane == 31) misc[kRdTot] = run;
        if (lane == 0) misc[kRdMax] = most;
      }
      __syncthreads();
      const uint32_t rd_total = misc[kRdTot];
      const uint32_t rd_share = (rd_total + G - 1) / G;
      const int rd_cap = static_cast<int>(union_bytes(p.g_cap_pad, p.cand_cap) / 4 / kWarps);
      // spread only lists that are skewed (a warp holds over twice its share):
      // even lists (rows of a few levels spread over the whole row) gain nothing
      // from it but its cost; cluster-uniform
      const bool rd = gv == 1 && G > 1 && misc[kRdMax] > 2u * rd_share + 32u &&
                      rd_share <= static_cast<uint32_t>(rd_cap);
      // Without spreading, the dead granule-maximum / candidate region keeps each
      // listed block's masks from the count pass (2 bytes per list entry), so the
      // write pass reads a block again only for the values it cannot tell from K*.
      const bool keep_masks = !rd && gv == 1 && union_bytes(p.g_cap_pad, p.cand_cap) >= 2 * static_cast<int64_t>(p.list_cap);
      uint16_t* vmask = reinterpret_cast<uint16_t*>(uni) + warp * segm;
      uint32_t* ra = reinterpret_cast<uint32_t*>(uni) + warp * rd_cap;  // this warp's share: row vector indices
      int rn = 0;
      if (rd) {
        const uint32_t g = static_cast<uint32_t>(rank * kWarps + warp);
        const uint32_t a = static_cast<uint32_t>(static_cast<uint64_t>(g) * rd_total / G);
        const uint32_t b = static_cast<uint32_t>(static_cast<uint64_t>(g + 1) * rd_total / G);
        rn = static_cast<int>(b - a);
        for (uint32_t j = a + lane; j < b; j += 32) {
          int lo = 0, hi = G - 1;  // the last (CTA, warp) whose list starts at or before j
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gpre[mid] <= j) lo = mid;
            else hi = mid - 1;
          }
          const int orank = lo / kWarps, ow = lo % kWarps;
          const int64_t onv = min(p.vec_per_cta, p.nvec - orank * p.vec_per_cta);  // vectors of its slice
          const int osegm = round_up32(static_cast<int>((onv + kWarps - 1) / kWarps));
          const uint16_t* ol = list + ow * osegm + (j - gpre[lo]);
          uint32_t e;
          if constexpr (S > 1) e = dsmem_ld_u16(ol, static_cast<uint32_t>(orank));
          else e = *ol;
          ra[j - a] = static_cast<uint32_t>(orank * p.vec_per_cta) + e;
        }
        __syncwarp();
      }
      const int lcnt = rd ? rn : lc;  // this warp's listed granules, after spreading
      auto vec_at = [&](int j) -> int {  // row vector index of the warp's j-th listed granule
        return rd ? static_cast<int>(ra[j]) : static_cast<int>(v0) + static_cast<int>(wlist[j]);
      };
      auto visit = [&](auto&& f) {
        if (gv == 1) {  // 4 listed vectors in flight per lane (row vector indices fit 32 bits)
          constexpr int UV = 4;
          const int ilen = static_cast<int>(p.len);
          const int ilead = lead;
          for (int jb = 0; jb < lcnt; jb += 32 * UV) {
            uint4 w[UV];
            int v[UV];
#pragma unroll
            for (int u = 0; u < UV; ++u) {
              const int j = jb + 32 * u + lane;
              v[u] = j < lcnt ? vec_at(j) : -1;
              w[u] = make_uint4(T::kNegInfWord, T::kNegInfWord, T::kNegInfWord, T::kNegInfWord);
              if (v[u] >= 0) w[u] = blk(v[u]);
            }
#pragma unroll
            for (int u = 0; u < UV; ++u) {
              const bool vok = v[u] >= 0;
#pragma unroll
              for (int e = 0; e < VEC; ++e) {
                const uint32_t eb = elem_bits<ES>(w[u], e);
                const uint32_t key = key_of<ES>(eb);
                const int idx = v[u] * VEC + e - ilead;
                f(key, vok && idx >= 0 && idx < ilen && (key >= T_full || is_nan_bits<ES>(eb)));
              }
            }
          }
          return;
        }
        if constexpr (!GV1) {  // granules of several vectors
          for (int j = lane; j < round_up32(lc); j += 32) {
            const bool gok = j < lc;
            for (int q = 0; q < gv; ++q) {
              const int64_t v = gok ? v0 + static_cast<int64_t>(wlist[j]) * gv + q : v1;
              const bool vok = v < v1;
              uint4 w = make_uint4(T::kNegInfWord, T::kNegInfWord, T::kNegInfWord, T::kNegInfWord);
              if (vok) w = blk(v);
#pragma unroll
              for (int e = 0; e < VEC; ++e) {
                const uint32_t eb = elem_bits<ES>(w, e);
                const uint32_t key = key_of<ES>(eb);
                const int64_t idx = v * VEC + e - lead;
                f(key, vok && idx >= 0 && idx < p.len && (key >= T_full || is_nan_bits<ES>(eb)));
              }
            }
          }
        }
      };
      uint32_t need = k, kstar = 0;
      if (KB == 16 && row_max16 == t16) {
        // at least k granule maxima equal the row's largest key, so at least k
        // elements do: that key is the k-th key, and the lowest-index k of the
        // elements holding it are the row's top k (rows of a few repeated levels)
        kstar = t16;
      } else {
        {
          // the 256 top-16 key values from t16 up, with a count of the keys above
          const uint32_t wbase = t16;
          CL.begin();
          uint32_t* h = CL.loc();
          uint32_t lover = 0;
          visit([&](uint32_t key, bool ok) {
            const uint32_t k16v = key >> (KB - 16);
            ok = ok && k16v >= wbase;
            const uint32_t d = k16v - wbase;
            hist_add(h, d, ok && d < 256u);
            lover += __popc(__ballot_sync(kFull, ok && d >= 256u));
          });
          if (lane == 0 && lover) atomicAdd(CL.ov(), lover);
          const LevelResult r = CL.finish<S>(lvl++, need);
          if (r.shift && wbase + 256u <= 0xFFFFu) {
            // the k-th key lies above the window (t far below it, e.g. when k exceeds
            // the number of granules with a finite maximum): two 8-bit levels over
            // the top 16 key bits of the keys above the window
            const uint32_t lo16 = wbase + 256u;
            CL.begin();
            h = CL.loc();
            visit([&](uint32_t key, bool ok) {
              const uint32_t k16v = key >> (KB - 16);
              hist_add(h, k16v >> 8, ok && k16v >= lo16);
            });
            const LevelResult ra = CL.finish<S>(lvl++, need);
            need -= ra.above;
            CL.begin();
            h = CL.loc();
            visit([&](uint32_t key, bool ok) {
              const uint32_t k16v = key >> (KB - 16);
              hist_add(h, k16v & 0xFFu, ok && k16v >= lo16 && (k16v >> 8) == ra.digit);
            });
            const LevelResult rb = CL.finish<S>(lvl++, need);
            need -= rb.above;
            kstar = ((ra.digit << 8) | rb.digit) << (KB - 16);
          } else {
            kstar = (wbase + r.digit) << (KB - 16);
            need -= r.above;
          }
        }
        if constexpr (KB == 32) {
  #pragma unroll 1
          for (int j = 0; j < 2; ++j) {
            const int shift = 8 - 8 * j;
            CL.begin();
            uint32_t* h = CL.loc();
            const uint32_t pre = kstar >> (shift + 8);
            visit([&](uint32_t key, bool ok) {
              hist_add(h, (key >> shift) & 0xFFu, ok && (key >> (shift + 8)) == pre);
            });
            const LevelResult r = CL.finish<S>(lvl++, need);
            kstar |= r.digit << shift;
            need -= r.above;
          }
        }
      }
      const uint32_t r_ties = need;
      // Per vector, the row elements above K* (mg) and equal to it (mq) as bit
      // masks; every such element also reaches the threshold t. Elements outside
      // the row read as -inf, which can equal K*, so partly covered blocks are
      // masked to the row.
      auto kstar_masks = [&](const uint4& w, int64_t v, bool vok, uint32_t& mg, uint32_t& mq) {
        mg = 0u;
        mq = 0u;
        if (!vok) return;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const uint32_t key = key_of<ES>(elem_bits<ES>(w, e));
          mg |= static_cast<uint32_t>(key > kstar) << e;
          mq |= static_cast<uint32_t>(key == kstar) << e;
        }
        const int64_t e0 = v * VEC - lead;  // row index of the block's element 0
        if (e0 < 0 || e0 + VEC > p.len) {
          uint32_t inrow = 0u;
#pragma unroll
          for (int e = 0; e < VEC; ++e) inrow |= static_cast<uint32_t>(e0 + e >= 0 && e0 + e < p.len) << e;
          mg &= inrow;
          mq &= inrow;
        }
      };
      // The listed vectors of this warp, g(w, v, vok) for each, in list order.
      auto visit_vecs = [&](auto&& g) {
        if (gv == 1) {
          constexpr int UV = 4;
          for (int jb = 0; jb < lcnt; jb += 32 * UV) {
            uint4 w[UV];
            int64_t v[UV];
#pragma unroll
            for (int u = 0; u < UV; ++u) {
              const int j = jb + 32 * u + lane;
              v[u] = j < lcnt ? static_cast<int64_t>(vec_at(j)) : -1;
              w[u] = make_uint4(T::kNegInfWord, T::kNegInfWord, T::kNegInfWord, T::kNegInfWord);
              if (v[u] >= 0) w[u] = blk(v[u]);
            }
#pragma unroll
            for (int u = 0; u < UV; ++u) g(w[u], v[u], v[u] >= 0, jb + 32 * u + lane);
          }
          return;
        }
        if constexpr (!GV1) {
          for (int j = lane; j < lc; j += 32)
            for (int q = 0; q < gv; ++q) {
              const int64_t v = v0 + static_cast<int64_t>(wlist[j]) * gv + q;
              if (v < v1) g(blk(v), v, true, j);
            }
        }
      };
      // counts of this warp's list, then prefixes over warps and cluster CTAs
      uint32_t l_gt = 0, l_eq = 0;
      visit_vecs([&](const uint4& w, int64_t v, bool vok, int j) {
        uint32_t mg, mq;
        kstar_masks(w, v, vok, mg, mq);
        l_gt += __popc(mg);
        l_eq += __popc(mq);
        if (keep_masks && vok) vmask[j] = static_cast<uint16_t>(mg | (mq << 8));
      });
      const uint32_t c_gt = warp_sum(l_gt), c_eq = warp_sum(l_eq);
      if (lane == 0) {
        wtot[warp] = c_gt;
        wtot[kWarps + warp] = c_eq;
      }
      __syncthreads();
      uint32_t base_gt = 0, base_eq = 0, cta_gt = 0, cta_eq = 0;
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t tg = wtot[w], te = wtot[kWarps + w];
        if (w < warp) {
          base_gt += tg;
          base_eq += te;
        }
        cta_gt += tg;
        cta_eq += te;
      }
      if constexpr (S > 1) {
        if (tid > rank && tid < S) {  // push this CTA's counts to every later rank
          dsmem_red_add_u32(misc + kXpreGt, static_cast<uint32_t>(tid), cta_gt);
          dsmem_red_add_u32(misc + kXpreEq, static_cast<uint32_t>(tid), cta_eq);
        }
        cg::this_cluster().sync();
        base_gt += misc[kXpreGt];
        base_eq += misc[kXpreEq];
      }
      // write pass: one granule per lane, lanes in index order. Positions only
      // grow from base_gt + min(base_eq, r_ties): when that is already k, this
      // warp has nothing to write.
      const bool none_here = base_gt + min(base_eq, r_ties) >= k;
      // the value bits of K* itself, unless it is the key of zero (whose sign only
      // the input holds)
      uint32_t tie_bits = 0u;
      const bool tie_known = bits_of_key<ES>(kstar, &tie_bits);
      // writes the elements of masks mg / mq of vector v in index order, from the
      // lane's running positions bg (above K*) and bq (ties); values from w, or
      // (have_w false: ties only, with tie_known) the bits of K*
      auto put_masked = [&](const uint4& w, bool have_w, int64_t v, uint32_t mg, uint32_t mq, uint32_t& bg,
                            uint32_t& bq) {
        const int64_t e0 = v * VEC - lead;
        uint32_t m = mg | mq;
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          uint32_t pos = 0xFFFFFFFFu;
          if ((mg >> e) & 1u) {
            pos = bg + min(bq, r_ties);
            ++bg;
          } else {
            if (bq < r_ties) pos = bg + bq;
            ++bq;
          }
          if (pos < k) {
            put_index(p.out_indices, out_base + pos, e0 + e, p.idx64);
            if (out_val) out_val[pos] = static_cast<VT>(have_w ? elem_bits<ES>(w, e) : tie_bits);
          }
        }
      };
      if (gv == 1 && keep_masks) {
        // the masks kept by the count pass, 8 list entries per lane at a time; a
        // block is read again only for values above K* (or ties at the key of zero)
        constexpr int UM = 8;
        for (int jb = 0; jb < (none_here ? 0 : lcnt); jb += 32 * UM) {
          uint32_t mg[UM], mq[UM], sc[UM];
#pragma unroll
          for (int u = 0; u < UM; ++u) {
            const int j = jb + 32 * u + lane;
            const uint32_t m16 = j < lcnt ? vmask[j] : 0u;
            mg[u] = m16 & 0xFFu;
            mq[u] = m16 >> 8;
            sc[u] = static_cast<uint32_t>(__popc(mg[u])) | (static_cast<uint32_t>(__popc(mq[u])) << 16);
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int u = 0; u < UM; ++u) {
              const uint32_t t = __shfl_up_sync(kFull, sc[u], o);
              if (lane >= o) sc[u] += t;
            }
          }
#pragma unroll
          for (int u = 0; u < UM; ++u) {
            const uint32_t tot = __shfl_sync(kFull, sc[u], 31);
            uint32_t bg = base_gt + (sc[u] & 0xFFFFu) - static_cast<uint32_t>(__popc(mg[u]));
            uint32_t bq = base_eq + (sc[u] >> 16) - static_cast<uint32_t>(__popc(mq[u]));
            if ((mg[u] | mq[u]) != 0u && bg + min(bq, r_ties) < k) {
              const int64_t v = vec_at(jb + 32 * u + lane);
              const bool have_w = out_val != nullptr && (mg[u] != 0u || !tie_known);
              uint4 w = make_uint4(0u, 0u, 0u, 0u);
              if (have_w) w = blk(v);
              put_masked(w, have_w, v, mg[u], mq[u], bg, bq);
            }
            base_gt += tot & 0xFFFFu;
            base_eq += tot >> 16;
          }
          if (base_gt + min(base_eq, r_ties) >= k) break;
        }
      } else if (gv == 1) {
        // 4 listed vectors in flight per lane, one vector per lane at a time, in
        // list order; stop once every later output would land at or beyond k
        constexpr int UV = 4;
        for (int jb = 0; jb < (none_here ? 0 : lcnt); jb += 32 * UV) {
          uint4 w[UV];
          int64_t v[UV];
#pragma unroll
          for (int u = 0; u < UV; ++u) {
            const int j = jb + 32 * u + lane;
            v[u] = j < lcnt ? static_cast<int64_t>(vec_at(j)) : -1;
            w[u] = make_uint4(T::kNegInfWord, T::kNegInfWord, T::kNegInfWord, T::kNegInfWord);
            if (v[u] >= 0) w[u] = blk(v[u]);
          }
          // the UV vectors' counts (above | ties << 16: at most 256 each over the
          // warp) scanned over the lanes side by side; positions follow list order,
          // all lanes' vector u before their vector u + 1
          uint32_t mg[UV], mq[UV], sc[UV];
#pragma unroll
          for (int u = 0; u < UV; ++u) {
            kstar_masks(w[u], v[u], v[u] >= 0, mg[u], mq[u]);
            sc[u] = static_cast<uint32_t>(__popc(mg[u])) | (static_cast<uint32_t>(__popc(mq[u])) << 16);
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int u = 0; u < UV; ++u) {
              const uint32_t t = __shfl_up_sync(kFull, sc[u], o);
              if (lane >= o) sc[u] += t;
            }
          }
#pragma unroll
          for (int u = 0; u < UV; ++u) {
            const uint32_t tot = __shfl_sync(kFull, sc[u], 31);
            uint32_t bg = base_gt + (sc[u] & 0xFFFFu) - static_cast<uint32_t>(__popc(mg[u]));
            uint32_t bq = base_eq + (sc[u] >> 16) - static_cast<uint32_t>(__popc(mq[u]));
            put_masked(w[u], true, v[u], mg[u], mq[u], bg, bq);
            base_gt += tot & 0xFFFFu;
            base_eq += tot >> 16;
          }
          if (base_gt + min(base_eq, r_ties) >= k) break;
        }
      } else {
        // one granule of gv vectors per lane: its counts first, so that positions
        // follow index order (granule by granule, then vector by vector)
        for (int j0 = 0; j0 < (none_here ? 0 : lc); j0 += 32) {
          const int j = j0 + lane;
          const int64_t vb = j < lc ? v0 + static_cast<int64_t>(wlist[j]) * gv : v1;
          uint32_t lg = 0, lq = 0;
          for (int q = 0; q < gv; ++q)
            if (vb + q < v1) {
              uint32_t mg, mq;
              kstar_masks(blk(vb + q), vb + q, true, mg, mq);
              lg += __popc(mg);
              lq += __popc(mq);
            }
          uint32_t bg = base_gt + warp_excl_scan(lg);
          uint32_t bq = base_eq + warp_excl_scan(lq);
          base_gt += warp_sum(lg);
          base_eq += warp_sum(lq);
          if (lg + lq != 0) {
            for (int q = 0; q < gv; ++q)
              if (vb + q < v1) {
                const uint4 w = blk(vb + q);
                uint32_t mg, mq;
                kstar_masks(w, vb + q, true, mg, mq);
                put_masked(w, true, vb + q, mg, mq, bg, bq);
              }
          }
          if (base_gt + min(base_eq, r_ties) >= k) break;  // warp-uniform
        }
      }
    }
    // the next row reuses every shared buffer; cluster peers may still read ours,
    // and the words they push into must be clear before anyone starts the next row
    if constexpr (S > 1) {
      __syncthreads();
      if (tid < 4) misc[kXmax + tid] = 0;
      cg::this_cluster().sync();
    } else {
      __syncthreads();
    }
  }
}

}  // namespace ds_topk_dev
