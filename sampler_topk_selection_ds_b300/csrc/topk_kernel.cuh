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
//  B   exact k-th key K* among the elements >= t: 8-bit radix levels from the
//      most significant digit (2 levels for bf16 keys, 4 for fp32), histograms
//      aggregated per warp with match.any and summed over the cluster through
//      distributed shared memory.
//  C   ordered compaction: every element with key > K*, plus the lowest-index
//      elements with key == K* until k are taken, written in ascending index
//      order (so sorted_index costs nothing).
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
  int32_t g_cap_pad;     // per-CTA granule array size (multiple of 8)
  int32_t cache_vecs;    // capacity of the shared-memory copy of listed granules (vectors)
  int32_t cand_cap;      // capacity of the dense candidate array (elements)
  int32_t k;
  int32_t return_value;
  void* out_values;
  int32_t* out_indices;
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

// Vector v of a row (elements [v*VEC, v*VEC+VEC)). Elements at or beyond len are
// not read; their lanes hold -inf (only maxima see them; every element pass
// also tests the index against len).
template <int ES>
__device__ __forceinline__ uint4 load_vec(const char* rowp, int64_t v, int64_t len) {
  constexpr int VEC = Traits<ES>::kVec;
  const int64_t e0 = v * VEC;
  if (e0 + VEC <= len) return ld_nc_v4(rowp + v * 16);
  uint32_t w[4] = {Traits<ES>::kNegInfWord, Traits<ES>::kNegInfWord, Traits<ES>::kNegInfWord,
                   Traits<ES>::kNegInfWord};
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    if (e0 + e < len) {
      if constexpr (ES == 2) {
        const uint32_t h = *reinterpret_cast<const uint16_t*>(rowp + (e0 + e) * 2);
        const int sh = (e & 1) * 16;
        w[e >> 1] = (w[e >> 1] & ~(0xFFFFu << sh)) | (h << sh);
      } else {
        w[e] = *reinterpret_cast<const uint32_t*>(rowp + (e0 + e) * 4);
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
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

// Sum of a shared u32 over the cluster (after a row_sync made it visible).
template <int S>
__device__ __forceinline__ uint32_t cluster_sum(const uint32_t* w) {
  if constexpr (S > 1) {
    uint32_t t = 0;
#pragma unroll 1
    for (int r = 0; r < S; ++r) t += dsmem_ld_u32(w, static_cast<uint32_t>(r));
    return t;
  } else {
    return *w;
  }
}

struct LevelResult {
  uint32_t digit;  // bin holding the need-th largest key
  uint32_t above;  // keys above that bin (including the window's overflow count)
  bool found;      // false: fewer than `need` keys in the window and above it
  bool shift;      // true: the need-th largest key lies above the window
};

// Completes one histogram level: makes every CTA's histogram h (256 bins) and
// overflow count *ov (keys above the window) visible, sums them over the
// cluster, and locates the bin d with  ov + sum(h[> d]) < need <= ov + sum(h[>= d]).
template <int S>
__device__ __forceinline__ LevelResult finish_level(uint32_t* h, uint32_t* ov, uint32_t* hsum,
                                                    uint32_t* bc, uint32_t need) {
  row_sync<S>();
  const int tid = threadIdx.x;
  if (tid < kRadix) {
    uint32_t s = 0;
    if constexpr (S > 1) {
#pragma unroll 4
      for (int r = 0; r < S; ++r) s += dsmem_ld_u32(h + tid, static_cast<uint32_t>(r));
    } else {
      s = h[tid];
    }
    hsum[tid] = s;
  }
  const uint32_t over = cluster_sum<S>(ov);
  __syncthreads();
  if (tid < 32 && over < need) {
    const int lane = tid;
    const uint32_t n2 = need - over;
    const uint4 c0 = reinterpret_cast<const uint4*>(hsum)[lane * 2];
    const uint4 c1 = reinterpret_cast<const uint4*>(hsum)[lane * 2 + 1];
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
  return r;
}

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

// Shared-memory footprint of one CTA (bytes) for a plan.
__host__ __device__ constexpr int64_t smem_bytes(int64_t g_cap_pad, int64_t cache_vecs,
                                                 int64_t cand_cap) {
  return g_cap_pad * 2 * 2 + (3 * kRadix + kMiscWords) * 4 + cache_vecs * 16 + cand_cap * 8 +
         ((cache_vecs + 15) & ~int64_t(15));
}

// Threshold reuse across rows: a persistent CTA (or cluster) first tries the
// previous row's threshold lowered by this many top-16 key units; the guess is
// kept only if it provably holds for the new row (at least k granule maxima
// reach it) and is not too loose (at most max(2k, k + 1024) of them do).
constexpr uint32_t kGuessMargin = 4;

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// The listed granules' vectors, read either from the CTA's shared-memory copy
// (when they fit) or again from global memory (L2).
template <int ES>
struct ListedVectors {
  const char* rowp;
  const uint4* cache;
  const uint16_t* list;
  int64_t v0, v1, len;
  int gv;
  bool cached;

  // q-th vector of the li-th listed granule; v = its vector index in the row.
  __device__ __forceinline__ uint4 get(int li, int q, int64_t& v, bool& valid) const {
    v = v0 + static_cast<int64_t>(list[li]) * gv + q;
    valid = v < v1;
    if (cached) return cache[li * gv + q];
    if (valid) return load_vec<ES>(rowp, v, len);
    return make_uint4(Traits<ES>::kNegInfWord, Traits<ES>::kNegInfWord, Traits<ES>::kNegInfWord,
                      Traits<ES>::kNegInfWord);
  }
};

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

// Bit e set iff element e of the vector is a candidate: not below the
// threshold value, or NaN (unordered comparison), so a granule whose maximum
// reaches the threshold always contributes at least one candidate.
template <int ES>
__device__ __forceinline__ uint32_t cand_mask(const uint4& w, float tval) {
  uint32_t m = 0;
  if constexpr (ES == 2) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m |= static_cast<uint32_t>(!(__uint_as_float(ws[j] << 16) < tval)) << (2 * j);
      m |= static_cast<uint32_t>(!(__uint_as_float(ws[j] & 0xFFFF0000u) < tval)) << (2 * j + 1);
    }
  } else {
    m = static_cast<uint32_t>(!(__uint_as_float(w.x) < tval)) |
        static_cast<uint32_t>(!(__uint_as_float(w.y) < tval)) << 1 |
        static_cast<uint32_t>(!(__uint_as_float(w.z) < tval)) << 2 |
        static_cast<uint32_t>(!(__uint_as_float(w.w) < tval)) << 3;
  }
  return m;
}

// 8 consecutive u16 granule maxima starting at `base` (a multiple of 8).
__device__ __forceinline__ void load_m8(const uint16_t* M, int base, uint32_t m[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(M + base);
  m[0] = q.x & 0xFFFFu; m[1] = q.x >> 16;
  m[2] = q.y & 0xFFFFu; m[3] = q.y >> 16;
  m[4] = q.z & 0xFFFFu; m[5] = q.z >> 16;
  m[6] = q.w & 0xFFFFu; m[7] = q.w >> 16;
}

// Bit e set iff M[base+e] >= t16 and base+e < end.
__device__ __forceinline__ uint32_t m8_mask(const uint16_t* M, int base, int end, uint32_t t16) {
  if (base >= end) return 0u;
  uint32_t m[8];
  load_m8(M, base, m);
  uint32_t mask = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) mask |= static_cast<uint32_t>(base + e < end && m[e] >= t16) << e;
  return mask;
}

// misc[] layout (u32 words)
constexpr int kBc = 0;        // [0..2] level result: digit, above, found
constexpr int kXchg = 4;      // [4..7] cluster exchange: gt, eq, granule count, max key
constexpr int kOver = 8;      // [8..9] per-parity overflow counters of windowed levels
constexpr int kWtot = 16;     // [16..16+2*kWarps) per-warp totals

template <int ES, int S>
__global__ void __launch_bounds__(kThreads, 3) topk_rows_kernel(const Params p) {
  using T = Traits<ES>;
  constexpr int VEC = T::kVec;
  constexpr int KB = T::kKeyBits;
  constexpr uint32_t kFull = 0xFFFFFFFFu;
  static_assert(kWtot + 2 * kWarps <= kMiscWords, "misc layout");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* M = reinterpret_cast<uint16_t*>(smem_raw);
  uint16_t* list = M + p.g_cap_pad;
  uint32_t* hist = reinterpret_cast<uint32_t*>(list + p.g_cap_pad);  // 2 x kRadix
  uint32_t* hsum = hist + 2 * kRadix;                                 // kRadix
  uint32_t* misc = hsum + kRadix;                                     // kMiscWords
  uint32_t* bc = misc + kBc;
  uint32_t* xchg = misc + kXchg;
  uint32_t* wtot = misc + kWtot;
  uint4* cache = reinterpret_cast<uint4*>(misc + kMiscWords);         // cache_vecs
  uint32_t* craw = reinterpret_cast<uint32_t*>(cache + p.cache_vecs); // cand_cap raw bits
  uint32_t* cidx = craw + p.cand_cap;                                 // cand_cap indices
  uint8_t* vmask = reinterpret_cast<uint8_t*>(cidx + p.cand_cap);     // cache_vecs masks

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t lt_mask = lanemask_lt();
  int rank = 0;
  if constexpr (S > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
  const int64_t v0 = rank * p.vec_per_cta;
  const int64_t v1 = min(v0 + p.vec_per_cta, p.nvec);
  const int64_t nv = v1 > v0 ? v1 - v0 : 0;
  const int gv = p.gv;
  const int G = static_cast<int>((nv + gv - 1) / gv);
  const uint32_t k = static_cast<uint32_t>(p.k);
  const int64_t row_step = gridDim.x / S;
  // warp segments of the granule array, 256 granules (8 per lane) per step
  const int segm = ((G + kWarps - 1) / kWarps + 255) & ~255;
  const int sb = min(warp * segm, G);
  const int se = min(sb + segm, G);

  bool have_guess = false;
  uint32_t t_guess = 0;

#pragma unroll 1
  for (int64_t row = blockIdx.x / S; row < p.batch; row += row_step) {
    const char* rowp = p.x + row * p.row_stride_bytes;
    if (tid == 0) {  // level results start defined even if a NaN row breaks the counts
      bc[0] = 0;
      bc[1] = 0;
      bc[2] = 0;
    }

    // ---- P1: granule maxima + NaN test ------------------------------------------
    uint32_t nan_acc = T::kNegInfWord;  // NaN-propagating running max of everything seen
    uint32_t mmax = 0;                  // largest granule key seen by this thread
    if (gv == 1) {
      // vectors entirely inside [0, len) take the batched 16-byte path; the one
      // ragged vector at the end of the row (if any) is read element by element.
      const int64_t full_end = min(v1, max(v0, p.len / VEC));
      const int Gf = static_cast<int>(full_end - v0);
      constexpr int U = 8;
      const uint4* base = reinterpret_cast<const uint4*>(rowp) + v0;
      for (int g0 = tid; g0 < Gf; g0 += kThreads * U) {
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * kThreads;
          if (g < Gf) w[u] = ld_nc_v4(base + g);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int g = g0 + u * kThreads;
          if (g < Gf) {
            const uint32_t acc = max_acc<ES>(T::kNegInfWord, w[u]);
            nan_acc = max_packed<ES>(nan_acc, acc);
            const uint32_t mk = key_of<ES>(finish_max<ES>(acc)) >> (KB - 16);
            mmax = max(mmax, mk);
            M[g] = static_cast<uint16_t>(mk);
          }
        }
      }
      if (tid == 0 && Gf < G) {
        const uint32_t acc = max_acc<ES>(T::kNegInfWord, load_vec<ES>(rowp, full_end, p.len));
        nan_acc = max_packed<ES>(nan_acc, acc);
        const uint32_t mk = key_of<ES>(finish_max<ES>(acc)) >> (KB - 16);
        mmax = max(mmax, mk);
        M[Gf] = static_cast<uint16_t>(mk);
      }
    } else {
      for (int g = tid; g < G; g += kThreads) {
        const int64_t vb = v0 + static_cast<int64_t>(g) * gv;
        const int64_t ve = min(vb + gv, v1);
        uint32_t acc = T::kNegInfWord;
        for (int64_t v = vb; v < ve; ++v) acc = max_acc<ES>(acc, load_vec<ES>(rowp, v, p.len));
        nan_acc = max_packed<ES>(nan_acc, acc);
        const uint32_t mk = key_of<ES>(finish_max<ES>(acc)) >> (KB - 16);
        mmax = max(mmax, mk);
        M[g] = static_cast<uint16_t>(mk);
      }
    }
    mmax = __reduce_max_sync(kFull, mmax);
    if (lane == 0) wtot[warp] = mmax;
    if (__syncthreads_or(is_nan_bits<ES>(finish_max<ES>(nan_acc))) && tid == 0)
      atomicOr(p.flag, DS_TOPK_FLAG_NAN);
    mmax = 0;
    for (int w = 0; w < kWarps; ++w) mmax = max(mmax, wtot[w]);

    // ---- A: safe threshold t16 (at least k granule maxima reach it) -----------------
    int lvl = 0;
    uint32_t t16 = 0;
    bool accepted = false;
    if (have_guess) {
      t16 = t_guess;
      uint32_t wcount = 0;
      for (int b0 = sb; b0 < se; b0 += 256) wcount += __popc(m8_mask(M, b0 + lane * 8, se, t16));
      wcount = warp_sum(wcount);
      __syncthreads();  // wtot (warp maxima) read by everyone
      if (lane == 0) wtot[warp] = wcount;
      __syncthreads();
      uint32_t total = 0;
      for (int w = 0; w < kWarps; ++w) total += wtot[w];
      if constexpr (S > 1) {
        if (tid == 0) xchg[2] = total;
        cg::this_cluster().sync();
        total = cluster_sum<S>(xchg + 2);
      }
      const uint32_t cap = max(2u * k, k + 1024u);
      accepted = total >= k && total <= cap;
    }
    if (!accepted && p.g_total >= static_cast<int64_t>(k)) {
      // the k-th largest granule maximum, from a histogram over the 256 key
      // values just below the row's largest granule maximum
      if constexpr (S > 1) {
        if (tid == 0) xchg[3] = mmax;
        cg::this_cluster().sync();
#pragma unroll 1
        for (int r = 0; r < S; ++r) mmax = max(mmax, dsmem_ld_u32(xchg + 3, static_cast<uint32_t>(r)));
      }
      const uint32_t wbase = mmax > 255u ? mmax - 255u : 0u;
      uint32_t* h = hist + (lvl & 1) * kRadix;
      uint32_t* ov = misc + kOver + (lvl & 1);
      if (tid < kRadix) h[tid] = 0;
      if (tid == 0) *ov = 0;
      __syncthreads();
      for (int b0 = sb; b0 < se; b0 += 256) {
        const int base = b0 + lane * 8;
        if (base < se) {
          uint32_t m[8];
          load_m8(M, base, m);
#pragma unroll
          for (int e = 0; e < 8; ++e) hist_add(h, m[e] - wbase, base + e < se && m[e] >= wbase);
        }
      }
      LevelResult r = finish_level<S>(h, ov, hsum, bc, k);
      ++lvl;
      if (r.found) {
        t16 = wbase + r.digit;
      } else {
        // fewer than k maxima within 256 keys of the largest: two 8-bit levels
        h = hist + (lvl & 1) * kRadix;
        ov = misc + kOver + (lvl & 1);
        if (tid < kRadix) h[tid] = 0;
        if (tid == 0) *ov = 0;
        __syncthreads();
        for (int b0 = sb; b0 < se; b0 += 256) {
          const int base = b0 + lane * 8;
          if (base < se) {
            uint32_t m[8];
            load_m8(M, base, m);
#pragma unroll
            for (int e = 0; e < 8; ++e) hist_add(h, m[e] >> 8, base + e < se);
          }
        }
        const LevelResult r1 = finish_level<S>(h, ov, hsum, bc, k);
        ++lvl;
        const uint32_t d1 = r1.digit, a1 = r1.above;
        h = hist + (lvl & 1) * kRadix;
        ov = misc + kOver + (lvl & 1);
        if (tid < kRadix) h[tid] = 0;
        if (tid == 0) *ov = 0;
        __syncthreads();
        for (int b0 = sb; b0 < se; b0 += 256) {
          const int base = b0 + lane * 8;
          if (base < se) {
            uint32_t m[8];
            load_m8(M, base, m);
#pragma unroll
            for (int e = 0; e < 8; ++e) hist_add(h, m[e] & 0xFFu, base + e < se && (m[e] >> 8) == d1);
          }
        }
        const LevelResult r2 = finish_level<S>(h, ov, hsum, bc, k - a1);
        ++lvl;
        t16 = (d1 << 8) | r2.digit;
      }
      t_guess = t16 > 0x0080u + kGuessMargin ? t16 - kGuessMargin : 0u;
      have_guess = true;
    } else if (!accepted) {
      t16 = 0;  // fewer granules than k: every element is a candidate
    }

    // ---- L: ordered list of granules whose maximum reaches t16 ---------------------
    uint32_t wcount = 0;
    for (int b0 = sb; b0 < se; b0 += 256) wcount += __popc(m8_mask(M, b0 + lane * 8, se, t16));
    wcount = warp_sum(wcount);
    __syncthreads();  // wtot may still be read above
    if (lane == 0) wtot[warp] = wcount;
    __syncthreads();
    int nlist = 0;
    {
      uint32_t off = 0;
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = wtot[w];
        if (w < warp) off += t;
        nlist += static_cast<int>(t);
      }
      for (int b0 = sb; b0 < se; b0 += 256) {
        const int base = b0 + lane * 8;
        uint32_t mask = m8_mask(M, base, se, t16);
        const uint32_t c = __popc(mask);
        uint32_t pos = off + warp_excl_scan(c);
        off += warp_sum(c);
        while (mask) {
          const int e = __ffs(mask) - 1;
          mask &= mask - 1;
          list[pos++] = static_cast<uint16_t>(base + e);
        }
      }
    }
    __syncthreads();

    // ---- copy the listed granules into shared memory when they fit -------------------
    ListedVectors<ES> src;
    src.rowp = rowp;
    src.cache = cache;
    src.list = list;
    src.v0 = v0;
    src.v1 = v1;
    src.len = p.len;
    src.gv = gv;
    src.cached = static_cast<int64_t>(nlist) * gv <= p.cache_vecs;
    if (src.cached) {
      const int nvecs = nlist * gv;
      for (int i = tid; i < nvecs; i += kThreads) {
        int li = i, q = 0;
        if (gv > 1) {
          li = i / gv;
          q = i - li * gv;
        }
        const int64_t v = v0 + static_cast<int64_t>(list[li]) * gv + q;
        if (v < v1 && (v + 1) * VEC <= p.len) {
          cp_async_16(&cache[i], rowp + v * 16);
        } else {
          // ragged or absent vector: lanes outside [0, len) hold a NaN pattern and
          // are masked off by index in the candidate test below
          uint32_t wv[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
          if (v < v1) {
            const uint4 f = load_vec<ES>(rowp, v, p.len);
            const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (v * VEC + e < p.len) {
                if constexpr (ES == 2) {
                  const int sh = (e & 1) * 16;
                  wv[e >> 1] = (wv[e >> 1] & ~(0xFFFFu << sh)) | (fw[e >> 1] & (0xFFFFu << sh));
                } else {
                  wv[e] = fw[e];
                }
              }
            }
          }
          cache[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
      cp_async_wait_all();
      __syncthreads();
    }

    const uint32_t T_full = (KB == 16) ? t16 : (t16 << 16);
    const float tval = key_threshold_value<ES>(T_full);
    // Each warp owns a contiguous, index-ordered segment of the list.
    const int segl = round_up32((nlist + kWarps - 1) / kWarps);
    const int lb = min(warp * segl, nlist);
    const int le = min(lb + segl, nlist);

    // ---- D: dense, index-ordered array of the candidates -----------------------------
    // Candidate = key >= t or NaN. Built from the shared-memory copy with fp32
    // comparisons against the threshold's value (bf16 widens exactly); the
    // per-vector candidate masks are kept so the write pass does not retest.
    bool dense = src.cached;
    int ncand = 0;
    if (dense) {
      uint32_t wc = 0;
      for (int i = lb + lane; i < le; i += 32) {
        for (int q = 0; q < gv; ++q) {
          const int ci = i * gv + q;
          const int64_t v = v0 + static_cast<int64_t>(list[i]) * gv + q;
          uint32_t m = cand_mask<ES>(cache[ci], tval);
          if ((v + 1) * VEC > p.len) {  // ragged last vector of the row (or past it)
            const int64_t valid = v * VEC < p.len ? p.len - v * VEC : 0;
            m &= (1u << valid) - 1u;
          }
          vmask[ci] = static_cast<uint8_t>(m);
          wc += __popc(m);
        }
      }
      wc = warp_sum(wc);
      if (lane == 0) wtot[kWarps + warp] = wc;
      __syncthreads();
      uint32_t base = 0;
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = wtot[kWarps + w];
        if (w < warp) base += t;
        ncand += static_cast<int>(t);
      }
      dense = ncand <= p.cand_cap;
      if (dense) {
        for (int i0 = lb; i0 < le; i0 += 32) {
          const int i = i0 + lane;
          uint32_t c = 0;
          if (i < le)
            for (int q = 0; q < gv; ++q) c += __popc(vmask[i * gv + q]);
          uint32_t pos = base + warp_excl_scan(c);
          base += warp_sum(c);
          if (c == 0) continue;
          const int64_t vg = v0 + static_cast<int64_t>(list[i]) * gv;
          for (int q = 0; q < gv; ++q) {
            const int ci = i * gv + q;
            uint32_t m = vmask[ci];
            const uint32_t ibase = static_cast<uint32_t>((vg + q) * VEC);
            while (m) {
              const int e = __ffs(m) - 1;
              m &= m - 1;
              if constexpr (ES == 2) {
                craw[pos] = reinterpret_cast<const uint16_t*>(cache + ci)[e];
              } else {
                craw[pos] = reinterpret_cast<const uint32_t*>(cache + ci)[e];
              }
              cidx[pos] = ibase + e;
              ++pos;
            }
          }
        }
      }
      __syncthreads();  // candidates visible; wtot free again
    }

    // ---- B: exact k-th key among the candidates ---------------------------------------
    // visit(f): calls f(key, valid) for every candidate, warp-uniformly.
    auto visit = [&](auto&& f) {
      if (dense) {
        const int nw = round_up32(ncand);
        for (int c = tid; c < nw; c += kThreads) {
          const bool ok = c < ncand;
          f(key_of<ES>(ok ? craw[c] : 0u), ok);
        }
      } else {
        const int nw = round_up32(nlist);
        for (int i = tid; i < nw; i += kThreads) {
          const bool gok = i < nlist;
          for (int q = 0; q < gv; ++q) {
            int64_t v = 0;
            bool vok = false;
            uint4 w = make_uint4(T::kNegInfWord, T::kNegInfWord, T::kNegInfWord, T::kNegInfWord);
            if (gok) w = src.get(i, q, v, vok);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const uint32_t eb = elem_bits<ES>(w, e);
              const uint32_t key = key_of<ES>(eb);
              f(key, vok && (v * VEC + e < p.len) && (key >= T_full || is_nan_bits<ES>(eb)));
            }
          }
        }
      }
    };

    // Windowed level on the top 16 key bits: bins [wbase, wbase + 256), keys above
    // the window counted apart. The window starts at t16 (every candidate except a
    // NaN is at or above it) and moves up until it holds the k-th largest.
    uint32_t need = k, cnt_gt = 0, kstar = 0;
    {
      uint32_t wbase = t16;
#pragma unroll 1
      while (true) {
        uint32_t* h = hist + (lvl & 1) * kRadix;
        uint32_t* ov = misc + kOver + (lvl & 1);
        if (tid < kRadix) h[tid] = 0;
        if (tid == 0) *ov = 0;
        __syncthreads();
        uint32_t lover = 0;
        visit([&](uint32_t key, bool ok) {
          const uint32_t k16v = key >> (KB - 16);
          ok = ok && k16v >= wbase;
          const uint32_t d = k16v - wbase;
          hist_add(h, d, ok && d < 256u);
          lover += __popc(__ballot_sync(kFull, ok && d >= 256u));
        });
        if (lane == 0 && lover) atomicAdd(ov, lover);
        const LevelResult r = finish_level<S>(h, ov, hsum, bc, need);
        ++lvl;
        if (r.shift && wbase + 256u <= 0xFFFFu) {
          wbase += 256u;
          continue;
        }
        kstar = (wbase + r.digit) << (KB - 16);
        cnt_gt += r.above;
        need -= r.above;
        break;
      }
    }
    if constexpr (KB == 32) {
      // the low 16 bits of K*: two 8-bit levels among candidates with its top 16 bits
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        const int shift = 8 - 8 * j;
        uint32_t* h = hist + (lvl & 1) * kRadix;
        uint32_t* ov = misc + kOver + (lvl & 1);
        if (tid < kRadix) h[tid] = 0;
        if (tid == 0) *ov = 0;
        __syncthreads();
        const uint32_t pre = kstar >> (shift + 8);
        visit([&](uint32_t key, bool ok) {
          hist_add(h, (key >> shift) & 0xFFu, ok && (key >> (shift + 8)) == pre);
        });
        const LevelResult r = finish_level<S>(h, ov, hsum, bc, need);
        ++lvl;
        kstar |= r.digit << shift;
        cnt_gt += r.above;
        need -= r.above;
      }
    }
    const uint32_t r_ties = need;    // how many elements equal to K* are taken
    const uint32_t k16 = kstar >> (KB - 16);

    // ---- C: ordered compaction of the selected elements -------------------------------
    // Counts per warp segment, prefix over warps (and over the cluster's CTAs), then
    // every selected element is written at (#selected elements before it).
    const int segc = round_up32((ncand + kWarps - 1) / kWarps);
    const int cb = dense ? min(warp * segc, ncand) : lb;
    const int ce = dense ? min(cb + segc, ncand) : le;
    uint32_t c_gt = 0, c_eq = 0;
    if (dense) {
      for (int c0 = cb; c0 < ce; c0 += 32) {
        const int c = c0 + lane;
        const uint32_t key = key_of<ES>(c < ce ? craw[c] : 0u);
        c_gt += __popc(__ballot_sync(kFull, c < ce && key > kstar));
        c_eq += __popc(__ballot_sync(kFull, c < ce && key == kstar));
      }
    } else {
      for (int i = lb + lane; i < le; i += 32) {
        if (M[list[i]] < k16) continue;
        for (int q = 0; q < gv; ++q) {
          int64_t v;
          bool vok;
          const uint4 w = src.get(i, q, v, vok);
          if (!vok) continue;
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const uint32_t eb = elem_bits<ES>(w, e);
            const uint32_t key = key_of<ES>(eb);
            if (v * VEC + e < p.len && (key >= T_full || is_nan_bits<ES>(eb))) {
              c_gt += key > kstar;
              c_eq += key == kstar;
            }
          }
        }
      }
      c_gt = warp_sum(c_gt);
      c_eq = warp_sum(c_eq);
    }
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
      if (tid == 0) {
        xchg[0] = cta_gt;
        xchg[1] = cta_eq;
      }
      cg::this_cluster().sync();
#pragma unroll 1
      for (int r = 0; r < rank; ++r) {
        base_gt += dsmem_ld_u32(xchg, static_cast<uint32_t>(r));
        base_eq += dsmem_ld_u32(xchg + 1, static_cast<uint32_t>(r));
      }
    }

    int32_t* out_idx = p.out_indices + row * static_cast<int64_t>(k);
    using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
    VT* out_val = p.return_value ? reinterpret_cast<VT*>(p.out_values) + row * static_cast<int64_t>(k) : nullptr;
    if (dense) {
      for (int c0 = cb; c0 < ce; c0 += 32) {
        const int c = c0 + lane;
        const bool ok = c < ce;
        const uint32_t bits = ok ? craw[c] : 0u;
        const uint32_t key = key_of<ES>(bits);
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
          out_idx[pos] = static_cast<int32_t>(cidx[c]);
          if (out_val) out_val[pos] = static_cast<VT>(bits);
        }
      }
    } else {
      for (int i0 = lb; i0 < le; i0 += 32) {
        const int i = i0 + lane;
        const bool live = i < le && M[list[i < le ? i : lb]] >= k16;
        uint32_t lg = 0, lq = 0;
        if (live) {
          for (int q = 0; q < gv; ++q) {
            int64_t v;
            bool vok;
            const uint4 w = src.get(i, q, v, vok);
            if (!vok) continue;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const uint32_t eb = elem_bits<ES>(w, e);
              const uint32_t key = key_of<ES>(eb);
              if (v * VEC + e < p.len && (key >= T_full || is_nan_bits<ES>(eb))) {
                lg += key > kstar;
                lq += key == kstar;
              }
            }
          }
        }
        uint32_t bg = base_gt + warp_excl_scan(lg);
        uint32_t bq = base_eq + warp_excl_scan(lq);
        base_gt += warp_sum(lg);
        base_eq += warp_sum(lq);
        if (lg + lq == 0) continue;
        for (int q = 0; q < gv; ++q) {
          int64_t v;
          bool vok;
          const uint4 w = src.get(i, q, v, vok);
          if (!vok) continue;
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const int64_t idx = v * VEC + e;
            const uint32_t bits = elem_bits<ES>(w, e);
            const uint32_t key = key_of<ES>(bits);
            if (idx < p.len && (key >= T_full || is_nan_bits<ES>(bits))) {
              uint32_t pos = 0xFFFFFFFFu;
              if (key > kstar) {
                pos = bg + min(bq, r_ties);
                ++bg;
              } else if (key == kstar) {
                if (bq < r_ties) pos = bg + bq;
                ++bq;
              }
              if (pos < k) {
                out_idx[pos] = static_cast<int32_t>(idx);
                if (out_val) out_val[pos] = static_cast<VT>(bits);
              }
            }
          }
        }
      }
    }
    // the next row reuses every shared buffer; cluster peers may still read xchg
    if constexpr (S > 1) {
      cg::this_cluster().sync();
    } else {
      __syncthreads();
    }
  }
}

}  // namespace ds_topk_dev
