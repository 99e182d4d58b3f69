// unaligned_kernel.cuh — TopK of rows that do not start on a 16-byte boundary
// (x only element-aligned, or row_stride * sizeof(dtype) not a multiple of 16).
//
// The other paths read a row with 16-byte loads or bulk copies starting at its
// first element, so they need every row to start on a 16-byte boundary. The
// pages' kernel asks the same of its callers (they may pad the rows); this path
// takes such rows as they are. One CTA handles one row at a time and reads it
// through the 16-byte aligned vectors that overlap it: a vector that lies wholly
// inside the row is one 16-byte load, and the at most two vectors that straddle
// the row's ends are read element by element at in-row columns only. No byte
// outside the row's [0, len) is read.
//
// Per row:
//  G  threshold guess t: the previous row's k-th key less a margin (a CTA walks
//     rows with a stride), or, for a CTA's first row, a key near the
//     (1.5 k f + 16)-th largest of a strided sample holding a fraction f of the row.
//  F  filter pass: vectors whose maximum (NaN-propagating, so every NaN is seen)
//     is below t are skipped; keys >= t are appended to a shared-memory candidate
//     buffer and counted. If at least k and at most `cap` keys reach t, the k-th
//     key lies among the candidates.
//  R  exact radix select on the order key, most significant 8-bit digit first:
//     each level builds a 256-bin histogram of the next digit over the keys whose
//     higher digits equal the prefix found so far, and picks the bin holding the
//     kr-th largest (kr starts at k and loses the count of every bin above the
//     chosen one). It stops when the chosen bin is taken whole (every key >=
//     prefix << shift is selected) or at the last digit (the prefix is the k-th
//     key K* and kr of its ties are taken). R runs over the candidates, or over
//     the whole row when the guess failed (too few or too many candidates).
//  C  ordered compaction: keys above the threshold, and the lowest-index ties
//     until k are taken, written in ascending index order (vectors whose maximum
//     is below the threshold are skipped).
//
// Sources: deepseek-v4-pro.uk (zh-tw), "深入 DeepSeek V4.1 全新開放推論工具包",
// section "DeepSelect：快速且刻意狹義的 TopK": rows need a specific alignment and
// callers may pad them (this path removes the need); deepseek.csdn.net,
// "DeepSeek 一次开源三个仓库", section 三 (算子层): the top-K of each row by a
// threshold filter into a candidate buffer and a compaction to K.
#pragma once

#include "topk_kernel.cuh"

namespace ds_topk_dev {

constexpr int kUaThreads = 512;      // threads per CTA (>= 256: one per histogram bin)
constexpr int kUaWarps = kUaThreads / 32;
constexpr int kUaUnroll = 4;         // vectors in flight per thread in a row pass
constexpr int kUaOutVecs = 4;        // consecutive vectors per thread in a compaction tile
constexpr int kUaSampleKeys = 8192;  // most keys in a first-row sample (cap >= this)
constexpr int kUaGuessMargin = 6;    // previous-row guess: k-th key less 6 bf16 steps

struct UaParams {
  const char* x;
  int64_t batch;
  int64_t row_stride_bytes;
  int64_t len;
  int32_t k;
  int32_t cap;  // candidate slots in dynamic shared memory (uint32 keys), >= kUaSampleKeys
  int32_t return_value;
  void* out_values;
  void* out_indices;  // int32 or int64 (idx64)
  int32_t idx64;
  int32_t* flag;
};

struct UaShared {
  uint32_t hist[256];
  uint32_t tot[2][kUaWarps];  // per-warp scan totals (double-buffered)
  uint32_t bin, above, count;
  int nan;
};

// Aligned vector q of a row whose column 0 lies `lead` elements after the
// 16-byte boundary `abase`: lane e holds column q * VEC + e - lead. `valid` gets
// the lanes that are columns of the row; only those are read.
template <int ES>
__device__ __forceinline__ uint4 ua_load(const char* abase, int64_t q, int lead, int64_t len, uint32_t& valid) {
  constexpr int VEC = Traits<ES>::kVec;
  const int64_t c0 = q * VEC - lead;
  if (c0 >= 0 && c0 + VEC <= len) {
    valid = (1u << VEC) - 1u;
    return ld_nc_v4(abase + q * 16);
  }
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  valid = 0u;
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    const int64_t c = c0 + e;
    if (c >= 0 && c < len) {
      valid |= 1u << e;
      const char* ep = abase + (q * VEC + e) * ES;  // = column c of the row
      if constexpr (ES == 2) {
        w[e >> 1] |= static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(ep)) << ((e & 1) * 16);
      } else {
        w[e] = *reinterpret_cast<const uint32_t*>(ep);
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Order key of a full vector's largest element; a NaN anywhere gives the key of
// the canonical (positive) NaN, above every number's key.
template <int ES>
__device__ __forceinline__ uint32_t ua_vmax_key(const uint4& w) {
  if constexpr (ES == 2) {
    const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w));
    return max(key_of<2>(m & 0xFFFFu), key_of<2>(m >> 16));
  } else {
    return key_of<4>(f32_max_nan(f32_max_nan(w.x, w.y), f32_max_nan(w.z, w.w)));
  }
}

// The bin of sh.hist holding the kr-th largest key: thread t takes bin 255 - t,
// so an inclusive scan over t counts the keys in that bin and every bin above.
// Every thread gets the bin, the count above it and the count in it.
__device__ __forceinline__ void ua_pick(UaShared& sh, uint32_t kr, uint32_t& b, uint32_t& above, uint32_t& in_bin) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t h = 0u, s = 0u;
  if (tid < 256) {
    h = sh.hist[255 - tid];
    s = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += t;
    }
    if (lane == 31) sh.tot[0][warp] = s;
  }
  __syncthreads();
  if (tid < 256) {
    uint32_t a = s - h;
    for (int w2 = 0; w2 < warp; ++w2) a += sh.tot[0][w2];
    if (a < kr && kr <= a + h) {  // exactly one bin: the counts cover kr
      sh.bin = 255u - tid;
      sh.above = a;
    }
  }
  __syncthreads();
  b = sh.bin;
  above = sh.above;
  in_bin = sh.hist[b];
}

// Radix select of the kr-th largest key of a set, at most `levels` 8-bit levels
// from the top. accumulate(prefix, shift, first) adds to sh.hist the digit
// (key >> shift) & 255 of every key of the set whose digits above shift + 8
// equal prefix (every key when first). On return: prefix holds the digits
// found, kr the rank left among the keys sharing them, shift the last level's
// shift, and whole says that the last chosen bin is taken whole. Ends with a
// barrier, so sh may be reused at once.
template <int W, class Acc>
__device__ __forceinline__ void ua_radix(UaShared& sh, Acc&& accumulate, int levels, uint32_t& prefix,
                                         uint32_t& kr, int& shift, bool& whole) {
  prefix = 0u;
  whole = false;
  shift = W - 8;
  for (int l = 0; l < levels; ++l) {
    shift = W - 8 - 8 * l;
    for (int i = threadIdx.x; i < 256; i += kUaThreads) sh.hist[i] = 0u;
    __syncthreads();
    accumulate(prefix, shift, l == 0);
    __syncthreads();
    uint32_t b, above, in_bin;
    ua_pick(sh, kr, b, above, in_bin);
    kr -= above;
    prefix = (prefix << 8) | b;
    __syncthreads();  // sh.hist, sh.bin and sh.above are rewritten next
    if (in_bin == kr) {
      whole = true;
      return;
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kUaThreads, 2) topk_unaligned_kernel(const UaParams p) {
  constexpr int VEC = Traits<ES>::kVec;
  constexpr int W = Traits<ES>::kKeyBits;
  constexpr uint32_t kFull = (1u << VEC) - 1u;
  constexpr uint32_t kMargin = static_cast<uint32_t>(kUaGuessMargin) << (W - 16);
  using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
  __shared__ UaShared sh;
  extern __shared__ __align__(16) uint32_t cand[];  // p.cap keys
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t k = static_cast<uint32_t>(p.k);
  const uint32_t cap = static_cast<uint32_t>(p.cap);
  bool have_last = false;  // same value in every thread of the CTA
  uint32_t last_T = 0u;

  for (int64_t row = blockIdx.x; row < p.batch; row += gridDim.x) {
    const char* rowp = p.x + row * p.row_stride_bytes;
    const int lead = static_cast<int>((reinterpret_cast<uintptr_t>(rowp) & 15u) / ES);
    const char* abase = rowp - lead * ES;
    const int64_t nq = (lead + p.len + VEC - 1) / VEC;  // aligned vectors overlapping the row
    if (tid == 0) {
      sh.nan = 0;
      sh.count = 0u;
    }
    __syncthreads();

    // ---- G: threshold guess ----
    bool guess = false;
    uint32_t t = 0u;
    if (have_last) {
      guess = true;
      t = last_T > kMargin ? last_T - kMargin : 0u;
    } else {
      // strided sample of m full vectors (column 0 of vector q is q*VEC - lead)
      const int64_t q_lo = lead ? 1 : 0;
      const int64_t q_hi = (lead + p.len) / VEC;  // exclusive: vectors below it are full
      const int64_t nfull = q_hi - q_lo;
      const int64_t m = kUaSampleKeys / VEC;
      if (nfull >= 4 * m) {
        const uint32_t ns = static_cast<uint32_t>(m * VEC);
        // the q-th largest of the sample: about 1.5 k rows' worth, plus 16
        const uint32_t q = static_cast<uint32_t>((3 * static_cast<int64_t>(k) * ns) / (2 * p.len)) + 16u;
        if (q <= ns) {
          for (int64_t j = tid; j < m; j += kUaThreads) {
            const uint4 w = ld_nc_v4(abase + (q_lo + j * nfull / m) * 16);
#pragma unroll
            for (int e = 0; e < VEC; ++e) cand[j * VEC + e] = key_of<ES>(elem_bits<ES>(w, e));
          }
          __syncthreads();
          uint32_t prefix, kr = q;
          int shift;
          bool whole;
          ua_radix<W>(sh, [&](uint32_t pre, int sft, bool first) {
            for (uint32_t i = tid; i < ns; i += kUaThreads) {
              const uint32_t key = cand[i];
              if (first || (key >> (sft + 8)) == pre) atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
            }
          }, 2, prefix, kr, shift, whole);
          guess = true;
          t = prefix << shift;  // at most the sample's q-th largest key
        }
      }
    }

    // ---- F: filter pass, candidates >= t ----
    uint32_t T = 0u, r = 0u;
    bool exact = false;
    if (guess) {
      bool nan_seen = false;
      // the threshold as a value, for packed compares that mark a superset of the
      // elements with key >= t (every NaN included); each is then checked by key
      const float tval = key_threshold_value<ES>(t);
      const uint32_t tv2 = (__float_as_uint(tval) >> 16) * 0x00010001u;
      for (int64_t qb = 0; qb < nq; qb += static_cast<int64_t>(kUaThreads) * kUaUnroll) {
        uint4 w[kUaUnroll];
        uint32_t val[kUaUnroll];
#pragma unroll
        for (int u = 0; u < kUaUnroll; ++u) {
          const int64_t q = qb + u * kUaThreads + tid;
          val[u] = 0u;
          w[u] = make_uint4(0u, 0u, 0u, 0u);
          if (q < nq) w[u] = ua_load<ES>(abase, q, lead, p.len, val[u]);
        }
#pragma unroll
        for (int u = 0; u < kUaUnroll; ++u) {
          if (val[u] == 0u || (val[u] == kFull && ua_vmax_key<ES>(w[u]) < t)) continue;
          uint32_t m = cand_mask<ES>(w[u], tval, tv2) & val[u];
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1u;
            const uint32_t bits = elem_bits<ES>(w[u], e);
            nan_seen |= is_nan_bits<ES>(bits);
            const uint32_t key = key_of<ES>(bits);
            if (key >= t) {
              const uint32_t pos = atomicAdd(&sh.count, 1u);
              if (pos < cap) cand[pos] = key;
            }
          }
        }
      }
      if (nan_seen) sh.nan = 1;
      __syncthreads();
      const uint32_t n = sh.count;
      if (n >= k && n <= cap) {
        uint32_t prefix, kr = k;
        int shift;
        bool whole;
        ua_radix<W>(sh, [&](uint32_t pre, int sft, bool first) {
          for (uint32_t i = tid; i < n; i += kUaThreads) {
            const uint32_t key = cand[i];
            if (first || (key >> (sft + 8)) == pre) atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
          }
        }, W / 8, prefix, kr, shift, whole);
        // a bin taken whole holds only candidates: its keys below t are not selected
        T = whole ? max(prefix << shift, t) : prefix;
        r = whole ? 0xFFFFFFFFu : kr;
        exact = true;
      }
    }

    // ---- R over the whole row (no guess, or the guess missed) ----
    if (!exact) {
      uint32_t prefix, kr = k;
      int shift;
      bool whole;
      ua_radix<W>(sh, [&](uint32_t pre, int sft, bool first) {
        bool nan_seen = false;
        for (int64_t qb = 0; qb < nq; qb += static_cast<int64_t>(kUaThreads) * kUaUnroll) {
          uint4 w[kUaUnroll];
          uint32_t val[kUaUnroll];
#pragma unroll
          for (int u = 0; u < kUaUnroll; ++u) {
            const int64_t q = qb + u * kUaThreads + tid;
            val[u] = 0u;
            w[u] = make_uint4(0u, 0u, 0u, 0u);
            if (q < nq) w[u] = ua_load<ES>(abase, q, lead, p.len, val[u]);
          }
#pragma unroll
          for (int u = 0; u < kUaUnroll; ++u) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (!((val[u] >> e) & 1u)) continue;
              const uint32_t bits = elem_bits<ES>(w[u], e);
              const uint32_t key = key_of<ES>(bits);
              if (first) {
                nan_seen |= is_nan_bits<ES>(bits);
                atomicAdd(&sh.hist[key >> sft], 1u);
              } else if ((key >> (sft + 8)) == pre) {
                atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
              }
            }
          }
        }
        if (nan_seen) sh.nan = 1;
      }, W / 8, prefix, kr, shift, whole);
      T = whole ? prefix << shift : prefix;
      r = whole ? 0xFFFFFFFFu : kr;
    }
    if (tid == 0 && sh.nan) atomicOr(p.flag, DS_TOPK_FLAG_NAN);
    have_last = true;
    last_T = T;

    // ---- C: ordered compaction, keys > T, then ties == T by ascending index ----
    uint32_t base_gt = 0u, base_eq = 0u;
    const int64_t row_out = row * static_cast<int64_t>(k);
    VT* ov = p.return_value ? static_cast<VT*>(p.out_values) + row_out : nullptr;
    const float Tval = key_threshold_value<ES>(T);
    const uint32_t Tv2 = (__float_as_uint(Tval) >> 16) * 0x00010001u;
    int par = 0;
    for (int64_t tb = 0; tb < nq; tb += static_cast<int64_t>(kUaThreads) * kUaOutVecs, par ^= 1) {
      const int64_t q0 = tb + static_cast<int64_t>(tid) * kUaOutVecs;
      uint4 w[kUaOutVecs];
      uint32_t val[kUaOutVecs];
#pragma unroll
      for (int u = 0; u < kUaOutVecs; ++u) {
        val[u] = 0u;
        w[u] = make_uint4(0u, 0u, 0u, 0u);
        if (q0 + u < nq) {
          w[u] = ua_load<ES>(abase, q0 + u, lead, p.len, val[u]);
          if (val[u] == kFull && ua_vmax_key<ES>(w[u]) < T) val[u] = 0u;  // nothing selected here
          // from here on val[u] marks a superset of the lanes with key >= T
          if (val[u] != 0u) val[u] &= cand_mask<ES>(w[u], Tval, Tv2);
        }
      }
      uint32_t cg = 0u, ce = 0u;
#pragma unroll
      for (int u = 0; u < kUaOutVecs; ++u) {
        uint32_t m = val[u];
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          const uint32_t key = key_of<ES>(elem_bits<ES>(w[u], e));
          cg += key > T;
          ce += key == T;
        }
      }
      // block-wide exclusive scan of (cg, ce), packed in 16-bit halves (a tile
      // holds at most 512 * 4 * 8 = 16384 elements)
      const uint32_t v = cg | (ce << 16);
      uint32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t tt = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += tt;
      }
      if (lane == 31) sh.tot[par][warp] = incl;
      __syncthreads();
      uint32_t before = incl - v, tile = 0u;
#pragma unroll
      for (int w2 = 0; w2 < kUaWarps; ++w2) {
        const uint32_t tt = sh.tot[par][w2];
        if (w2 < warp) before += tt;
        tile += tt;
      }
      uint32_t gtb = base_gt + (before & 0xFFFFu), eqb = base_eq + (before >> 16);
      if (v != 0u) {
#pragma unroll
        for (int u = 0; u < kUaOutVecs; ++u) {
          uint32_t m = val[u];
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1u;
            const uint32_t bits = elem_bits<ES>(w[u], e);
            const uint32_t key = key_of<ES>(bits);
            const int64_t col = (q0 + u) * VEC + e - lead;
            int64_t pos = -1;
            if (key > T) {
              pos = gtb + min(eqb, r);
              ++gtb;
            } else if (key == T) {
              if (eqb < r) pos = gtb + eqb;
              ++eqb;
            }
            if (pos >= 0 && pos < k) {  // exactly k are selected; the bound keeps writes in the row
              put_index(p.out_indices, row_out + pos, col, p.idx64);
              if (ov) ov[pos] = static_cast<VT>(bits);
            }
          }
        }
      }
      base_gt += tile & 0xFFFFu;
      base_eq += tile >> 16;
      if (base_gt + min(base_eq, r) >= k) break;  // all k written (same decision in every thread)
    }
    __syncthreads();  // sh and cand are reused by the next row
  }
}

}  // namespace ds_topk_dev
