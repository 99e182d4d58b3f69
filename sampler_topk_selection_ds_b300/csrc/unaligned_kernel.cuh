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
// Selection is an exact radix select on the order key, most significant 8-bit
// digit first. Each level builds a 256-bin shared-memory histogram of the next
// digit over the elements whose higher digits equal the prefix found so far,
// and picks the bin that holds the kr-th largest of them (kr starts at k and
// loses the count of every bin above the chosen one). It stops early when the
// chosen bin is taken whole, so every key >= (prefix << shift) is selected, and
// otherwise at the last digit, where the prefix is the k-th key K* and kr is the
// number of K*-ties to take. A final pass is the ordered compaction: keys above
// the threshold, and the lowest-index ties until k are taken, written in
// ascending index order. Each level re-reads the row (from L2 after the first
// pass: a resident CTA holds one row at a time).
//
// Sources: deepseek-v4-pro.uk (zh-tw), "深入 DeepSeek V4.1 全新開放推論工具包",
// section "DeepSelect：快速且刻意狹義的 TopK": rows need a specific alignment and
// callers may pad them (this path removes the need); deepseek.csdn.net,
// "DeepSeek 一次开源三个仓库", section 三 (算子层): the top-K of each row, whose
// compaction here is a digit-by-digit threshold search instead of the
// candidate-buffer scheme.
#pragma once

#include "topk_kernel.cuh"

namespace ds_topk_dev {

constexpr int kUaThreads = 512;  // threads per CTA (>= 256: one per histogram bin)
constexpr int kUaWarps = kUaThreads / 32;
constexpr int kUaUnroll = 4;     // vectors in flight per thread in a histogram pass
constexpr int kUaOutVecs = 4;    // consecutive vectors per thread in a compaction tile

struct UaParams {
  const char* x;
  int64_t batch;
  int64_t row_stride_bytes;
  int64_t len;
  int32_t k;
  int32_t return_value;
  void* out_values;
  void* out_indices;  // int32 or int64 (idx64)
  int32_t idx64;
  int32_t* flag;
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

template <int ES>
__global__ void __launch_bounds__(kUaThreads, 2) topk_unaligned_kernel(const UaParams p) {
  constexpr int VEC = Traits<ES>::kVec;
  constexpr int W = Traits<ES>::kKeyBits;
  using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t tot_s[2][kUaWarps];  // per-warp scan totals (double-buffered)
  __shared__ uint32_t bin_s, above_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t k = static_cast<uint32_t>(p.k);

  for (int64_t row = blockIdx.x; row < p.batch; row += gridDim.x) {
    const char* rowp = p.x + row * p.row_stride_bytes;
    const int lead = static_cast<int>((reinterpret_cast<uintptr_t>(rowp) & 15u) / ES);
    const char* abase = rowp - lead * ES;
    const int64_t nq = (lead + p.len + VEC - 1) / VEC;  // aligned vectors overlapping the row

    // ---- radix levels: threshold T and ties to take r ----
    uint32_t prefix = 0u, kr = k, T = 0u, r = 0u;
    for (int shift = W - 8;; shift -= 8) {
      const bool first = shift == W - 8;
      for (int i = tid; i < 256; i += kUaThreads) hist[i] = 0u;
      __syncthreads();
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
              atomicAdd(&hist[key >> shift], 1u);
            } else if ((key >> (shift + 8)) == prefix) {
              atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
          }
        }
      }
      const int any_nan = __syncthreads_or(nan_seen);
      if (first && any_nan && tid == 0) atomicOr(p.flag, DS_TOPK_FLAG_NAN);
      // The bin holding the kr-th largest: thread t takes bin 255 - t, so an
      // inclusive scan over t counts the elements in that bin and every bin above.
      uint32_t h = 0u, s = 0u;
      if (tid < 256) {
        h = hist[255 - tid];
        s = h;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, s, o);
          if (lane >= o) s += t;
        }
        if (lane == 31) tot_s[0][warp] = s;
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t above = s - h;
        for (int w2 = 0; w2 < warp; ++w2) above += tot_s[0][w2];
        if (above < kr && kr <= above + h) {  // exactly one bin: the counts cover kr
          bin_s = 255u - tid;
          above_s = above;
        }
      }
      __syncthreads();
      const uint32_t b = bin_s;
      const uint32_t in_bin = hist[b];
      kr -= above_s;
      prefix = (prefix << 8) | b;
      if (in_bin == kr) {  // the whole bin is taken: select every key >= prefix << shift
        T = prefix << shift;
        r = 0xFFFFFFFFu;
        break;
      }
      if (shift == 0) {  // the last digit: T = K*, and kr of its ties are taken
        T = prefix;
        r = kr;
        break;
      }
      __syncthreads();  // hist, bin_s and above_s are rewritten by the next level
    }

    // ---- ordered compaction: keys > T, then ties == T by ascending index ----
    uint32_t base_gt = 0u, base_eq = 0u;
    const int64_t row_out = row * static_cast<int64_t>(k);
    VT* ov = p.return_value ? static_cast<VT*>(p.out_values) + row_out : nullptr;
    int par = 0;
    for (int64_t tb = 0; tb < nq; tb += static_cast<int64_t>(kUaThreads) * kUaOutVecs, par ^= 1) {
      const int64_t q0 = tb + static_cast<int64_t>(tid) * kUaOutVecs;
      uint4 w[kUaOutVecs];
      uint32_t val[kUaOutVecs];
#pragma unroll
      for (int u = 0; u < kUaOutVecs; ++u) {
        val[u] = 0u;
        w[u] = make_uint4(0u, 0u, 0u, 0u);
        if (q0 + u < nq) w[u] = ua_load<ES>(abase, q0 + u, lead, p.len, val[u]);
      }
      uint32_t cg = 0u, ce = 0u;
#pragma unroll
      for (int u = 0; u < kUaOutVecs; ++u) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          if (!((val[u] >> e) & 1u)) continue;
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
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) tot_s[par][warp] = incl;
      __syncthreads();
      uint32_t before = incl - v, tile = 0u;
#pragma unroll
      for (int w2 = 0; w2 < kUaWarps; ++w2) {
        const uint32_t t = tot_s[par][w2];
        if (w2 < warp) before += t;
        tile += t;
      }
      uint32_t gtb = base_gt + (before & 0xFFFFu), eqb = base_eq + (before >> 16);
      if (v != 0u) {
#pragma unroll
        for (int u = 0; u < kUaOutVecs; ++u) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            if (!((val[u] >> e) & 1u)) continue;
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
            if (pos >= 0) {
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
    __syncthreads();  // hist, tot_s and the shared words are reused by the next row
  }
}

}  // namespace ds_topk_dev
