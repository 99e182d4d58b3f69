// value_order_kernel.cuh — optional output order by value (sorted_index = 2).
//
// For value order, a sort kernel runs after the selection on the same stream and
// reorders each row's k outputs in place. It reads the k selected elements (from
// the values the selection wrote, or gathered from x when no values are
// returned) as sort words and sorts them descending with a bitonic network:
//  - one CTA per row (any k <= 4096): 64-bit words (order key << 32 | ~index) in
//    at most 32 KB of shared memory; strides below 64 run in registers with warp
//    shuffles, so only the wider ones pay a CTA barrier;
//  - one warp per row (many bf16 rows of at most 65536 elements, k <= 1024):
//    32-bit words (16-bit key << 16 | ~16-bit index) in registers.
// Descending words give value descending, and equal values by ascending index
// (the complement of the index sorts the lower index first), which is the
// selection's own total order; every word is distinct, so no stability is
// needed. Value bits follow from the sorted keys, except for zeros, whose sign
// is read back from x, so -0.0 stays -0.0.
//
// Source: github-research.aiutil.com, "deepseek-ai/DeepSelect", section
// 关键技术亮点 (item 2): the output may be ordered by index or by value, and either
// order costs speed, so it is off unless asked for.
#pragma once

#include "sampler_kernel.cuh"

namespace ds_topk_dev {

struct OrderParams {
  const char* x;
  int64_t batch;
  int64_t row_stride_bytes;
  int64_t len;
  int32_t k;
  int32_t n2;  // k rounded up to a power of two, at least 64 (sort width)
  int32_t return_value;
  void* out_values;
  void* out_indices;  // int32 or int64 (idx64)
  int32_t idx64;
  // sampler tail drawn by the CTA sort right after it (tokens null: none)
  int32_t* tokens;
  const float* u;
  float inv_temperature;
  float top_p;
};

// The value of a sort word's order key (the key of zero gives +0: a weight does
// not see the sign).
template <int ES>
__device__ __forceinline__ float word_value(unsigned long long w) {
  uint32_t bits = 0u;
  if (!bits_of_key<ES>(static_cast<uint32_t>(w >> 32), &bits)) bits = 0u;
  return __uint_as_float(ES == 2 ? (bits << 16) : bits);
}

template <int ES>
__device__ __forceinline__ uint32_t load_bits(const char* rowp, int64_t i) {
  if constexpr (ES == 2) return *reinterpret_cast<const uint16_t*>(rowp + i * 2);
  return *reinterpret_cast<const uint32_t*>(rowp + i * 4);
}

// One compare-exchange step of the bitonic network on the two words a lane
// holds (elements e0 = base + 2 lane and e0 + 1 of its warp's 64-word block).
__device__ __forceinline__ void reg_step(unsigned long long& x0, unsigned long long& x1, int e0, int size,
                                         int stride) {
  const bool desc = (e0 & size) == 0;
  if (stride == 1) {
    if (desc ? (x0 < x1) : (x0 > x1)) {
      const unsigned long long t = x0;
      x0 = x1;
      x1 = t;
    }
    return;
  }
  const int lm = stride >> 1;  // partner lane distance
  const unsigned long long y0 = __shfl_xor_sync(0xFFFFFFFFu, x0, lm);
  const unsigned long long y1 = __shfl_xor_sync(0xFFFFFFFFu, x1, lm);
  const bool keep_max = ((e0 & stride) == 0) == desc;
  x0 = keep_max ? (x0 > y0 ? x0 : y0) : (x0 < y0 ? x0 : y0);
  x1 = keep_max ? (x1 > y1 ? x1 : y1) : (x1 < y1 ? x1 : y1);
}

template <int ES>
__global__ void __launch_bounds__(1024) topk_value_order_kernel(const OrderParams p) {
  // let the next kernel in the stream be scheduled; wait for the previous one
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(16) unsigned long long sw[];
  __shared__ float d_warp_tot[32];  // the sampler tail's scratch
  __shared__ float d_cm;
  __shared__ int d_m, d_t;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nt = blockDim.x;  // min(n2 / 2, 1024)
  const int n2 = p.n2;        // >= 64
  const int nwarps = nt >> 5;
  const int nblk = n2 >> 6;   // 64-word blocks, each handled by one warp at a time
  using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
  for (int64_t row = blockIdx.x; row < p.batch; row += gridDim.x) {
    const char* rowp = p.x + row * p.row_stride_bytes;
    const int64_t ob = row * static_cast<int64_t>(p.k);
    VT* ov = p.return_value ? static_cast<VT*>(p.out_values) + row * static_cast<int64_t>(p.k) : nullptr;
    for (int j = tid; j < n2; j += nt) {
      unsigned long long w = 0ull;  // padding sorts last
      if (j < p.k) {
        int64_t idx = get_index(p.out_indices, ob + j, p.idx64);
        if (idx < 0 || idx >= p.len) idx = 0;  // never read outside the row
        // values already written by the selection are read in order; else gather
        const uint32_t bits = ov ? static_cast<uint32_t>(ov[j]) : load_bits<ES>(rowp, idx);
        const uint32_t key = key_of<ES>(bits);
        w = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
      }
      sw[j] = w;
    }
    __syncthreads();
    // bitonic network, descending overall: strides below 64 run in registers
    // (each warp owns 64 consecutive words), larger strides through shared memory
    for (int blk = tid >> 5; blk < nblk; blk += nwarps) {
      const int e0 = blk * 64 + 2 * lane;
      unsigned long long x0 = sw[e0], x1 = sw[e0 + 1];
      for (int size = 2; size <= 64; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) reg_step(x0, x1, e0, size, stride);
      sw[e0] = x0;
      sw[e0 + 1] = x1;
    }
    __syncthreads();
    for (int size = 128; size <= n2; size <<= 1) {
      for (int stride = size >> 1; stride >= 64; stride >>= 1) {
        for (int i = tid; i < (n2 >> 1); i += nt) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const unsigned long long a = sw[lo], b = sw[hi];
          const bool desc = (lo & size) == 0;
          if (desc ? (a < b) : (a > b)) {
            sw[lo] = b;
            sw[hi] = a;
          }
        }
        __syncthreads();
      }
      for (int blk = tid >> 5; blk < nblk; blk += nwarps) {
        const int e0 = blk * 64 + 2 * lane;
        unsigned long long x0 = sw[e0], x1 = sw[e0 + 1];
        for (int stride = 32; stride > 0; stride >>= 1) reg_step(x0, x1, e0, size, stride);
        sw[e0] = x0;
        sw[e0 + 1] = x1;
      }
      __syncthreads();
    }
    for (int j = tid; j < p.k; j += nt) {
      const unsigned long long w = sw[j];
      const uint32_t idx = 0xFFFFFFFFu - static_cast<uint32_t>(w);
      put_index(p.out_indices, ob + j, idx, p.idx64);
      if (ov) {
        uint32_t bits;
        if (!bits_of_key<ES>(static_cast<uint32_t>(w >> 32), &bits)) bits = load_bits<ES>(rowp, idx);
        ov[j] = static_cast<VT>(bits);
      }
    }
    if (p.tokens) {
      // The sampler tail, on the sorted words still in shared memory: the weights
      // of the k survivors, their block-wide inclusive scan C, the nucleus end m
      // (first C_j >= top_p C_{k-1}) and the draw t (first j <= m with C_j > u C_m),
      // as in topk_sample_kernel, thread tid holding the consecutive j of [j0, j0 + per).
      constexpr int kMaxPer = 4;  // k <= 4096 over at least k / 4 threads
      const int per = (p.k + nt - 1) / nt;
      const int j0 = tid * per;
      const float v0 = word_value<ES>(sw[0]);
      float c[kMaxPer];
      float run = 0.f;
#pragma unroll
      for (int e = 0; e < kMaxPer; ++e) {
        const int j = j0 + e;
        if (e < per && j < p.k) run += sample_weight(word_value<ES>(sw[j]), v0, j, p.inv_temperature);
        c[e] = run;
      }
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) d_warp_tot[tid >> 5] = incl;
      if (tid == 0) {
        d_m = p.k - 1;
        d_t = 0x7FFFFFFF;
      }
      __syncthreads();
      float before = incl - run, total = 0.f;
      for (int w = 0; w < nwarps; ++w) {
        if (w < (tid >> 5)) before += d_warp_tot[w];
        total += d_warp_tot[w];
      }
      const float mass = p.top_p * total;
#pragma unroll
      for (int e = 0; e < kMaxPer; ++e) {
        const int j = j0 + e;
        if (e < per && j < p.k && before + c[e] >= mass) {
          atomicMin(&d_m, j);
          break;
        }
      }
      __syncthreads();
      const int m = d_m;
#pragma unroll
      for (int e = 0; e < kMaxPer; ++e)
        if (e < per && j0 + e == m) d_cm = before + c[e];
      __syncthreads();
      const float target = p.u[row] * d_cm;
#pragma unroll
      for (int e = 0; e < kMaxPer; ++e) {
        const int j = j0 + e;
        if (e < per && j <= m && before + c[e] > target) {
          atomicMin(&d_t, j);
          break;
        }
      }
      __syncthreads();
      if (tid == 0) {
        const int t = d_t <= m ? d_t : 0;  // a NaN row finds no step: any in-range choice
        p.tokens[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(sw[t]));
      }
    }
    __syncthreads();  // the next row reuses sw (and the draw's shared words)
  }
}


// ---- one warp per row: bf16 rows of at most 65536 elements, k <= 1024 ----------------
// A sort word is 32 bits, the 16-bit order key above the complemented 16-bit
// index, so descending words are value descending, equal values by ascending
// index. Lane l holds E = n2 / 32 of them in registers (n2 = k rounded up to a
// power of two, at least 32) and no CTA barrier is involved, so a CTA sorts
// several rows at once. (With 64-bit words, as fp32 keys need, the register
// sort costs more than the CTA sort above, which those rows keep.)
// Input word j is read by lane j mod 32 (coalesced) into sort position
// (j mod 32) E + j / 32: where a word starts does not change the sorted result.
// The sorted words go out through a per-warp shared-memory stage, written at the
// lane's sort positions and read back at output position j = e 32 + lane, with one
// pad word after every 32 so that both sides are free of bank conflicts.
constexpr int kVoMaxK = 1024;
constexpr int kVoMaxLen = 65536;
constexpr int kVoWarps = 8;

// Descending bitonic sort of the 32 E words of a warp, word e of lane l at sort
// position i = l E + e, in the form where every comparator points the same way:
// for each block size 2, 4, .., 32 E, position i of a block first pairs with its
// mirror i ^ (size - 1), then (half-cleaners) with i ^ stride for stride = size /
// 4, .., 1; the lower position of a pair keeps the larger word. Pairs inside a
// lane (stride < E) are compile-time (one max, one min); wider ones exchange
// through shuffles, the lane's role (lower or upper) being one predicate per step.
template <typename W>
__device__ __forceinline__ W vo_max(W a, W b) { return a > b ? a : b; }
template <typename W>
__device__ __forceinline__ W vo_min(W a, W b) { return a > b ? b : a; }
// The larger of a and the partner's word b if `larger`, else the smaller: one
// compare folded with the predicate, one select.
template <typename W>
__device__ __forceinline__ W vo_keep(W a, W b, bool larger) { return (a > b) == larger ? a : b; }

template <typename W, int E>
__device__ __forceinline__ void vo_sort_desc(W (&x)[E], int lane) {
  constexpr int N = 32 * E;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
    if (size <= E) {  // mirror pairs inside the lane
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & (size >> 1)) == 0) {
          const int f = e ^ (size - 1);
          const W a = x[e], b = x[f];
          x[e] = vo_max(a, b);
          x[f] = vo_min(a, b);
        }
      }
    } else {  // the mirror of word e sits in lane l ^ m as word E - 1 - e
      const int m = (size - 1) / E;
      const bool lower = (lane & ((size >> 1) / E)) == 0;
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const W ya = __shfl_xor_sync(0xFFFFFFFFu, x[E - 1 - e], m);
        const W yb = __shfl_xor_sync(0xFFFFFFFFu, x[e], m);
        x[e] = vo_keep(x[e], ya, lower);
        x[E - 1 - e] = vo_keep(x[E - 1 - e], yb, lower);
      }
      if (E == 1) x[0] = vo_keep(x[0], __shfl_xor_sync(0xFFFFFFFFu, x[0], m), lower);
    }
#pragma unroll
    for (int stride = size >> 2; stride > 0; stride >>= 1) {
      if (stride < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & stride) == 0) {
            const W a = x[e], b = x[e | stride];
            x[e] = vo_max(a, b);
            x[e | stride] = vo_min(a, b);
          }
        }
      } else {
        const int d = stride / E;
        const bool lower = (lane & d) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          x[e] = vo_keep(x[e], __shfl_xor_sync(0xFFFFFFFFu, x[e], d), lower);
        }
      }
    }
  }
}

template <int E, bool IDX64, bool RETV>
__global__ void __launch_bounds__(32 * kVoWarps) topk_value_order_warp_kernel(const OrderParams p) {
  // let the next kernel in the stream be scheduled; wait for the previous one
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the selection's outputs
  constexpr int N = 32 * E;
  __shared__ uint32_t stage[kVoWarps][N + N / 32];
  const int lane = threadIdx.x & 31;
  uint32_t* st = stage[threadIdx.x >> 5];
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kVoWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kVoWarps + (threadIdx.x >> 5); row < p.batch; row += nw) {
    const char* rowp = p.x + row * p.row_stride_bytes;
    const int64_t ob = row * static_cast<int64_t>(p.k);
    uint16_t* ov = RETV ? static_cast<uint16_t*>(p.out_values) + ob : nullptr;
    uint32_t x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int j = e * 32 + lane;
      uint32_t w = 0u;  // padding sorts last
      if (j < p.k) {
        int64_t idx = get_index(p.out_indices, ob + j, IDX64);
        if (idx < 0 || idx >= p.len) idx = 0;  // never read outside the row
        const uint32_t bits = RETV ? static_cast<uint32_t>(ov[j]) : load_bits<2>(rowp, idx);
        w = (key_of<2>(bits) << 16) | (0xFFFFu - static_cast<uint32_t>(idx));
      }
      x[e] = w;
    }
    vo_sort_desc<uint32_t, E>(x, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = lane * E + e;
      st[i + i / 32] = x[e];
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int j = e * 32 + lane;
      if (j < p.k) {
        const uint32_t w = st[j + j / 32];
        const uint32_t idx = 0xFFFFu - (w & 0xFFFFu);
        put_index(p.out_indices, ob + j, idx, IDX64);
        if constexpr (RETV) {
          uint32_t bits;
          if (!bits_of_key<2>(w >> 16, &bits)) bits = load_bits<2>(rowp, idx);
          ov[j] = static_cast<uint16_t>(bits);
        }
      }
    }
    __syncwarp();  // the next row rewrites the stage
  }
}

}  // namespace ds_topk_dev
