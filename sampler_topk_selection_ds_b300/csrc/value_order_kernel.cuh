// value_order_kernel.cuh — optional output order by value (sorted_index = 2).
//
// The selection kernels write each row's k outputs in ascending index order.
// For value order, this kernel runs after them on the same stream: one CTA per
// row reads the k selected elements (from the values the selection wrote, or
// gathered from x when no values are returned), forms 64-bit sort words (order
// key << 32 | ~index) and sorts them descending with a bitonic network (k <=
// 4096: at most 32 KB of shared memory); strides below 64 run in registers with
// warp shuffles, so only the wider ones pay a CTA barrier.
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

#include "topk_kernel.cuh"

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
};

template <int ES>
__device__ __forceinline__ uint32_t load_bits(const char* rowp, int64_t i) {
  if constexpr (ES == 2) return *reinterpret_cast<const uint16_t*>(rowp + i * 2);
  return *reinterpret_cast<const uint32_t*>(rowp + i * 4);
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
  // the selection kernel's outputs must be complete before they are read
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(16) unsigned long long sw[];
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
    __syncthreads();  // the next row reuses sw
  }
}

}  // namespace ds_topk_dev
