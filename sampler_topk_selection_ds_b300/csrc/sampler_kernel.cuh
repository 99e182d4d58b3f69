// sampler_kernel.cuh — the sampler tail after TopK: temperature softmax over the
// k selected logits, the top-p nucleus, and one draw from it.
//
// Runs after the value-ordered selection (sorted_index = DS_TOPK_SORT_VALUE with
// values) on the same stream, one CTA per row, when that value order was the
// one-warp-per-row sort; the CTA sort draws the same way itself (its draw uses
// sample_weight below). Per row, in fp32:
//   w_j = exp((v_j - v_0) / T)   (v_0 the largest value, so w_0 = 1; when v_0 is
//                                 +inf the +inf values weigh 1 and the rest 0)
//   C_j = w_0 + ... + w_j        (block-wide inclusive scan)
//   m   = first j with C_j >= top_p * C_{k-1}        (the nucleus is [0, m])
//   t   = first j <= m with C_j > u * C_m            (inverse CDF, u in [0, 1))
// and the token is the column of the t-th selected element. The uniform number
// u is the caller's (one per row): nothing random happens here.
//
// Sources: github-research.aiutil.com, "deepseek-ai/DeepSelect", section
// 关键技术亮点: the sampler path of TopK, whose k survivors the sampler draws the
// next token from; deepseek.csdn.net, "DeepSeek 一次开源三个仓库": temperature and
// top_p as the request's sampling parameters.
#pragma once

#include <cmath>

#include "topk_kernel.cuh"

namespace ds_topk_dev {

constexpr int kSampleThreads = 256;

struct SampleParams {
  int64_t batch;
  int32_t k;
  float inv_temperature;
  float top_p;
  const float* u;
  const void* values;      // [batch, k] value-ordered top-k values
  const int32_t* indices;  // [batch, k] their columns
  int32_t* tokens;         // [batch]
};

template <int ES>
__device__ __forceinline__ float value_at(const void* values, int64_t i) {
  if constexpr (ES == 2) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(values)[i]) << 16);
  return static_cast<const float*>(values)[i];
}

// Weight of the j-th value-ordered survivor v given the largest v0 (see above).
__device__ __forceinline__ float sample_weight(float v, float v0, int j, float inv_temperature) {
  if (isinf(v0) && v0 > 0.f) return v == v0 ? 1.f : 0.f;
  if (isinf(v0)) return j == 0 ? 1.f : 0.f;  // every value is -inf
  return expf((v - v0) * inv_temperature);
}

template <int ES>
__global__ void __launch_bounds__(kSampleThreads) topk_sample_kernel(const SampleParams p) {
  // let the next kernel in the stream be scheduled; wait for the previous one
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the value-ordered selection
  constexpr int kMaxPer = (DS_TOPK_MAX_K + kSampleThreads - 1) / kSampleThreads;
  __shared__ float warp_tot[kSampleThreads / 32];
  __shared__ float cm;
  __shared__ int m_s, t_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.k;
  const int per = (k + kSampleThreads - 1) / kSampleThreads;
  const int j0 = tid * per;  // this thread's consecutive elements [j0, j0 + per)
  for (int64_t row = blockIdx.x; row < p.batch; row += gridDim.x) {
    const int64_t base = row * k;
    const float v0 = value_at<ES>(p.values, base);
    float c[kMaxPer];
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxPer; ++e) {
      const int j = j0 + e;
      float w = 0.f;
      if (e < per && j < k) w = sample_weight(value_at<ES>(p.values, base + j), v0, j, p.inv_temperature);
      run += w;
      c[e] = run;  // inclusive within the thread
    }
    // exclusive prefix of the thread totals over the block
    float incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    if (tid == 0) {
      m_s = k - 1;
      t_s = 0x7FFFFFFF;
    }
    __syncthreads();
    float before = incl - run, total = 0.f;
    for (int w = 0; w < kSampleThreads / 32; ++w) {
      if (w < warp) before += warp_tot[w];
      total += warp_tot[w];
    }
    // nucleus end m: first j with C_j >= top_p * total
    const float mass = p.top_p * total;
#pragma unroll
    for (int e = 0; e < kMaxPer; ++e) {
      const int j = j0 + e;
      if (e < per && j < k && before + c[e] >= mass) {
        atomicMin(&m_s, j);
        break;
      }
    }
    __syncthreads();
    const int m = m_s;
#pragma unroll
    for (int e = 0; e < kMaxPer; ++e)
      if (e < per && j0 + e == m) cm = before + c[e];
    __syncthreads();
    // the draw: first j <= m with C_j > u * C_m
    const float target = p.u[row] * cm;
#pragma unroll
    for (int e = 0; e < kMaxPer; ++e) {
      const int j = j0 + e;
      if (e < per && j <= m && before + c[e] > target) {
        atomicMin(&t_s, j);
        break;
      }
    }
    __syncthreads();
    if (tid == 0) {
      const int t = t_s <= m ? t_s : 0;  // a NaN row finds no step: any in-range choice
      p.tokens[row] = p.indices[base + t];
    }
    __syncthreads();  // m_s, t_s, cm and warp_tot are reused by the next row
  }
}

}  // namespace ds_topk_dev
