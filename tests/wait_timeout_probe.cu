// wait_timeout_probe.cu — test-only probe of the bounded mbarrier wait used by
// the one-warp-per-row kernel's streaming ring. Built by the test with a short
// DS_TOPK_WAIT_LIMIT; never part of libds_topk.so.
//
// One warp initialises an mbarrier for one arrival. With `arrive` set, lane 0
// arrives once, so phase 0 completes and the wait must succeed. Without it
// nothing ever arrives and no copy is issued (nothing is in flight), so the
// wait must give up after the poll limit; the kernel then ORs
// DS_TOPK_FLAG_TIMEOUT into *flag and returns, as the streaming ring does.
#include <cuda_runtime.h>

#include "warp_rows_kernel.cuh"

namespace {

__global__ void wait_probe_kernel(int arrive, int32_t* flag, int32_t* waited) {
  __shared__ __align__(8) uint64_t bar;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    ds_topk_dev::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (arrive && lane == 0) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ds_topk_dev::smem_addr(&bar)) : "memory");
  }
  __syncwarp();
  const bool ok = __all_sync(0xFFFFFFFFu, ds_topk_dev::mbar_wait(&bar, 0u));
  if (lane == 0) {
    *waited = 1;
    if (!ok) atomicOr(flag, DS_TOPK_FLAG_TIMEOUT);
  }
}

}  // namespace

extern "C" int wait_probe(int arrive, int32_t* flag, int32_t* waited) {
  wait_probe_kernel<<<1, 32>>>(arrive, flag, waited);
  if (cudaGetLastError() != cudaSuccess) return 1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}

extern "C" unsigned wait_probe_limit(void) { return ds_topk_dev::kWrWaitLimit; }
