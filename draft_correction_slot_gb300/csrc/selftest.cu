// selftest.cu -- a check of the failure path every bounded wait shares.
//
// The kernels' waits on mbarriers (weight and row tiles, MMA completion) end
// after a time limit, record kErrTimeout in the handle's device status word
// and let the kernel return; the host reads the word with
// dcoco_get_device_status.  dcoco_selftest_wait_timeout runs that exact wait
// (tc::mbar_wait) on an mbarrier that nothing completes, with a short limit,
// so that a test can see the status word set and the context still usable,
// without faulting or hanging the GPU.
#include <cuda_runtime.h>

#include "../../include/dcoco.h"
#include "common.cuh"
#include "tc.cuh"

namespace dc {
namespace {

__global__ void k_wait_timeout(unsigned long long limit_ns, int *err) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // nothing arrives on `bar`: the wait gives up after limit_ns
  if (threadIdx.x == 0) tc::mbar_wait(tc::smem_u32(&bar), 0, &s_abort, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout(unsigned long long limit_ns, int *err, cudaStream_t st) {
  k_wait_timeout<<<1, 32, 0, st>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace dc
