// A self-test of the failure path every pipeline wait of the library shares: one
// warp waits on an mbarrier that nothing arrives on, gives up after the wait
// budget (about a second), records where (kernel id 4) and sets
// PFA_DEVERR_TIMEOUT in the device error word. Nothing traps and the context
// stays usable, which the GPU tests check by running the attention kernels
// afterwards.
#include "pfa_device.cuh"
#include "pfa_internal.h"

namespace pfa {
namespace {

__global__ void __launch_bounds__(32, 1) wait_probe_kernel(int* err, unsigned long long* site) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const WaitCtl ctl{&abort_flag, err, site, b, 4u};
  (void)wait_warp(b, 0, ctl);
}

}  // namespace

cudaError_t launch_wait_probe(int* err, unsigned long long* site, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, site);
  return cudaGetLastError();
}

}  // namespace pfa
