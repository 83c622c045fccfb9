// Self-test of the failure path of the bounded waits.
//
// Every spin-wait in the library's kernels (the mbarrier waits of the TMA and
// tensor-core pipelines) gives up after a time limit, sets FP4MOE_ERR_TIMEOUT
// in the error word and lets its kernel return, so a lost arrival never hangs
// the GPU. This kernel drives that routine into its limit on purpose: it waits
// on an mbarrier that nothing arrives at. It faults nothing and traps nothing;
// the host then sees the error bit, and later calls that share the error word
// see the abort bit and skip their work until the word is cleared.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

__global__ void selftest_wait_kernel(uint32_t* err, uint64_t limit_ns, uint32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
    // parity 0 completes only after one arrival, and none comes
    const bool ok = mbar_try_wait(b, 0) || mbar_wait_slow(b, 0, err, limit_ns);
    *result = ok ? 1u : 0u;
  }
}

}  // namespace

fp4moe_status selftest_wait_launch(uint32_t* err, int64_t limit_ns, uint32_t* result, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(err, (uint64_t)limit_ns, result);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
