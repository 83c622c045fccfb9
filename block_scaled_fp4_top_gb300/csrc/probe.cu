// Dense FP4 tensor-core throughput probe: the peak that the prefill GEMMs'
// tensor-pipe utilisation is reported against.
//
// One CTA per SM. Each stages one K atom of A (128 rows) and B (n rows) of
// pseudo-random codes in shared memory with the 128-byte swizzle, sets its
// block scales in TMEM to 1.0,
// and then one thread issues `iters` x 4 back-to-back
// tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X (M = 128,
// N = n, K = 64) into one TMEM accumulator: the grouped GEMMs' instruction at
// the largest single-CTA shape, with no global traffic at all. The caller
// times the launch; the work is SMs x iters x 4 x 2 x 128 x n x 64 flops.
// The final commit is awaited with the library's bounded wait.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int kProbeSmem = 1024 + 16384 + 32768 + 512;

__global__ void __launch_bounds__(128, 1) tensor_peak_kernel(int n, int iters, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t a_s = smem, b_s = smem + 16384u, sf_s = smem + 16384u + 32768u;
  const int warp = threadIdx.x >> 5;
  // operands: pseudo-random codes (every E2M1 value, as real data has them; zeros could take a cheaper path
  // through the tensor core); scales: all 0x38 (1.0), so every product stays finite
  uint32_t* base = reinterpret_cast<uint32_t*>(smem_raw + (smem - smem_u32(smem_raw)));
  for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x) base[i] = (uint32_t)i * 2654435761u ^ 0x5bd1e995u;
  for (int i = threadIdx.x; i < 512 / 4; i += blockDim.x) base[(16384 + 32768) / 4 + i] = 0x38383838u;
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  const uint32_t bar = smem_u32(&s_bar);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (threadIdx.x == 0) {
    // scales 1.0: A's at columns 256..271, B's at 384..447 (room for any N up to 256)
    for (int c = 0; c < 4; ++c) tc_cp_scales(tmem + 256 + 4 * c, desc_scales(sf_s));
    for (int c = 0; c < 16; ++c) tc_cp_scales(tmem + 384 + 4 * c, desc_scales(sf_s));
    const uint32_t idesc = n == 256 ? idesc_nvf4(128, 256) : idesc_nvf4(128, 128);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
        tc_mma_nvf4(tmem, desc_sw128(a_s + 32 * a), desc_sw128(b_s + 32 * a), idesc, tmem + 256 + 4 * a,
                    tmem + 384 + 4 * a, (it | a) != 0 ? 1u : 0u);
    }
    tc_commit(bar);
    if (!mbar_wait(bar, 0, err)) drain_wait(bar, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

fp4moe_status tensor_peak_launch(int32_t n, int32_t iters, uint32_t* err, cudaStream_t st) {
  static int ok = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(tensor_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) ==
                 cudaSuccess
             ? 1
             : 0;
  });
  if (ok != 1) return FP4MOE_CUDA_ERROR;
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  tensor_peak_kernel<<<nsm, 128, kProbeSmem, st>>>(n, iters, err);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
