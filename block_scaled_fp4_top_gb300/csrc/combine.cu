// Weighted top-k combine: y[t] = bf16( sum_{j=0..k-1} w[t,j] * o[t*k+j] ), plus the shared
// expert's row o_shared[t] (weight 1, added last) when the layer has one.
//
// This is the scatter_add of "Current Bug: CuTeDSLMoERunner" ("Data Flow"),
// restated as a gather. The second GEMM stores one fp32 row per (token, k)
// pair and drops padding rows ("Bug 14"). Every token then sums its k rows in
// a fixed j order, so the result has no atomics and is run-to-run
// deterministic. One thread owns 8 consecutive columns, loaded and stored as
// 128-bit vectors. Inputs written by the kernels just before are read through
// L2 (ld.global.cg): with programmatic dependent launch this kernel may start
// before they finish.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__global__ void __launch_bounds__(256) combine_kernel(int H, int k, const float* __restrict__ o,
                                                      const float* __restrict__ w,
                                                      const int32_t* __restrict__ slot_of_pair,
                                                      const float* __restrict__ o_shared,
                                                      uint16_t* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (col >= H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    if (slot_of_pair != nullptr && __ldcg(slot_of_pair + (size_t)t * k + j) < 0) continue;  // not held here
    const float wj = __ldcg(w + (size_t)t * k + j);
    const float4* src = reinterpret_cast<const float4*>(o + ((size_t)t * k + j) * H + col);
    const float4 a = __ldcg(src), b = __ldcg(src + 1);
    acc[0] = fmaf(wj, a.x, acc[0]);
    acc[1] = fmaf(wj, a.y, acc[1]);
    acc[2] = fmaf(wj, a.z, acc[2]);
    acc[3] = fmaf(wj, a.w, acc[3]);
    acc[4] = fmaf(wj, b.x, acc[4]);
    acc[5] = fmaf(wj, b.y, acc[5]);
    acc[6] = fmaf(wj, b.z, acc[6]);
    acc[7] = fmaf(wj, b.w, acc[7]);
  }
  if (o_shared != nullptr) {  // the shared expert, weight 1, after the routed terms
    const float4* src = reinterpret_cast<const float4*>(o_shared + (size_t)t * H + col);
    const float4 a = __ldcg(src), b = __ldcg(src + 1);
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
  }
  *reinterpret_cast<uint4*>(y + (size_t)t * H + col) =
      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                 pack_bf16x2(acc[6], acc[7]));
}

}  // namespace

fp4moe_status combine_launch(const fp4moe_config& cfg, int32_t T, const float* o_pairs, const float* w,
                             const int32_t* slot_of_pair, const float* o_shared, uint16_t* y, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden;
  return launch_pdl(combine_kernel, dim3((H / 8 + 255) / 256, T), dim3(256), 0, st, H, cfg.top_k, o_pairs, w,
                    slot_of_pair, o_shared, y) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
