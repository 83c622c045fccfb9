// Weighted top-k combine: y[t] = bf16( sum_{j=0..k-1} w[t,j] * o[t*k+j] ), plus the shared
// expert's row o_shared[t] (weight 1, added last) when the layer has one.
//
// This is the scatter_add of "Current Bug: CuTeDSLMoERunner" ("Data Flow"),
// restated as a gather. The second GEMM stores one bf16 row per (token, k)
// pair (l2_out is BF16 there) and drops padding rows ("Bug 14"). Every token
// then sums its k rows in fp32 in a fixed j order, so the result has no
// atomics and is run-to-run deterministic. One thread owns 8 consecutive
// columns: one 128-bit load per pair row, one 128-bit store of y. Inputs written by the kernels just before are read through
// L2 (ld.global.cg): with programmatic dependent launch this kernel may start
// before they finish.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {

int sm_count();

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

// Eight bf16 values through L2 as fp32.
__device__ __forceinline__ void ld8_bf16_cg(const uint16_t* p, float (&v)[8]) {
  const uint4 q = __ldcg(reinterpret_cast<const uint4*>(p));
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

// Eight fp32 values through L2: one 256-bit load (sm_100 and later) when the address is 32-byte aligned.
template <bool V8>
__device__ __forceinline__ void ld8_cg(const float* p, float (&v)[8]) {
  if constexpr (V8) {
    asm volatile("ld.global.cg.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(p)
                 : "memory");
  } else {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p)), b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// V8: the shared expert's fp32 rows are 32-byte aligned. BATCH: a grid of one wave (decode). The token's k
// weights and slots are loaded first, then the rows of up
// to 8 pairs at a time, all in flight before the sums. Otherwise many waves (prefill) keep the memory system
// busy instead, and a lean loop keeps more CTAs resident. Either way the sum runs in pair order and a pair
// held by no local expert (it has no row) is skipped.
template <bool V8, bool BATCH>
__global__ void __launch_bounds__(256) combine_kernel(int H, int k, const uint16_t* __restrict__ o,
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
  if constexpr (!BATCH) {
    for (int j = 0; j < k; ++j) {
      if (slot_of_pair != nullptr && __ldcg(slot_of_pair + (size_t)t * k + j) < 0) continue;
      const float wj = __ldcg(w + (size_t)t * k + j);
      float v[8];
      ld8_bf16_cg(o + ((size_t)t * k + j) * H + col, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
    }
  } else {
    float wj[kMaxTopK];
    bool held[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      held[j] = j < k && (slot_of_pair == nullptr || __ldcg(slot_of_pair + (size_t)t * k + j) >= 0);
      wj[j] = j < k ? __ldcg(w + (size_t)t * k + j) : 0.0f;
    }
#pragma unroll
    for (int j0 = 0; j0 < kMaxTopK; j0 += 8) {
      if (j0 >= k) break;
      float v[8][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (held[j0 + jj]) ld8_bf16_cg(o + ((size_t)t * k + j0 + jj) * H + col, v[jj]);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (held[j0 + jj]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j0 + jj], v[jj][i], acc[i]);
        }
      }
    }
  }
  if (o_shared != nullptr) {  // the shared expert, weight 1, after the routed terms
    float v[8];
    ld8_cg<V8>(o_shared + (size_t)t * H + col, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
  *reinterpret_cast<uint4*>(y + (size_t)t * H + col) =
      make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                 pack_bf16x2(acc[6], acc[7]));
}

}  // namespace

fp4moe_status combine_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* o_pairs, const float* w,
                             const int32_t* slot_of_pair, const float* o_shared, uint16_t* y, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden;
  // 256-bit loads of the shared expert's fp32 rows when every row start is 32-byte aligned (H % 256 == 0)
  const bool v8 = (reinterpret_cast<uintptr_t>(o_shared) & 31u) == 0;
  const dim3 grid((H / 8 + 255) / 256, T);
  const bool batch = (int64_t)grid.x * grid.y <= sm_count();  // one wave: latency rules
  cudaError_t r;
  if (v8) {
    r = batch ? launch_pdl(combine_kernel<true, true>, grid, dim3(256), 0, st, H, cfg.top_k, o_pairs, w, slot_of_pair,
                           o_shared, y)
              : launch_pdl(combine_kernel<true, false>, grid, dim3(256), 0, st, H, cfg.top_k, o_pairs, w,
                           slot_of_pair, o_shared, y);
  } else {
    r = batch ? launch_pdl(combine_kernel<false, true>, grid, dim3(256), 0, st, H, cfg.top_k, o_pairs, w,
                           slot_of_pair, o_shared, y)
              : launch_pdl(combine_kernel<false, false>, grid, dim3(256), 0, st, H, cfg.top_k, o_pairs, w,
                           slot_of_pair, o_shared, y);
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
