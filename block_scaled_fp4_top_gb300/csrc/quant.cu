// NVFP4 quantisation kernels: activation quantise-and-scatter into slot order,
// weight quantisation (with the W1 gate/up tile interleave), amax reductions,
// global scales and alpha tables.
//
// Per 16-element block this is quantize_activation_nvfp4 on "Current Bug:
// CuTeDSLMoERunner" ("Data Flow"). The scale assembly is the graph-safe
// per-expert swizzle of "Bug 1", "Bug 11" and "Bug 14". Every expert's rows
// start on a 128-row boundary, so writing each scale byte straight to its
// 128x4 tile position gives exactly the concatenation of independently
// swizzled per-expert blocks. The kernel needs no second scale pass and no
// staging buffer.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

// Set `bit` in `*word` if any active lane of the warp asks for it: one atomic per warp, and none once the bit
// is already set (a stale scale can make every block of a large batch saturate).
__device__ __forceinline__ void warp_flag(bool want, uint32_t* word, uint32_t bit) {
  const unsigned m = __activemask();
  const unsigned b = __ballot_sync(m, want);
  if (b != 0u && (threadIdx.x & 31u) == (unsigned)(__ffs(b) - 1) && !(*(volatile uint32_t*)word & bit))
    atomicOr(word, bit);
}

// One thread per 16-element block: thread i quantises block i % (H/16) of
// token i / (H/16) once and writes it to the token's k slot rows. Consecutive
// threads cover consecutive blocks of a row, so loads and code stores are
// contiguous. Padding rows are never touched. A block whose scale saturates
// (s = RN(RN(amax/6) * gs1) rounds above 448 in E4M3, s > 464) sets
// FP4MOE_SAT_L1 in `status`; a NaN in x sets FP4MOE_ERR_NAN in `err`.
__global__ void __launch_bounds__(256) quant_scatter_kernel(int T, int H, int k, const uint16_t* __restrict__ x,
                                                            const float* __restrict__ gs1,
                                                            const int32_t* __restrict__ slot_of_pair,
                                                            uint8_t* __restrict__ a1, uint8_t* __restrict__ a1_sf,
                                                            uint32_t* status, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int C = H >> 4;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)T * C) return;
  const int t = (int)(i / C), b = (int)(i - (int64_t)t * C);
  // every load is issued before the first use: the token's k slots, the global scale and the block
  int rows[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rows[j] = j < k ? __ldcg(slot_of_pair + (size_t)t * k + j) : -1;
  const float g = __ldg(gs1);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H) + 2 * b;
  const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
  const float v[16] = {bf16_lo(u0.x), bf16_hi(u0.x), bf16_lo(u0.y), bf16_hi(u0.y), bf16_lo(u0.z), bf16_hi(u0.z),
                       bf16_lo(u0.w), bf16_hi(u0.w), bf16_lo(u1.x), bf16_hi(u1.x), bf16_lo(u1.y), bf16_hi(u1.y),
                       bf16_lo(u1.z), bf16_hi(u1.z), bf16_lo(u1.w), bf16_hi(u1.w)};
  uint32_t lo, hi;
  float s;
  const uint32_t sf = quant_block16(v, g, lo, hi, s);
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) nan |= (v[i] != v[i]);
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    const int row = rows[j];
    if (row < 0) continue;  // past k, or held by no local expert
    *reinterpret_cast<uint2*>(a1 + (size_t)row * (H >> 1) + b * 8) = make_uint2(lo, hi);
    a1_sf[sf_offset(row, b, C)] = (uint8_t)sf;
  }
  warp_flag(s > kE4M3SatAbove, status, FP4MOE_SAT_L1);
  warp_flag(nan, err, FP4MOE_ERR_NAN);
}

// Byte offset of code byte `kbyte` of kernel row o in the pre-tiled weight
// layout. Blocks of 128 rows x 128 bytes (16 KB) are ordered
// [group][row tile][k stage]. Inside a block, row i's 16-byte chunk j sits at
// i*128 + (j ^ (i % 8))*16: the 128-byte swizzle that the tensor cores read.
__device__ __forceinline__ size_t tiled_offset(int64_t grp, int o, int kbyte, int n_row_tiles, int k_stages) {
  return ((size_t)(grp * n_row_tiles + (o >> 7)) * k_stages + (kbyte >> 7)) * 16384u + (size_t)(o & 127) * 128u +
         ((((kbyte & 127) >> 4) ^ (o & 7)) << 4) + (kbyte & 15);
}

// Generic fp32 row quantiser. Row gr belongs to group gr / rows_per_group,
// and its output row inside the group is either the same row or, when
// inter > 0, the W1 kernel order: gate feature f -> 128*(f/64) + f%64,
// up feature f -> 128*(f/64) + 64 + f%64. With tiled != 0, the codes go to the
// pre-tiled weight layout instead of row-major [row][K/2].
__global__ void __launch_bounds__(256) quant_rows_kernel(int64_t n_rows, int K, int rows_per_group, int inter,
                                                         int tiled, const float* __restrict__ in,
                                                         const float* __restrict__ g, int g_div,
                                                         uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gr = (int64_t)blockIdx.x * 8 + warp;
  if (gr >= n_rows) return;
  const int64_t grp = gr / rows_per_group;
  int i = (int)(gr - grp * rows_per_group);
  if (inter > 0) {
    const int up = i >= inter;
    const int f = up ? i - inter : i;
    i = 128 * (f >> 6) + 64 * up + (f & 63);
  }
  const int C = K >> 4;
  const float gg = __ldg(g + gr / g_div);
  const float4* src = reinterpret_cast<const float4*>(in + gr * K);
  uint8_t* dst = codes + (grp * rows_per_group + i) * (int64_t)(K >> 1);
  uint8_t* sdst = sf + grp * (int64_t)rows_per_group * C;
  const int n_row_tiles = rows_per_group >> 7, k_stages = (K + 255) >> 8;
  for (int b = lane; b < C; b += 32) {
    const float4 a = __ldg(src + 4 * b), c = __ldg(src + 4 * b + 1), d = __ldg(src + 4 * b + 2),
                 e = __ldg(src + 4 * b + 3);
    const float v[16] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w, e.x, e.y, e.z, e.w};
    uint32_t lo, hi;
    const uint32_t s = quant_block16(v, gg, lo, hi);
    uint8_t* cd = tiled ? codes + tiled_offset(grp, i, b * 8, n_row_tiles, k_stages) : dst + b * 8;
    *reinterpret_cast<uint2*>(cd) = make_uint2(lo, hi);
    sdst[sf_offset(i, b, C)] = (uint8_t)s;
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

// amax over each group of `per_group` fp32 values (grid.y = group). Result via an unsigned max on the
// bit patterns of non-negative floats, which orders them correctly. The caller zeroes amax first.
__global__ void __launch_bounds__(256) amax_f32_kernel(int64_t per_group, const float* __restrict__ in,
                                                       float* __restrict__ amax) {
  const float* base = in + (int64_t)blockIdx.y * per_group;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per_group; i += (int64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(base[i]));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax + blockIdx.y), __float_as_uint(m));
}

__global__ void __launch_bounds__(256) amax_bf16_kernel(int64_t n, const uint16_t* __restrict__ in,
                                                        float* __restrict__ amax) {
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(__uint_as_float((uint32_t)in[i] << 16)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(m));
}

__global__ void gs_from_amax_kernel(int n, float* inout) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) inout[i] = global_scale_from_amax(inout[i]);
}

__global__ void make_alpha_kernel(int n, const float* __restrict__ gs_act, const float* __restrict__ gs_w,
                                  float* __restrict__ alpha) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) alpha[i] = __fdiv_rn(1.0f, __fmul_rn(gs_act[0], gs_w[i]));
}

inline fp4moe_status last_status() { return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR; }

// The L1 activation global scale of the batch in hand: gs1 = RN(2688 / amax|x|) and
// alpha1[e] = RN(1 / RN(gs1 * gw1[e])), in one launch. Every CTA folds its part of the amax into `acc`
// (float bits compare as unsigned for non-negative values); the last CTA to arrive reads and clears it,
// writes gs1 and the alpha table, and clears the arrival counter, so both words are zero again afterwards.
__global__ void __launch_bounds__(256) batch_gs1_kernel(int64_t n, const uint16_t* __restrict__ x, int E,
                                                        const float* __restrict__ gw1, float* __restrict__ gs1,
                                                        float* __restrict__ alpha1, unsigned int* acc,
                                                        unsigned int* done) {
  pdl_wait();
  pdl_trigger();
  __shared__ bool s_last;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(__uint_as_float((uint32_t)x[i] << 16)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(acc, __float_as_uint(m));
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ float s_g;
  if (threadIdx.x == 0) {
    s_g = global_scale_from_amax(__uint_as_float(atomicExch(acc, 0u)));
    gs1[0] = s_g;
    *done = 0u;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) alpha1[e] = __fdiv_rn(1.0f, __fmul_rn(s_g, gw1[e]));
}

// gs2 = RN(2688 / amax) from the running amax|h| of the W1 epilogues, and alpha2[e] = RN(1 / RN(gs2 * gw2[e])),
// in one CTA; then the running amax is cleared. With no h since the last refresh (amax 0) gs2 and alpha2 stay.
__global__ void __launch_bounds__(256) refresh_gs2_kernel(int E, float* amax_run, const float* __restrict__ gw2,
                                                          float* gs2, float* __restrict__ alpha2) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_g;
  if (threadIdx.x == 0) {
    const float a = *(volatile float*)amax_run;
    s_g = a > 0.0f ? global_scale_from_amax(a) : 0.0f;
    if (a > 0.0f) gs2[0] = s_g;
  }
  __syncthreads();
  if (s_g > 0.0f)
    for (int e = threadIdx.x; e < E; e += blockDim.x) alpha2[e] = __fdiv_rn(1.0f, __fmul_rn(s_g, gw2[e]));
  __syncthreads();
  if (threadIdx.x == 0) *amax_run = 0.0f;
}

}  // namespace

fp4moe_status refresh_gs2_launch(int32_t E, float* amax_run, const float* gw2, float* gs2, float* alpha2,
                                 cudaStream_t st) {
  return launch_pdl(refresh_gs2_kernel, dim3(1), dim3(256), 0, st, (int)E, amax_run, gw2, gs2, alpha2) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

fp4moe_status batch_gs1_launch(int32_t T, int32_t H, const uint16_t* x, int32_t E, const float* gw1, float* gs1,
                               float* alpha1, unsigned int* acc, unsigned int* done, cudaStream_t st) {
  const int64_t n = (int64_t)T * H;
  const int64_t want = (n + 256 * 16 - 1) / (256 * 16);
  const unsigned bx = (unsigned)(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  return launch_pdl(batch_gs1_kernel, dim3(bx), dim3(256), 0, st, n, x, (int)E, gw1, gs1, alpha1, acc, done) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}


fp4moe_status quant_scatter_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const float* gs1,
                                   const int32_t* slot_of_pair, uint8_t* a1, uint8_t* a1_sf, uint32_t* status,
                                   uint32_t* err, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int64_t threads = (int64_t)T * (cfg.hidden / 16);
  return launch_pdl(quant_scatter_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, T, cfg.hidden,
                    cfg.top_k, x, gs1, slot_of_pair, a1, a1_sf, status, err) == cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

fp4moe_status quant_rows_launch(int64_t n_rows_total, int32_t K, int32_t rows_per_group, int32_t inter,
                                int32_t tiled, const float* in, const float* g, int32_t g_div, uint8_t* codes,
                                uint8_t* sf, cudaStream_t st) {
  if (n_rows_total == 0) return FP4MOE_OK;
  const int64_t blocks = (n_rows_total + 7) / 8;
  quant_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(n_rows_total, K, rows_per_group, inter, tiled, in, g, g_div,
                                                      codes, sf);
  return last_status();
}

fp4moe_status amax_f32_launch(int32_t n_groups, int64_t per_group, const float* in, float* amax, cudaStream_t st) {
  if (n_groups == 0) return FP4MOE_OK;
  if (cudaMemsetAsync(amax, 0, sizeof(float) * n_groups, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  const int64_t want = (per_group + 256 * 16 - 1) / (256 * 16);
  const unsigned bx = (unsigned)(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  amax_f32_kernel<<<dim3(bx, n_groups), 256, 0, st>>>(per_group, in, amax);
  return last_status();
}

fp4moe_status amax_bf16_launch(int64_t n, const uint16_t* in, float* amax, cudaStream_t st) {
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  if (n == 0) return FP4MOE_OK;
  const int64_t want = (n + 256 * 16 - 1) / (256 * 16);
  const unsigned bx = (unsigned)(want < 1 ? 1 : (want > 2048 ? 2048 : want));
  amax_bf16_kernel<<<bx, 256, 0, st>>>(n, in, amax);
  return last_status();
}

fp4moe_status gs_from_amax_launch(int32_t n, float* inout, cudaStream_t st) {
  if (n == 0) return FP4MOE_OK;
  gs_from_amax_kernel<<<(n + 255) / 256, 256, 0, st>>>(n, inout);
  return last_status();
}

fp4moe_status make_alpha_launch(int32_t n, const float* gs_act, const float* gs_w, float* alpha, cudaStream_t st) {
  if (n == 0) return FP4MOE_OK;
  make_alpha_kernel<<<(n + 255) / 256, 256, 0, st>>>(n, gs_act, gs_w, alpha);
  return last_status();
}

}  // namespace fp4moe
