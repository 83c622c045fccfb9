// GPU twin of the seeded generator in synthgen/__init__.py.
//
// It draws the same numbers, bit for bit, so that large synthetic tensors can
// be made directly in device memory. The definitions are the ones documented
// in the Python module:
//   SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) counter streams:
//     key = mix64(seed * GOLDEN + tensor_id),
//     word(i) = mix64(key + (i + 1) * GOLDEN)
//   Irwin-Hall(4 x 16 bit) unit normal: z = f32(S - 131070) * f32(sqrt(3)/65536)
//   value = f32(z * sigma). Optional Bernoulli(p) outlier mask from a second
//   stream (high 32 bits < thr) multiplies by `mult`. bf16 output uses RNE.
// This module holds no arithmetic of the MoE layer.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint32_t kIhScaleBits = 0x37DDB3D7u;  // fp32 sqrt(3)/65536
constexpr int64_t kIhCentre = 131070;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float unit_normal(uint64_t key, uint64_t i) {
  const uint64_t r = mix64(key + (i + 1) * kGolden);
  const int64_t s = (int64_t)(r & 0xFFFF) + (int64_t)((r >> 16) & 0xFFFF) + (int64_t)((r >> 32) & 0xFFFF) +
                    (int64_t)(r >> 48);
  return __fmul_rn(__int2float_rn((int)(s - kIhCentre)), __uint_as_float(kIhScaleBits));
}

__global__ void normal_f32_kernel(uint64_t key, uint64_t start, uint64_t count, float sigma, float* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = __fmul_rn(unit_normal(key, start + i), sigma);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t okey, uint32_t thr, float mult, uint64_t start,
                                   uint64_t count, float sigma, uint16_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count;
       i += (uint64_t)gridDim.x * blockDim.x) {
    float v = __fmul_rn(unit_normal(key, start + i), sigma);
    if (thr != 0u && (uint32_t)(mix64(okey + (start + i + 1) * kGolden) >> 32) < thr) v = __fmul_rn(v, mult);
    out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

inline unsigned grid_for(uint64_t count) {
  const uint64_t g = (count + 255) / 256;
  return (unsigned)(g < 1 ? 1 : (g > 65536 ? 65536 : g));
}

}  // namespace

extern "C" {

uint64_t synth_stream_key(uint64_t seed, uint64_t tensor_id) { return mix64(seed * kGolden + tensor_id); }

// out[i] = sigma * N(start + i) of stream (seed, tensor_id); returns a cudaError_t value.
int synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count, float sigma, float* out,
                     void* stream) {
  if (count == 0) return 0;
  normal_f32_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(synth_stream_key(seed, tensor_id), start,
                                                                        count, sigma, out);
  return (int)cudaGetLastError();
}

// bf16 bits of sigma * N(...), times `mult` where the outlier stream (seed, outlier_id) word is below thr.
int synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t outlier_id, uint32_t thr, float mult,
                      uint64_t start, uint64_t count, float sigma, uint16_t* out, void* stream) {
  if (count == 0) return 0;
  normal_bf16_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(
      synth_stream_key(seed, tensor_id), synth_stream_key(seed, outlier_id), thr, mult, start, count, sigma, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
