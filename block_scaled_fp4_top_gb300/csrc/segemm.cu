// The shared expert: a dense SwiGLU FFN with block-FP8 weights, beside the routed experts.
//
// DeepSeek-V4-Flash has one shared expert of intermediate size 2048 ("Lucifer-CUTLASS TP3
// virtual-padding audit", "TP3 shape plan"; 768 per rank under TP3). Its weights and scales are
// block-FP8 ("Paths that already appear compatible"), and it runs in the same captured step as
// the router and the routed MoE ("DSV4 -> vLLM: CUDA-Graph Safety", Graph B). Block-FP8 is read
// as in the DeepSeek-V3 technical report's FP8 recipe: E4M3 values with one fp32 scale per
// 128 x 128 weight block and one per 1 x 128 activation group along K, s = RN(amax / 448).
//
// Three kernels:
//   se_quant_x_kernel   x (bf16) -> E4M3 codes and fp32 scales per 1 x 128 group, one warp per group.
//   se_gemm_kernel<0>   W1: [g | u] = x~ W1~^T, the clamped SwiGLU, and h requantised per 1 x 128 group.
//   se_gemm_kernel<1>   W2: o = h~ W2~^T as fp32 rows [T][H], added by the combine.
//
// The GEMM is a dense contraction over fp32-scaled blocks, so the tensor cores multiply the E4M3
// codes (tcgen05.mma kind::f8f6f4, fp32 accumulation) one 128-wide K block at a time, and the
// epilogue warps apply the two scales and accumulate on the CUDA cores:
//   acc[t, n] += sa[t, kb] * sw[n / 128, kb] * P_kb[t, n],  P_kb = sum over the block of qa * qw.
// A tile is 128 tokens x 256 weight rows. W1's kernel row order puts the gate and up rows of the
// same 128 features in one tile (rows 256 j .. 256 j + 127 are gate features 128 j .., the next
// 128 are up), so the SwiGLU and the h group amax stay inside one CTA.
//   producer (warp 8)      TMA: the activation block (128 rows x 128 bytes) and the weight block
//                          (256 rows x 128 bytes), both 128-byte swizzled, into a 4-stage ring.
//   MMA issuer (warp 9)    4 MMAs of K = 32 per block into one of two TMEM partial buffers
//                          (256 columns each); a fresh accumulation for every K block.
//   epilogue (warps 0-7)   warp w reads TMEM lanes 32 (w % 4) .. +31 (its token rows) and half
//                          w / 4 of the columns: 128 fp32 accumulators per thread in registers.
// Every wait is bounded, as in the routed GEMMs; a timeout sets FP4MOE_ERR_TIMEOUT and skips work.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {

bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows);

namespace {

constexpr int SE_BM = 128;                       // token rows per tile (MMA M)
constexpr int SE_BN = 256;                       // weight rows per tile (MMA N)
constexpr int SE_BK = 128;                       // K elements (bytes) per block: one swizzle atom
constexpr int SE_A_BYTES = SE_BM * SE_BK;        // 16 KB
constexpr int SE_B_BYTES = SE_BN * SE_BK;        // 32 KB
constexpr int SE_STAGE = SE_A_BYTES + SE_B_BYTES;
constexpr int SE_STAGES = 4;
constexpr int SE_BAR_OFF = SE_STAGES * SE_STAGE;
constexpr int SE_SMEM = SE_BAR_OFF + 256 + 1024;  // barriers + 1024-byte alignment slack
constexpr int SE_THREADS = 320;                  // 8 epilogue warps, producer, MMA issuer
constexpr uint32_t SE_TMEM_COLS = 512;           // two 256-column partial products
static_assert(SE_STAGE % 1024 == 0 && SE_A_BYTES % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(SE_SMEM + 2 * SE_BM * 4 + 64 <= 232448, "shared memory budget (dynamic + static)");

struct SeMaps {
  CUtensorMap a;  // activation codes [T][K] u8, box 128 rows x 128 bytes
  CUtensorMap b;  // weight codes [N][K] u8, box 256 rows x 128 bytes
};

struct SeParams {
  int T, KB, tcap;
  float limit;
  const float* a_scale;  // [KB][tcap]
  const float* w_scale;  // [N / 128][KB], kernel row-block order
  uint8_t* h_codes;      // W1: [tcap][I] E4M3
  float* h_scale;        // W1: [I / 128][tcap]
  int I;
  float* out;            // W2: [T][H] fp32
  int H;
  uint32_t* err;
};

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 with fp32 accumulation (kind::f8f6f4, K = 32).
__device__ __forceinline__ void tc_mma_f8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor: kind::f8f6f4 with fp32 D, A and B E4M3 (format 0), both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) { return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24); }

// silu(min(g, L)) * clamp(u, -L, L), as in the routed experts
__device__ __forceinline__ float swiglu(float g, float u, float L) {
  const float gc = fmaxf(fminf(g, L), -80.0f);
  const float uc = fminf(fmaxf(u, -L), L);
  return __fdividef(gc, 1.0f + __expf(-gc)) * uc;
}

// Two E4M3 codes (RNE, satfinite) of lo / s and hi / s in the low 16 bits, lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_scaled(float lo, float hi, float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(__fdiv_rn(hi, s)), "f"(__fdiv_rn(lo, s)));
  return r;
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// One warp per (token, 1 x 128 group): s = RN(amax / 448), codes E4M3(RN(v / s)), 0 where s == 0.
__global__ void __launch_bounds__(256) se_quant_x_kernel(int T, int H, int tcap, const uint16_t* __restrict__ x,
                                                         uint8_t* __restrict__ qx, float* __restrict__ sx) {
  pdl_wait();
  pdl_trigger();
  const int G = H / 128;
  const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (gw >= (int64_t)T * G) return;
  const int t = (int)(gw / G), g = (int)(gw - (int64_t)t * G);
  const int lane = threadIdx.x & 31;
  const size_t off = (size_t)t * H + (size_t)g * 128 + 4 * lane;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + off));
  const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
  float a = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  const float s = __fdiv_rn(a, 448.0f);
  const uint32_t c = s == 0.0f ? 0u : (e4m3x2_scaled(v0, v1, s) | (e4m3x2_scaled(v2, v3, s) << 16));
  *reinterpret_cast<uint32_t*>(qx + off) = c;
  if (lane == 0) sx[(size_t)g * tcap + t] = s;
}

template <int MODE>
__global__ void __launch_bounds__(SE_THREADS, 1)
    se_gemm_kernel(const __grid_constant__ SeMaps maps, const SeParams prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ float s_amax[2][SE_BM];  // W1: amax of each half of a row's 128 h features

  pdl_wait();
  pdl_trigger();
  if (*(volatile uint32_t*)prm.err & kAbortMask) return;
  const int nt = blockIdx.x, mt = blockIdx.y, KB = prm.KB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem + SE_BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * SE_STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * SE_STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;

  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), SE_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int s = 0; s < SE_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 8);  // one arrive per epilogue warp
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = policy_evict_normal();                              // read by every n-tile
    const uint64_t pol_b = gridDim.y == 1 ? policy_evict_first() : policy_evict_last();  // re-read per m-tile
    int kb = 0;
    for (; kb < KB; ++kb) {
      const int s = kb % SE_STAGES;
      if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(kb / SE_STAGES) & 1u) ^ 1u, prm.err)) break;
      const uint32_t st = smem + s * SE_STAGE;
      mbar_arrive_expect_tx(bar_full + 8 * s, SE_STAGE);  // rows past T are zero-filled and still counted
      tma_load_2d(st, &maps.a, bar_full + 8 * s, kb * SE_BK, mt * SE_BM, pol_a);
      tma_load_2d(st + SE_A_BYTES, &maps.b, bar_full + 8 * s, kb * SE_BK, nt * SE_BN, pol_b);
    }
    // on every path, let the copies already issued land before the CTA exits
    for (int j = max(0, kb - SE_STAGES); j < kb; ++j)
      drain_wait(bar_full + 8 * (j % SE_STAGES), (uint32_t)(j / SE_STAGES) & 1u);
  } else if (warp == 9 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_e4m3(SE_BM, SE_BN);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % SE_STAGES, b = kb & 1;
      if (!mbar_wait(bar_tempty + 8 * b, ((uint32_t)(kb >> 1) & 1u) ^ 1u, prm.err)) break;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(kb / SE_STAGES) & 1u, prm.err)) break;
      tc_fence_after();
      const uint32_t st = smem + (uint32_t)s * SE_STAGE;
#pragma unroll
      for (int q = 0; q < 4; ++q)  // K = 32 E4M3 = 32 bytes per MMA
        tc_mma_f8(tmem + 256u * b, desc_sw128(st + 32 * q), desc_sw128(st + SE_A_BYTES + 32 * q), idesc,
                  q > 0 ? 1u : 0u);
      tc_commit(bar_empty + 8 * s);
      tc_commit(bar_tfull + 8 * b);
    }
    tc_commit(bar_drain);
    drain_wait(bar_drain, 0);  // no MMA may still write TMEM when it is freed
  } else if (warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3, hf = warp >> 2;
    const int row = mt * SE_BM + quad * 32 + lane;  // token
    const int rs = min(row, prm.tcap - 1);          // scale rows past T exist but hold no token
    // weight row blocks of this thread's columns: W1 gate block 2 nt and up block 2 nt + 1 (kernel order);
    // W2 block 2 nt + hf
    const int blk0 = MODE == 0 ? 2 * nt : 2 * nt + hf;
    const int blk1 = MODE == 0 ? 2 * nt + 1 : blk0;
    // this thread's four 32-column pieces of the 256: W1 gate 64 hf + 0/32, up 128 + 64 hf + 0/32;
    // W2 128 hf + 0/32/64/96
    const uint32_t c0 = MODE == 0 ? 64u * hf : 128u * hf;
    const uint32_t cols[4] = {c0, c0 + 32u, MODE == 0 ? 128u + c0 : c0 + 64u, MODE == 0 ? 160u + c0 : c0 + 96u};
    float acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
    bool ok = true;
    float sa_next = __ldg(prm.a_scale + rs);
    for (int kb = 0; kb < KB; ++kb) {
      const float sa = sa_next;
      if (kb + 1 < KB) sa_next = __ldg(prm.a_scale + (size_t)(kb + 1) * prm.tcap + rs);
      const float f0 = sa * __ldg(prm.w_scale + (size_t)blk0 * KB + kb);
      const float f1 = sa * __ldg(prm.w_scale + (size_t)blk1 * KB + kb);
      const int b = kb & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull + 8 * b, (uint32_t)(kb >> 1) & 1u, prm.err) ? 1 : 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + 256u * b + ((uint32_t)(quad * 32) << 16);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tb + cols[c], v);
        tmem_ld_wait();
        const float f = c < 2 ? f0 : f1;
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * c + i] = fmaf(v[i], f, acc[32 * c + i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
    }
    if constexpr (MODE == 0) {
      // h for features 128 nt + 64 hf .. + 63: gate in acc[0..63], up in acc[64..127]
      const float L = prm.limit;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        acc[i] = swiglu(acc[i], acc[64 + i], L);
        amax = fmaxf(amax, fabsf(acc[i]));
      }
      s_amax[hf][quad * 32 + lane] = amax;
      named_sync(1, 256);  // every epilogue warp comes here exactly once, also after a timeout
      amax = fmaxf(amax, s_amax[hf ^ 1][quad * 32 + lane]);
      const float s = __fdiv_rn(amax, 448.0f);
      if (ok && row < prm.T) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = s == 0.0f ? 0u
                           : (e4m3x2_scaled(acc[4 * i], acc[4 * i + 1], s) |
                              (e4m3x2_scaled(acc[4 * i + 2], acc[4 * i + 3], s) << 16));
        uint4* dst = reinterpret_cast<uint4*>(prm.h_codes + (size_t)row * prm.I + 128 * nt + 64 * hf);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        if (hf == 0) prm.h_scale[(size_t)nt * prm.tcap + row] = s;
      }
    } else {
      if (ok && row < prm.T) {
        float4* dst = reinterpret_cast<float4*>(prm.out + (size_t)row * prm.H + SE_BN * nt + 128 * hf);
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, SE_TMEM_COLS);
  }
}

// One CTA per 128 x 128 weight block: s = RN(amax / 448), codes E4M3(RN(w / s)), 0 where s == 0.
// W1 (inter > 0): logical rows [0, I) gate and [I, 2I) up go to kernel row blocks 2 j and 2 j + 1.
__global__ void __launch_bounds__(256) se_quant_weights_kernel(int K, int inter, const float* __restrict__ w,
                                                               uint8_t* __restrict__ codes, float* __restrict__ scales) {
  __shared__ float s_red[8];
  const int KB = K / 128;
  const int bi = blockIdx.y, bk = blockIdx.x;  // logical row block, K block
  int kbi = bi;                                // kernel row block
  if (inter > 0) {
    const int ib = inter / 128;
    kbi = bi < ib ? 2 * bi : 2 * (bi - ib) + 1;
  }
  // thread: row 128 bi + threadIdx.x / 2, 64 elements from column 128 bk + 64 (threadIdx.x & 1)
  const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
  const float* src = w + ((size_t)bi * 128 + r) * K + (size_t)bk * 128 + 64 * h;
  float v[64];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(src + i));
    v[i] = q.x;
    v[i + 1] = q.y;
    v[i + 2] = q.z;
    v[i + 3] = q.w;
    a = fmaxf(a, fmaxf(fmaxf(fabsf(q.x), fabsf(q.y)), fmaxf(fabsf(q.z), fabsf(q.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = s_red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, s_red[i]);
  const float s = __fdiv_rn(a, 448.0f);
  uint32_t out[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    out[i] = s == 0.0f ? 0u : (e4m3x2_scaled(v[4 * i], v[4 * i + 1], s) | (e4m3x2_scaled(v[4 * i + 2], v[4 * i + 3], s) << 16));
  uint4* dst = reinterpret_cast<uint4*>(codes + ((size_t)kbi * 128 + r) * K + (size_t)bk * 128 + 64 * h);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
  if (threadIdx.x == 0) scales[(size_t)kbi * KB + bk] = s;
}

template <int MODE>
bool configure_se() {
  static int ok = -1;
  if (ok < 0)
    ok = cudaFuncSetAttribute(se_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SE_SMEM) ==
                 cudaSuccess
             ? 1
             : 0;
  return ok == 1;
}

}  // namespace

size_t se_tcap(const fp4moe_config& cfg) {
  const size_t t = (size_t)(cfg.max_tokens > 0 ? cfg.max_tokens : 1);
  return (t + SE_BM - 1) / SE_BM * SE_BM;
}

fp4moe_status se_quant_weights_launch(const fp4moe_config& cfg, int32_t which, const float* w, uint8_t* codes,
                                      float* scales, cudaStream_t st) {
  const int Is = cfg.shared_inter, H = cfg.hidden;
  const int rows = which == 1 ? 2 * Is : H, K = which == 1 ? H : Is;
  se_quant_weights_kernel<<<dim3(K / 128, rows / 128), 256, 0, st>>>(K, which == 1 ? Is : 0, w, codes, scales);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

fp4moe_status se_forward_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint8_t* w1,
                                const float* s1, const uint8_t* w2, const float* s2, uint8_t* qx, float* sx,
                                uint8_t* qh, float* sh, float* out, uint32_t* err, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden, Is = cfg.shared_inter;
  const int tcap = (int)se_tcap(cfg);
  const int64_t groups = (int64_t)T * (H / 128);
  if (launch_pdl(se_quant_x_kernel, dim3((unsigned)((groups + 7) / 8)), dim3(256), 0, st, T, H, tcap, x, qx, sx) !=
      cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  if (!configure_se<0>() || !configure_se<1>()) return FP4MOE_CUDA_ERROR;
  const unsigned mt = (unsigned)((T + SE_BM - 1) / SE_BM);
  SeMaps m1, m2;
  if (!encode_u8_sw128(&m1.a, qx, (uint64_t)H, (uint64_t)T, SE_BM) ||
      !encode_u8_sw128(&m1.b, w1, (uint64_t)H, (uint64_t)2 * Is, SE_BN) ||
      !encode_u8_sw128(&m2.a, qh, (uint64_t)Is, (uint64_t)T, SE_BM) ||
      !encode_u8_sw128(&m2.b, w2, (uint64_t)Is, (uint64_t)H, SE_BN))
    return FP4MOE_CUDA_ERROR;
  SeParams p{};
  p.T = T;
  p.tcap = tcap;
  p.limit = cfg.swiglu_limit;
  p.I = Is;
  p.H = H;
  p.err = err;
  p.KB = H / 128;
  p.a_scale = sx;
  p.w_scale = s1;
  p.h_codes = qh;
  p.h_scale = sh;
  if (launch_pdl(se_gemm_kernel<0>, dim3((unsigned)(2 * Is / SE_BN), mt), dim3(SE_THREADS), SE_SMEM, st, m1, p) !=
      cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  p.KB = Is / 128;
  p.a_scale = sh;
  p.w_scale = s2;
  p.out = out;
  return launch_pdl(se_gemm_kernel<1>, dim3((unsigned)(H / SE_BN), mt), dim3(SE_THREADS), SE_SMEM, st, m2, p) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
