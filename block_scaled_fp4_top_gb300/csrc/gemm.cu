// Block-scaled NVFP4 grouped GEMMs on the 5th-generation tensor cores (tcgen05).
//
// This is the grouped GEMM of "Current Bug: CuTeDSLMoERunner" ("Data Flow":
// run_nvfp4_grouped_gemm for L1 and L2). The A operand is slot-ordered
// activations: each expert's rows start on a 128-row boundary, and the
// scales are swizzled per 128-row block ("Bug 1", "Bug 14"). The B operand is
// each expert's K-major weights. Tile -> expert uses
// searchsorted(padded_offsets, row, right=True) on offsets with no leading 0
// ("Bug 2", "Bug 4").
//
// One CTA computes one 128 (rows) x 128 (weight rows) output tile:
//   warp 4      TMA producer. FP4 tiles come in by cp.async.bulk.tensor with
//               the 128-byte swizzle, and the 512-byte scale tiles by plain
//               cp.async.bulk, all into a STAGES-deep shared-memory ring.
//   warp 5      MMA issuer. tcgen05.cp moves the scale tiles into TMEM, then
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X issues
//               (K = 64 per instruction, fp32 accumulator in TMEM), and
//               tcgen05.commit frees the ring slot.
//   warps 0-3   epilogue. tcgen05.ld brings one accumulator row per thread.
//     W1: alpha, then the clamped SwiGLU (gate columns 0-63, up columns
//         64-127, from the W1 kernel row order), then NVFP4 requantisation
//         into the L2 slot buffers ("Bug 6", "Bug 7").
//     W1 amax: the same SwiGLU, reduced to amax|h| for calibration.
//     W2: alpha, then fp32 rows stored per (token, k) pair. Padding rows are
//         dropped ("Bug 14").
// Every spin-wait is bounded (mbar_wait). A timeout sets FP4MOE_ERR_TIMEOUT
// in the error word. The CTA then drains its in-flight copies and MMAs,
// frees its TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int BM = 128;            // activation rows per tile (MMA M)
constexpr int BN = 128;            // weight rows per tile (MMA N)
constexpr int KBYTES = 128;        // K bytes per stage: 256 FP4 elements = 4 MMAs of K = 64
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * KBYTES;
constexpr int B_BYTES = BN * KBYTES;
constexpr int SF_TILE = 512;       // one 128x4 scale tile
constexpr int SFA_OFF = A_BYTES + B_BYTES;
constexpr int SFB_OFF = SFA_OFF + 4 * SF_TILE;
constexpr int STAGE_BYTES = SFB_OFF + 4 * SF_TILE;  // 36864, a multiple of 1024
constexpr int BAR_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;    // barriers + 1024-byte alignment slack
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t ACC_COL = 0;    // accumulator: columns [0, 128)
constexpr uint32_t SF_COL = 128;   // per stage: 32 columns, [0,16) A scales, [16,32) B scales
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(SF_COL + STAGES * 32 <= TMEM_COLS, "TMEM budget");

struct Params {
  int E, K, b_rows, NT, k, cap, I, H;
  float limit;
  const int32_t* poff;
  const int32_t* pair_of_row;
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const float* alpha;
  const float* gs2;
  uint8_t* out_codes;
  uint8_t* out_sf;
  float* amax;
  float* o_pairs;
  uint32_t* err;
};

// Bounded wait that ignores other CTAs' aborts: used only while draining.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ float swiglu(float g, float u, float L) {
  const float gc = fminf(g, L);
  const float uc = fminf(fmaxf(u, -L), L);
  return __fmul_rn(__fdiv_rn(gc, __fadd_rn(1.0f, expf(-gc))), uc);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 2)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;

  if (*(volatile uint32_t*)prm.err & kAbortMask) return;  // an earlier timeout poisons the call

  // ---- tile -> (expert, n-tile, m-tile): experts in order, then n-tiles, then the expert's m-tiles
  const int E = prm.E, NT = prm.NT;
  const int R = min(__ldg(prm.poff + E - 1), prm.cap);
  const int tau = blockIdx.x;
  if (tau >= (R / BM) * NT) return;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((__ldg(prm.poff + mid) / BM) * NT > tau) hi = mid;
    else lo = mid + 1;
  }
  const int e = lo;
  const int mt_end = __ldg(prm.poff + e) / BM;
  const int mt_start = e > 0 ? __ldg(prm.poff + e - 1) / BM : 0;
  const int m_e = mt_end - mt_start;
  const int local = tau - mt_start * NT;
  const int nt = local / m_e;
  const int mt = mt_start + local % m_e;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem + BAR_OFF;         // STAGES x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * STAGES;  // STAGES x 8 bytes
  const uint32_t bar_acc = bar_empty + 8 * STAGES;
  const uint32_t bar_drain = bar_acc + 8;

  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    mbar_init(bar_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  const int K = prm.K;
  const int KB = (K + 255) / 256;   // stages of 256 elements
  const int katoms_total = K / 64;  // 64-element scale atoms along K

  if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();  // weights stream through once
    const uint64_t pol_a = policy_evict_last();   // activations are re-read by every n-tile
    const int a_row = mt * BM;
    const int b_row = e * prm.b_rows + nt * BN;
    const uint8_t* sfa = prm.a_sf + (size_t)mt * katoms_total * SF_TILE;
    const uint8_t* sfb = prm.b_sf + ((size_t)e * (prm.b_rows / 128) + nt) * katoms_total * SF_TILE;
    int issued = 0;
    bool ok = true;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
      if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, prm.err)) {
        ok = false;
        break;
      }
      const int atoms = min(4, katoms_total - kb * 4);
      const uint32_t st = smem + s * STAGE_BYTES;
      mbar_arrive_expect_tx(bar_full + 8 * s, A_BYTES + B_BYTES + 2 * atoms * SF_TILE);
      tma_load_2d(st, &tmA, bar_full + 8 * s, kb * KBYTES, a_row, pol_a);
      tma_load_2d(st + A_BYTES, &tmB, bar_full + 8 * s, kb * KBYTES, b_row, pol_w);
      bulk_load(st + SFA_OFF, sfa + (size_t)kb * 4 * SF_TILE, atoms * SF_TILE, bar_full + 8 * s, pol_a);
      bulk_load(st + SFB_OFF, sfb + (size_t)kb * 4 * SF_TILE, atoms * SF_TILE, bar_full + 8 * s, pol_w);
      issued = kb + 1;
    }
    (void)ok;  // on every path, let the copies already issued land before the CTA exits
    for (int kb = max(0, issued - STAGES); kb < issued; ++kb)
      drain_wait(bar_full + 8 * (kb % STAGES), (uint32_t)(kb / STAGES) & 1u);
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_nvf4(BM, BN);
    bool ok = true, any = false;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
      if (!mbar_wait(bar_full + 8 * s, ph, prm.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int atoms = min(4, katoms_total - kb * 4);
      const uint32_t st = smem + s * STAGE_BYTES;
      const uint32_t sfa_t = tmem + SF_COL + 32 * s;
      const uint32_t sfb_t = sfa_t + 16;
      for (int a = 0; a < atoms; ++a) {
        tc_cp_scales(sfa_t + 4 * a, desc_scales(st + SFA_OFF + a * SF_TILE));
        tc_cp_scales(sfb_t + 4 * a, desc_scales(st + SFB_OFF + a * SF_TILE));
      }
      for (int a = 0; a < atoms; ++a) {
        tc_mma_nvf4(tmem + ACC_COL, desc_sw128(st + a * 32), desc_sw128(st + A_BYTES + a * 32), idesc, sfa_t + 4 * a,
                    sfb_t + 4 * a, (kb > 0 || a > 0) ? 1u : 0u);
      }
      any = true;
      tc_commit(bar_empty + 8 * s);
    }
    if (ok) {
      tc_commit(bar_acc);
      drain_wait(bar_acc, 0);  // no MMA may still write TMEM when it is freed
    } else if (any) {
      tc_commit(bar_drain);
      drain_wait(bar_drain, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int r = mt * BM + warp * 32 + lane;
    const int p = __ldg(prm.pair_of_row + r);
    const float alpha = __ldg(prm.alpha + e);
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16) + ACC_COL;
    // the whole warp takes one decision: tcgen05.ld is warp-collective
    if (__all_sync(0xFFFFFFFFu, mbar_wait(bar_acc, 0, prm.err) ? 1 : 0)) {
      tc_fence_after();
      if constexpr (MODE == kW2Rows) {
        float* dst = prm.o_pairs + (size_t)(p < 0 ? 0 : p) * prm.H + nt * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tl + c * 32, v);
          tmem_ld_wait();
          if (p >= 0) {
            float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              d4[q] = make_float4(__fmul_rn(v[4 * q], alpha), __fmul_rn(v[4 * q + 1], alpha),
                                  __fmul_rn(v[4 * q + 2], alpha), __fmul_rn(v[4 * q + 3], alpha));
          }
        }
      } else {
        const float L = prm.limit;
        const float g2 = (MODE == kW1SwiGLU) ? __ldg(prm.gs2) : 1.0f;
        uint32_t codes[8];
        uint32_t sfw = 0;
        float hmax = 0.0f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float g[32], u[32];
          tmem_ld32(tl + half * 32, g);
          tmem_ld32(tl + 64 + half * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              h[j] = swiglu(__fmul_rn(g[blk * 16 + j], alpha), __fmul_rn(u[blk * 16 + j], alpha), L);
            if constexpr (MODE == kW1Amax) {
#pragma unroll
              for (int j = 0; j < 16; ++j) hmax = fmaxf(hmax, fabsf(h[j]));
            } else {
              uint32_t lo2, hi2;
              const uint32_t sf = quant_block16(h, g2, lo2, hi2);
              codes[half * 4 + blk * 2] = lo2;
              codes[half * 4 + blk * 2 + 1] = hi2;
              sfw |= sf << (8 * (half * 2 + blk));
            }
          }
        }
        if constexpr (MODE == kW1Amax) {
          if (p < 0) hmax = 0.0f;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) hmax = fmaxf(hmax, __shfl_xor_sync(0xFFFFFFFFu, hmax, off));
          if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(prm.amax), __float_as_uint(hmax));
        } else {
          if (p < 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) codes[q] = 0u;
            sfw = 0u;
          }
          uint4* dst = reinterpret_cast<uint4*>(prm.out_codes + (size_t)r * (prm.I >> 1) + nt * 32);
          dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
          dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
          *reinterpret_cast<uint32_t*>(prm.out_sf + sf_offset(r, nt * 4, prm.I >> 4)) = sfw;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------ host side --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor [rows][inner_bytes], 128-byte-swizzled boxes of box_rows x 128 bytes.
bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {(cuuint32_t)KBYTES, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
bool configure_once() {
  static int ok = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) ==
                 cudaSuccess
             ? 1
             : 0;
  });
  return ok == 1;
}

}  // namespace

fp4moe_status gemm_launch(GemmMode mode, const fp4moe_config& cfg, int32_t T, const uint8_t* a_codes,
                          const uint8_t* a_sf, const int32_t* poff, const int32_t* pair_of_row,
                          const uint8_t* b_codes, const uint8_t* b_sf, const float* alpha, const float* gs2,
                          uint8_t* out_codes, uint8_t* out_sf, float* amax, float* o_pairs, uint32_t* err,
                          cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const bool w2 = (mode == kW2Rows);
  Params prm;
  prm.E = cfg.num_experts;
  prm.K = w2 ? cfg.inter : cfg.hidden;
  prm.b_rows = w2 ? cfg.hidden : 2 * cfg.inter;
  prm.NT = prm.b_rows / BN;
  prm.k = cfg.top_k;
  prm.cap = (int)capacity_rows(cfg, T);
  prm.I = cfg.inter;
  prm.H = cfg.hidden;
  prm.limit = cfg.swiglu_limit;
  prm.poff = poff;
  prm.pair_of_row = pair_of_row;
  prm.a_sf = a_sf;
  prm.b_sf = b_sf;
  prm.alpha = alpha;
  prm.gs2 = gs2;
  prm.out_codes = out_codes;
  prm.out_sf = out_sf;
  prm.amax = amax;
  prm.o_pairs = o_pairs;
  prm.err = err;
  CUtensorMap tmA, tmB;
  if (!encode_u8_sw128(&tmA, a_codes, (uint64_t)prm.K / 2, (uint64_t)prm.cap, BM)) return FP4MOE_CUDA_ERROR;
  if (!encode_u8_sw128(&tmB, b_codes, (uint64_t)prm.K / 2, (uint64_t)prm.E * prm.b_rows, BN))
    return FP4MOE_CUDA_ERROR;
  const unsigned grid = (unsigned)((prm.cap / BM) * prm.NT);
  switch (mode) {
    case kW1SwiGLU:
      if (!configure_once<kW1SwiGLU>()) return FP4MOE_CUDA_ERROR;
      grouped_gemm_kernel<kW1SwiGLU><<<grid, THREADS, SMEM_BYTES, st>>>(tmA, tmB, prm);
      break;
    case kW1Amax:
      if (!configure_once<kW1Amax>()) return FP4MOE_CUDA_ERROR;
      grouped_gemm_kernel<kW1Amax><<<grid, THREADS, SMEM_BYTES, st>>>(tmA, tmB, prm);
      break;
    case kW2Rows:
      if (!configure_once<kW2Rows>()) return FP4MOE_CUDA_ERROR;
      grouped_gemm_kernel<kW2Rows><<<grid, THREADS, SMEM_BYTES, st>>>(tmA, tmB, prm);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
