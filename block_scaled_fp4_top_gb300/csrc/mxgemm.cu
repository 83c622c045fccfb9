// Grouped GEMMs with MXFP4 expert weights and bf16 activations.
//
// This is the TP3 shard variant of "Lucifer-CUTLASS TP3 virtual-padding
// audit". Its section "Remaining kernel assumptions" fixes the case: BF16
// activations with MXFP4 weights, hidden 4096, logical local intermediate
// 704 in a kernel-local width of 768, 256 experts, top-k 6, swiglu_limit 10.
// The weights stay MXFP4 in HBM: E2M1 codes with one E8M0 scale per 32
// elements along K (OCP Microscaling v1.0). An E2M1 value times a power of
// two is exact in bf16, so four converter warps expand each weight tile to
// bf16 in shared memory. The tensor cores then multiply bf16 x bf16 with fp32
// accumulation (tcgen05.mma kind::f16). The products are the exact ones, and
// only the fp32 accumulation rounds.
//
// The tile order, the persistent CTAs and the real-row activation boxes are
// those of the NVFP4 kernel (gemm.cu, tiles.cuh). A ring stage is one
// 64-element K atom:
//   producer (warp 4)      TMA: the atom's activation rows (bf16, 128-byte
//                          swizzle); bulk copies: the weight atom's 4 KB of
//                          codes and 256 B of scales.
//   converters (warps 6-13) two threads expand weight row j into 128 bytes of
//                          bf16 in the tensor cores' 128-byte-swizzled layout:
//                          byte permutes map eight codes at a time to their
//                          exact bf16 patterns (integer ALU work, no
//                          conversion unit), and a bf16x2 multiply by the
//                          power of two applies the scale exactly.
//   MMA issuer (warp 5)    4 MMAs of K = 16 per atom into a TMEM accumulator
//                          (two buffers).
//   epilogue (warps 0-3)   W1: the clamped SwiGLU on gate columns 0-63 and up
//                          columns 64-127 (kernel row order), h rounded to
//                          bf16 into the W2 activation rows. W2: fp32 rows
//                          per (token, k) pair. Padding rows are skipped.
// Every wait is bounded, as in gemm.cu.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace fp4moe {

int sm_count();
bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows);

namespace {

constexpr int MX_BM = 128;                  // activation rows per tile
constexpr int MX_BN = 128;                  // weight rows per tile
constexpr int MX_A_OFF = 0;                 // bf16 activation atom: 128 rows x 128 bytes
constexpr int MX_BC_OFF = 16384;            // weight codes of the atom: 128 rows x 32 bytes
constexpr int MX_BS_OFF = 20480;            // weight scales of the atom: 128 rows x 2 bytes
constexpr int MX_BB_OFF = 24576;            // the converted bf16 weight atom: 128 rows x 128 bytes
constexpr int MX_BC_BYTES = MX_BN * 32;
constexpr int MX_BS_BYTES = MX_BN * 2;
constexpr int MX_STAGE = 40960;
constexpr int MX_STAGES = 5;
constexpr int MX_BAR_OFF = MX_STAGES * MX_STAGE;
constexpr int MX_SMEM = MX_BAR_OFF + 256 + 1024;
constexpr int MX_THREADS = 448;            // 4 epilogue, producer, MMA, 8 converter warps
constexpr uint32_t MX_TMEM_COLS = 256;      // two 128-column accumulators
static_assert(MX_STAGE % 1024 == 0 && MX_BB_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(MX_SMEM + 4 * kMaxExperts + 1024 + 64 <= 232448, "shared memory budget (dynamic + static)");

struct MxAMaps {
  CUtensorMap box[4];  // bf16 activation rows, boxes 16, 32, 64 and 128 rows high, 128 bytes wide
};

struct MxParams {
  int E, K, KA, NT, cap, I, H;
  float limit;
  const int32_t* poff;
  const int32_t* pair_of_row;
  const uint8_t* b_codes;
  const uint8_t* b_sf;
  uint16_t* out_bf16;  // W1: h rows [cap][I] bf16
  uint16_t* o_pairs;   // W2: bf16 rows [T*k][H]
  uint32_t* err;
};

__device__ __forceinline__ void cta_range(int total, int& tau0, int& tau1) {
  tau0 = (int)(((long long)total * blockIdx.x) / gridDim.x);
  tau1 = (int)(((long long)total * (blockIdx.x + 1)) / gridDim.x);
}

// Eight E2M1 codes (w, element i in bits 4i .. 4i+3) as eight bf16 values: out[i] holds elements 2i (low
// half) and 2i + 1. The magnitude index (bits 0-2) picks the low and the high byte of each bf16 pattern
// from two 8-byte tables with byte permutes; a multiply by a sum of two powers of two moves each code's
// sign bit (bit 3) to bit 15 or bit 31 of its word. The tables hold 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t (&out)[4]) {
  constexpr uint32_t kLo03 = 0xC0800000u, kLo47 = 0xC0804000u;  // low bytes of the bf16 patterns
  constexpr uint32_t kHi03 = 0x3F3F3F00u, kHi47 = 0x40404040u;  // high bytes
  const uint32_t m = w & 0x77777777u;                           // selector nibbles stay below 8
  const uint32_t lo0 = __byte_perm(kLo03, kLo47, m), hi0 = __byte_perm(kHi03, kHi47, m);
  const uint32_t lo1 = __byte_perm(kLo03, kLo47, m >> 16), hi1 = __byte_perm(kHi03, kHi47, m >> 16);
  const uint32_t wh = w >> 16;
  out[0] = __byte_perm(lo0, hi0, 0x5140) | (((w & 0x88u) * 0x01001000u) & 0x80008000u);
  out[1] = __byte_perm(lo0, hi0, 0x7362) | (((w & 0x8800u) * 0x00010010u) & 0x80008000u);
  out[2] = __byte_perm(lo1, hi1, 0x5140) | (((wh & 0x88u) * 0x01001000u) & 0x80008000u);
  out[3] = __byte_perm(lo1, hi1, 0x7362) | (((wh & 0x8800u) * 0x00010010u) & 0x80008000u);
}

// bf16x2 product; exact here, since one factor is a power of two
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

// bf16 bit pattern of the E8M0 scale 2^(s - 127) (255 is NaN; 0 is the subnormal 2^-127)
__device__ __forceinline__ uint32_t e8m0_bf16_bits(uint32_t s) {
  if (s == 255u) return 0x7FC0u;
  if (s == 0u) return 0x0040u;
  return s << 7;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

template <int MODE>
__global__ void __launch_bounds__(MX_THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ MxAMaps tmA, const MxParams prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_poff[kMaxExperts];

  pdl_wait();
  pdl_trigger();
  if (*(volatile uint32_t*)prm.err & kAbortMask) return;
  const int E = prm.E, NT = prm.NT, KA = prm.KA;
  const int R = min(__ldcg(prm.poff + E - 1), prm.cap);
  const int r128 = R / MX_BM;
  int tau0, tau1;
  cta_range(r128 * NT, tau0, tau1);
  if (tau0 >= tau1) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem - smem_u32(smem_raw));
  const uint32_t bar_full = smem + MX_BAR_OFF;
  const uint32_t bar_conv = bar_full + 8 * MX_STAGES;
  const uint32_t bar_empty = bar_conv + 8 * MX_STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * MX_STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;

  for (int e = threadIdx.x; e < E; e += MX_THREADS) s_poff[e] = __ldcg(prm.poff + e);
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), MX_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < MX_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_conv + 8 * s, 8);   // one arrive per converter warp
      mbar_init(bar_empty + 8 * s, 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);  // one arrive per epilogue warp
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_stages = (tau1 - tau0) * KA;

  if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_reuse = policy_evict_normal();
    TileCursor cur;
    cur.seek(tau0, s_poff, E, NT, r128);
    int it = 0, prev_mt = -1, a_box = 3;
    bool ok = true;
    for (int tau = tau0; tau < tau1 && ok; ++tau) {
      if (tau > tau0) cur.step(s_poff, E, NT, r128);
      const Tile t = cur.tile();
      const bool one = (t.me == 1);
      const uint64_t pol_w = one ? pol_once : pol_reuse;
      const uint64_t pol_a = one ? pol_keep : pol_reuse;
      const int a_row = t.mt * MX_BM;
      if (t.mt != prev_mt) {
        prev_mt = t.mt;
        a_box = 3;
        if (t.last) {  // the first padding row bounds the rows this m-tile needs (rows < R are all written)
          const int32_t* por = prm.pair_of_row + a_row;
          const int p16 = __ldcg(por + 16), p32 = __ldcg(por + 32), p64 = __ldcg(por + 64);
          a_box = p16 < 0 ? 0 : (p32 < 0 ? 1 : (p64 < 0 ? 2 : 3));
        }
      }
      const uint32_t a_bytes = (16u << a_box) * 128u;
      const size_t wblk = (size_t)(t.e * NT + t.nt) * KA;
      for (int kb = 0; kb < KA; ++kb, ++it) {
        const int s = it % MX_STAGES;
        if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(it / MX_STAGES) & 1u) ^ 1u, prm.err)) {
          ok = false;
          break;
        }
        const uint32_t st = smem + s * MX_STAGE;
        mbar_arrive_expect_tx(bar_full + 8 * s, a_bytes + MX_BC_BYTES + MX_BS_BYTES);
        tma_load_2d(st + MX_A_OFF, &tmA.box[a_box], bar_full + 8 * s, kb * 128, a_row, pol_a);
        bulk_load(st + MX_BC_OFF, prm.b_codes + (wblk + kb) * MX_BC_BYTES, MX_BC_BYTES, bar_full + 8 * s, pol_w);
        bulk_load(st + MX_BS_OFF, prm.b_sf + (wblk + kb) * MX_BS_BYTES, MX_BS_BYTES, bar_full + 8 * s, pol_w);
      }
    }
    // on every path, let the copies already issued land before the CTA exits
    for (int j = max(0, it - MX_STAGES); j < it; ++j)
      drain_wait(bar_full + 8 * (j % MX_STAGES), (uint32_t)(j / MX_STAGES) & 1u);
  } else if (warp >= 6) {
    // ------------------------------------------------------------ converters
    // thread t: weight row j = t % 128, elements 32 g .. 32 g + 31 (one E8M0 group) with g = t / 128
    const int t = threadIdx.x - 192;
    const int j = t & 127, g = t >> 7;
    for (int it = 0; it < n_stages; ++it) {
      const int s = it % MX_STAGES;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / MX_STAGES) & 1u, prm.err)) break;
      const uint8_t* stg = smem_gen + s * MX_STAGE;
      const uint4 cw = *reinterpret_cast<const uint4*>(stg + MX_BC_OFF + 32 * j + 16 * g);
      const uint32_t b = e8m0_bf16_bits(stg[MX_BS_OFF + 2 * j + g]);
      const uint32_t scl = b | (b << 16);
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
      uint8_t* dst_row = smem_gen + s * MX_STAGE + MX_BB_OFF + 128 * j;
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16-byte chunk c = 4 g + q holds elements 8c .. 8c + 7
        const int c = 4 * g + q;
        uint32_t o[4];
        e2m1x8_to_bf16(words[q], o);
        *reinterpret_cast<uint4*>(dst_row + ((c ^ (j & 7)) << 4)) =
            make_uint4(bf16x2_mul(o[0], scl), bf16x2_mul(o[1], scl), bf16x2_mul(o[2], scl), bf16x2_mul(o[3], scl));
      }
      fence_proxy_async_smem();  // the tensor cores read these bytes through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_conv + 8 * s);
    }
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(MX_BM, MX_BN);
    int tl = 0, s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tau = tau0; tau < tau1 && ok; ++tau, ++tl) {
      const int b = tl & 1;
      const uint32_t use = (uint32_t)(tl >> 1);
      if (!mbar_wait(bar_tempty + 8 * b, (use & 1u) ^ 1u, prm.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + 128u * b;
      for (int kb = 0; kb < KA; ++kb) {
        // the converters arrive only after the stage's copies landed and its weights were expanded
        if (!mbar_wait(bar_conv + 8 * s, ph, prm.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem + (uint32_t)s * MX_STAGE;
#pragma unroll
        for (int q = 0; q < 4; ++q)  // K = 16 bf16 = 32 bytes per MMA
          tc_mma_bf16(acc, desc_sw128(st + MX_A_OFF + 32 * q), desc_sw128(st + MX_BB_OFF + 32 * q), idesc,
                      (kb > 0 || q > 0) ? 1u : 0u);
        tc_commit(bar_empty + 8 * s);
        if (++s == MX_STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) tc_commit(bar_tfull + 8 * b);
    }
    tc_commit(bar_drain);
    drain_wait(bar_drain, 0);  // no MMA may still write TMEM when it is freed
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    int tl = 0;
    TileCursor cur;
    cur.seek(tau0, s_poff, E, NT, r128);
    for (int tau = tau0; tau < tau1; ++tau, ++tl) {
      if (tau > tau0) cur.step(s_poff, E, NT, r128);
      const Tile t = cur.tile();
      const int r = t.mt * MX_BM + warp * 32 + lane;
      const int p = __ldcg(prm.pair_of_row + r);
      const bool any_real = __any_sync(0xFFFFFFFFu, p >= 0);
      const int b = tl & 1;
      const uint32_t use = (uint32_t)(tl >> 1);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull + 8 * b, use & 1u, prm.err) ? 1 : 0)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + 128u * b + ((uint32_t)(warp * 32) << 16);
      // 32-column pieces keep the register footprint small enough for 448 threads; the accumulator is
      // released after the last piece (the other buffer takes the next tile meanwhile)
      if (any_real) {
        if constexpr (MODE == 0) {
          const float L = prm.limit;
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {  // features 32 q .. 32 q + 31 of this n-tile's 64
            float gv[32], uv[32];
            tmem_ld32(tacc + 32 * q, gv);
            tmem_ld32(tacc + 64 + 32 * q, uv);
            tmem_ld_wait();
            if (p >= 0) {
              uint32_t hw[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                hw[i] = pack_bf16x2(swiglu_clamped(gv[2 * i], uv[2 * i], L),
                                    swiglu_clamped(gv[2 * i + 1], uv[2 * i + 1], L));
              uint4* dst = reinterpret_cast<uint4*>(prm.out_bf16 + (size_t)r * prm.I + t.nt * 64 + 32 * q);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
            }
          }
        } else {
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            float v[32];
            tmem_ld32(tacc + 32 * q, v);
            tmem_ld_wait();
            if (p >= 0) {
              uint4* d4 = reinterpret_cast<uint4*>(prm.o_pairs + (size_t)p * prm.H + t.nt * MX_BN + 32 * q);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                   pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, MX_TMEM_COLS);
  }
}

template <int MODE>
bool configure_mx() {
  static int ok = -1;
  if (ok < 0)
    ok = cudaFuncSetAttribute(mx_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, MX_SMEM) ==
                 cudaSuccess
             ? 1
             : 0;
  return ok == 1;
}

// One thread per (row, 32-element block): the OCP MX scale X = floor(log2(amax)) - 2 (clamped to
// [-127, 127]; an all-zero block takes -127), E2M1 codes of v / 2^X with round-to-nearest-even and
// saturation, written into the atom-tiled weight layout.
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(int64_t n_rows, int K, int rows_per_group, int inter,
                                                            const float* __restrict__ in, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf) {
  const int nb = K / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rows * nb) return;
  const int64_t row = idx / nb;
  const int blk = (int)(idx - row * nb);
  const int64_t g = row / rows_per_group;
  const int lr = (int)(row - g * rows_per_group);
  int kr = lr;  // row in kernel order: W1 gate/up interleaved per 64 features
  if (inter > 0) {
    const bool up = lr >= inter;
    const int f = up ? lr - inter : lr;
    kr = 128 * (f / 64) + (up ? 64 : 0) + f % 64;
  }
  const float* src = in + row * (int64_t)K + blk * 32;
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 q = *reinterpret_cast<const float4*>(src + i);
    v[i] = q.x;
    v[i + 1] = q.y;
    v[i + 2] = q.z;
    v[i + 3] = q.w;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int X = -127;
  if (amax > 0.0f) {
    int e;
    frexpf(amax, &e);  // amax = m 2^e, m in [0.5, 1)
    X = min(127, max(-127, (e - 1) - 2));
  }
  const float inv = ldexpf(1.0f, -X);  // exact power of two
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t pair = cvt_e2m1x2(v[i] * inv, v[i + 1] * inv);
    w[i / 8] |= pair << (8 * ((i / 2) % 4));
  }
  const int ka = K / 64, rt = kr / 128, rr = kr % 128, atom = blk / 2;
  const size_t blk_idx = ((size_t)g * (rows_per_group / 128) + rt) * ka + atom;
  *reinterpret_cast<uint4*>(codes + blk_idx * MX_BC_BYTES + 32 * rr + 16 * (blk & 1)) = make_uint4(w[0], w[1], w[2], w[3]);
  sf[blk_idx * MX_BS_BYTES + 2 * rr + (blk & 1)] = (uint8_t)(X + 127);
}

// One rank's kernel-local shard cut from an already quantised full-width MXFP4 checkpoint ("Lucifer-CUTLASS
// TP3 virtual-padding audit", "Packed W2 weight is wrong", "W2 E8M0 scales are wrong", "Required loader
// changes"). The slice is counted in logical elements and read in each tensor's own storage unit: W13 in
// unpacked rows, packed W2 codes in bytes of 2 elements, E8M0 scales in groups of 32. Destinations past the
// rank's logical count get zero codes and zero scale bytes. One thread moves one 32-element group (16 code
// bytes and one scale byte) into the atom-tiled layout that the MX GEMMs read.
//   W13 (w1 = true): src codes [n][2 I_full][K / 2], scales [n][2 I_full][K / 32]; dest logical row lr of
//     [0, 2 Ik): gate rows [0, Ik), up rows [Ik, 2 Ik); the source row of kernel feature f < count is
//     (up ? I_full : 0) + first + f.
//   W2 (w1 = false): src codes [n][rows][I_full / 2], scales [n][rows][I_full / 32]; dest group b < Ik / 32
//     holds source elements first + 32 b .. first + 32 b + 31 when 32 b < count.
__global__ void __launch_bounds__(256) mx_shard_kernel(int64_t n_items, bool w1, int rows, int Kd, int Ik,
                                                       int full_inter, int src_row_elems, int first, int count,
                                                       const uint8_t* __restrict__ src_codes,
                                                       const uint8_t* __restrict__ src_sf,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int nb = Kd / 32;  // destination groups per row
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_items) return;
  const int64_t row = idx / nb;  // destination row over all experts
  const int blk = (int)(idx - row * nb);
  const int64_t g = row / rows;
  const int lr = (int)(row - g * rows);
  int kr = lr;  // row in kernel order
  int64_t src_row = -1, src_elem = 0;  // source row (over all experts) and element offset inside it
  if (w1) {
    const bool up = lr >= Ik;
    const int f = up ? lr - Ik : lr;
    kr = 128 * (f / 64) + (up ? 64 : 0) + f % 64;
    if (f < count) {
      src_row = g * 2 * (int64_t)full_inter + (up ? full_inter : 0) + first + f;
      src_elem = 32 * (int64_t)blk;
    }
  } else if (32 * blk < count) {
    src_row = row;
    src_elem = first + 32 * (int64_t)blk;
  }
  uint4 c = make_uint4(0u, 0u, 0u, 0u);
  uint8_t s = 0;
  if (src_row >= 0) {
    c = *reinterpret_cast<const uint4*>(src_codes + src_row * (src_row_elems / 2) + src_elem / 2);
    s = src_sf[src_row * (src_row_elems / 32) + src_elem / 32];
  }
  const int ka = Kd / 64, rt = kr / 128, rr = kr % 128, atom = blk / 2;
  const size_t blk_idx = ((size_t)g * (rows / 128) + rt) * ka + atom;
  *reinterpret_cast<uint4*>(codes + blk_idx * MX_BC_BYTES + 32 * rr + 16 * (blk & 1)) = c;
  sf[blk_idx * MX_BS_BYTES + 2 * rr + (blk & 1)] = s;
}

// MXFP4 weights in the NVFP4 operand form, for the block-scaled FP4 MMA of the NVFP4 layer. An MX scale
// 2^X is a power of two, and E4M3 holds every power of two from 2^-9 (0x01) to 2^8 (0x78), so with one
// factor per matrix, G = X_max - 8, the value e2m1(q) * 2^X is exactly e2m1(q) * e4m3(2^(X - G)) / gw with
// gw = 2^-G, for every block within 17 binades of the matrix's largest.
// Kernel 1: the largest E8M0 byte of each expert's matrix -> gw[e] (1 for a matrix of all-zero blocks).
__global__ void __launch_bounds__(256) mx_gw_kernel(int64_t per_expert, const uint8_t* __restrict__ sf, float* gw,
                                                    uint32_t* err) {
  const uint8_t* p = sf + (size_t)blockIdx.x * per_expert;
  uint32_t m = 0;
  bool nan = false;
  for (int64_t i = threadIdx.x; i < per_expert; i += blockDim.x) {
    const uint32_t b = p[i];
    nan |= (b == 0xFFu);
    m = max(m, b);
  }
  __shared__ uint32_t s_m[8];
  __shared__ int s_nan;
  if (threadIdx.x == 0) s_nan = 0;
  __syncthreads();
  if (nan) s_nan = 1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_m[w]);
    m = max(m, s_m[0]);
    if (s_nan) raise_error(err, FP4MOE_ERR_SCALE_RANGE);
    // X_max = m - 127 (m = 0: no live block); G = X_max - 8; gw = 2^-G
    // (clamped so that gw stays a normal fp32; a matrix that needs more raises the error in kernel 2)
    const int G = (m == 0u || m == 0xFFu) ? 0 : max(-126, min(126, (int)m - 127 - 8));
    gw[blockIdx.x] = ldexpf(1.0f, -G);
  }
}

// Kernel 2: one thread per (row, 32-element block): its 16 code bytes move from the atom-tiled MXFP4 layout
// to the pre-tiled NVFP4 layout, and its scale becomes E4M3(2^(X - G)) in both 16-element scale columns of
// the NVFP4 scale layout. E8M0 byte 0 (an all-zero block) gives scale 0. A NaN byte, nonzero codes under byte
// 0, or a block outside the 18-binade window sets FP4MOE_ERR_SCALE_RANGE (and takes scale 0, or the nearest
// power of two in the window).
__global__ void __launch_bounds__(256) mx_as_nvfp4_kernel(int64_t n_items, int rows, int K,
                                                          const uint8_t* __restrict__ mx_codes,
                                                          const uint8_t* __restrict__ mx_sf, const float* gw,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                          uint32_t* err) {
  const int nb = K / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_items) return;
  const int64_t row = idx / nb;
  const int blk = (int)(idx - row * nb);
  const int64_t e = row / rows;
  const int lr = (int)(row - e * rows);
  const int ka = K / 64, rt = lr / 128, rr = lr % 128;
  const size_t src_blk = ((size_t)e * (rows / 128) + rt) * ka + blk / 2;
  const uint4 c = *reinterpret_cast<const uint4*>(mx_codes + src_blk * MX_BC_BYTES + 32 * rr + 16 * (blk & 1));
  const uint32_t b = mx_sf[src_blk * MX_BS_BYTES + 2 * rr + (blk & 1)];
  uint32_t out = 0u;
  if (b == 0xFFu || (b == 0u && ((c.x | c.y | c.z | c.w) & 0x77777777u) != 0u)) {
    raise_error(err, FP4MOE_ERR_SCALE_RANGE);  // NaN scale, or nonzero codes under the all-zero block's byte 0
  } else if (b != 0u) {
    const int G = -ilogbf(__ldg(gw + e));
    int d = (int)b - 127 - G;
    if (d < -9 || d > 8) {
      raise_error(err, FP4MOE_ERR_SCALE_RANGE);
      d = max(-9, min(8, d));
    }
    out = d >= -6 ? (uint32_t)(d + 7) << 3 : 1u << (d + 9);  // E4M3 of 2^d: normal, else subnormal m / 8 * 2^-6
  }
  // pre-tiled NVFP4 codes: 16 KB blocks [expert][row tile][k stage of 256], row i 128 bytes, 16-byte chunk j
  // at i * 128 + (j ^ (i % 8)) * 16
  const int kst = (K + 255) / 256, stage = blk / 8, j = blk % 8;
  const size_t dst_blk = ((size_t)e * (rows / 128) + rt) * kst + stage;
  *reinterpret_cast<uint4*>(codes + dst_blk * 16384 + rr * 128 + ((j ^ (rr & 7)) * 16)) = c;
  // NVFP4 scales: 128 x 4 tiles per expert, C = K / 16 columns; columns 2 blk and 2 blk + 1 are adjacent
  const int C = K / 16, col = 2 * blk;
  const size_t so = (size_t)e * rows * C + ((size_t)(lr >> 7) * (C >> 2) + (col >> 2)) * 512 + (lr & 31) * 16 +
                    ((lr & 127) >> 5) * 4 + (col & 3);
  *reinterpret_cast<uint16_t*>(sf + so) = (uint16_t)(out | (out << 8));
}

// bf16 activation rows into slot order: each token's row goes to its k slots.
__global__ void __launch_bounds__(256) scatter_rows_bf16_kernel(int H, int k, const uint16_t* __restrict__ x,
                                                                const int32_t* __restrict__ slot_of_pair,
                                                                uint16_t* __restrict__ a1) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;  // 16-byte chunk
  if (c >= H / 8) return;
  int s[kMaxTopK];  // the k slots and the chunk are all loaded before the first store
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) s[j] = j < k ? __ldcg(slot_of_pair + (size_t)t * k + j) : -1;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c);
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (s[j] >= 0) reinterpret_cast<uint4*>(a1 + (size_t)s[j] * H)[c] = v;  // -1: held by no local expert
}

}  // namespace

fp4moe_status mx_gemm_launch(bool w2, const fp4moe_config& cfg, int32_t T, const uint16_t* a_bf16,
                             const int32_t* poff, const int32_t* pair_of_row, const uint8_t* b_codes,
                             const uint8_t* b_sf, uint16_t* out_bf16, uint16_t* o_pairs, uint32_t* err,
                             cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  MxParams prm;
  prm.E = local_experts(cfg);
  prm.K = w2 ? cfg.inter : cfg.hidden;
  prm.KA = prm.K / 64;
  prm.NT = (w2 ? cfg.hidden : 2 * cfg.inter) / MX_BN;
  prm.cap = (int)capacity_rows(cfg, T);
  prm.I = cfg.inter;
  prm.H = cfg.hidden;
  prm.limit = cfg.swiglu_limit;
  prm.poff = poff;
  prm.pair_of_row = pair_of_row;
  prm.b_codes = b_codes;
  prm.b_sf = b_sf;
  prm.out_bf16 = out_bf16;
  prm.o_pairs = o_pairs;
  prm.err = err;
  MxAMaps maps;
  for (int b = 0; b < 4; ++b)
    if (!encode_u8_sw128(&maps.box[b], a_bf16, (uint64_t)prm.K * 2, (uint64_t)prm.cap, 16u << b))
      return FP4MOE_CUDA_ERROR;
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  const int max_tiles = (prm.cap / MX_BM) * prm.NT;
  const unsigned grid = (unsigned)(max_tiles < nsm ? max_tiles : nsm);
  cudaError_t r;
  if (w2) {
    if (!configure_mx<1>()) return FP4MOE_CUDA_ERROR;
    r = launch_pdl(mx_gemm_kernel<1>, dim3(grid), dim3(MX_THREADS), MX_SMEM, st, maps, prm);
  } else {
    if (!configure_mx<0>()) return FP4MOE_CUDA_ERROR;
    r = launch_pdl(mx_gemm_kernel<0>, dim3(grid), dim3(MX_THREADS), MX_SMEM, st, maps, prm);
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

fp4moe_status mx_quant_rows_launch(int64_t n_rows, int32_t K, int32_t rows_per_group, int32_t inter, const float* in,
                                   uint8_t* codes, uint8_t* sf, cudaStream_t st) {
  if (n_rows == 0) return FP4MOE_OK;
  const int64_t n = n_rows * (K / 32);
  mx_quant_rows_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n_rows, K, rows_per_group, inter, in, codes, sf);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

fp4moe_status mx_shard_launch(int32_t n_experts, bool w1, int32_t rows, int32_t Kd, int32_t Ik, int32_t full_inter,
                              int32_t src_row_elems, int32_t first, int32_t count, const uint8_t* src_codes,
                              const uint8_t* src_sf, uint8_t* codes, uint8_t* sf, cudaStream_t st) {
  const int64_t n = (int64_t)n_experts * rows * (Kd / 32);
  if (n == 0) return FP4MOE_OK;
  mx_shard_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n, w1, rows, Kd, Ik, full_inter, src_row_elems, first,
                                                              count, src_codes, src_sf, codes, sf);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

fp4moe_status mx_as_nvfp4_launch(int32_t n_experts, int32_t rows, int32_t K, const uint8_t* mx_codes,
                                 const uint8_t* mx_sf, uint8_t* codes, uint8_t* sf, float* gw, uint32_t* err,
                                 cudaStream_t st) {
  if (n_experts == 0) return FP4MOE_OK;
  mx_gw_kernel<<<n_experts, 256, 0, st>>>((int64_t)rows * (K / 32), mx_sf, gw, err);
  if (cudaGetLastError() != cudaSuccess) return FP4MOE_CUDA_ERROR;
  if (K % 256 != 0 &&  // the last k-stage of every block is padded with zero codes
      cudaMemsetAsync(codes, 0, (size_t)n_experts * rows * ((K + 255) / 256) * 128, st) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  const int64_t n = (int64_t)n_experts * rows * (K / 32);
  mx_as_nvfp4_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n, rows, K, mx_codes, mx_sf, gw, codes, sf, err);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

fp4moe_status scatter_rows_bf16_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x,
                                       const int32_t* slot_of_pair, uint16_t* a1, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden;
  return launch_pdl(scatter_rows_bf16_kernel, dim3((H / 8 + 255) / 256, T), dim3(256), 0, st, H, cfg.top_k, x,
                    slot_of_pair, a1) == cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
