// Shared device helpers for the block-scaled FP4 MoE kernels (sm_103a).
//
// Inline PTX wrappers for mbarrier, TMA and tcgen05, plus the NVFP4 block
// quantiser that every kernel uses. The quantiser is the per-16-element
// procedure on "Current Bug: CuTeDSLMoERunner", "Data Flow"
// (quantize_activation_nvfp4). Its scale arithmetic is fixed to IEEE fp32 RNE:
//   a = max|v|, s = RN(RN(a/6)*g), sf = E4M3_satfinite(s),
//   inv = sf ? RN(g/sf) : 0, q = E2M1_satfinite(RN(v*inv)).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4moe.h"

namespace fp4moe {

// ------------------------------------------------------------------ limits --
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kRouteChunk = 64;          // tokens per histogram chunk
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;  // bounded spin-wait: 200 ms
constexpr uint32_t kAbortMask = FP4MOE_ERR_TIMEOUT;

// ------------------------------------------------------ workspace header --
// byte offsets inside the first 256 bytes of the workspace
constexpr size_t kWsErr = 0;        // uint32 error word
constexpr size_t kWsAmaxH = 16;     // float, calibration scratch (amax of h)
constexpr size_t kWsAmaxX = 20;     // float, calibration scratch (amax of x)
// int pairs {chunks taken, CTAs finished} of the W1 and W2 GEMMs' schedules (dynamic chunks or the static
// pool): zero between launches, the last CTA of each launch zeroes its pair
constexpr size_t kWsSchedW1 = 64;
constexpr size_t kWsSchedW2 = 72;
constexpr size_t kWsBatchAmax = 40; // uint, batch amax accumulator of fp4moe_batch_gs1 (zero between calls)
constexpr size_t kWsBatchDone = 44; // uint, its CTA arrival counter (zero between calls)
constexpr size_t kWsScaleFlags = 48;  // uint, sticky FP4MOE_SAT_* bits (fp4moe_read_scale_status)
constexpr size_t kWsAmaxHRun = 52;    // float, amax|h| of the W1 epilogues since the last refresh or clear
constexpr size_t kWsHeader = 256;

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

// ------------------------------------------------------------- bf16/fp32 --
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values as bf16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// ----------------------------------------------------------- FP8/FP4 cvt --
// E4M3 (satfinite, RNE) of a non-negative fp32; returns the byte.
__device__ __forceinline__ uint32_t cvt_e4m3(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return r & 0xFFu;
}
// Exact decode of an E4M3 byte that is not NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
  return (b & 0x80u) ? -v : v;
}
// Two E2M1 codes (RNE, satfinite) packed in a byte: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// NVFP4 quantisation of one 16-element block under global scale g.
// Returns the E4M3 scale byte; codes_lo/codes_hi get the 8 packed code bytes
// (element 2i in the low nibble of byte i; bytes 0-3 in codes_lo, 4-7 in codes_hi).
// s_out receives the unrounded block scale s. s > kE4M3SatAbove means the
// E4M3 scale saturated: s rounds above the largest finite E4M3 value, so the
// global scale g no longer covers this block.
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float g, uint32_t& codes_lo,
                                                  uint32_t& codes_hi, float& s_out) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  const float s = __fmul_rn(__fdiv_rn(a, 6.0f), g);
  s_out = s;
  const uint32_t sf = cvt_e4m3(s);
  const float inv = (sf == 0u) ? 0.0f : __fdiv_rn(g, e4m3_to_f32(sf));
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= cvt_e2m1x2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    hi |= cvt_e2m1x2(__fmul_rn(v[8 + 2 * i], inv), __fmul_rn(v[8 + 2 * i + 1], inv)) << (8 * i);
  codes_lo = lo;
  codes_hi = hi;
  return sf;
}
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float g, uint32_t& codes_lo,
                                                  uint32_t& codes_hi) {
  float s;
  return quant_block16(v, g, codes_lo, codes_hi, s);
}

// max that propagates NaN (fmaxf returns the other operand instead).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The clamped SwiGLU of the routed and shared experts: silu(min(g, L)) * clamp(u, -L, L).
// A NaN gate or up gives a NaN h: the comparisons are written so that NaN
// passes through (fminf/fmaxf would replace it by a clamp bound). The gate's
// floor at -80 only keeps the exponential finite (silu(-80) is about -1e-33).
// The exponential and the division use the fast hardware approximations (a
// few ulp): h only feeds a requantiser or a bf16 rounding and the
// tolerance-checked output.
__device__ __forceinline__ float swiglu_clamped(float g, float u, float L) {
  float gc = g > L ? L : g;
  gc = gc < -80.0f ? -80.0f : gc;
  const float uc = u > L ? L : (u < -L ? -L : u);
  return __fdividef(gc, 1.0f + __expf(-gc)) * uc;
}

// E4M3 round-to-nearest-even takes s above 448 (to the 480 that the format lacks) exactly when s > 464, the
// midpoint; ties go to 448, the even code. A block scale beyond it saturates.
constexpr float kE4M3SatAbove = 464.0f;

// Byte offset of scale (r, c) in the 128x4 tile layout of a matrix with C scale columns.
__device__ __forceinline__ uint32_t sf_offset(uint32_t r, uint32_t c, uint32_t C) {
  return ((r >> 7) * (C >> 2) + (c >> 2)) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u + (c & 3u);
}

// Quant-direction global scale from an amax: RN(2688 / amax), 1 when amax == 0.
__device__ __forceinline__ float global_scale_from_amax(float amax) {
  return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
}

// ------------------------------------------------ programmatic dependent launch --
// Kernels on the hot path are launched with programmatic stream serialisation
// (launch_pdl in the host code). Each one lets its successor start early,
// which hides the launch gap, and waits for its predecessor's results before
// reading them. Without a programmatic predecessor both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- PTX: misc --
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------- PTX: mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Slow path of mbar_wait: spin with a time limit.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint32_t* err,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*(volatile uint32_t*)err & kAbortMask) return false;
      if (globaltimer() - t0 > limit_ns) {
        raise_error(err, FP4MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
// Bounded wait for the phase with `parity` to complete. It returns false if
// kWaitLimitNs passes first (setting FP4MOE_ERR_TIMEOUT), or if another CTA
// has already raised an abort bit in the error word. The common case, a phase
// that has already completed, stays inline.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, err);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Bounded wait that ignores other CTAs' aborts: used only while draining
// copies or MMAs already in flight before a CTA frees what they touch.
static __device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (TMA stores, tcgen05.mma operands) of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- PTX: TMA --
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], "
      "[%2], %5;" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// Pull `bytes` (multiple of 16, 16-byte aligned) into L2 ahead of a later bulk load.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 32 bytes to a 32-byte-aligned global address in one 256-bit store (sm_100 and later), so a thread writing a
// row fills whole L2 sectors; the line is not allocated in L1.
__device__ __forceinline__ void st_global_v8(float* p, float a, float b, float c, float d, float e, float f, float g,
                                             float h) {
  asm volatile("st.global.L1::no_allocate.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a), "f"(b),
               "f"(c), "f"(d), "f"(e), "f"(f), "f"(g), "f"(h)
               : "memory");
}

// ----------------------------------------------------------- PTX: tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrive on `bar` once every tcgen05 op this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Copy one 512-byte 128x4 scale tile (32 rows of 16 bytes) from shared memory
// into 4 TMEM columns, replicated into all four 32-lane groups.
__device__ __forceinline__ void tc_cp_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, NVFP4 x NVFP4 with UE4M3 scales per 16 elements (K = 64).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,"
      "%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte
// swizzle: 8-row x 128-byte atoms, 1024 bytes apart along M/N.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of a 512-byte scale tile for tcgen05.cp: no swizzle, core
// matrices of 8 rows x 16 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t desc_scales(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 x bf16 with fp32 accumulation (kind::f16, K = 16).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor: kind::f16 with fp32 D, A and B bf16, both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------- PTX: clusters --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Full-cluster barrier: every thread of every CTA in the cluster arrives, with
// release/acquire ordering of shared-memory writes across the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address `saddr` of this CTA, mapped into CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t caddr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
  return v;
}

// Instruction descriptor: kind::mxf4nvf4, A and B E2M1, UE4M3 scales, both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace fp4moe
