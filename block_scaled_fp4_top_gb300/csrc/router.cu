// Router logits and softmax top-k, in two passes.
//
// The routing of "Current Bug: CuTeDSLMoERunner" ("Data Flow": route, then
// sort by expert), with the top-k decided on fp32 logits l = RN(x . w_e):
// the exact bf16 x bf16 dot product rounded once to fp32. Only the top-k ids
// and their softmax weights leave the layer, so only the experts that can
// still reach the top k need their exact logit.
//
// Pass 1, router_mma_kernel: approximate logits on the tensor cores.
//   tcgen05.mma kind::f16 (bf16 x bf16, fp32 accumulate in TMEM). A tile is
//   128 tokens x 128 experts, and K may be split over a thread-block cluster
//   of S CTAs. The S partial tiles are summed through distributed shared
//   memory, in rank order, so the result is run-to-run deterministic without
//   atomics or a global partial buffer. While the MMAs run, the four
//   epilogue warps read the same shared-memory stages and accumulate the
//   squared norms |x_t|^2 and |w_e|^2 needed by the error bound.
// Pass 2, router_refine_kernel: one CTA per token.
//   a. bounds: lo/hi = l~ -/+ d with d = C |x_t| |w_e| + 2^-21 |l~|
//      (Cauchy-Schwarz bounds sum |x_h w_h|; C covers the tensor-core
//      accumulation, with a fourfold margin over 256 K-steps of 2^-22
//      relative error each);
//   b. tau = the k-th largest lo; every expert whose hi reaches tau is a
//      candidate (every expert that can be in the top k is one);
//   c. candidates get their exact logit: a compensated (two-sum) fp32 dot
//      product in a fixed order, within an ulp of the exact sum rounded once;
//   d. the top k of the candidates by exact logit, ties to the lower expert
//      id, and the renormalised softmax over them.
// The final ids and weights equal those of an all-exact computation. In
// logits_out the candidates hold their exact logit and the other experts the
// pass-1 approximation, which lies within its bound d.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

int sm_count();
bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows);

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int RT_BM = 128;                 // tokens per tile (MMA M)
constexpr int RT_BN = 128;                 // experts per tile (MMA N)
constexpr int RT_KBYTES = 128;             // one 64-element bf16 K atom per row (128-byte swizzle)
constexpr int RT_HALF = RT_BM * RT_KBYTES; // 16 KB
constexpr int RT_STAGE = 2 * RT_HALF;      // x tile + w tile of one K atom
constexpr int RT_STAGES = 4;
constexpr int RT_BAR_OFF = RT_STAGES * RT_STAGE;
constexpr int RT_SMEM = RT_BAR_OFF + 128 + 1024;
constexpr int RT_THREADS = 192;
constexpr int RT_RS = RT_BN + 4;           // row stride (floats) of the cluster-reduction tile
constexpr int RT_MAX_SPLIT = 8;            // portable cluster size
static_assert(RT_BM * RT_RS * 4 + 2 * RT_BM * 4 <= RT_BAR_OFF, "reduction tile must fit in the ring");
// d = kBoundRel |x||w| + kBoundAbsRel |l~|: 2^-12 and 2^-21
constexpr float kBoundRel = 2.44140625e-4f;
constexpr float kBoundUlp = 4.76837158203125e-7f;

struct RouterParams {
  int T, H, E, S;
  float* lt;     // [T][E] approximate logits (no bias)
  float* nx2;    // [T] |x_t|^2
  float* nw2;    // [E] |w_e|^2
  uint32_t* err;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) return;
  }
}

// sum of squares of 8 bf16 values packed in a uint4
__device__ __forceinline__ float sumsq8(uint4 v, float a) {
  a = fmaf(bf16_lo(v.x), bf16_lo(v.x), a);
  a = fmaf(bf16_hi(v.x), bf16_hi(v.x), a);
  a = fmaf(bf16_lo(v.y), bf16_lo(v.y), a);
  a = fmaf(bf16_hi(v.y), bf16_hi(v.y), a);
  a = fmaf(bf16_lo(v.z), bf16_lo(v.z), a);
  a = fmaf(bf16_hi(v.z), bf16_hi(v.z), a);
  a = fmaf(bf16_lo(v.w), bf16_lo(v.w), a);
  a = fmaf(bf16_hi(v.w), bf16_hi(v.w), a);
  return a;
}

// grid (ceil(T/128), ceil(E/128), S), cluster (1, 1, S), 192 threads.
// warp 4: TMA producer; warp 5: MMA issuer; warps 0-3: norms, then epilogue.
// Every CTA reaches both cluster barriers on every path: a bounded wait that
// expires only skips work.
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_mma_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  pdl_wait();
  pdl_trigger();
  const int mt = blockIdx.x, nt = blockIdx.y, split = blockIdx.z, S = p.S;
  const int atoms = p.H / 64;
  const int a0 = split * atoms / S, a1 = (split + 1) * atoms / S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem - smem_u32(smem_raw));
  const uint32_t bar_full = smem + RT_BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * RT_STAGES;
  const uint32_t bar_done = bar_empty + 8 * RT_STAGES;

  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 128);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < RT_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + 4);  // the MMA commit and one arrive per norm warp
    }
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  float acc[RT_BN];
  float sx = 0.0f, sw = 0.0f;
  bool ok = true;
  if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_last();  // x and w are each read by several CTAs
    int issued = a0;
    for (int j = a0; j < a1; ++j, ++issued) {
      const int it = j - a0, s = it % RT_STAGES;
      if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(it / RT_STAGES) & 1u) ^ 1u, p.err)) {
        ok = false;
        break;
      }
      const uint32_t st = smem + s * RT_STAGE;
      mbar_arrive_expect_tx(bar_full + 8 * s, RT_STAGE);
      tma_load_2d(st, &tmX, bar_full + 8 * s, j * RT_KBYTES, mt * RT_BM, pol);
      tma_load_2d(st + RT_HALF, &tmW, bar_full + 8 * s, j * RT_KBYTES, nt * RT_BN, pol);
    }
    // on every path, let the copies already issued land before the ring is reused or the CTA exits
    for (int j = max(a0, issued - RT_STAGES); j < issued; ++j) {
      const int it = j - a0;
      drain_wait(bar_full + 8 * (it % RT_STAGES), (uint32_t)(it / RT_STAGES) & 1u);
    }
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16(RT_BM, RT_BN);
    for (int j = a0; j < a1 && ok; ++j) {
      const int it = j - a0, s = it % RT_STAGES;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / RT_STAGES) & 1u, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st = smem + s * RT_STAGE;
#pragma unroll
      for (int q = 0; q < 4; ++q)  // K = 16 bf16 = 32 bytes per MMA
        tc_mma_bf16(tmem, desc_sw128(st + 32 * q), desc_sw128(st + RT_HALF + 32 * q), idesc,
                    (it > 0 || q > 0) ? 1u : 0u);
      tc_commit(bar_empty + 8 * s);
    }
    tc_commit(bar_done);
  } else if (warp < 4) {
    // ------------------------------------------------ norms, then epilogue
    // thread i owns token row i of the x tile and expert row i of the w tile; the 128-byte swizzle only
    // permutes 16-byte chunks inside a row's 128 bytes, so a row's sum of squares reads them in place
    const int i = threadIdx.x;
    for (int j = a0; j < a1 && ok; ++j) {
      const int it = j - a0, s = it % RT_STAGES;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / RT_STAGES) & 1u, p.err)) {
        ok = false;
        break;
      }
      const uint4* xa = reinterpret_cast<const uint4*>(smem_gen + s * RT_STAGE + i * RT_KBYTES);
      const uint4* wa = reinterpret_cast<const uint4*>(smem_gen + s * RT_STAGE + RT_HALF + i * RT_KBYTES);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        sx = sumsq8(xa[c], sx);
        sw = sumsq8(wa[c], sw);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (ok && a1 > a0) ok = mbar_wait(bar_done, 0, p.err);
    tc_fence_after();
    if (ok && a1 > a0) {
      const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
      for (int c = 0; c < RT_BN / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) acc[32 * c + q] = v[q];
      }
    } else {
#pragma unroll
      for (int c = 0; c < RT_BN; ++c) acc[c] = 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();  // the ring is idle from here on: every copy landed and every MMA completed

  const int i = threadIdx.x;
  const int t_row = mt * RT_BM + i;  // token of row i
  const int e_row = nt * RT_BN + i;  // expert of row i
  if (S == 1) {
    if (i < RT_BM) {
      if (t_row < p.T) {
        float* dst = p.lt + (size_t)t_row * p.E + nt * RT_BN;
        const int ne = min(RT_BN, p.E - nt * RT_BN);
#pragma unroll
        for (int c = 0; c < RT_BN; ++c)
          if (c < ne) dst[c] = acc[c];
        if (nt == 0) p.nx2[t_row] = sx;
      }
      if (mt == 0 && e_row < p.E) p.nw2[e_row] = sw;
    }
  } else {
    // every CTA of the cluster parks its partial tile in its own (idle) ring memory
    float* red = reinterpret_cast<float*>(smem_gen);
    float* red_nx = red + RT_BM * RT_RS;
    float* red_nw = red_nx + RT_BM;
    if (i < RT_BM) {
#pragma unroll
      for (int c = 0; c < RT_BN; c += 4)
        *reinterpret_cast<float4*>(red + i * RT_RS + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
      red_nx[i] = sx;
      red_nw[i] = sw;
    }
    cluster_sync();
    // CTA r sums rows [r R, (r + 1) R) of the S partial tiles, in rank order
    const uint32_t rank = cluster_ctarank();
    const int R = RT_BM / S;
    const uint32_t red_s = smem;
    for (int idx = threadIdx.x; idx < R * (RT_BN / 4); idx += RT_THREADS) {
      const int row = (int)rank * R + idx / (RT_BN / 4);
      const int c = (idx % (RT_BN / 4)) * 4;
      const uint32_t off = (uint32_t)(row * RT_RS + c) * 4u;
      float4 a = ld_cluster_f4(map_cluster(red_s + off, 0));
      for (int q = 1; q < S; ++q) {
        const float4 b = ld_cluster_f4(map_cluster(red_s + off, (uint32_t)q));
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      const int t = mt * RT_BM + row, e = nt * RT_BN + c;
      if (t < p.T) {
        float* dst = p.lt + (size_t)t * p.E + e;
        if (e + 0 < p.E) dst[0] = a.x;
        if (e + 1 < p.E) dst[1] = a.y;
        if (e + 2 < p.E) dst[2] = a.z;
        if (e + 3 < p.E) dst[3] = a.w;
      }
    }
    if (rank == 0 && i < RT_BM) {
      const uint32_t onx = (uint32_t)(RT_BM * RT_RS + i) * 4u, onw = onx + RT_BM * 4u;
      float nx = ld_cluster_f32(map_cluster(red_s + onx, 0));
      float nw = ld_cluster_f32(map_cluster(red_s + onw, 0));
      for (int q = 1; q < S; ++q) {
        nx += ld_cluster_f32(map_cluster(red_s + onx, (uint32_t)q));
        nw += ld_cluster_f32(map_cluster(red_s + onw, (uint32_t)q));
      }
      if (nt == 0 && t_row < p.T) p.nx2[t_row] = nx;
      if (mt == 0 && e_row < p.E) p.nw2[e_row] = nw;
    }
    cluster_sync();  // no CTA leaves while another still reads its shared memory
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Error-free transformation a + b = s + e (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Add the exact bf16 x bf16 product to the compensated pair (s, c).
__device__ __forceinline__ void acc_prod(float& s, float& c, float xv, float wv) {
  float e;
  two_sum(s, __fmul_rn(xv, wv), s, e);  // the product is exact in fp32 (8-bit significands)
  c = __fadd_rn(c, e);
}

// Exact-sum-rounded-once logit (within an ulp) of token row x and expert row w, by one warp. Lane l takes
// the 16-byte chunks l, l + 32, ... with two compensated accumulators; a fixed butterfly merges the lanes.
__device__ float warp_exact_dot(const uint4* __restrict__ xr, const uint4* __restrict__ wrow, int nchunks) {
  const int lane = threadIdx.x & 31;
  float s0 = 0.0f, c0 = 0.0f, s1 = 0.0f, c1 = 0.0f;
#pragma unroll 2
  for (int ch = lane; ch < nchunks; ch += 32) {
    const uint4 xv = __ldg(xr + ch);
    const uint4 wv = __ldg(wrow + ch);
    acc_prod(s0, c0, bf16_lo(xv.x), bf16_lo(wv.x));
    acc_prod(s1, c1, bf16_hi(xv.x), bf16_hi(wv.x));
    acc_prod(s0, c0, bf16_lo(xv.y), bf16_lo(wv.y));
    acc_prod(s1, c1, bf16_hi(xv.y), bf16_hi(wv.y));
    acc_prod(s0, c0, bf16_lo(xv.z), bf16_lo(wv.z));
    acc_prod(s1, c1, bf16_hi(xv.z), bf16_hi(wv.z));
    acc_prod(s0, c0, bf16_lo(xv.w), bf16_lo(wv.w));
    acc_prod(s1, c1, bf16_hi(xv.w), bf16_hi(wv.w));
  }
  float s, e0;
  two_sum(s0, s1, s, e0);
  float c = __fadd_rn(__fadd_rn(c0, c1), e0);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float so = __shfl_xor_sync(kFull, s, off);
    const float co = __shfl_xor_sync(kFull, c, off);
    float ns, ne;
    two_sum(s, so, ns, ne);
    s = ns;
    c = __fadd_rn(__fadd_rn(c, co), ne);
  }
  return __fadd_rn(s, c);
}

// One warp picks the k largest of key[list[0..n)] (descending, ties to the lower expert id): writes the
// picks to sel_e / sel_v (lane 0's registers are authoritative) and returns the k-th value, or NaN when
// fewer than k finite-or-infinite keys exist.
__device__ float warp_select(const float* key, const int* list, int n, int k, int* sel_e, float* sel_v) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit q: item lane + 32 q already picked
  float kth = __int_as_float(0x7FC00000);
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX, bq = -1;
    for (int q = 0; lane + 32 * q < n; ++q) {
      if ((taken >> q) & 1u) continue;
      const int e = list ? list[lane + 32 * q] : lane + 32 * q;
      const float v = key[e];
      if (v > bv || (v == bv && e < be)) {
        bv = v;
        be = e;
        bq = q;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oe = __shfl_xor_sync(kFull, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be == INT_MAX) return __int_as_float(0x7FC00000);  // only NaN keys remain
    // the lane that holds the winner marks it taken
    if (bq >= 0 && (list ? list[lane + 32 * bq] : lane + 32 * bq) == be) taken |= 1u << bq;
    sel_e[j] = be;
    sel_v[j] = bv;
    kth = bv;
  }
  return kth;
}

// One CTA of 256 threads per token.
__global__ void __launch_bounds__(256) router_refine_kernel(int H, int E, int k, const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ wr,
                                                            const float* __restrict__ bias,
                                                            const float* __restrict__ nx2,
                                                            const float* __restrict__ nw2, float* logits,
                                                            int32_t* __restrict__ ids_out,
                                                            float* __restrict__ w_out, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_l[kMaxExperts];
  __shared__ float s_lo[kMaxExperts];
  __shared__ float s_hi[kMaxExperts];
  __shared__ int s_cand[kMaxExperts];
  __shared__ int s_m;
  __shared__ float s_tau;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* lrow = logits + (size_t)t * E;
  const float nx = sqrtf(__ldcg(nx2 + t));
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float l = __ldcg(lrow + e);
    if (bias != nullptr) l = __fadd_rn(l, bias[e]);
    // the fp32 norms are low by at most ~3e-4 relative: the (1 + 2^-10) factor keeps the bound above it
    const float d = fmaf(kBoundRel * 1.0009765625f, nx * sqrtf(__ldcg(nw2 + e)), kBoundUlp * fabsf(l));
    s_l[e] = l;
    s_lo[e] = __fsub_rd(l, d);
    s_hi[e] = __fadd_ru(l, d);
  }
  if (threadIdx.x == 0) s_m = 0;
  __syncthreads();
  if (warp == 0) {
    int se[kMaxTopK];
    float sv[kMaxTopK];
    const float tau = warp_select(s_lo, nullptr, E, k, se, sv);
    if (lane == 0) s_tau = tau;
  }
  __syncthreads();
  const float tau = s_tau;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    // NaN tau (NaN logits) makes every expert a candidate; the selection below then reports the NaNs
    if (!(s_hi[e] < tau)) s_cand[atomicAdd(&s_m, 1)] = e;
  }
  __syncthreads();
  const int m = s_m;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int c = warp; c < m; c += blockDim.x / 32) {
    const int e = s_cand[c];
    float l = warp_exact_dot(xr, reinterpret_cast<const uint4*>(wr + (size_t)e * H), H / 8);
    if (bias != nullptr) l = __fadd_rn(l, bias[e]);
    if (lane == 0) s_l[e] = l;
  }
  __syncthreads();
  if (warp == 0) {
    int se[kMaxTopK];
    float sv[kMaxTopK];
    const float kth = warp_select(s_l, s_cand, m, k, se, sv);
    if (lane == 0) {
      if (kth != kth) {  // fewer than k comparable logits: NaN input
        raise_error(err, FP4MOE_ERR_EXPERT_ID);
        for (int j = 0; j < k; ++j) {
          ids_out[(size_t)t * k + j] = 0;
          w_out[(size_t)t * k + j] = 0.0f;
        }
      } else {
        const float lmax = sv[0];
        float ex[kMaxTopK];
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) {
          ex[j] = expf(__fsub_rn(sv[j], lmax));
          sum = __fadd_rn(sum, ex[j]);
        }
        for (int j = 0; j < k; ++j) {
          ids_out[(size_t)t * k + j] = se[j];
          w_out[(size_t)t * k + j] = __fdiv_rn(ex[j], sum);
        }
      }
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) lrow[e] = s_l[e];
}

bool configure_router() {
  static int ok = -1;
  if (ok < 0)
    ok = cudaFuncSetAttribute(router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RT_SMEM) ==
                 cudaSuccess
             ? 1
             : 0;
  return ok == 1;
}

}  // namespace

fp4moe_status router_topk_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* wr,
                                 const float* bias, float* logits, float* nx2, float* nw2, int32_t* ids, float* w,
                                 uint32_t* err, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden, E = cfg.num_experts, k = cfg.top_k;
  if (!configure_router()) return FP4MOE_CUDA_ERROR;
  CUtensorMap tmX, tmW;
  if (!encode_u8_sw128(&tmX, x, (uint64_t)H * 2, (uint64_t)T, RT_BM)) return FP4MOE_CUDA_ERROR;
  if (!encode_u8_sw128(&tmW, wr, (uint64_t)H * 2, (uint64_t)E, RT_BN)) return FP4MOE_CUDA_ERROR;
  const int n_mt = (T + RT_BM - 1) / RT_BM, n_nt = (E + RT_BN - 1) / RT_BN;
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  // split K over a cluster while the tiles alone leave SMs idle; at least 2 K atoms per split
  int S = 1;
  while (S * 2 <= RT_MAX_SPLIT && n_mt * n_nt * S * 2 <= nsm && (H / 64) >= 4 * S) S *= 2;
  RouterParams prm;
  prm.T = T;
  prm.H = H;
  prm.E = E;
  prm.S = S;
  prm.lt = logits;
  prm.nx2 = nx2;
  prm.nw2 = nw2;
  prm.err = err;

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_mt, n_nt, S);
  lc.blockDim = dim3(RT_THREADS);
  lc.dynamicSmemBytes = RT_SMEM;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = S;
  lc.attrs = attr;
  lc.numAttrs = 2;
  if (cudaLaunchKernelEx(&lc, router_mma_kernel, tmX, tmW, prm) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  return launch_pdl(router_refine_kernel, dim3(T), dim3(256), 0, st, H, E, k, x, wr, bias,
                    (const float*)nx2, (const float*)nw2, logits, ids, w, err) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
