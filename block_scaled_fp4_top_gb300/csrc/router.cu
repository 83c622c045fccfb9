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
//   128 experts x up to 256 tokens. With a single tile of tokens (decode), K
//   is split over up to 16 independent CTAs that write fp32 partial tiles to
//   the workspace, and pass 2 sums them in split order. With more tiles, K
//   may be split over a thread-block cluster of S CTAs whose partial tiles
//   are summed through distributed shared memory in rank order. Either way
//   the sum has a fixed order, so the result is run-to-run deterministic
//   without atomics. While the MMAs run, the four
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
constexpr int RT_BM = 128;                 // experts per tile (MMA M)
constexpr int RT_MAX_BN = 256;             // tokens per tile (MMA N): min(256, T rounded up to 32)
constexpr int RT_KBYTES = 128;             // one 64-element bf16 K atom per row (128-byte swizzle)
constexpr int RT_A = RT_BM * RT_KBYTES;    // w tile of one K atom: 16 KB
constexpr int RT_MAX_STAGE = RT_A + RT_MAX_BN * RT_KBYTES;  // + x tile: 48 KB at most
constexpr int RT_BAR_OFF = 4 * RT_MAX_STAGE;  // the ring: 4 stages of the largest tile, more of smaller ones
constexpr int RT_MAX_STAGES = 8;
constexpr int RT_SMEM = RT_BAR_OFF + 16 * RT_MAX_STAGES + 8 + 1024;
constexpr int RT_THREADS = 192;
constexpr int RT_RS = RT_MAX_BN + 4;       // row stride (floats) of the cluster-reduction tile
constexpr int RT_MAX_SPLIT = 8;            // portable cluster size
constexpr int RT_MAX_PART_SPLIT = 16;      // one tile of tokens: K split over independent CTAs
constexpr int kWarpRefineMinT = 4096;  // from this many tokens on, one warp (not one CTA) per token (measured: T = 512 is faster with a CTA per token, T = 8192 with a warp)
static_assert(RT_BM * RT_RS * 4 + RT_BM * 4 <= RT_BAR_OFF, "reduction tile must fit in the ring");
// d = kBoundRel |x||w| + kBoundUlp |l~|: 2^-12 and 2^-21
constexpr float kBoundRel = 2.44140625e-4f;
constexpr float kBoundUlp = 4.76837158203125e-7f;

struct RouterParams {
  int T, H, E, S, BN;
  int partial;    // 1: the S CTAs of a K split write partial tiles lt[split][T][E], nw2[split][E]; no cluster
  int NS, stage;  // ring stages and bytes per stage (RT_A + BN * RT_KBYTES, a multiple of 4 KB)
  float* lt;     // [T][E] approximate logits (no bias)
  float* nw2;    // [E] |w_e|^2
  uint32_t* err;
};

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

// Sum of squares of one 128-byte row of a 128-byte-swizzled tile. The swizzle
// only permutes the row's eight 16-byte chunks, so any order covers them; thread
// i starts at chunk i % 8, which keeps the eight threads of each shared-memory
// phase on distinct banks.
__device__ __forceinline__ float row_sumsq(const uint8_t* row, int i, float a) {
#pragma unroll
  for (int c = 0; c < 8; ++c) a = sumsq8(*reinterpret_cast<const uint4*>(row + (((c + i) & 7) << 4)), a);
  return a;
}

// grid (ceil(E/128), ceil(T/BN), S), cluster (1, 1, S) (no cluster for partial tiles), 192 threads. The tile
// is 128 experts (MMA M, TMEM lanes) x BN tokens (MMA N, TMEM columns).
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
  const int et = blockIdx.x, tt = blockIdx.y, split = blockIdx.z, S = p.S, BN = p.BN;
  const int atoms = p.H / 64;
  const int a0 = split * atoms / S, a1 = (split + 1) * atoms / S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem - smem_u32(smem_raw));
  const int NS = p.NS, STAGE = p.stage;
  const uint32_t bar_full = smem + RT_BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * RT_MAX_STAGES;
  const uint32_t bar_done = bar_empty + 8 * RT_MAX_STAGES;

  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), RT_MAX_BN);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < NS; ++s) {
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

  const int i = threadIdx.x;
  // squared norm of expert row i, accumulated by the CTAs of the first token tile
  float sw = 0.0f;
  const bool do_w = (tt == 0);
  bool ok = true;
  if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_last();  // x and w are each read by several CTAs
    int issued = a0;
    for (int j = a0; j < a1; ++j, ++issued) {
      const int it = j - a0, s = it % NS;
      if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(it / NS) & 1u) ^ 1u, p.err)) {
        ok = false;
        break;
      }
      const uint32_t st = smem + s * STAGE;
      mbar_arrive_expect_tx(bar_full + 8 * s, RT_A + BN * RT_KBYTES);
      tma_load_2d(st, &tmW, bar_full + 8 * s, j * RT_KBYTES, et * RT_BM, pol);
      tma_load_2d(st + RT_A, &tmX, bar_full + 8 * s, j * RT_KBYTES, tt * BN, pol);
    }
    // on every path, let the copies already issued land before the ring is reused or the CTA exits
    for (int j = max(a0, issued - NS); j < issued; ++j) {
      const int it = j - a0;
      drain_wait(bar_full + 8 * (it % NS), (uint32_t)(it / NS) & 1u);
    }
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(RT_BM, BN);
    for (int j = a0; j < a1 && ok; ++j) {
      const int it = j - a0, s = it % NS;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / NS) & 1u, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st = smem + s * STAGE;
#pragma unroll
      for (int q = 0; q < 4; ++q)  // K = 16 bf16 = 32 bytes per MMA
        tc_mma_bf16(tmem, desc_sw128(st + 32 * q), desc_sw128(st + RT_A + 32 * q), idesc,
                    (it > 0 || q > 0) ? 1u : 0u);
      tc_commit(bar_empty + 8 * s);
    }
    tc_commit(bar_done);
    drain_wait(bar_done, 0);  // no MMA may still write TMEM when it is read or freed
  } else if (warp < 4) {
    // ------------------------------------------------------------------ norms
    for (int j = a0; j < a1 && ok; ++j) {
      const int it = j - a0, s = it % NS;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / NS) & 1u, p.err)) {
        ok = false;
        break;
      }
      if (do_w) sw = row_sumsq(smem_gen + s * STAGE + i * RT_KBYTES, i, sw);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (ok) ok = mbar_wait(bar_done, 0, p.err);
    tc_fence_after();
  }
  __syncthreads();  // the ring is idle from here on: every copy landed and every MMA completed

  const int e_row = et * RT_BM + i;  // expert of TMEM lane / thread i (i < 128)
  const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  if (S == 1 || p.partial) {
    float* lt = p.lt + (size_t)split * p.T * p.E;  // split is 0 without a K split
    float* nw2 = p.nw2 + (size_t)split * p.E;
    if (warp < 4) {
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);
        tmem_ld_wait();
        if (ok && e_row < p.E) {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int t = tt * BN + c + q;
            if (t < p.T) lt[(size_t)t * p.E + e_row] = v[q];  // a warp stores 32 consecutive experts
          }
        }
      }
      if (do_w && e_row < p.E) nw2[e_row] = sw;
    }
  } else {
    // every CTA of the cluster parks its partial tile in its own (idle) ring memory
    float* red = reinterpret_cast<float*>(smem_gen);
    float* red_nw = red + RT_BM * RT_RS;
    if (warp < 4) {
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; q += 4)
          *reinterpret_cast<float4*>(red + i * RT_RS + c + q) =
              ok ? make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      red_nw[i] = sw;
    }
    cluster_sync();
    // CTA r sums expert rows [r R, (r + 1) R) of the S partial tiles, in rank order. Consecutive threads take
    // consecutive experts of the same 4 tokens, so each store of a warp covers consecutive addresses.
    const uint32_t rank = cluster_ctarank();
    const int R = RT_BM / S;
    const uint32_t red_s = smem;
    for (int idx = threadIdx.x; idx < R * (BN / 4); idx += RT_THREADS) {
      const int row = (int)rank * R + idx % R;
      const int c = (idx / R) * 4;
      const uint32_t off = (uint32_t)(row * RT_RS + c) * 4u;
      // all S loads are in flight before the first add; the sum still runs in rank order
      float4 b[RT_MAX_SPLIT];
#pragma unroll
      for (int q = 0; q < RT_MAX_SPLIT; ++q)
        if (q < S) b[q] = ld_cluster_f4(map_cluster(red_s + off, (uint32_t)q));
      float4 a = b[0];
#pragma unroll
      for (int q = 1; q < RT_MAX_SPLIT; ++q) {
        if (q < S) {
          a.x += b[q].x;
          a.y += b[q].y;
          a.z += b[q].z;
          a.w += b[q].w;
        }
      }
      const int e = et * RT_BM + row, t = tt * BN + c;
      if (e < p.E) {
        float* dst = p.lt + (size_t)t * p.E + e;
        if (t + 0 < p.T) dst[0] = a.x;
        if (t + 1 < p.T) dst[(size_t)p.E] = a.y;
        if (t + 2 < p.T) dst[(size_t)2 * p.E] = a.z;
        if (t + 3 < p.T) dst[(size_t)3 * p.E] = a.w;
      }
    }
    if (rank == 0 && warp < 4 && do_w) {
      const uint32_t onw = (uint32_t)(RT_BM * RT_RS + i) * 4u;
      float b[RT_MAX_SPLIT];
#pragma unroll
      for (int q = 0; q < RT_MAX_SPLIT; ++q)
        if (q < S) b[q] = ld_cluster_f32(map_cluster(red_s + onw, (uint32_t)q));
      float nw = b[0];
#pragma unroll
      for (int q = 1; q < RT_MAX_SPLIT; ++q)
        if (q < S) nw += b[q];
      if (e_row < p.E) p.nw2[e_row] = nw;
    }
    cluster_sync();  // no CTA leaves while another still reads its shared memory
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, RT_MAX_BN);
  }
}

// Error-free transformation a + b = s + e (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Two fp32 lanes in one 64-bit register, lane 0 in the low word, for the packed f32x2 add, sub and mul of
// sm_100 and later. Each lane rounds to nearest even exactly as the scalar instruction would, so a packed chain
// gives the same bits as two scalar chains, one per lane, in half the instructions.
typedef unsigned long long f32x2_t;

__device__ __forceinline__ f32x2_t add_x2(f32x2_t a, f32x2_t b) {
  f32x2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2_t sub_x2(f32x2_t a, f32x2_t b) {
  f32x2_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2_t mul_x2(f32x2_t a, f32x2_t b) {
  f32x2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// The two bf16 of a 32-bit word as fp32 lanes: the low half in lane 0, the high half in lane 1.
__device__ __forceinline__ f32x2_t bf16x2_widen(uint32_t w) {
  return (static_cast<f32x2_t>(w & 0xFFFF0000u) << 32) | static_cast<f32x2_t>(w << 16);
}
__device__ __forceinline__ float lane0(f32x2_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float lane1(f32x2_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// Add the exact bf16 x bf16 products of the word pair (xw, ww) to the compensated pairs (s, c), lane by lane:
// Knuth's two-sum on each lane. Each product is exact in fp32 (8-bit significands).
__device__ __forceinline__ void acc_prod_x2(f32x2_t& s, f32x2_t& c, uint32_t xw, uint32_t ww) {
  const f32x2_t p = mul_x2(bf16x2_widen(xw), bf16x2_widen(ww));
  const f32x2_t sn = add_x2(s, p);
  const f32x2_t bb = sub_x2(sn, s);
  const f32x2_t e = add_x2(sub_x2(s, sub_x2(sn, bb)), sub_x2(p, bb));
  s = sn;
  c = add_x2(c, e);
}

constexpr int kMaxChunksPerLane = 18;  // H <= 4608: 576 16-byte chunks over 32 lanes

// Exact-sum-rounded-once logit (within an ulp) of the token row xs (in shared memory) and expert row w, by
// one warp. Lane l takes the 16-byte chunks l, l + 32, ..., all of whose loads are issued before the
// arithmetic, with two compensated accumulators (the low and the high bf16 of each word, the lanes of one
// packed pair); a fixed butterfly merges the lanes.
__device__ float warp_exact_dot(const uint4* xs, const uint4* __restrict__ wrow, int nchunks) {
  const int lane = threadIdx.x & 31;
  uint4 wv[kMaxChunksPerLane];
#pragma unroll
  for (int j = 0; j < kMaxChunksPerLane; ++j)
    if (lane + 32 * j < nchunks) wv[j] = __ldg(wrow + lane + 32 * j);
  f32x2_t S = 0ull, C = 0ull;
#pragma unroll
  for (int j = 0; j < kMaxChunksPerLane; ++j) {
    if (lane + 32 * j < nchunks) {
      const uint4 xv = xs[lane + 32 * j];
      acc_prod_x2(S, C, xv.x, wv[j].x);
      acc_prod_x2(S, C, xv.y, wv[j].y);
      acc_prod_x2(S, C, xv.z, wv[j].z);
      acc_prod_x2(S, C, xv.w, wv[j].w);
    }
  }
  float s, e0;
  two_sum(lane0(S), lane1(S), s, e0);
  float c = __fadd_rn(__fadd_rn(lane0(C), lane1(C)), e0);
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

// The rank of the item (v, e) among the n items key[list[j]]: how many of them come before it in the order
// value descending, expert id ascending. A NaN item comes before nothing, and a NaN v is never ranked. The
// items of a top-k pick are those of rank < k, and rank r goes to place r, so every thread can rank its own
// items at once; the ranks do not depend on the order of the list.
__device__ __forceinline__ int rank_among(const float* key, const int* list, int n, float v, int e) {
  int r = 0;
  for (int j = 0; j < n; ++j) {
    const int f = list[j];
    const float u = key[f];
    r += (u > v || (u == v && f < e)) ? 1 : 0;
  }
  return r;
}

// One CTA of 256 threads per token.
// part (null without a K split over independent CTAs): S partial logit tiles [S][T][E], then S partial norm
// rows [S][E], summed here in split order.
__global__ void __launch_bounds__(256) router_refine_kernel(int T, int H, int E, int k, int S,
                                                            const float* __restrict__ part,
                                                            const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ wr,
                                                            const float* __restrict__ bias,
                                                            const float* __restrict__ nw2, float* logits,
                                                            int32_t* __restrict__ ids_out,
                                                            float* __restrict__ w_out, uint32_t* err) {
  __shared__ uint4 s_x[kMaxChunksPerLane * 32];
  __shared__ float s_l[kMaxExperts];
  __shared__ float s_lo[kMaxExperts];
  __shared__ float s_hi[kMaxExperts];
  __shared__ int s_cand[kMaxExperts];
  __shared__ float s_part[8];
  __shared__ float s_wmax[8];
  __shared__ int s_m, s_n2;
  __shared__ float s_tau;
  __shared__ int s_sel_e[kMaxTopK];
  __shared__ float s_sel_v[kMaxTopK];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = H / 8;
  float* lrow = logits + (size_t)t * E;
  // The token row goes to shared memory once; its squared norm is a fixed-order block sum. x is the
  // layer's input: router_mma, the launch this one follows, began only after whatever wrote x had
  // finished, so x is read before the wait on router_mma.
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  float sq = 0.0f;
  for (int c = threadIdx.x; c < nchunks; c += blockDim.x) {
    const uint4 v = __ldg(xr + c);
    s_x[c] = v;
    sq = sumsq8(v, sq);
  }
  pdl_wait();  // the partial tiles, logits and norms of router_mma from here on
  pdl_trigger();
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(kFull, sq, off);
  if (lane == 0) s_part[warp] = sq;
  if (threadIdx.x == 0) {
    s_m = 0;
    s_n2 = 0;
    s_tau = __int_as_float(0x7FC00000);  // stays NaN when fewer than k lower ends are numbers
  }
  if (threadIdx.x < kMaxTopK) s_sel_e[threadIdx.x] = -1;
  __syncthreads();
  float nx2 = 0.0f;
#pragma unroll
  for (int w8 = 0; w8 < 8; ++w8) nx2 += s_part[w8];
  const float nx = sqrtf(nx2);
  float wmax = -INFINITY;  // this warp's largest lower end (a NaN never wins)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float l, nw;
    if (part != nullptr) {  // every load in flight before the sums, which run in split order
      const float* pl = part + (size_t)t * E + e;
      const float* pn = part + (size_t)S * T * E + e;
      float vl[RT_MAX_PART_SPLIT], vn[RT_MAX_PART_SPLIT];
#pragma unroll
      for (int s = 0; s < RT_MAX_PART_SPLIT; ++s) {
        if (s < S) {
          vl[s] = __ldcg(pl + (size_t)s * T * E);
          vn[s] = __ldcg(pn + (size_t)s * E);
        }
      }
      l = vl[0];
      nw = vn[0];
#pragma unroll
      for (int s = 1; s < RT_MAX_PART_SPLIT; ++s) {
        if (s < S) {
          l += vl[s];
          nw += vn[s];
        }
      }
    } else {
      l = __ldcg(lrow + e);
      nw = __ldcg(nw2 + e);
    }
    if (bias != nullptr) l = __fadd_rn(l, bias[e]);
    // the fp32 norms are low by at most ~3e-4 relative: the (1 + 2^-10) factor keeps the bound above it
    const float d = fmaf(kBoundRel * 1.0009765625f, nx * sqrtf(nw), kBoundUlp * fabsf(l));
    const float lo = __fsub_rd(l, d);
    s_l[e] = l;
    s_lo[e] = lo;
    s_hi[e] = __fadd_ru(l, d);
    wmax = fmaxf(wmax, lo);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(kFull, wmax, off));
  if (lane == 0) s_wmax[warp] = wmax;
  __syncthreads();
  // theta <= tau: the k-th largest of the eight warp maxima. Each is the lower end of a different expert, so
  // when theta is a number at least k experts reach it, and so does the k-th largest lower end. A warp with
  // no number has the maximum -inf; if theta is -inf, every expert whose lower end is a number is kept.
  float theta = -INFINITY;
  if (k <= 8) {
    const int q0 = lane & 7;
    const float mq = s_wmax[q0];
    int r = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float o = s_wmax[q];
      r += (o > mq || (o == mq && q < q0)) ? 1 : 0;
    }
    const unsigned b = __ballot_sync(kFull, lane < 8 && r == k - 1);
    theta = __shfl_sync(kFull, mq, __ffs(b) - 1);
  }
  // tau = the k-th largest lower end: the one of rank k - 1 among those that reach theta (a NaN never does)
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (s_lo[e] >= theta) s_cand[atomicAdd(&s_n2, 1)] = e;
  __syncthreads();
  const int n2 = s_n2;
  for (int c = threadIdx.x; c < n2; c += blockDim.x) {
    const int e = s_cand[c];
    if (rank_among(s_lo, s_cand, n2, s_lo[e], e) == k - 1) s_tau = s_lo[e];
  }
  __syncthreads();
  const float tau = s_tau;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    // NaN tau (NaN logits) makes every expert a candidate; the selection below then reports the NaNs
    if (!(s_hi[e] < tau)) s_cand[atomicAdd(&s_m, 1)] = e;
  }
  __syncthreads();
  const int m = s_m;
  for (int c = warp; c < m; c += blockDim.x / 32) {
    const int e = s_cand[c];
    float l = warp_exact_dot(s_x, reinterpret_cast<const uint4*>(wr + (size_t)e * H), nchunks);
    if (bias != nullptr) l = __fadd_rn(l, bias[e]);
    if (lane == 0) s_l[e] = l;
  }
  __syncthreads();
  // the top k of the candidates by exact logit: the candidate of rank r < k takes place r
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    const int e = s_cand[c];
    const float v = s_l[e];
    if (v == v) {
      const int r = rank_among(s_l, s_cand, m, v, e);
      if (r < k) {
        s_sel_e[r] = e;
        s_sel_v[r] = v;
      }
    }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) lrow[e] = s_l[e];
  __syncthreads();
  if (threadIdx.x == 0) {
    bool bad = false;
    for (int j = 0; j < k; ++j) bad |= s_sel_e[j] < 0;
    if (bad) {  // fewer than k comparable logits: NaN input
      raise_error(err, FP4MOE_ERR_EXPERT_ID);
      for (int j = 0; j < k; ++j) {
        ids_out[(size_t)t * k + j] = 0;
        w_out[(size_t)t * k + j] = 0.0f;
      }
    } else {
      const float lmax = s_sel_v[0];
      float ex[kMaxTopK];
      float sum = 0.0f;
      for (int j = 0; j < k; ++j) {
        ex[j] = expf(__fsub_rn(s_sel_v[j], lmax));
        sum = __fadd_rn(sum, ex[j]);
      }
      for (int j = 0; j < k; ++j) {
        ids_out[(size_t)t * k + j] = s_sel_e[j];
        w_out[(size_t)t * k + j] = __fdiv_rn(ex[j], sum);
      }
    }
  }
}

// Argmax over this warp's register arrays (item lane + 32 q is expert lane + 32 q): the largest v among the
// items whose bit is set in `eligible`, ties to the lower expert id. Returns INT_MAX in be when no eligible
// item compares (only NaNs left).
template <int MAXV>
__device__ __forceinline__ void warp_argmax(const float (&v)[MAXV], uint32_t eligible, int& be_out, float& bv_out) {
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int be = INT_MAX;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int e = lane + 32 * q;
    if (((eligible >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < be))) {
      bv = v[q];
      be = e;
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
  be_out = be;
  bv_out = bv;
}

// The compensated dot product of warp_exact_dot, with the token row read from global memory (it stays in
// L1 across the candidates of a token). Lane l takes chunks l, l + 32, ... in batches of 2 per lane, the
// next batch's loads in flight while the current one is summed, into four independent compensated pairs
// (more independent dependency chains per lane) held as two packed pairs: the words x and z of a chunk go
// to the first, y and w to the second. Two-sums merge the four at the end.
__device__ __forceinline__ void acc_chunk(f32x2_t (&s)[2], f32x2_t (&c)[2], const uint4& xv, const uint4& wv) {
  acc_prod_x2(s[0], c[0], xv.x, wv.x);
  acc_prod_x2(s[1], c[1], xv.y, wv.y);
  acc_prod_x2(s[0], c[0], xv.z, wv.z);
  acc_prod_x2(s[1], c[1], xv.w, wv.w);
}

__device__ __noinline__ float warp_exact_dot_global(const uint4* __restrict__ xr, const uint4* __restrict__ wrow,
                                                   int nchunks) {
  const int lane = threadIdx.x & 31;
  constexpr int B = 2;          // chunks per lane per batch
  const int n = nchunks >> 5;   // chunks per lane: H is a multiple of 256, so nchunks = H / 8 is a multiple of 32
  const int nb = n - n % B;     // those in whole batches; an odd last chunk is summed after them
  xr += lane;
  wrow += lane;
  f32x2_t s[2] = {0ull, 0ull}, c[2] = {0ull, 0ull};
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 xv[B], wv[B], xn[B], wn[B];
#pragma unroll
  for (int j = 0; j < B; ++j) {
    xv[j] = wv[j] = xn[j] = wn[j] = zero;
    if (j < nb) {
      xv[j] = __ldg(xr + 32 * j);
      wv[j] = __ldg(wrow + 32 * j);
    }
  }
  for (int it = 0; it < nb; it += B) {
    if (it + B < nb) {  // the next batch, in flight while this one is summed (the same branch in every lane)
#pragma unroll
      for (int j = 0; j < B; ++j) {
        xn[j] = __ldg(xr + 32 * (it + B + j));
        wn[j] = __ldg(wrow + 32 * (it + B + j));
      }
    }
#pragma unroll
    for (int j = 0; j < B; ++j) acc_chunk(s, c, xv[j], wv[j]);
#pragma unroll
    for (int j = 0; j < B; ++j) {
      xv[j] = xn[j];
      wv[j] = wn[j];
    }
  }
  if (nb < n) acc_chunk(s, c, __ldg(xr + 32 * nb), __ldg(wrow + 32 * nb));
  float a, ea, b, eb, sum, e;
  two_sum(lane0(s[0]), lane1(s[0]), a, ea);
  two_sum(lane0(s[1]), lane1(s[1]), b, eb);
  two_sum(a, b, sum, e);
  float cc = __fadd_rn(__fadd_rn(__fadd_rn(lane0(c[0]), lane1(c[0])), __fadd_rn(lane0(c[1]), lane1(c[1]))),
                       __fadd_rn(__fadd_rn(ea, eb), e));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float so = __shfl_xor_sync(kFull, sum, off);
    const float co = __shfl_xor_sync(kFull, cc, off);
    float ns, ne;
    two_sum(sum, so, ns, ne);
    sum = ns;
    cc = __fadd_rn(__fadd_rn(cc, co), ne);
  }
  return __fadd_rn(sum, cc);
}

// One warp per token, 8 tokens per CTA, no block barriers: for large T, where throughput matters more than
// the latency of a single token. The same four steps as router_refine_kernel, on register arrays (expert
// lane + 32 q in slot q of each lane), with the exact dot products of a token's candidates done one after
// another by its warp.
template <int MAXV>
__global__ void __launch_bounds__(256, 3) router_refine_warp_kernel(int T, int H, int E, int k,
                                                                 const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ wr,
                                                                 const float* __restrict__ bias,
                                                                 const float* __restrict__ nw2, float* logits,
                                                                 int32_t* __restrict__ ids_out,
                                                                 float* __restrict__ w_out, uint32_t* err) {
  __shared__ int s_ce[8][32];          // each warp's candidates (at most 32 on the ranking path): experts
  __shared__ float s_cv[8][32];        // and their exact logits
  __shared__ int s_pe[8][kMaxTopK];    // each warp's k picks in order: experts
  __shared__ float s_pv[8][kMaxTopK];  // and their exact logits
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;  // the whole warp leaves; nothing below synchronises beyond the warp
  const int nchunks = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  float sq = 0.0f;
  for (int c = lane; c < nchunks; c += 32) sq = sumsq8(__ldg(xr + c), sq);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(kFull, sq, off);
  const float nx = sqrtf(sq);
  float* lrow = logits + (size_t)t * E;
  float l[MAXV], d[MAXV];
  uint32_t valid = 0;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int e = lane + 32 * q;
    l[q] = -INFINITY;
    d[q] = 0.0f;
    if (e < E) {
      float v = __ldcg(lrow + e);
      if (bias != nullptr) v = __fadd_rn(v, bias[e]);
      // the fp32 norms are low by at most ~3e-4 relative: the (1 + 2^-10) factor keeps the bound above it
      d[q] = fmaf(kBoundRel * 1.0009765625f, nx * sqrtf(__ldcg(nw2 + e)), kBoundUlp * fabsf(v));
      l[q] = v;
      valid |= 1u << q;
    }
  }
  // tau = the k-th largest lower end
  float lo[MAXV];
#pragma unroll
  for (int q = 0; q < MAXV; ++q) lo[q] = __fsub_rd(l[q], d[q]);
  float tau = __int_as_float(0x7FC00000);
  {
    uint32_t left = valid;
    for (int j = 0; j < k; ++j) {
      int be;
      float bv;
      warp_argmax<MAXV>(lo, left, be, bv);
      if (be == INT_MAX) {
        tau = __int_as_float(0x7FC00000);
        break;
      }
      if ((be & 31) == lane) left &= ~(1u << (be >> 5));
      tau = bv;
    }
  }
  // candidates (all valid experts when tau is NaN), each given its exact logit
  uint32_t cand = 0;
#pragma unroll
  for (int q = 0; q < MAXV; ++q)
    if (((valid >> q) & 1u) && !(__fadd_ru(l[q], d[q]) < tau)) cand |= 1u << q;
  // one call site of the (out-of-line) dot product keeps the kernel small enough for the instruction cache
  for (int q = 0; q < MAXV; ++q) {
    uint32_t ball = __ballot_sync(kFull, (cand >> q) & 1u);
    while (ball != 0u) {
      const int src = __ffs(ball) - 1;
      ball &= ball - 1u;
      const int e = src + 32 * q;
      float lv = warp_exact_dot_global(xr, reinterpret_cast<const uint4*>(wr + (size_t)e * H), nchunks);
      if (bias != nullptr) lv = __fadd_rn(lv, bias[e]);
      if (lane == src) {
#pragma unroll
        for (int qq = 0; qq < MAXV; ++qq)
          if (qq == q) l[qq] = lv;
      }
    }
  }
  // the top k of the candidates by exact logit: value descending, ties to the lower id, a NaN never taken. Pick
  // j goes to place j of this warp's list s_pe/s_pv.
  bool bad = false;
  int nc = 0;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) nc += __popc(__ballot_sync(kFull, (cand >> q) & 1u));
  if (nc <= 32) {
    // the usual case (about k candidates): candidate p to lane p, each ranked against all of them at once (the
    // count of candidates ahead of it in that order); rank r is pick r
    int pos = 0;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const bool mine = (cand >> q) & 1u;
      const uint32_t ball = __ballot_sync(kFull, mine);
      if (mine) {
        const int p = pos + __popc(ball & ((1u << lane) - 1u));
        s_ce[warp][p] = lane + 32 * q;
        s_cv[warp][p] = l[q];
      }
      pos += __popc(ball);
    }
    __syncwarp();
    const bool have = lane < nc;
    const int ce = have ? s_ce[warp][lane] : INT_MAX;
    const float cv = have ? s_cv[warp][lane] : __int_as_float(0x7FC00000);
    int rank = 0;
    for (int i = 0; i < nc; ++i) {
      const float vi = __shfl_sync(kFull, cv, i);
      const int ei = __shfl_sync(kFull, ce, i);
      rank += (vi > cv || (vi == cv && ei < ce)) ? 1 : 0;  // a NaN is ahead of nothing
    }
    const bool num = have && cv == cv;  // the numbers' ranks are 0, 1, ..., one each
    bad = __popc(__ballot_sync(kFull, num)) < k;
    if (num && rank < k) {
      s_pe[warp][rank] = ce;
      s_pv[warp][rank] = cv;
    }
  } else {  // more (a NaN bound, or many ties): k passes of a warp argmax
    uint32_t left = cand;
    for (int j = 0; j < k; ++j) {
      int be;
      float bv;
      warp_argmax<MAXV>(l, left, be, bv);
      if (be == INT_MAX) {
        bad = true;
        break;
      }
      if ((be & 31) == lane) left &= ~(1u << (be >> 5));
      if (lane == 0) {
        s_pe[warp][j] = be;
        s_pv[warp][j] = bv;
      }
    }
  }
  __syncwarp();
  // the softmax over the k picks, lane j taking pick j; the sum runs in pick order
  if (bad) {  // fewer than k comparable logits: NaN input
    if (lane == 0) raise_error(err, FP4MOE_ERR_EXPERT_ID);
    if (lane < k) {
      ids_out[(size_t)t * k + lane] = 0;
      w_out[(size_t)t * k + lane] = 0.0f;
    }
  } else {
    const int pe = lane < k ? s_pe[warp][lane] : 0;
    const float pv = lane < k ? s_pv[warp][lane] : 0.0f;
    const float lmax = __shfl_sync(kFull, pv, 0);
    const float ex = lane < k ? expf(__fsub_rn(pv, lmax)) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(kFull, ex, j));
    if (lane < k) {
      ids_out[(size_t)t * k + lane] = pe;
      w_out[(size_t)t * k + lane] = __fdiv_rn(ex, sum);
    }
  }
#pragma unroll
  for (int q = 0; q < MAXV; ++q)
    if ((valid >> q) & 1u) lrow[lane + 32 * q] = l[q];
}

template <int MAXV>
cudaError_t launch_refine_warp(int T, int H, int E, int k, const uint16_t* x, const uint16_t* wr, const float* bias,
                               const float* nw2, float* logits, int32_t* ids, float* w, uint32_t* err,
                               cudaStream_t st) {
  return launch_pdl(router_refine_warp_kernel<MAXV>, dim3((T + 7) / 8), dim3(256), 0, st, T, H, E, k, x, wr, bias,
                    nw2, logits, ids, w, err);
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

// Enough for every T <= min(max_tokens, 256) (a single tile of tokens), so the split chosen below depends only
// on T, E and H, never on the buffer.
size_t router_partial_bytes(const fp4moe_config& cfg) {
  const size_t Tt = (size_t)std::min(cfg.max_tokens, RT_MAX_BN);
  return (size_t)RT_MAX_PART_SPLIT * (Tt + 1) * (size_t)cfg.num_experts * 4;
}

fp4moe_status router_topk_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* wr,
                                 const float* bias, float* logits, float* nw2, float* part, size_t part_bytes,
                                 int32_t* ids, float* w, uint32_t* err, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  const int H = cfg.hidden, E = cfg.num_experts, k = cfg.top_k;
  if (!configure_router()) return FP4MOE_CUDA_ERROR;
  const int BN = T >= RT_MAX_BN ? RT_MAX_BN : (T + 31) / 32 * 32;  // tokens per tile: a multiple of 32
  CUtensorMap tmX, tmW;
  if (!encode_u8_sw128(&tmX, x, (uint64_t)H * 2, (uint64_t)T, (uint32_t)BN)) return FP4MOE_CUDA_ERROR;
  if (!encode_u8_sw128(&tmW, wr, (uint64_t)H * 2, (uint64_t)E, RT_BM)) return FP4MOE_CUDA_ERROR;
  const int n_et = (E + RT_BM - 1) / RT_BM, n_tt = (T + BN - 1) / BN;
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  // One tile of tokens: split K over up to 16 independent CTAs with at least 4 K atoms each, whose partial
  // tiles the refine sums. Otherwise split K over a cluster while the tiles alone leave SMs idle, keeping at
  // least 2 K atoms per split, and sum through distributed shared memory.
  int S = 1;
  bool partial = false;
  if (n_tt == 1 && part != nullptr) {
    while (S * 2 <= RT_MAX_PART_SPLIT && n_et * S * 2 <= nsm && (H / 64) >= 4 * S * 2 &&
           (size_t)S * 2 * ((size_t)T + 1) * E * 4 <= part_bytes)
      S *= 2;
    partial = S > 1;
  }
  if (!partial) {
    S = 1;
    while (S * 2 <= RT_MAX_SPLIT && n_et * n_tt * S * 2 <= nsm && (H / 64) >= 4 * S) S *= 2;
  }
  RouterParams prm;
  prm.T = T;
  prm.H = H;
  prm.E = E;
  prm.S = S;
  prm.BN = BN;
  prm.stage = RT_A + BN * RT_KBYTES;
  prm.NS = RT_BAR_OFF / prm.stage < RT_MAX_STAGES ? RT_BAR_OFF / prm.stage : RT_MAX_STAGES;
  prm.partial = partial ? 1 : 0;
  prm.lt = partial ? part : logits;
  prm.nw2 = partial ? part + (size_t)S * T * E : nw2;
  prm.err = err;

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_et, n_tt, S);
  lc.blockDim = dim3(RT_THREADS);
  lc.dynamicSmemBytes = RT_SMEM;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = partial ? 1 : S;
  lc.attrs = attr;
  lc.numAttrs = 2;
  if (cudaLaunchKernelEx(&lc, router_mma_kernel, tmX, tmW, prm) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  cudaError_t r;
  if (T < kWarpRefineMinT) {  // latency-bound: one CTA per token spreads its exact dot products over 8 warps
    r = launch_pdl(router_refine_kernel, dim3(T), dim3(256), 0, st, (int)T, H, E, k, partial ? S : 1,
                   partial ? (const float*)part : nullptr, x, wr, bias, (const float*)nw2, logits, ids, w, err);
  } else {
    const int maxv = (E + 31) / 32;
    const float* cnw2 = nw2;
    if (maxv <= 2) r = launch_refine_warp<2>(T, H, E, k, x, wr, bias, cnw2, logits, ids, w, err, st);
    else if (maxv <= 4) r = launch_refine_warp<4>(T, H, E, k, x, wr, bias, cnw2, logits, ids, w, err, st);
    else if (maxv <= 8) r = launch_refine_warp<8>(T, H, E, k, x, wr, bias, cnw2, logits, ids, w, err, st);
    else if (maxv <= 16) r = launch_refine_warp<16>(T, H, E, k, x, wr, bias, cnw2, logits, ids, w, err, st);
    else r = launch_refine_warp<32>(T, H, E, k, x, wr, bias, cnw2, logits, ids, w, err, st);
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
