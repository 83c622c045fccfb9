// Routing: router logits, softmax top-k, per-expert counts, offsets and
// 128-row-padded slots.
//
// This is the device-native routing of "CUDA-Graph Safety / GPU-Native
// Requirements" (SECTION B: counts by scatter-add into a preallocated buffer,
// no bincount; SECTION C row 4: expert offsets stay on the GPU). The layout
// rules come from "Current Bug: CuTeDSLMoERunner": offsets without a leading 0
// ("Bug 4"), searchsorted(right=True) ownership ("Bug 2") and 128-row-aligned
// expert slots ("Bug 14").
//
// Launches, each with a fixed grid chosen from the host-known T:
//   1. logits_topk   grid (T, ceil(E/64)), 1024 threads. Each CTA computes 64
//                    logits of one token, with a compensated fp32 dot product
//                    per expert (4 H-quarters x 8 expert groups of warps). The
//                    last CTA of the token to finish (an arrival counter)
//                    takes the softmax top-k of all E logits.
//   then, for T*k <= kSmallPairs (decode):
//   2. layout_small  1 CTA: counts, offsets, padded offsets, slot ranks and
//                    pair_of_row
//   otherwise (prefill):
//   2. hist          grid (chunks of 64 tokens): per-chunk expert histograms
//   3. scan          1 CTA: chunk prefix per expert, counts, offsets, padded offsets
//   4. slots         grid (chunks): slot ranks in ascending pair order
// Every output is run-to-run deterministic: integer atomics only count, and
// ranks never depend on the order of atomics. Results of the previous launch
// are read through L2 (ld.global.cg), because with programmatic dependent
// launch a kernel can start before its predecessor ends.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kExpertsPerCta = 64;   // logits_topk: 8 warps x 8 experts
constexpr int kSmallPairs = 4096;    // single-CTA layout up to this many (token, k) pairs

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

// Top-k of one token's E logits by one warp: descending logit, ties to the
// lower expert id. Then the renormalised softmax weights (lane 0 writes).
template <int MAXV>
__device__ void warp_topk(const float* __restrict__ l, int E, int k, int32_t* ids_out, float* w_out, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  float v[MAXV];
  uint32_t taken = 0;
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int e = q * 32 + lane;
    v[q] = (e < E) ? __ldcg(l + e) : 0.0f;
    if (e >= E) taken |= 1u << q;
  }
  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int e = q * 32 + lane;
      if (!((taken >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < be))) {
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
    if (be >= E) {  // only possible with NaN logits
      if (lane == 0) raise_error(err, FP4MOE_ERR_EXPERT_ID);
      be = 0;
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sel_v[j] = bv;
    sel_e[j] = be;
  }
  if (lane == 0) {
    const float lmax = sel_v[0];
    float ex[kMaxTopK];
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(__fsub_rn(sel_v[j], lmax));
      sum = __fadd_rn(sum, ex[j]);
    }
    for (int j = 0; j < k; ++j) {
      ids_out[j] = sel_e[j];
      w_out[j] = __fdiv_rn(ex[j], sum);
    }
  }
}

// grid (T, ceil(E/64)), 1024 threads. Warp w of CTA (t, g) computes, for the
// 8 experts 64g + 8(w % 8) .. +7, the compensated partial sum over H-quarter
// w / 8. Inside the quarter each lane covers a fixed strided set of elements
// with two independent compensated accumulators, and a fixed butterfly
// combines the lanes. The 4 quarters are then summed in quarter order with
// two-sums. The last CTA of the token to arrive takes the top-k.
template <int MAXV>
__global__ void __launch_bounds__(1024) logits_topk_kernel(int T, int H, int E, int k, const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ wr,
                                                           const float* __restrict__ bias, float* __restrict__ logits,
                                                           int32_t* __restrict__ cnt, int32_t* __restrict__ ids_out,
                                                           float* __restrict__ w_out, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_part[4][kExpertsPerCta][2];
  __shared__ int s_last;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp & 7, quarter = warp >> 3;
  // 256 elements per warp iteration; quarter q takes iterations [q n / 4, (q + 1) n / 4) of n = H / 256
  const int n_it = H >> 8;
  const int it0 = quarter * n_it / 4, it1 = (quarter + 1) * n_it / 4;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {
    const int el = grp * 8 + q;  // expert index inside this CTA's 64
    const int e = blockIdx.y * kExpertsPerCta + el;
    float s = 0.0f, c = 0.0f;
    if (e < E) {
      const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
      float s0 = 0.0f, c0 = 0.0f, s1 = 0.0f, c1 = 0.0f;
#pragma unroll 2
      for (int it = it0; it < it1; ++it) {
        const uint4 xv = __ldg(xr + it * 32 + lane);
        const uint4 wv = __ldg(wrow + it * 32 + lane);
        acc_prod(s0, c0, bf16_lo(xv.x), bf16_lo(wv.x));
        acc_prod(s1, c1, bf16_hi(xv.x), bf16_hi(wv.x));
        acc_prod(s0, c0, bf16_lo(xv.y), bf16_lo(wv.y));
        acc_prod(s1, c1, bf16_hi(xv.y), bf16_hi(wv.y));
        acc_prod(s0, c0, bf16_lo(xv.z), bf16_lo(wv.z));
        acc_prod(s1, c1, bf16_hi(xv.z), bf16_hi(wv.z));
        acc_prod(s0, c0, bf16_lo(xv.w), bf16_lo(wv.w));
        acc_prod(s1, c1, bf16_hi(xv.w), bf16_hi(wv.w));
      }
      float e0;
      two_sum(s0, s1, s, e0);
      c = __fadd_rn(__fadd_rn(c0, c1), e0);
    }
    // fixed butterfly; every lane ends with the same (s, c)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float so = __shfl_xor_sync(kFull, s, off);
      const float co = __shfl_xor_sync(kFull, c, off);
      float ns, ne;
      two_sum(s, so, ns, ne);
      s = ns;
      c = __fadd_rn(__fadd_rn(c, co), ne);
    }
    if (lane == 0) {
      s_part[quarter][el][0] = s;
      s_part[quarter][el][1] = c;
    }
  }
  __syncthreads();
  if (threadIdx.x < kExpertsPerCta) {
    const int el = threadIdx.x;
    const int e = blockIdx.y * kExpertsPerCta + el;
    if (e < E) {
      float s = s_part[0][el][0], c = s_part[0][el][1];
#pragma unroll
      for (int qq = 1; qq < 4; ++qq) {
        float ns, ne;
        two_sum(s, s_part[qq][el][0], ns, ne);
        s = ns;
        c = __fadd_rn(__fadd_rn(c, s_part[qq][el][1]), ne);
      }
      float l = __fadd_rn(s, c);
      if (bias != nullptr) l = __fadd_rn(l, bias[e]);
      logits[(size_t)t * E + e] = l;
    }
  }
  // the last CTA of this token to arrive takes the top-k (threadfence-reduction pattern)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(cnt + t, 1) == (int)gridDim.y - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp == 0) {
    warp_topk<MAXV>(logits + (size_t)t * E, E, k, ids_out + (size_t)t * k, w_out + (size_t)t * k, err);
    if (lane == 0) cnt[t] = 0;  // ready for the next call
  }
}

__device__ __forceinline__ int block_inclusive_scan(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, w, off);
      if (lane >= off) w += o;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int r = v + (warp > 0 ? s_warp[warp - 1] : 0);
  __syncthreads();
  return r;
}

// Counts, inclusive offsets and padded offsets for expert e = threadIdx.x
// (1024 threads), given its count c; pads its padding rows with -1.
// Returns the first row of the expert's block in `start`.
// All padded rows [0, min(R, cap)) get -1 with coalesced stores; real rows
// are overwritten by the slot pass that follows.
__device__ __forceinline__ void offsets_and_pads(int E, int cap, int c, int* s_warp, int32_t* counts, int32_t* offsets,
                                                 int32_t* poff, int32_t* pair_of_row, uint32_t* err, int& start) {
  __shared__ int s_R;
  const int e = threadIdx.x;
  const int P = (c + 127) & ~127;
  const int oc = block_inclusive_scan(c, s_warp);
  const int op = block_inclusive_scan(P, s_warp);
  start = op - P;
  if (e < E) {
    counts[e] = c;
    offsets[e] = oc;
    poff[e] = op;
  }
  if (e == E - 1) {
    s_R = op;
    if (op > cap) raise_error(err, FP4MOE_ERR_CAPACITY);
  }
  __syncthreads();
  const int R = min(s_R, cap);
  for (int r = threadIdx.x; r < R; r += blockDim.x) pair_of_row[r] = -1;
  __syncthreads();
}

// Decode-sized layout in one CTA of 1024 threads: histogram, offsets, pads,
// and slots in ascending pair order (warp 0 walks the pairs 32 at a time;
// lanes sharing an expert rank themselves by lane order).
__global__ void __launch_bounds__(1024) layout_small_kernel(int npairs, int E, int cap,
                                                            const int32_t* __restrict__ ids,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ poff,
                                                            int32_t* __restrict__ slot_of_pair,
                                                            int32_t* __restrict__ pair_of_row, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_warp[32];
  __shared__ int s_ids[kSmallPairs];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    int e = __ldcg(ids + p);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    else {
      raise_error(err, FP4MOE_ERR_EXPERT_ID);
      e = -1;
    }
    s_ids[p] = e;
  }
  __syncthreads();
  const int c = (threadIdx.x < E) ? s_cnt[threadIdx.x] : 0;
  int start;
  offsets_and_pads(E, cap, c, s_warp, counts, offsets, poff, pair_of_row, err, start);
  if (threadIdx.x < E) s_base[threadIdx.x] = start;
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  for (int pb = 0; pb < npairs; pb += 32) {
    const int p = pb + lane;
    const int e = (p < npairs) ? s_ids[p] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int slot = s_base[e] + rank;
      slot_of_pair[p] = slot;
      if (slot < cap) pair_of_row[slot] = p;
      else raise_error(err, FP4MOE_ERR_CAPACITY);
    }
    __syncwarp();
    if (e >= 0 && rank == 0) s_base[e] += __popc(peers);
    __syncwarp();
  }
}

// Per-chunk expert histograms (64 tokens per chunk), for large T.
__global__ void __launch_bounds__(256) hist_kernel(int T, int E, int k, const int32_t* __restrict__ ids,
                                                   int32_t* __restrict__ hist, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sh[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kRouteChunk * k;
  const int p1 = min(T, (blockIdx.x + 1) * kRouteChunk) * k;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = __ldcg(ids + p);
    if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
    else raise_error(err, FP4MOE_ERR_EXPERT_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
}

// One CTA of 1024 threads, thread e = expert e: exclusive prefix of the chunk
// histograms (in place), then counts, offsets, padded offsets and pads.
__global__ void __launch_bounds__(1024) scan_kernel(int E, int nchunks, int cap, int32_t* __restrict__ hist,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ poff, int32_t* __restrict__ pair_of_row,
                                                    uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
    for (int b = 0; b < nchunks; ++b) {
      const int h = __ldcg(hist + (size_t)b * E + e);
      hist[(size_t)b * E + e] = c;
      c += h;
    }
  }
  int start;
  offsets_and_pads(E, cap, c, s_warp, counts, offsets, poff, pair_of_row, err, start);
}

// Slot of every pair of one 64-token chunk, in ascending pair order.
__global__ void __launch_bounds__(256) slots_kernel(int T, int E, int k, int cap, const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ poff,
                                                    const int32_t* __restrict__ chunk_base,
                                                    int32_t* __restrict__ slot_of_pair,
                                                    int32_t* __restrict__ pair_of_row, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int base[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = __ldcg(chunk_base + (size_t)blockIdx.x * E + e) + (__ldcg(poff + e) - ((__ldcg(counts + e) + 127) & ~127));
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int p0 = blockIdx.x * kRouteChunk * k;
  const int p1 = min(T, (blockIdx.x + 1) * kRouteChunk) * k;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    int e = (p < p1) ? __ldcg(ids + p) : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int slot = base[e] + rank;
      slot_of_pair[p] = slot;
      if (slot < cap) pair_of_row[slot] = p;
      else raise_error(err, FP4MOE_ERR_CAPACITY);
    }
    __syncwarp();
    if (e >= 0 && rank == 0) base[e] += __popc(peers);
    __syncwarp();
  }
}

template <int MAXV>
cudaError_t launch_logits_topk(int T, int H, int E, int k, const uint16_t* x, const uint16_t* wr, const float* bias,
                               float* logits, int32_t* cnt, int32_t* ids, float* w, uint32_t* err, cudaStream_t st) {
  return launch_pdl(logits_topk_kernel<MAXV>, dim3(T, (E + kExpertsPerCta - 1) / kExpertsPerCta), dim3(1024), 0, st,
                    T, H, E, k, x, wr, bias, logits, cnt, ids, w, err);
}

}  // namespace

fp4moe_status route_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                           const float* bias, float* logits, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* poff, int32_t* slot_of_pair, int32_t* pair_of_row,
                           int32_t* hist, int32_t* cnt, uint32_t* err, cudaStream_t st) {
  const int E = cfg.num_experts, H = cfg.hidden, k = cfg.top_k;
  const int cap = (int)capacity_rows(cfg, T);
  const int npairs = T * k;
  cudaError_t r = cudaSuccess;
  if (T > 0) {
    const int maxv = (E + 31) / 32;
    if (maxv <= 1) r = launch_logits_topk<1>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    else if (maxv <= 2) r = launch_logits_topk<2>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    else if (maxv <= 4) r = launch_logits_topk<4>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    else if (maxv <= 8) r = launch_logits_topk<8>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    else if (maxv <= 16) r = launch_logits_topk<16>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    else r = launch_logits_topk<32>(T, H, E, k, x, router_w, bias, logits, cnt, ids, w, err, st);
    if (r != cudaSuccess) return FP4MOE_CUDA_ERROR;
  }
  if (npairs <= kSmallPairs) {
    r = launch_pdl(layout_small_kernel, dim3(1), dim3(1024), 0, st, npairs, E, cap, (const int32_t*)ids, counts,
                   offsets, poff, slot_of_pair, pair_of_row, err);
  } else {
    const int nchunks = (T + kRouteChunk - 1) / kRouteChunk;
    r = launch_pdl(hist_kernel, dim3(nchunks), dim3(256), 0, st, T, E, k, (const int32_t*)ids, hist, err);
    if (r == cudaSuccess)
      r = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, st, E, nchunks, cap, hist, counts, offsets, poff,
                     pair_of_row, err);
    if (r == cudaSuccess)
      r = launch_pdl(slots_kernel, dim3(nchunks), dim3(256), 0, st, T, E, k, cap, (const int32_t*)ids,
                     (const int32_t*)counts, (const int32_t*)poff, (const int32_t*)hist, slot_of_pair, pair_of_row,
                     err);
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
