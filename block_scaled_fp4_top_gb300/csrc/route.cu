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
// Four launches, each with a fixed grid chosen from the host-known T:
//   1. router_logits  grid (ceil(E/32), T): a compensated fp32 dot product per (t, e)
//   2. topk_hist      grid (chunks of 64 tokens): warp top-k, softmax, chunk histogram
//   3. scan           1 CTA: chunk prefix per expert, counts, offsets, padded offsets
//   4. slots          grid (chunks): ranks in ascending pair order, one warp per chunk
// Nothing here depends on the order of floating-point atomics. The
// histogram uses integer atomics only, so every output is run-to-run
// deterministic.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Error-free transformation a + b = s + e (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void acc_pair(float& s, float& c, uint32_t xw, uint32_t ww) {
  // bf16 x bf16 products are exact in fp32 (8-bit significands)
  float e0, e1, s0;
  const float p0 = __fmul_rn(bf16_lo(xw), bf16_lo(ww));
  const float p1 = __fmul_rn(bf16_hi(xw), bf16_hi(ww));
  two_sum(s, p0, s0, e0);
  two_sum(s0, p1, s, e1);
  c = __fadd_rn(c, __fadd_rn(e0, e1));
}

// One warp per (token, expert), 4 experts per warp, 8 warps per CTA.
__global__ void __launch_bounds__(256) router_logits_kernel(int H, int E, const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ wr,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits) {
  const int t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const int nit = H >> 8;  // 256 elements per warp iteration
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    const int e = blockIdx.x * 32 + warp * 4 + q;
    if (e >= E) break;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    float s = 0.0f, c = 0.0f;
#pragma unroll 4
    for (int it = 0; it < nit; ++it) {
      const uint4 xv = __ldg(xr + it * 32 + lane);
      const uint4 wv = __ldg(wrow + it * 32 + lane);
      acc_pair(s, c, xv.x, wv.x);
      acc_pair(s, c, xv.y, wv.y);
      acc_pair(s, c, xv.z, wv.z);
      acc_pair(s, c, xv.w, wv.w);
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
      float l = __fadd_rn(s, c);
      if (bias != nullptr) l = __fadd_rn(l, bias[e]);
      logits[(size_t)t * E + e] = l;
    }
  }
}

// Top-k per token (one warp per token), renormalised softmax weights, and the
// per-chunk expert histogram.
template <int MAXV>
__global__ void __launch_bounds__(256) topk_hist_kernel(int T, int E, int k, const float* __restrict__ logits,
                                                        int32_t* __restrict__ ids_out, float* __restrict__ w_out,
                                                        int32_t* __restrict__ hist, uint32_t* err) {
  __shared__ int sh[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int i = 0; i < kRouteChunk / 8; ++i) {
    const int t = blockIdx.x * kRouteChunk + i * 8 + warp;
    if (t >= T) break;
    float v[MAXV];
    uint32_t taken = 0;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int e = q * 32 + lane;
      v[q] = (e < E) ? logits[(size_t)t * E + e] : 0.0f;
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
        ids_out[(size_t)t * k + j] = sel_e[j];
        w_out[(size_t)t * k + j] = __fdiv_rn(ex[j], sum);
        atomicAdd(&sh[sel_e[j]], 1);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
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

// One CTA of 1024 threads, thread e = expert e.
__global__ void __launch_bounds__(1024) scan_kernel(int E, int nchunks, int cap, int32_t* __restrict__ hist,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ poff, int32_t* __restrict__ pair_of_row,
                                                    uint32_t* err) {
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
    for (int b = 0; b < nchunks; ++b) {  // exclusive prefix over chunks, in place
      const int h = hist[(size_t)b * E + e];
      hist[(size_t)b * E + e] = c;
      c += h;
    }
  }
  const int P = (c + 127) & ~127;
  const int oc = block_inclusive_scan(c, s_warp);
  const int op = block_inclusive_scan(P, s_warp);
  if (e < E) {
    counts[e] = c;
    offsets[e] = oc;
    poff[e] = op;
    const int start = op - P;
    for (int r = start + c; r < op && r < cap; ++r) pair_of_row[r] = -1;
    if (e == E - 1 && op > cap) raise_error(err, FP4MOE_ERR_CAPACITY);
  }
}

// Slot of every pair in ascending pair order: warp 0 walks its chunk 32 pairs
// at a time, and lanes that share an expert rank themselves by lane order.
__global__ void __launch_bounds__(256) slots_kernel(int T, int E, int k, int cap, const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ poff,
                                                    const int32_t* __restrict__ chunk_base,
                                                    int32_t* __restrict__ slot_of_pair,
                                                    int32_t* __restrict__ pair_of_row, uint32_t* err) {
  __shared__ int base[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = chunk_base[(size_t)blockIdx.x * E + e] + (poff[e] - ((counts[e] + 127) & ~127));
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int p0 = blockIdx.x * kRouteChunk * k;
  const int p1 = min(T, (blockIdx.x + 1) * kRouteChunk) * k;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    int e = (p < p1) ? ids[p] : -1;
    if (p < p1 && (e < 0 || e >= E)) {
      raise_error(err, FP4MOE_ERR_EXPERT_ID);
      e = -1;
    }
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
void launch_topk(int nchunks, cudaStream_t st, int T, int E, int k, const float* logits, int32_t* ids, float* w,
                 int32_t* hist, uint32_t* err) {
  topk_hist_kernel<MAXV><<<nchunks, 256, 0, st>>>(T, E, k, logits, ids, w, hist, err);
}

}  // namespace

fp4moe_status route_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                           const float* bias, float* logits, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* poff, int32_t* slot_of_pair, int32_t* pair_of_row,
                           int32_t* hist, uint32_t* err, cudaStream_t st) {
  const int E = cfg.num_experts, H = cfg.hidden, k = cfg.top_k;
  const int cap = (int)capacity_rows(cfg, T);
  const int nchunks = (T + kRouteChunk - 1) / kRouteChunk;
  if (T > 0) {
    router_logits_kernel<<<dim3((E + 31) / 32, T), 256, 0, st>>>(H, E, x, router_w, bias, logits);
    const int maxv = (E + 31) / 32;
    if (maxv <= 1) launch_topk<1>(nchunks, st, T, E, k, logits, ids, w, hist, err);
    else if (maxv <= 2) launch_topk<2>(nchunks, st, T, E, k, logits, ids, w, hist, err);
    else if (maxv <= 4) launch_topk<4>(nchunks, st, T, E, k, logits, ids, w, hist, err);
    else if (maxv <= 8) launch_topk<8>(nchunks, st, T, E, k, logits, ids, w, hist, err);
    else if (maxv <= 16) launch_topk<16>(nchunks, st, T, E, k, logits, ids, w, hist, err);
    else launch_topk<32>(nchunks, st, T, E, k, logits, ids, w, hist, err);
  }
  scan_kernel<<<1, 1024, 0, st>>>(E, nchunks, cap, hist, counts, offsets, poff, pair_of_row, err);
  if (T > 0)
    slots_kernel<<<nchunks, 256, 0, st>>>(T, E, k, cap, ids, counts, poff, hist, slot_of_pair, pair_of_row, err);
  return cudaGetLastError() == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
