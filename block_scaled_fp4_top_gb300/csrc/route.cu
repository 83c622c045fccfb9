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
//   1-2. router_mma + router_refine (router.cu): logits and softmax top-k.
//   then, for T*k <= kSmallPairs (decode):
//   3. layout_small  8 CTAs, one slice of rows each: counts, offsets, padded offsets, slot ranks and
//                    pair_of_row
//   otherwise (prefill):
//   3. hist          grid (chunks of 64 tokens): per-chunk expert histograms
//   4. scan          1 CTA: chunk prefix per expert, counts, offsets, padded offsets
//   5. slots         grid (chunks): slot ranks in ascending pair order
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
constexpr int kSmallPairs = 4096;    // one-launch layout up to this many (token, k) pairs
constexpr int kSmallParts = 8;       // its CTAs, one slice of the padded rows each
constexpr int kSmallHist = 8192;     // its per-chunk expert histogram: at most min(32, 8192 / E) chunks
static_assert(kMaxExperts <= 8192 && kMaxExperts <= 32767, "a chunk row fits the histogram; ids fit int16");

// Inclusive block scans of two values at once (one set of barriers for both); s_warp holds 64 ints.
__device__ __forceinline__ int2 block_inclusive_scan2(int2 v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ox = __shfl_up_sync(kFull, v.x, off);
    const int oy = __shfl_up_sync(kFull, v.y, off);
    if (lane >= off) {
      v.x += ox;
      v.y += oy;
    }
  }
  if (lane == 31) {
    s_warp[warp] = v.x;
    s_warp[32 + warp] = v.y;
  }
  __syncthreads();
  if (warp == 0) {
    const bool in = lane < (int)(blockDim.x >> 5);
    int wx = in ? s_warp[lane] : 0, wy = in ? s_warp[32 + lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ox = __shfl_up_sync(kFull, wx, off);
      const int oy = __shfl_up_sync(kFull, wy, off);
      if (lane >= off) {
        wx += ox;
        wy += oy;
      }
    }
    s_warp[lane] = wx;
    s_warp[32 + lane] = wy;
  }
  __syncthreads();
  const int2 r = make_int2(v.x + (warp > 0 ? s_warp[warp - 1] : 0), v.y + (warp > 0 ? s_warp[32 + warp - 1] : 0));
  __syncthreads();
  return r;
}

// Counts, inclusive offsets and padded offsets for expert e = threadIdx.x
// (1024 threads), given its count c. Returns the first row of the expert's
// block in `start`. The R padded rows are cut into nparts slices, a multiple
// of 4 rows apart; this CTA (part) alone writes the rows [r_lo, r_hi): here
// every one of them below cap gets -1 with coalesced stores, and the slot
// pass that follows overwrites the real ones. Part 0 writes counts, offsets
// and padded offsets.
__device__ __forceinline__ void offsets_and_pads(int E, int cap, int c, int* s_warp, int32_t* counts, int32_t* offsets,
                                                 int32_t* poff, int32_t* pair_of_row, uint32_t* err, int part,
                                                 int nparts, int& start, int& r_lo, int& r_hi) {
  __shared__ int s_R;
  const int e = threadIdx.x;
  const int P = (c + 127) & ~127;
  const int2 sc = block_inclusive_scan2(make_int2(c, P), s_warp);
  const int oc = sc.x, op = sc.y;
  start = op - P;
  if (e < E && part == 0) {
    counts[e] = c;
    offsets[e] = oc;
    poff[e] = op;
  }
  if (e == E - 1) {
    s_R = op;
    if (op > cap && part == 0) raise_error(err, FP4MOE_ERR_CAPACITY);
  }
  __syncthreads();
  const int R = s_R;
  r_lo = (int)((long long)(R / 4) * part / nparts) * 4;
  r_hi = part + 1 == nparts ? R : (int)((long long)(R / 4) * (part + 1) / nparts) * 4;
  const int R0 = min(r_lo, cap), R1 = pair_of_row != nullptr ? min(r_hi, cap) : R0;  // no map: no row fill
  int r0 = R0;
  if ((reinterpret_cast<uintptr_t>(pair_of_row) & 15u) == 0) {  // four rows per store where aligned
    const int4 m1 = make_int4(-1, -1, -1, -1);
    for (int q = R0 / 4 + threadIdx.x; q < R1 / 4; q += blockDim.x) reinterpret_cast<int4*>(pair_of_row)[q] = m1;
    r0 = max(R0, R1 & ~3);
  }
  for (int r = r0 + threadIdx.x; r < R1; r += blockDim.x) pair_of_row[r] = -1;
  __syncthreads();
}

// Local expert of global id g: g - first for the experts [first, first + E) this layer holds, -1 for an
// expert held elsewhere (its pair is masked out, "Bug 8"), -2 for an id outside [0, Eg) (an error).
__device__ __forceinline__ int local_expert(int g, int Eg, int first, int E) {
  if (g < 0 || g >= Eg) return -2;
  const int l = g - first;
  return (l >= 0 && l < E) ? l : -1;
}

// Decode-sized layout in kSmallParts CTAs of 1024 threads: each builds the
// whole histogram, offsets and slot ranks (a few thousand pairs at most) and
// writes only the rows of its own slice, so no CTA waits for another and no
// row has two writers. Slots run in ascending pair order. Each warp walks its own contiguous chunk
// of pairs 32 at a time from its chunk's per-expert base; lanes sharing an
// expert rank themselves by lane order.
__global__ void __launch_bounds__(1024) layout_small_kernel(int npairs, int Eg, int first, int E, int cap,
                                                            const int32_t* __restrict__ ids,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ poff,
                                                            int32_t* __restrict__ slot_of_pair,
                                                            int32_t* __restrict__ pair_of_row, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  // The pairs are cut into nch contiguous chunks, one per warp; s_hist[ch * E + e] counts expert e in chunk
  // ch, then holds the chunk's first slot for e. Slots stay in ascending pair order.
  __shared__ int s_hist[kSmallHist];
  __shared__ int s_warp[64];
  __shared__ int16_t s_ids[kSmallPairs];  // local expert ids (E <= 1024), -1 for a masked pair
  // at most one chunk of 32 pairs per warp keeps the per-expert chunk walks below short
  const int nch = max(1, min(min(32, kSmallHist / E), (npairs + 31) / 32));
  const int len = (npairs + nch - 1) / nch;
  for (int i = threadIdx.x; i < nch * E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int e = local_expert(__ldcg(ids + p), Eg, first, E);
    if (e >= 0) atomicAdd(&s_hist[(p / len) * E + e], 1);
    else if (e == -2) raise_error(err, FP4MOE_ERR_EXPERT_ID);
    s_ids[p] = (int16_t)(e < 0 ? -1 : e);
  }
  __syncthreads();
  int c = 0;
  if (threadIdx.x < E)
    for (int ch = 0; ch < nch; ++ch) c += s_hist[ch * E + threadIdx.x];
  int start;
  int r_lo, r_hi;
  offsets_and_pads(E, cap, c, s_warp, counts, offsets, poff, pair_of_row, err, blockIdx.x, gridDim.x, start, r_lo,
                   r_hi);
  if (threadIdx.x < E) {
    int base = start;
    for (int ch = 0; ch < nch; ++ch) {
      const int n = s_hist[ch * E + threadIdx.x];
      s_hist[ch * E + threadIdx.x] = base;
      base += n;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= nch) return;
  int* base = s_hist + warp * E;
  const int p1 = min(npairs, (warp + 1) * len);
  for (int pb = warp * len; pb < p1; pb += 32) {
    const int p = pb + lane;
    const int e = (p < p1) ? s_ids[p] : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int slot = base[e] + rank;
      if (slot >= r_lo && slot < r_hi) {  // the slice that holds the slot writes both maps
        slot_of_pair[p] = slot;
        if (slot < cap) pair_of_row[slot] = p;
        else raise_error(err, FP4MOE_ERR_CAPACITY);
      }
    } else if (p < p1 && blockIdx.x == 0) {
      slot_of_pair[p] = -1;  // held by no local expert: no slot
    }
    __syncwarp();
    if (e >= 0 && rank == 0) base[e] += __popc(peers);
    __syncwarp();
  }
}

// Per-chunk expert histograms (64 tokens per chunk), for large T.
__global__ void __launch_bounds__(256) hist_kernel(int T, int Eg, int first, int E, int k,
                                                   const int32_t* __restrict__ ids, int32_t* __restrict__ hist,
                                                   uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sh[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kRouteChunk * k;
  const int p1 = min(T, (blockIdx.x + 1) * kRouteChunk) * k;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = local_expert(__ldcg(ids + p), Eg, first, E);
    if (e >= 0) atomicAdd(&sh[e], 1);
    else if (e == -2) raise_error(err, FP4MOE_ERR_EXPERT_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
}

// One CTA of 1024 threads: exclusive prefix of the chunk histograms over the chunks (in place), then
// counts, offsets and padded offsets (slots_kernel marks the padding rows). Each expert's column is split among tpe = 1024 / E threads
// (a power of two, at most 32, so one warp holds them all): every part loads its run of chunk counts at
// once, the parts' sums are scanned across their lanes, and each part rewrites its run from its own base.
// For E = 256 that is four parts of 32 chunks at T = 8192: one round trip to L2 instead of eight.
__global__ void __launch_bounds__(1024) scan_kernel(int E, int nchunks, int cap, int32_t* __restrict__ hist,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ poff, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_warp[64];
  __shared__ int s_c[kMaxExperts];
  int tpe = 1;
  while (tpe < 32 && tpe * 2 * E <= 1024) tpe *= 2;
  const int e = threadIdx.x / tpe, q = threadIdx.x % tpe;
  const int per = (nchunks + tpe - 1) / tpe, b0 = q * per, b1 = min(nchunks, b0 + per);
  int sum = 0;
  if (e < E) {
    // this part's chunk counts, 16 loads in flight at a time
    for (int bb = b0; bb < b1; bb += 16) {
      int h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = (bb + i < b1) ? __ldcg(hist + (size_t)(bb + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) sum += h[i];
    }
  }
  // exclusive prefix of the parts' sums across the tpe lanes of expert e (one warp holds them all)
  int incl = sum;
  for (int off = 1; off < tpe; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off, tpe);
    if (q >= off) incl += o;
  }
  int run = incl - sum;
  if (e < E) {
    for (int bb = b0; bb < b1; bb += 16) {
      int h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = (bb + i < b1) ? __ldcg(hist + (size_t)(bb + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (bb + i < b1) hist[(size_t)(bb + i) * E + e] = run;
        run += h[i];
      }
    }
    if (q == tpe - 1) s_c[e] = incl;  // the expert's total count
  }
  __syncthreads();
  const int c = threadIdx.x < E ? s_c[threadIdx.x] : 0;
  int start;
  int r_lo, r_hi;
  // the padding rows' -1 is left to slots_kernel, spread over its CTAs: one CTA writing all R rows here took
  // longer than the rest of this kernel
  offsets_and_pads(E, cap, c, s_warp, counts, offsets, poff, nullptr, err, 0, 1, start, r_lo, r_hi);
}

// Slot of every pair of one 64-token chunk, in ascending pair order. The chunk's pairs are cut into one
// contiguous run per warp. Each warp counts its run's pairs per expert into its own shared-memory row; a
// prefix over the warp rows then gives every warp, for every expert, the first slot after the pairs of the
// chunk's earlier runs; within a run, lanes that share an expert rank themselves by lane order, 32 pairs at
// a time. No slot depends on the order of atomics. The CTAs also mark the padding rows -1, expert by expert.
constexpr int kSlotWarps = 8;
__global__ void __launch_bounds__(32 * kSlotWarps) slots_kernel(int T, int Eg, int first, int E, int k, int cap,
                                                                const int32_t* __restrict__ ids,
                                                                const int32_t* __restrict__ counts,
                                                                const int32_t* __restrict__ poff,
                                                                const int32_t* __restrict__ chunk_base,
                                                                int32_t* __restrict__ slot_of_pair,
                                                                int32_t* __restrict__ pair_of_row, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int s_cnt[];  // [kSlotWarps][E]: pairs of each warp's run per expert, then its first slot
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kSlotWarps * E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kRouteChunk * k;
  const int p1 = min(T, (blockIdx.x + 1) * kRouteChunk) * k;
  const int per = ((p1 - p0) + kSlotWarps - 1) / kSlotWarps;
  const int w0 = min(p1, p0 + warp * per), w1 = min(p1, w0 + per);
  for (int p = w0 + lane; p < w1; p += 32) {
    const int e = local_expert(__ldcg(ids + p), Eg, first, E);
    if (e >= 0) atomicAdd(&s_cnt[warp * E + e], 1);
  }
  __syncthreads();
  // per expert: the chunk's base slot, then each warp row's first slot (exclusive prefix over the warps)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = __ldcg(chunk_base + (size_t)blockIdx.x * E + e) + (__ldcg(poff + e) - ((__ldcg(counts + e) + 127) & ~127));
#pragma unroll
    for (int w = 0; w < kSlotWarps; ++w) {
      const int c = s_cnt[w * E + e];
      s_cnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int* base = s_cnt + warp * E;
  for (int pb = w0; pb < w1; pb += 32) {
    const int p = pb + lane;
    int e = (p < w1) ? local_expert(__ldcg(ids + p), Eg, first, E) : -1;
    if (e < 0) e = -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int slot = base[e] + rank;
      slot_of_pair[p] = slot;
      if (slot < cap) pair_of_row[slot] = p;
      else raise_error(err, FP4MOE_ERR_CAPACITY);
    } else if (p < w1) {
      slot_of_pair[p] = -1;  // held by no local expert: no slot
    }
    __syncwarp();
    if (e >= 0 && rank == 0) base[e] += __popc(peers);
    __syncwarp();
  }
  // the padding rows of experts blockIdx.x, blockIdx.x + gridDim.x, ...: -1 (rows from cap on are not written)
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int n = __ldcg(counts + e), pe = __ldcg(poff + e);
    const int end = min(pe, cap);
    for (int r = pe - (((n + 127) & ~127) - n) + threadIdx.x; r < end; r += blockDim.x) pair_of_row[r] = -1;
  }
}

}  // namespace

fp4moe_status route_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                           const float* bias, float* logits, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* poff, int32_t* slot_of_pair, int32_t* pair_of_row,
                           int32_t* hist, float* nw2, float* part, size_t part_bytes, uint32_t* err,
                           cudaStream_t st) {
  const int Eg = cfg.num_experts, first = cfg.ep_count > 0 ? cfg.ep_first : 0, E = local_experts(cfg);
  const int k = cfg.top_k;
  const int cap = (int)capacity_rows(cfg, T);
  const int npairs = T * k;
  const fp4moe_status rs =
      router_topk_launch(cfg, T, x, router_w, bias, logits, nw2, part, part_bytes, ids, w, err, st);
  if (rs != FP4MOE_OK) return rs;
  cudaError_t r = cudaSuccess;
  if (npairs <= kSmallPairs) {
    r = launch_pdl(layout_small_kernel, dim3(kSmallParts), dim3(1024), 0, st, npairs, Eg, first, E, cap, (const int32_t*)ids,
                   counts, offsets, poff, slot_of_pair, pair_of_row, err);
  } else {
    const int nchunks = (T + kRouteChunk - 1) / kRouteChunk;
    r = launch_pdl(hist_kernel, dim3(nchunks), dim3(256), 0, st, T, Eg, first, E, k, (const int32_t*)ids, hist, err);
    if (r == cudaSuccess)
      r = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, st, E, nchunks, cap, hist, counts, offsets, poff, err);
    if (r == cudaSuccess)
      r = launch_pdl(slots_kernel, dim3(nchunks), dim3(32 * kSlotWarps), (size_t)kSlotWarps * E * sizeof(int), st, T, Eg,
                     first, E, k, cap, (const int32_t*)ids,
                     (const int32_t*)counts, (const int32_t*)poff, (const int32_t*)hist, slot_of_pair, pair_of_row,
                     err);
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
