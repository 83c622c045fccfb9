// Tile schedules shared by the persistent grouped GEMMs (gemm.cu: 128 x 128 tiles, gemm_wide.cu: 128 x 256
// tiles): the dynamic chunk schedule, the per-role tile source and the static contiguous ranges. A kernel's
// parameter block P provides dyn, sched and err.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace fp4moe {

// Parameters of one grouped GEMM launch (both tile shapes). NT counts the kernel's own n-tiles.
struct GemmParams {
  int E, K, KB, b_rows, NT, k, cap, I, H, nacc;  // KB: ring stages per tile; nacc: accumulators (128 x 128 kernel)
  float limit;
  const int32_t* poff;
  const int32_t* pair_of_row;
  const uint8_t* b_codes;
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const float* alpha;
  const float* gs2;
  uint8_t* out_codes;
  uint8_t* out_sf;
  float* amax;       // W1 amax: the calibration maximum; W1 + SwiGLU: the running amax|h| (both non-negative)
  uint32_t* status;  // W1 + SwiGLU: sticky FP4MOE_SAT_* bits
  uint16_t* o_pairs;  // W2: bf16 rows [T*k][H] ("Data Flow": l2_out is BF16)
  uint32_t* err;
  int o_pairs32;  // W2: o_pairs is 32-byte aligned (every 128-column piece of a row is then)
  int dyn;     // 1: dynamic chunk schedule (large T); 0: contiguous static ranges (decode sizes)
  int steal;   // static schedule: the last tiles form a pool that CTAs take from `sched` once their range is done
  int* sched;  // {next chunk or pool tile, CTAs finished}: zero at launch, zeroed again by the launch's last CTA
};

// Tensor maps of the activation codes whose boxes are 16, 32, 64 and 128 rows
// high (128 bytes wide, 128-byte swizzle).
struct AMaps {
  CUtensorMap box[4];
};

// gemm_wide.cu: the 128 x 256 tile kernel. gemm_wide_fits: K and the weight rows suit it (K % 256, rows %
// 256). gemm_wide_launch takes the 128 x 128 kernel's parameters (NT, KB of 128-row tiles and 512-deep
// stages) and derives its own.
bool gemm_wide_fits(int K, int b_rows);
fp4moe_status gemm_wide_launch(GemmMode mode, const GemmParams& prm, const AMaps& tmA, cudaStream_t st);

namespace {

// Dynamic schedule. A chunk is at most kChunk tiles of one expert: for a one-m-tile expert, up to kChunk
// n-tiles (the activation tile fixed); otherwise one n-tile over up to kChunk m-tiles (the weight tile
// fixed). Chunks are numbered expert by expert (for several m-tiles: m-block, then n-tile), and CTAs take
// them in that order from a global counter. So the CTAs running at any moment share one expert's
// activation and weight tiles in L2, and the load balances itself.
constexpr int kChunk = 4;
constexpr int kSchedSlots = 4;  // chunk ids handed from the producer to the MMA issuer and the epilogue
constexpr int kPoolPerCta = 3;  // static schedule: pool tiles per CTA

// Static schedule with a pool: of the N tiles, the last ones (about three per CTA, at most a quarter) are not
// assigned. A CTA that has finished its contiguous range takes them one at a time from the counter, in tile
// order, so CTAs that stream slower than others (their place on the chip, the expert boundaries in their
// range) no longer hold up the whole launch. Fewer than four tiles per CTA: no pool.
__device__ __forceinline__ int tail_pool(int N, int G) {
  return N >= 4 * G ? min(kPoolPerCta * G, N / 4) : 0;
}

// Tiles per chunk of expert e: kChunk, except for the experts at the end of the order that hold the last
// two tiles per CTA or so, whose tiles go out one at a time. A chunk of four tiles taken last held the end of
// a launch up to its own length after the median CTA: a 35 us spread of CTA end times on the Zipf prefill W1.
__device__ __forceinline__ int chunk_tiles(int e, int e_tail) { return e >= e_tail ? 1 : kChunk; }

__device__ __forceinline__ int expert_chunks(int me, int NT, int sz) {
  return me == 0 ? 0 : (me == 1 ? (NT + sz - 1) / sz : ((me + sz - 1) / sz) * NT);
}

// m-tiles of expert e (its padded rows, up to r128 m-tiles in all)
__device__ __forceinline__ int expert_mtiles(const int* poff, int e, int r128) {
  return min(poff[e] >> 7, r128) - (e > 0 ? min(poff[e - 1] >> 7, r128) : 0);
}

// The dynamic schedule's chunk table, built by one warp: s_cstart[e] is the first chunk of expert e (empty
// experts share the next one's start), s_cstart[E] the number of chunks and s_cstart[E + 1] the first expert
// of the single-tile tail (the experts from the end of the order that hold at least 2 G tiles).
__device__ __forceinline__ void build_chunk_table(const int* s_poff, int* s_cstart, int E, int NT, int r128, int G,
                                                  int lane) {
  int e_tail = 0;
  if (lane == 0) {
    int tiles = 0, e = E;
    while (e > 0 && tiles < 2 * G) {
      --e;
      tiles += expert_mtiles(s_poff, e, r128) * NT;
    }
    e_tail = e;
  }
  e_tail = __shfl_sync(0xFFFFFFFFu, e_tail, 0);
  // per-lane sums over a block of experts, then a warp scan
  const int per = (E + 31) / 32, e0 = lane * per, e1 = min(E, e0 + per);
  int sum = 0;
  for (int e = e0; e < e1; ++e) sum += expert_chunks(expert_mtiles(s_poff, e, r128), NT, chunk_tiles(e, e_tail));
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
  for (int e = e0; e < e1; ++e) {
    s_cstart[e] = run;
    run += expert_chunks(expert_mtiles(s_poff, e, r128), NT, chunk_tiles(e, e_tail));
  }
  if (lane == 31) s_cstart[E] = incl;
  if (lane == 0) s_cstart[E + 1] = e_tail;
}

struct Chunk {
  int e, pm0, me;  // expert, its first m-tile, its m-tiles
  int n0, m0;      // first n-tile and m-tile of the chunk
  int count;       // tiles in the chunk
  bool along_n;    // one m-tile: walk n-tiles n0.. with m fixed; else m-tiles m0.. with n fixed

  __device__ __forceinline__ Tile tile(int i) const {
    const int mt = along_n ? m0 : m0 + i;
    return Tile{e, along_n ? n0 + i : n0, mt, me, mt == pm0 + me - 1};
  }
};

// Chunk c of the table of build_chunk_table.
__device__ __forceinline__ Chunk decode_chunk(int c, const int* s_cstart, const int* poff, int E, int NT, int r128) {
  int lo = 0, hi = E - 1;  // the last expert whose first chunk is <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_cstart[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  Chunk k;
  k.e = lo;
  k.pm0 = lo > 0 ? min(poff[lo - 1] >> 7, r128) : 0;
  k.me = min(poff[lo] >> 7, r128) - k.pm0;
  const int l = c - s_cstart[lo];
  const int sz = chunk_tiles(lo, s_cstart[E + 1]);
  k.along_n = (k.me == 1);
  if (k.along_n) {
    k.n0 = l * sz;
    k.m0 = k.pm0;
    k.count = min(sz, NT - k.n0);
  } else {
    k.n0 = l % NT;
    const int mb = l / NT;
    k.m0 = k.pm0 + mb * sz;
    k.count = min(sz, k.me - mb * sz);
  }
  return k;
}

// The schedule's counter pair is zero between launches: the last CTA of a launch to stop taking chunks zeroes
// both words. One thread per CTA calls this: the producer, once it takes no more chunks (off the critical
// path: the CTA's last tiles are still in flight), or thread 0 of a CTA with nothing to do.
__device__ __forceinline__ void sched_release(int* sched) {
  if (sched == nullptr) return;
  __threadfence();
  if (atomicAdd(sched + 1, 1) == (int)gridDim.x - 1) {
    atomicExch(sched, 0);
    atomicExch(sched + 1, 0);
  }
}

// Pool tile i of the static schedule (tile tau of the order) as a one-tile chunk.
__device__ __forceinline__ Chunk pool_tile(int tau, const int* poff, int E, int NT, int r128) {
  TileCursor c;
  c.seek(tau, poff, E, NT, r128);
  Chunk k;
  k.e = c.e;
  k.pm0 = c.pm0;
  k.me = c.me;
  k.n0 = c.nt;
  k.m0 = c.pm0 + c.ml;
  k.count = 1;
  k.along_n = true;
  return k;
}

// The tiles of one CTA, in order, as each role sees them: its contiguous share [tau0, tau1) of the tile
// order (static schedule), then, with a pool, the pool tiles it takes from the counter; or the chunks it
// takes from the global counter (dynamic schedule). Whatever comes from the counter, the producer takes and
// hands its id to the MMA issuer, the scale copiers and the epilogue warps through a small shared-memory
// ring; every role then walks the same tiles in the same order. n_chunks counts the chunks (dynamic) or the
// pool tiles (static), which are the last n_chunks of the r128 * NT tiles.
enum SourceRole { kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleCopier = 3 };

template <int ROLE>
struct TileSource {
  // static schedule
  TileCursor cur;
  int tau, tau1;
  // dynamic schedule
  Chunk ck;
  int ci, q;
  uint32_t qph;
  bool dyn, done;

  template <class P>
  __device__ __forceinline__ void init(const P& prm, int tau0_, int tau1_, const int* poff, int E, int NT,
                                       int r128) {
    dyn = prm.dyn != 0;
    tau = tau0_;
    tau1 = tau1_;
    if (!dyn && tau < tau1) cur.seek(tau, poff, E, NT, r128);
    ck.count = 0;
    ci = 0;
    q = 0;
    qph = 0;
    done = false;
  }

  // The next tile, or false at the end (or when a bounded wait gave up).
  template <class P>
  __device__ __forceinline__ bool next(Tile& t, const P& prm, int tau0, const int* poff, const int* cstart,
                                       int* s_sched, uint32_t bar_sfull, uint32_t bar_sempty, int n_chunks, int E,
                                       int NT, int r128) {
    if (!dyn) {
      if (tau < tau1) {
        if (tau > tau0) cur.step(poff, E, NT, r128);
        ++tau;
        t = cur.tile();
        return true;
      }
      if (n_chunks <= 0) return false;  // no pool
    }
    while (ci >= ck.count) {
      if (done) return false;
      int c;
      if constexpr (ROLE == kRoleProducer) {
        if (!mbar_wait(bar_sempty + 8 * q, qph ^ 1u, prm.err)) {  // the slot's previous id was read by all
          done = true;
          return false;
        }
        c = atomicAdd(prm.sched, 1);
        if (c >= n_chunks) c = -1;
        s_sched[q] = c;
        mbar_arrive(bar_sfull + 8 * q);
      } else if constexpr (ROLE == kRoleMma || ROLE == kRoleCopier) {
        if (!mbar_wait(bar_sfull + 8 * q, qph, prm.err)) {
          done = true;
          return false;
        }
        c = s_sched[q];
        mbar_arrive(bar_sempty + 8 * q);
      } else {
        // the whole warp takes one decision
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_sfull + 8 * q, qph, prm.err) ? 1 : 0)) {
          done = true;
          return false;
        }
        c = s_sched[q];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(bar_sempty + 8 * q);
      }
      if (++q == kSchedSlots) {
        q = 0;
        qph ^= 1u;
      }
      if (c < 0) {
        done = true;
        return false;
      }
      ck = dyn ? decode_chunk(c, cstart, poff, E, NT, r128) : pool_tile(r128 * NT - n_chunks + c, poff, E, NT, r128);
      ci = 0;
    }
    t = ck.tile(ci++);
    return true;
  }
};


// Contiguous share [tau0, tau1) of `total` tiles for CTA c of G.
__device__ __forceinline__ void cta_range(int total, int& tau0, int& tau1) {
  tau0 = (int)(((long long)total * blockIdx.x) / gridDim.x);
  tau1 = (int)(((long long)total * (blockIdx.x + 1)) / gridDim.x);
}


// The epilogue of one accumulator row: 128 columns of weight tile nt for activation row r, which holds pair
// p (p >= 0). W2: the alpha-scaled row of the pair, rounded once to bf16. W1: alpha, then the clamped SwiGLU (gate columns
// 0-63, up columns 64-127, from the W1 kernel row order) and its NVFP4 requantisation into the L2 slot
// buffers ("Bug 6", "Bug 7"). W1 amax: the same SwiGLU, reduced only. hrun keeps the NaN-propagating
// amax|h| of the thread's rows.
template <int MODE, class P>
__device__ __forceinline__ void epilogue_row(const P& prm, const float (&v)[128], int r, int p, int nt, float alpha,
                                             float& hrun) {
  if constexpr (MODE == kW2Rows) {
    uint16_t* d = prm.o_pairs + (size_t)p * prm.H + nt * 128;
    // the alpha-scaled row as bf16 pairs, 16 values (32 bytes) at a time
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = bf16x2_rn(__fmul_rn(v[16 * q + 2 * i], alpha), __fmul_rn(v[16 * q + 2 * i + 1], alpha));
      if (prm.o_pairs32) {  // whole 32-byte L2 sectors: half the write transactions of 16-byte stores
        st_global_v8(reinterpret_cast<float*>(d) + 8 * q, __uint_as_float(w[0]), __uint_as_float(w[1]),
                     __uint_as_float(w[2]), __uint_as_float(w[3]), __uint_as_float(w[4]), __uint_as_float(w[5]),
                     __uint_as_float(w[6]), __uint_as_float(w[7]));
      } else {  // a caller's buffer aligned to 16 bytes only
        uint4* d4 = reinterpret_cast<uint4*>(d) + 2 * q;
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  } else {
    // columns [0, 64): gate of features 64 nt .. 64 nt + 63; columns [64, 128): up of the same features
    const float L = prm.limit;
    if constexpr (MODE == kW1Amax) {
#pragma unroll
      for (int j = 0; j < 64; ++j)
        hrun = fmax_nan(hrun, fabsf(swiglu_clamped(__fmul_rn(v[j], alpha), __fmul_rn(v[64 + j], alpha), L)));
    } else {
      const float g2 = __ldg(prm.gs2);
      uint32_t codes[8];
      uint32_t sfw = 0;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float h[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          h[j] = swiglu_clamped(__fmul_rn(v[blk * 16 + j], alpha), __fmul_rn(v[64 + blk * 16 + j], alpha), L);
          hrun = fmax_nan(hrun, fabsf(h[j]));
        }
        const uint32_t sf = quant_block16(h, g2, codes[2 * blk], codes[2 * blk + 1]);
        sfw |= sf << (8 * blk);
      }
      uint4* dst = reinterpret_cast<uint4*>(prm.out_codes + (size_t)r * (prm.I >> 1) + nt * 32);
      dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      *reinterpret_cast<uint32_t*>(prm.out_sf + sf_offset(r, nt * 4, prm.I >> 4)) = sfw;
    }
  }
}

// One amax per warp once a CTA is done: NaN -> error bit; else the running (or calibration) maximum, and for
// the hot path the saturation test of the largest block, RN(RN(amax/6) * gs2) > 464, the quantiser's own
// arithmetic ("Bug 5", "Bug 6").
template <int MODE, class P>
__device__ __forceinline__ void epilogue_amax_flush(const P& prm, float hrun) {
  if constexpr (MODE != kW2Rows) {
    __syncwarp();
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) hrun = fmax_nan(hrun, __shfl_xor_sync(0xFFFFFFFFu, hrun, off));
    if ((threadIdx.x & 31) == 0) {
      if (hrun != hrun) {
        raise_error(prm.err, FP4MOE_ERR_NAN);
      } else if (hrun > 0.0f) {
        atomicMax(reinterpret_cast<unsigned int*>(prm.amax), __float_as_uint(hrun));
        if constexpr (MODE == kW1SwiGLU) {
          if (__fmul_rn(__fdiv_rn(hrun, 6.0f), __ldg(prm.gs2)) > kE4M3SatAbove) atomicOr(prm.status, FP4MOE_SAT_L2);
        }
      }
    }
  }
}
}  // namespace
}  // namespace fp4moe
