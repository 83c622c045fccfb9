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
// A tile is 128 tokens x 128 weight rows; its fp32 accumulator is 64 registers in each of the 256
// epilogue threads, which leaves room for two TMEM loads in flight per wait.
//   producer (warp 8)      TMA: the activation block and the weight block (128 rows x 128 bytes
//                          each, 128-byte swizzled) into a 6-stage ring.
//   MMA issuer (warp 9)    4 MMAs of K = 32 per block into one of four 128-column TMEM buffers;
//                          a fresh accumulation for every K block.
//   epilogue (warps 0-7)   warp w reads TMEM lanes 32 (w % 4) .. +31 (its token rows) and 64 of
//                          the 128 columns (half w / 4).
// W1's kernel row order interleaves gate and up per 64 features (tile j: gate features
// 64 j .. 64 j + 63, then their up rows), so the SwiGLU stays inside a tile. The 1 x 128 group of
// h spans two tiles, so W1 runs as clusters of 2 n-tiles that swap the per-row amax (or, when K
// is split, reduce both tiles together) through distributed shared memory.
//
// K split: with fewer tiles than half of the SMs (decode; the other half stays free for the routing that
// runs beside the shared expert), K is cut into S slices over the z dimension of the cluster. Each CTA leaves its fp32 partial tile in shared memory; after a cluster barrier each
// CTA sums a share of the rows over all slices, in slice order (deterministic), and runs the
// epilogue on them.
// Every wait is bounded, as in the routed GEMMs; a timeout sets FP4MOE_ERR_TIMEOUT and skips work.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {

bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows);
int sm_count();

namespace {

constexpr int SE_BM = 128;                       // token rows per tile (MMA M)
constexpr int SE_BN = 128;                       // weight rows per tile (MMA N)
constexpr int SE_BK = 128;                       // K elements (bytes) per block: one swizzle atom
constexpr int SE_A_BYTES = SE_BM * SE_BK;        // 16 KB
constexpr int SE_B_BYTES = SE_BN * SE_BK;        // 16 KB
constexpr int SE_STAGE = SE_A_BYTES + SE_B_BYTES;
constexpr int SE_STAGES = 6;
constexpr int SE_BAR_OFF = SE_STAGES * SE_STAGE;
constexpr int SE_SMEM = SE_BAR_OFF + 256 + 1024;  // barriers + 1024-byte alignment slack
constexpr int SE_THREADS = 320;                  // 8 epilogue warps, producer, MMA issuer
constexpr int SE_TBUF = 4;                       // TMEM partial buffers
constexpr uint32_t SE_TMEM_COLS = 512;           // four 128-column partial products
constexpr int SE_MAX_KB = 32;                    // K blocks of one matrix: H and Is up to 4096
constexpr int SE_MAX_CLUSTER = 8;                // portable cluster size
constexpr int SE_RED_STRIDE = SE_BN * 4 + 16;    // bytes per row of an fp32 partial tile in shared memory
static_assert(SE_STAGE % 1024 == 0 && SE_A_BYTES % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(SE_SMEM + SE_MAX_KB * SE_BM * 4 + 2 * SE_MAX_KB * 4 + 3 * SE_BM * 4 + 64 <= 232448,
              "shared memory budget (dynamic + static)");
static_assert(SE_BM * SE_RED_STRIDE <= SE_STAGES * SE_STAGE, "a partial tile fits the idle ring");
static_assert(8 * (2 * SE_STAGES + 2 * SE_TBUF + 1) <= 256, "barriers fit their area");

struct SeMaps {
  CUtensorMap a;  // activation codes [T][K] u8, box 128 rows x 128 bytes
  CUtensorMap b;  // weight codes [N][K] u8, box 128 rows x 128 bytes
};

struct SeParams {
  int T, KB, tcap;
  float limit;
  const float* a_scale;  // [KB][tcap]
  const float* w_scale;  // [N / 128][KB], logical block order (W1: gate blocks, then up blocks)
  int up_blk;            // W1: index of the first up block (Is / 128)
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
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Two E4M3 codes (RNE, satfinite) of lo / s and hi / s in the low 16 bits, lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_scaled(float lo, float hi, float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(__fdiv_rn(hi, s)), "f"(__fdiv_rn(lo, s)));
  return r;
}
// Four codes of v[0..3] / s in one word (all zero when s == 0).
__device__ __forceinline__ uint32_t e4m3x4_scaled(const float* v, float s) {
  return s == 0.0f ? 0u : (e4m3x2_scaled(v[0], v[1], s) | (e4m3x2_scaled(v[2], v[3], s) << 16));
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
  const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  const float s = __fdiv_rn(a, 448.0f);
  *reinterpret_cast<uint32_t*>(qx + off) = e4m3x4_scaled(v, s);
  if (lane == 0) sx[(size_t)g * tcap + t] = s;
}

// Grid (N / 128, ceil(T / 128), S); cluster (CX, 1, S) with CX = 2 for W1 (the two n-tiles of a
// 128-feature h group) and 1 for W2. A CTA's rank in its cluster is x % CX + CX * z.
template <int MODE>
__global__ void __launch_bounds__(SE_THREADS, 1)
    se_gemm_kernel(const __grid_constant__ SeMaps maps, const SeParams prm) {
  constexpr int CX = MODE == 0 ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ float s_sa[SE_MAX_KB][SE_BM];  // activation scales of this CTA's K blocks, per tile row
  __shared__ float s_sw[2][SE_MAX_KB];      // weight scales: W1 gate and up block, W2 the tile's block
  __shared__ float s_amax[3][SE_BM];        // W1: amax of each half of a row's 64 h features; [2]: both

  pdl_trigger();
  // The weights depend on no earlier kernel, so the producer starts streaming them before it waits
  // for the previous kernel (programmatic dependent launch); every other read of a predecessor's
  // output waits first. Every CTA runs to the end (cluster peers read its shared memory), so an
  // abort raised elsewhere only skips work.
  const int nt = blockIdx.x, mt = blockIdx.y, S = gridDim.z, z = blockIdx.z;
  const int px = nt % CX;  // position in the W1 pair
  const int KB = prm.KB, kb0 = KB * z / S, nk = KB * (z + 1) / S - kb0;
  const int rows_live = min(SE_BM, prm.T - mt * SE_BM);  // token rows of this tile, >= 1
  const int live_quads = (rows_live + 31) / 32;           // epilogue lane quadrants holding any token
  const bool go = (*(volatile uint32_t*)prm.err & kAbortMask) == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (smem - smem_u32(smem_raw));
  const uint32_t bar_full = smem + SE_BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * SE_STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * SE_STAGES;
  const uint32_t bar_tempty = bar_tfull + 8 * SE_TBUF;
  const uint32_t bar_drain = bar_tempty + 8 * SE_TBUF;

  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), SE_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int s = 0; s < SE_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);  // the MMA commit
    }
    for (int b = 0; b < SE_TBUF; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 2 * live_quads);  // one arrive per epilogue warp with tokens
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // epilogue state, used by warps 0-7 after the role split as well
  const int quad = warp & 3, hf = (warp >> 2) & 1;
  const int r = quad * 32 + lane;  // tile row
  const int row = mt * SE_BM + r;  // token
  // this thread's 64 columns: W1 gate 32 hf .. +31 and up 64 + 32 hf .. +31 (features 64 nt + 32 hf ..);
  // W2 64 hf .. +63
  const uint32_t ca = MODE == 0 ? 32u * hf : 64u * hf, cb = MODE == 0 ? 64u + 32u * hf : 64u * hf + 32u;
  float acc[64];
  bool ok = false;

  if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = policy_evict_normal();                              // read by every n-tile
    const uint64_t pol_b = gridDim.y == 1 ? policy_evict_first() : policy_evict_last();  // re-read per m-tile
    const int pre = go ? min(nk, SE_STAGES) : 0;
    for (int i = 0; i < pre; ++i) {  // fresh stages: weights first, activations once they exist
      mbar_arrive_expect_tx(bar_full + 8 * i, SE_STAGE);
      tma_load_2d(smem + i * SE_STAGE + SE_A_BYTES, &maps.b, bar_full + 8 * i, (kb0 + i) * SE_BK, nt * SE_BN, pol_b);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i)
      tma_load_2d(smem + i * SE_STAGE, &maps.a, bar_full + 8 * i, (kb0 + i) * SE_BK, mt * SE_BM, pol_a);
    int i = pre;
    for (; go && i < nk; ++i) {
      const int s = i % SE_STAGES;
      if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(i / SE_STAGES) & 1u) ^ 1u, prm.err)) break;
      const uint32_t st = smem + s * SE_STAGE;
      mbar_arrive_expect_tx(bar_full + 8 * s, SE_STAGE);  // rows past T are zero-filled and still counted
      tma_load_2d(st, &maps.a, bar_full + 8 * s, (kb0 + i) * SE_BK, mt * SE_BM, pol_a);
      tma_load_2d(st + SE_A_BYTES, &maps.b, bar_full + 8 * s, (kb0 + i) * SE_BK, nt * SE_BN, pol_b);
    }
    // on every path, let the copies already issued land before the CTA exits
    for (int j = max(0, i - SE_STAGES); j < i; ++j)
      drain_wait(bar_full + 8 * (j % SE_STAGES), (uint32_t)(j / SE_STAGES) & 1u);
  } else if (warp == 9 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_e4m3(SE_BM, SE_BN);
    for (int i = 0; go && i < nk; ++i) {
      const int s = i % SE_STAGES, b = i % SE_TBUF;
      if (!mbar_wait(bar_tempty + 8 * b, ((uint32_t)(i / SE_TBUF) & 1u) ^ 1u, prm.err)) break;
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(i / SE_STAGES) & 1u, prm.err)) break;
      tc_fence_after();
      const uint32_t st = smem + (uint32_t)s * SE_STAGE;
#pragma unroll
      for (int q = 0; q < 4; ++q)  // K = 32 E4M3 = 32 bytes per MMA
        tc_mma_f8(tmem + (uint32_t)SE_BN * b, desc_sw128(st + 32 * q), desc_sw128(st + SE_A_BYTES + 32 * q), idesc,
                  q > 0 ? 1u : 0u);
      tc_commit(bar_empty + 8 * s);
      tc_commit(bar_tfull + 8 * b);
    }
    tc_commit(bar_drain);
    drain_wait(bar_drain, 0);  // no MMA may still write TMEM when it is freed
  } else if (warp < 8) {
    // ------------------------------------------------------------ epilogue: the K loop
    pdl_wait();  // the activation scales come from the previous kernel
    for (int i = threadIdx.x; i < nk * SE_BM; i += 256) {
      const int kk = i / SE_BM, rr = i % SE_BM;
      const int srow = min(mt * SE_BM + rr, prm.tcap - 1);  // scale rows past T exist but hold no token
      s_sa[kk][rr] = __ldcg(prm.a_scale + (size_t)(kb0 + kk) * prm.tcap + srow);
    }
    // W1 tile nt holds gate and up features 64 nt .. 64 nt + 63: gate block nt / 2 and up block
    // up_blk + nt / 2. W2 tile nt is block nt.
    const int blk_a = MODE == 0 ? nt / 2 : nt, blk_b = MODE == 0 ? prm.up_blk + nt / 2 : nt;
    for (int i = threadIdx.x; i < 2 * nk; i += 256)
      s_sw[i / nk][i % nk] = __ldg(prm.w_scale + (size_t)(i < nk ? blk_a : blk_b) * KB + kb0 + i % nk);
    named_sync(2, 256);  // the eight epilogue warps
    const bool live = go && quad < live_quads;
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
    ok = live;
    for (int i = 0; live && i < nk; ++i) {
      const float sa = s_sa[i][r];
      const float fa = sa * s_sw[0][i], fb = sa * s_sw[1][i];
      const int b = i % SE_TBUF;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull + 8 * b, (uint32_t)(i / SE_TBUF) & 1u, prm.err) ? 1 : 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + (uint32_t)SE_BN * b + ((uint32_t)(quad * 32) << 16);
      float va[32], vb[32];
      tmem_ld32(tb + ca, va);
      tmem_ld32(tb + cb, vb);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);  // the buffer is in registers: the MMA may refill it
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(va[j], fa, acc[j]);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[32 + j] = fmaf(vb[j], fb, acc[32 + j]);
    }
  }
  __syncwarp();  // the producer and MMA warps reconverge: cluster barriers are warp-aligned instructions

  if (S == 1) {
    if constexpr (MODE == 0) {
      // h for features 64 nt + 32 hf .. + 31: gate in acc[0..31], up in acc[32..63]. The partner tile of
      // the cluster holds the other 64 features of the 128-feature group: swap the row amax with it.
      float amax = 0.0f;
      if (warp < 8) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = swiglu_clamped(acc[i], acc[32 + i], prm.limit);
          amax = fmaxf(amax, fabsf(acc[i]));
        }
        s_amax[hf][r] = amax;
        named_sync(1, 256);  // the eight epilogue warps
        if (hf == 0) s_amax[2][r] = fmaxf(amax, s_amax[1][r]);
      }
      cluster_sync();
      if (warp < 8) {
        amax = fmaxf(s_amax[2][r], ld_cluster_f32(map_cluster(smem_u32(&s_amax[2][r]), (uint32_t)(px ^ 1))));
        const float sc = __fdiv_rn(amax, 448.0f);
        if (ok && row < prm.T) {
          uint4* dst = reinterpret_cast<uint4*>(prm.h_codes + (size_t)row * prm.I + 64 * nt + 32 * hf);
#pragma unroll
          for (int i = 0; i < 2; ++i)
            dst[i] = make_uint4(e4m3x4_scaled(acc + 16 * i, sc), e4m3x4_scaled(acc + 16 * i + 4, sc),
                                e4m3x4_scaled(acc + 16 * i + 8, sc), e4m3x4_scaled(acc + 16 * i + 12, sc));
          if (px == 0 && hf == 0) prm.h_scale[(size_t)(nt / 2) * prm.tcap + row] = sc;
        }
      }
      cluster_sync();  // the partner has read this CTA's amax
    } else {
      if (warp < 8 && ok && row < prm.T) {
        float4* dst = reinterpret_cast<float4*>(prm.out + (size_t)row * prm.H + SE_BN * nt + 64 * hf);
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
    }
  } else {
    // this CTA's fp32 partial tile into the idle ring: row r at r * SE_RED_STRIDE (padded rows keep the
    // float4 stores of consecutive rows on distinct banks)
    if (warp < 8 && ok) {
      float* rowp = reinterpret_cast<float*>(smem_gen + (size_t)r * SE_RED_STRIDE);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        *reinterpret_cast<float4*>(rowp + ca + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        *reinterpret_cast<float4*>(rowp + cb + j) =
            make_float4(acc[32 + j], acc[32 + j + 1], acc[32 + j + 2], acc[32 + j + 3]);
      }
    }
    // every partial tile of the cluster is written; CTA rank c sums rows [r0, r1) of the tile over the S
    // slices in slice order (deterministic), then runs the epilogue on them
    cluster_sync();
    if (warp < 8 && go) {
      const int c = px + CX * z, nc = CX * S;
      const int r0 = rows_live * c / nc, r1 = rows_live * (c + 1) / nc;
      const int rr = threadIdx.x >> 4, part = threadIdx.x & 15;
      // W1: features 8 part .. +7 of the pair's 128 come from pair tile part / 8 (gate columns
      // 8 (part % 8) .., up columns 64 + 8 (part % 8) ..); W2: columns 8 part .. + 7
      const int src_x = MODE == 0 ? part / 8 : 0;
      const uint32_t ra = MODE == 0 ? 8u * (part % 8) : 8u * part, rb = MODE == 0 ? 64u + ra : ra + 4u;
      for (int base = r0; base < r1; base += 16) {  // uniform bounds: every lane takes part in the shuffles
        const int rt = base + rr;
        const bool have = rt < r1;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        if (have) {
          const uint32_t la = smem + (uint32_t)rt * SE_RED_STRIDE + 4u * ra;
          const uint32_t lb = smem + (uint32_t)rt * SE_RED_STRIDE + 4u * rb;
          // four slices' loads in flight at a time; the sums still run in slice order
          for (int z0 = 0; z0 < S; z0 += 4) {
            float4 q[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (z0 + j < S) {
                const uint32_t peer = (uint32_t)(src_x + CX * (z0 + j));
                const uint32_t pa = map_cluster(la, peer), pb = map_cluster(lb, peer);
                q[j][0] = ld_cluster_f4(pa);
                q[j][2] = ld_cluster_f4(pb);
                if (MODE == 0) {
                  q[j][1] = ld_cluster_f4(pa + 16);
                  q[j][3] = ld_cluster_f4(pb + 16);
                } else {
                  q[j][1] = q[j][3] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (z0 + j < S) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  v[4 * u] += q[j][u].x;
                  v[4 * u + 1] += q[j][u].y;
                  v[4 * u + 2] += q[j][u].z;
                  v[4 * u + 3] += q[j][u].w;
                }
              }
            }
          }
        }
        const int orow = mt * SE_BM + rt;
        if constexpr (MODE == 0) {
          // v[0..7] gate, v[8..15] up of features 128 (nt / 2) + 8 part ..
          float h[8], amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            h[i] = swiglu_clamped(v[i], v[8 + i], prm.limit);
            amax = fmaxf(amax, fabsf(h[i]));
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));  // 16 lanes
          const float sc = __fdiv_rn(amax, 448.0f);
          if (have && orow < prm.T) {
            *reinterpret_cast<uint2*>(prm.h_codes + (size_t)orow * prm.I + 128 * (nt / 2) + 8 * part) =
                make_uint2(e4m3x4_scaled(h, sc), e4m3x4_scaled(h + 4, sc));
            if (part == 0) prm.h_scale[(size_t)(nt / 2) * prm.tcap + orow] = sc;
          }
        } else {
          // v[0..3]: columns 8 part .. +3; v[8..11]: columns 8 part + 4 .. +7
          if (have && orow < prm.T) {
            float4* dst = reinterpret_cast<float4*>(prm.out + (size_t)orow * prm.H + SE_BN * nt + 8 * part);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[8], v[9], v[10], v[11]);
          }
        }
      }
    }
    cluster_sync();  // no CTA leaves while a peer still reads its partial tile
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, SE_TMEM_COLS);
  }
}

// One CTA per 128 x 128 weight block: s = RN(amax / 448), codes E4M3(RN(w / s)), 0 where s == 0.
// Scales stay in logical block order. W1 (inter > 0): the codes of gate row f go to kernel row
// 128 (f / 64) + f % 64 and those of up row f to 128 (f / 64) + 64 + f % 64.
__global__ void __launch_bounds__(256) se_quant_weights_kernel(int K, int inter, const float* __restrict__ w,
                                                               uint8_t* __restrict__ codes, float* __restrict__ scales) {
  __shared__ float s_red[8];
  const int KB = K / 128;
  const int bi = blockIdx.y, bk = blockIdx.x;  // logical row block, K block
  // thread: row 128 bi + threadIdx.x / 2, 64 elements from column 128 bk + 64 (threadIdx.x & 1)
  const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
  const int lr = bi * 128 + r;  // logical row
  int kr = lr;                  // kernel row
  if (inter > 0) {
    const bool up = lr >= inter;
    const int f = up ? lr - inter : lr;
    kr = 128 * (f / 64) + (up ? 64 : 0) + f % 64;
  }
  const float* src = w + (size_t)lr * K + (size_t)bk * 128 + 64 * h;
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
  uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)kr * K + (size_t)bk * 128 + 64 * h);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[i] = make_uint4(e4m3x4_scaled(v + 16 * i, s), e4m3x4_scaled(v + 16 * i + 4, s),
                        e4m3x4_scaled(v + 16 * i + 8, s), e4m3x4_scaled(v + 16 * i + 12, s));
  if (threadIdx.x == 0) scales[(size_t)bi * KB + bk] = s;
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

template <int MODE>
cudaLaunchConfig_t se_launch_config(dim3 grid, int S, cudaStream_t st, cudaLaunchAttribute (&attr)[2]) {
  constexpr int CX = MODE == 0 ? 2 : 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid.x, grid.y, S);
  lc.blockDim = dim3(SE_THREADS);
  lc.dynamicSmemBytes = SE_SMEM;
  lc.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CX;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = S;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return lc;
}

// Clusters of (CX, 1, S) CTAs (one per SM) that the device holds at once, per GEMM mode; cached per device.
template <int MODE>
int max_active_clusters(int S) {
  static int cache[64][SE_MAX_CLUSTER + 1];
  static bool init[64][SE_MAX_CLUSTER + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || S < 1 || S > SE_MAX_CLUSTER) return 0;
  if (!init[dev][S]) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t lc = se_launch_config<MODE>(dim3(MODE == 0 ? 2 : 1, 1), S, nullptr, attr);
    lc.numAttrs = 1;  // the cluster shape alone
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, se_gemm_kernel<MODE>, &lc) != cudaSuccess) n = 0;
    cache[dev][S] = n;
    init[dev][S] = true;
  }
  return cache[dev][S];
}

// K slices: with fewer tiles than SMs, split K over the cluster's z dimension (each CTA keeps >= 1 K block)
// so that the weights stream through more SMs, as long as every cluster of the grid is resident at once (a
// second wave would double the time).
template <int MODE>
int k_slices(int nx, int ny, int KB, int nsm) {
  constexpr int CX = MODE == 0 ? 2 : 1;
  for (int S = SE_MAX_CLUSTER / CX; S > 1; --S)
    if (nx * ny * S <= nsm && KB >= S && max_active_clusters<MODE>(S) >= nx / CX * ny) return S;
  return 1;
}

template <int MODE>
cudaError_t launch_se_gemm(dim3 grid, int S, cudaStream_t st, const SeMaps& maps, const SeParams& prm) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t lc = se_launch_config<MODE>(grid, S, st, attr);
  return cudaLaunchKernelEx(&lc, se_gemm_kernel<MODE>, maps, prm);
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
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  // The shared expert runs beside the routing on a side stream. Its K slices are capped at half of the SMs,
  // so the routing kernels and the routed W1 find free SMs while it runs. Uncapped (96 and 128 CTAs), it held
  // the routed chain back by about 15 us. Capped, the DSV4 decode layer took 460.8 us with it against 468.0
  // (453.7 us without the shared expert).
  const int se_sms = nsm / 2;
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
  p.up_blk = Is / 128;
  p.h_codes = qh;
  p.h_scale = sh;
  const dim3 g1((unsigned)(2 * Is / SE_BN), mt);
  if (launch_se_gemm<0>(g1, k_slices<0>((int)g1.x, (int)mt, p.KB, se_sms), st, m1, p) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  p.KB = Is / 128;
  p.a_scale = sh;
  p.w_scale = s2;
  p.out = out;
  const dim3 g2((unsigned)(H / SE_BN), mt);
  return launch_se_gemm<1>(g2, k_slices<1>((int)g2.x, (int)mt, p.KB, se_sms), st, m2, p) == cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
