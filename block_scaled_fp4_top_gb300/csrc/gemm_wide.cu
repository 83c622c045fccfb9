// Block-scaled NVFP4 grouped GEMMs with 128 x 256 output tiles: every W1, and every W2 whose K is a multiple
// of 256, under both tile schedules (static with its tail pool at decode sizes, dynamic chunks at prefill
// sizes; gemm_sched.cuh).
//
// The same GEMMs as gemm.cu ("Current Bug: CuTeDSLMoERunner", "Data Flow": run_nvfp4_grouped_gemm for L1
// and L2; searchsorted(right=True) tile ownership on offsets without a leading 0, "Bug 2" and "Bug 4"; per
// expert 128-row swizzled scales, "Bug 1" and "Bug 14"), with one difference: a tile covers 256 weight
// rows (two 128-row weight tiles) instead of 128. Every activation tile that reaches shared memory then
// feeds twice the MACs, and each tcgen05.mma (M = 128, N = 256, K = 64) does twice the work of the
// 128 x 128 one, so both the ring's bytes and the MMA instructions per MAC fall. At prefill sizes the
// 128 x 128 kernel is bound by neither alone but by the per-stage ring latency, the MMA issue and a
// four-warp epilogue together; this kernel attacks all three. At decode sizes, where both stream weights at
// the HBM rate, its half as many tiles start, hand over and finish with less idle time between kernels.
//
// The accumulator takes 256 of TMEM's 512 columns, so there is one of it, not two. The epilogue has eight
// warps (two per TMEM lane quarter, one per 128-column half) that move the whole accumulator to registers,
// free it, and only then compute, so the next tile's MMAs wait only for that move. Block scales stream
// through TMEM slots, one per ring stage (A: 4 columns per 64-element K atom; B: 8, the two 128-row halves
// side by side); no operand keeps its scales resident.
//   warps 0-7   epilogue (warp w: lanes 32 (w % 4) .., columns 128 (w / 4) ..).
//   warp 8      producer: a ring stage is one 256-element K atom: the activation block by
//               cp.async.bulk.tensor (128-byte swizzle, only the leading 16/32/64/128 rows that cover
//               the tile's real rows), the two pre-tiled 16 KB weight blocks and the three 2 KB scale
//               groups by cp.async.bulk.
//   warp 9      MMA issuer: tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X.
//   warps 10-11 scale copiers: tcgen05.cp of the stage's 12 scale tiles into its TMEM slot.
// Every spin-wait is bounded (mbar_wait); a timeout sets FP4MOE_ERR_TIMEOUT, each role stops, in-flight
// copies and MMAs are drained, and the CTA frees its TMEM and returns.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "gemm_sched.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace fp4moe {
namespace {

constexpr int WBM = 128;                   // activation rows per tile (MMA M)
constexpr int WBN = 256;                   // weight rows per tile (MMA N)
constexpr int WKBYTES = 128;               // bytes of K per stage: 256 FP4, 4 MMAs of K = 64
constexpr int WATOMS = 4;                  // 64-element scale atoms per stage
constexpr int WSTAGES = 4;
constexpr int WA_BYTES = WBM * WKBYTES;    // 16 KB
constexpr int WHALF_BYTES = 128 * WKBYTES; // one 128-row pre-tiled weight block: 16 KB
constexpr int WB_BYTES = 2 * WHALF_BYTES;  // 32 KB
constexpr int WSF_TILE = 512;              // one 128 x 4 scale tile
constexpr int WSFA_OFF = WA_BYTES + WB_BYTES;
constexpr int WSFB_OFF = WSFA_OFF + WATOMS * WSF_TILE;
constexpr int WSTAGE_BYTES = WSFB_OFF + 2 * WATOMS * WSF_TILE;  // 55296, a multiple of 1024
constexpr int WBAR_OFF = WSTAGES * WSTAGE_BYTES;
constexpr int WSMEM_BYTES = WBAR_OFF + 256 + 1024;  // barriers + 1024-byte alignment slack
constexpr int WNCOPY = 2;
constexpr int WEPI = 8;
constexpr int WTHREADS = 32 * (WEPI + 2 + WNCOPY);
constexpr int WPRODUCER = WEPI, WMMA = WEPI + 1, WCOPY0 = WEPI + 2;
constexpr uint32_t WTMEM_COLS = 512;
constexpr uint32_t WACC_COLS = 256;
constexpr uint32_t WSLOT_COLS = 4 * WATOMS + 8 * WATOMS;  // A 16, B 32 columns per ring stage
constexpr int WCOPIES = WATOMS * 3;                       // scale tiles per stage: 4 of A, 8 of B
static_assert(WSTAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(WSMEM_BYTES + 8 * kMaxExperts + 128 <= 232448, "shared memory budget (dynamic + static)");
static_assert(WACC_COLS + WSLOT_COLS * WSTAGES <= WTMEM_COLS, "accumulator and scale slots fit TMEM");
// full, empty, sready (STAGES each), tfull, tempty, drain, cdrain, sfull, sempty (kSchedSlots each)
static_assert(8 * (3 * WSTAGES + 4 + 2 * kSchedSlots) <= 256, "barriers fit their area");

// One tcgen05.mma of N = 256 reads the B scales of rows 0-127 from its sfb column and those of rows 128-255
// from the four columns after them.
constexpr bool kOneMmaN256 = true;

template <int MODE>
__global__ void __launch_bounds__(WTHREADS, 1)
    grouped_gemm_wide_kernel(const __grid_constant__ AMaps tmA, const GemmParams prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_poff[kMaxExperts];
  __shared__ int s_cstart[kMaxExperts + 2];  // dynamic schedule: the chunk table (build_chunk_table)
  __shared__ int s_sched[kSchedSlots];

  __shared__ int s_abort;

  // As in the 128 x 128 kernel: the set-up overlaps the previous kernel, and the schedule counter is zero at
  // launch and zeroed again by the last CTA to finish.
  const int E = prm.E, NT = prm.NT;  // NT: 256-row weight tiles
  const int R = min(__ldcg(prm.poff + E - 1), prm.cap);
  const int r128 = R / WBM;
  const int pool = (!prm.dyn && prm.steal) ? tail_pool(r128 * NT, (int)gridDim.x) : 0;
  int tau0, tau1;
  cta_range(r128 * NT - pool, tau0, tau1);
  if (tau0 >= tau1 && pool == 0 && !prm.dyn) {  // (with a pool every CTA has at least three tiles of its own)
    if (threadIdx.x == 0) sched_release(prm.sched);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem + WBAR_OFF;            // WSTAGES x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * WSTAGES;    // WSTAGES x 8 bytes
  const uint32_t bar_sready = bar_empty + 8 * WSTAGES;  // WSTAGES x 8: the stage's scales are in TMEM
  const uint32_t bar_tfull = bar_sready + 8 * WSTAGES;
  const uint32_t bar_tempty = bar_tfull + 8;
  const uint32_t bar_drain = bar_tempty + 8;
  const uint32_t bar_cdrain = bar_drain + 8;
  const uint32_t bar_sfull = bar_cdrain + 8;                 // kSchedSlots x 8: a chunk id was written
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedSlots;  // kSchedSlots x 8: it was read

  for (int e = threadIdx.x; e < E; e += WTHREADS) s_poff[e] = __ldcg(prm.poff + e);
  if (prm.dyn) {
    __syncthreads();
    if (warp == 0) build_chunk_table(s_poff, s_cstart, E, NT, r128, (int)gridDim.x, lane);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), WTMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32 * WPRODUCER) {
    for (int s = 0; s < WSTAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sready + 8 * s, WNCOPY);  // one commit per copier
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, WEPI);  // one arrive per epilogue warp
    mbar_init(bar_drain, 1);
    mbar_init(bar_cdrain, WNCOPY);
    for (int q = 0; q < kSchedSlots; ++q) {
      mbar_init(bar_sfull + 8 * q, 1);
      mbar_init(bar_sempty + 8 * q, 1 + WNCOPY + WEPI);  // the MMA issuer, the copiers and the epilogue warps
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  int n_chunks = prm.dyn ? s_cstart[E] : pool;
  const int KB = prm.KB;  // ring stages per tile: K / 256
  const int katoms_total = prm.K / 64;
  const int NT128 = 2 * NT;  // 128-row weight tiles of one expert
  pdl_wait();  // the activations and every other result of the previous launch are needed from here on
  pdl_trigger();
  if (threadIdx.x == 0) s_abort = (*(volatile uint32_t*)prm.err & kAbortMask) != 0;
  __syncthreads();
  if (s_abort) {  // an earlier timeout poisons the call: no role takes a tile
    tau1 = tau0;
    n_chunks = 0;
  }

  if (warp == WPRODUCER && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_once = policy_evict_first();  // weights of a one-m-tile expert are read once
    const uint64_t pol_keep = policy_evict_last();   // activations are re-read by every n-tile
    const uint64_t pol_reuse = policy_evict_normal();  // weights re-read by the next m-tiles of the expert
    const int wblocks = prm.K / 256;                  // 16 KB weight blocks per 128-row weight tile
    int it = 0, prev_mt = -1, a_box = 3;
    bool ok = true;
    TileSource<kRoleProducer> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    while (ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128)) {
      const bool res_a = (t.me == 1);  // one m-tile: the activation tile is the one re-read (along n)
      const int a_row = t.mt * WBM;
      if (t.mt != prev_mt) {
        prev_mt = t.mt;
        a_box = 3;
        if (t.last) {
          // the first padding row of the block bounds the rows this m-tile needs (rows < R are all written)
          const int32_t* por = prm.pair_of_row + a_row;
          const int p16 = __ldcg(por + 16), p32 = __ldcg(por + 32), p64 = __ldcg(por + 64);
          a_box = p16 < 0 ? 0 : (p32 < 0 ? 1 : (p64 < 0 ? 2 : 3));
        }
      }
      const uint32_t a_bytes = (uint32_t)(16 << a_box) * WKBYTES;
      const uint64_t pol_w = res_a ? pol_once : pol_reuse;
      const uint64_t pol_a = res_a ? pol_keep : pol_reuse;
      const size_t wt0 = (size_t)t.e * NT128 + 2 * t.nt;  // the tile's first 128-row weight tile
      const uint8_t* b0 = prm.b_codes + wt0 * wblocks * WHALF_BYTES;
      const uint8_t* b1 = b0 + (size_t)wblocks * WHALF_BYTES;
      const uint8_t* sfa = prm.a_sf + (size_t)t.mt * katoms_total * WSF_TILE;
      const uint8_t* sfb0 = prm.b_sf + wt0 * katoms_total * WSF_TILE;
      const uint8_t* sfb1 = sfb0 + (size_t)katoms_total * WSF_TILE;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % WSTAGES;
        const uint32_t ph = (uint32_t)(it / WSTAGES) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, prm.err)) {
          ok = false;
          break;
        }
        const uint32_t st = smem + s * WSTAGE_BYTES;
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, a_bytes + WB_BYTES + 3 * WATOMS * WSF_TILE);
        bulk_load(st + WA_BYTES, b0 + (size_t)kb * WHALF_BYTES, WHALF_BYTES, full, pol_w);
        bulk_load(st + WA_BYTES + WHALF_BYTES, b1 + (size_t)kb * WHALF_BYTES, WHALF_BYTES, full, pol_w);
        tma_load_2d(st, &tmA.box[a_box], full, kb * WKBYTES, a_row, pol_a);
        bulk_load(st + WSFA_OFF, sfa + (size_t)kb * WATOMS * WSF_TILE, WATOMS * WSF_TILE, full, pol_a);
        bulk_load(st + WSFB_OFF, sfb0 + (size_t)kb * WATOMS * WSF_TILE, WATOMS * WSF_TILE, full, pol_w);
        bulk_load(st + WSFB_OFF + WATOMS * WSF_TILE, sfb1 + (size_t)kb * WATOMS * WSF_TILE, WATOMS * WSF_TILE, full,
                  pol_w);
      }
    }
    sched_release(prm.sched);  // this CTA takes no more chunks
    // on every path, let the copies already issued land before the CTA exits
    for (int j = max(0, it - WSTAGES); j < it; ++j)
      drain_wait(bar_full + 8 * (j % WSTAGES), (uint32_t)(j / WSTAGES) & 1u);
  } else if (warp == WMMA && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // Shared-memory descriptors are built from full byte addresses (the 14-bit field wraps with the window).
    constexpr uint32_t idesc = kOneMmaN256 ? idesc_nvf4(WBM, WBN) : idesc_nvf4(WBM, 128);
    int tl = 0, s = 0;
    uint32_t ph = 0;
    bool ok = true;
    TileSource<kRoleMma> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    for (; ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128);
         ++tl) {
      // the epilogue has moved the previous tile's accumulator out of TMEM
      if (!mbar_wait(bar_tempty, ((uint32_t)tl & 1u) ^ 1u, prm.err)) {
        ok = false;
        break;
      }
      for (int kb = 0; kb < KB; ++kb) {
        // the operands are in shared memory and the copiers' scale copies for this stage have completed
        if (!mbar_wait(bar_full + 8 * s, ph, prm.err) || !mbar_wait(bar_sready + 8 * s, ph, prm.err)) {
          ok = false;
          break;
        }
        tc_fence_after();  // order the tensor-core reads after the waits that made the stage visible
        const uint32_t st = smem + (uint32_t)s * WSTAGE_BYTES;
        const uint32_t slot = tmem + WACC_COLS + WSLOT_COLS * s;
#pragma unroll
        for (int a = 0; a < WATOMS; ++a) {
          const uint32_t acc_flag = (kb > 0 || a > 0) ? 1u : 0u;
          if constexpr (kOneMmaN256) {
            tc_mma_nvf4(tmem, desc_sw128(st + 32 * a), desc_sw128(st + WA_BYTES + 32 * a), idesc, slot + 4 * a,
                        slot + 4 * WATOMS + 8 * a, acc_flag);
          } else {  // two N = 128 MMAs, one per 128-row half of the weight tile
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tc_mma_nvf4(tmem + 128 * h, desc_sw128(st + 32 * a), desc_sw128(st + WA_BYTES + WHALF_BYTES * h + 32 * a),
                          idesc, slot + 4 * a, slot + 4 * WATOMS + 8 * a + 4 * h, acc_flag);
          }
        }
        tc_commit(bar_empty + 8 * s);
        if (++s == WSTAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) tc_commit(bar_tfull);
    }
    // no MMA may still write TMEM when it is freed
    tc_commit(bar_drain);
    drain_wait(bar_drain, 0);
  } else if (warp >= WCOPY0 && warp < WCOPY0 + WNCOPY && lane == 0) {
    // ------------------------------------------------------------ scale copiers
    // Copier c takes copies i with i % WNCOPY == c of the stage's 12: A atoms 0-3, then B atom a, half h.
    // TMEM slot s is free again once stage s is full: the producer refilled the stage only after the MMAs
    // of the slot's previous use committed bar_empty.
    const int cpy = warp - WCOPY0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    TileSource<kRoleCopier> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    while (ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128)) {
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(bar_full + 8 * s, ph, prm.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem + (uint32_t)s * WSTAGE_BYTES;
        const uint32_t slot = tmem + WACC_COLS + WSLOT_COLS * s;
#pragma unroll
        for (int i = cpy; i < WCOPIES; i += WNCOPY) {
          if (i < WATOMS) {
            tc_cp_scales(slot + 4 * i, desc_scales(st + WSFA_OFF + i * WSF_TILE));
          } else {
            const int a = (i - WATOMS) >> 1, h = (i - WATOMS) & 1;
            tc_cp_scales(slot + 4 * WATOMS + 8 * a + 4 * h, desc_scales(st + WSFB_OFF + (h * WATOMS + a) * WSF_TILE));
          }
        }
        tc_commit(bar_sready + 8 * s);
        if (++s == WSTAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // no copy may still write TMEM when it is freed
    tc_commit(bar_cdrain);
    drain_wait(bar_cdrain, 0);
  } else if (warp < WEPI) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, half = warp >> 2;
    int tl = 0;
    float hrun = 0.0f;  // W1 modes: amax|h| of this thread's rows, NaN if any h was NaN
    TileSource<kRoleEpilogue> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    for (; src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128); ++tl) {
      const int r = t.mt * WBM + quarter * 32 + lane;
      // the row's pair and the expert's alpha are loaded before the accumulator wait, which hides them
      const int p = __ldcg(prm.pair_of_row + r);
      const float alpha = __ldg(prm.alpha + t.e);
      // the whole warp takes one decision: tcgen05.ld is warp-collective
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull, (uint32_t)tl & 1u, prm.err) ? 1 : 0)) break;
      tc_fence_after();
      const bool any_real = __any_sync(0xFFFFFFFFu, p >= 0);
      const uint32_t tacc = tmem + 128u * half + ((uint32_t)(quarter * 32) << 16);
      float v[128];
      if (any_real) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float q[32];
          tmem_ld32(tacc + c * 32, q);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[c * 32 + j] = q[j];
        }
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty);  // this warp's share of the accumulator is out of TMEM
      if (p < 0) continue;                      // padding rows carry nothing ("Bug 14")
      epilogue_row<MODE>(prm, v, r, p, 2 * t.nt + half, alpha, hrun);
    }
    epilogue_amax_flush<MODE>(prm, hrun);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, WTMEM_COLS);
  }
}

template <int MODE>
bool wide_configure_once() {
  static int ok = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(grouped_gemm_wide_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              WSMEM_BYTES) == cudaSuccess
             ? 1
             : 0;
  });
  return ok == 1;
}

}  // namespace

bool gemm_wide_fits(int K, int b_rows) { return K % 256 == 0 && b_rows % WBN == 0; }

fp4moe_status gemm_wide_launch(GemmMode mode, const GemmParams& prm128, const AMaps& tmA, cudaStream_t st) {
  if (!gemm_wide_fits(prm128.K, prm128.b_rows)) return FP4MOE_UNSUPPORTED;
  GemmParams prm = prm128;
  prm.NT = prm128.b_rows / WBN;
  prm.KB = prm128.K / 256;
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  const int max_tiles = (prm.cap / WBM) * prm.NT;
  const unsigned grid = (unsigned)(max_tiles < nsm ? max_tiles : nsm);
  cudaError_t r = cudaErrorInvalidValue;
  switch (mode) {
    case kW1SwiGLU:
      if (!wide_configure_once<kW1SwiGLU>()) return FP4MOE_CUDA_ERROR;
      r = launch_pdl(grouped_gemm_wide_kernel<kW1SwiGLU>, dim3(grid), dim3(WTHREADS), WSMEM_BYTES, st, tmA, prm);
      break;
    case kW1Amax:
      if (!wide_configure_once<kW1Amax>()) return FP4MOE_CUDA_ERROR;
      r = launch_pdl(grouped_gemm_wide_kernel<kW1Amax>, dim3(grid), dim3(WTHREADS), WSMEM_BYTES, st, tmA, prm);
      break;
    case kW2Rows:
      if (!wide_configure_once<kW2Rows>()) return FP4MOE_CUDA_ERROR;
      r = launch_pdl(grouped_gemm_wide_kernel<kW2Rows>, dim3(grid), dim3(WTHREADS), WSMEM_BYTES, st, tmA, prm);
      break;
  }
  return r == cudaSuccess ? FP4MOE_OK : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
