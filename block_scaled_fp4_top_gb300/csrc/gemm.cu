// Block-scaled NVFP4 grouped GEMMs on the 5th-generation tensor cores (tcgen05).
//
// This is the grouped GEMM of "Current Bug: CuTeDSLMoERunner" ("Data Flow":
// run_nvfp4_grouped_gemm for L1 and L2). The A operand is slot-ordered
// activations: each expert's rows start on a 128-row boundary, and the
// scales are swizzled per 128-row block ("Bug 1", "Bug 14"). The B operand is
// each expert's K-major weights. Tile -> expert uses
// searchsorted(padded_offsets, row, right=True) on offsets with no leading 0
// ("Bug 2", "Bug 4").
//
// This 128 x 128 kernel now serves only the W2 GEMM whose K (the intermediate
// width) is an odd multiple of 128. Every other grouped GEMM runs on the
// 128 x 256 kernel of gemm_wide.cu, which shares the tile schedules and the
// row epilogues (gemm_sched.cuh); this one still carries the W1 modes.
//
// Persistent kernel, one CTA per SM. Output tiles are 128 activation rows x
// 128 weight rows. They are numbered expert by expert; inside expert e, with
// M_e m-tiles, the n-tiles run slowest and the m-tiles fastest. CTA c takes
// the contiguous share [c*T/G, (c+1)*T/G) of the T tiles. So an expert with
// one m-tile (every expert at decode sizes) is walked across its n-tiles
// with the activation tile fixed, and a weight tile of a larger expert is
// used for all of the expert's m-tiles in a row, while it is still in L2.
// The fixed operand keeps its block scales resident in TMEM ("resident"),
// the other one streams them with every stage ("streamed"):
//   warp 4      producer. A ring stage covers 512 elements of K. Its two
//               consecutive 16 KB weight blocks arrive with one contiguous
//               cp.async.bulk: the weights are stored pre-tiled and
//               pre-swizzled (see fp4moe.h). The two activation blocks
//               arrive by cp.async.bulk.tensor with the 128-byte swizzle,
//               and the scale tiles by cp.async.bulk. Real rows lead every
//               expert block, so an m-tile loads only its first 16, 32, 64
//               or 128 rows: enough to cover the real ones. The rest of the
//               128-row shared tile keeps stale bytes; MMA rows are
//               independent and the epilogue drops those rows. At decode
//               sizes (a few tokens per expert) this cuts the activation
//               bytes re-read for every n-tile eightfold. Weight stages
//               are also pulled into L2 a few stages ahead
//               (cp.async.bulk.prefetch.L2). The shared-memory ring runs on
//               across tile boundaries, so the weight stream never stops.
//   warps 6-7   scale copiers. tcgen05.cp costs about the same per instruction
//               whatever its size, and holds its issuing thread (about 190
//               cycles), so two threads share each stage's copies. The
//               resident scales are copied into TMEM only once, for the whole
//               of K, and stay there while the operand is fixed. Each stage
//               then copies only its 8 streamed scale tiles, and each copier
//               commits its share to a per-stage barrier.
//   warp 5      MMA issuer. Once a stage's operands and scales are in place,
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64
//               each) accumulates in fp32 in TMEM, and tcgen05.commit frees the
//               ring slot and then hands the accumulator to the epilogue. The
//               copier works on the next stage meanwhile.
//   warps 0-3   epilogue. tcgen05.ld gives one accumulator row per thread. It
//               moves all 128 columns to registers, frees the accumulator for
//               the next tile's MMAs, then computes. Padding rows are skipped
//               ("Bug 14"), and warps whose 32 rows are all padding do not read
//               TMEM at all.
//     W1: alpha, then the clamped SwiGLU (gate columns 0-63, up columns
//         64-127, from the W1 kernel row order), then NVFP4 requantisation
//         into the L2 slot buffers ("Bug 6", "Bug 7"). Each thread also keeps
//         the amax of its h (NaN-propagating). When the CTA is done, each warp
//         folds it into the running amax|h| of the workspace, sets
//         FP4MOE_SAT_L2 if that amax made an E4M3 block scale saturate
//         under gs2 (a stale L2 scale, "Bug 5" and "Bug 6"), or
//         FP4MOE_ERR_NAN if an h was NaN.
//     W1 amax: the same SwiGLU, reduced to amax|h| for calibration.
//     W2: alpha, then fp32 rows stored per (token, k) pair.
// Every spin-wait is bounded (mbar_wait). A timeout sets FP4MOE_ERR_TIMEOUT
// in the error word. Each role then stops, waits for its in-flight copies and
// MMAs, and the CTA frees its TMEM and returns.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"
#include "gemm_sched.cuh"

namespace fp4moe {
namespace {

constexpr int BM = 128;            // activation rows per tile (MMA M)
constexpr int BN = 128;            // weight rows per tile (MMA N)
constexpr int KBYTES = 128;        // bytes of K in one 128-byte swizzle atom: 256 FP4 = 4 MMAs of K = 64
constexpr int HALVES = 2;          // K atoms per ring stage: 512 FP4 = 8 MMAs per stage
constexpr int ATOMS = 4 * HALVES;  // 64-element scale atoms per stage
constexpr int STAGES = 3;  // six half-size stages were slower: per-stage overhead outweighs the extra slack
constexpr int HALF_BYTES = BM * KBYTES;        // one 128-row x 128-byte swizzled block (16 KB)
constexpr int A_BYTES = HALVES * HALF_BYTES;
constexpr int B_BYTES = HALVES * HALF_BYTES;   // pre-tiled weight blocks of consecutive k-stages
constexpr int SF_TILE = 512;                   // one 128x4 scale tile
constexpr int RES_OFF = A_BYTES + B_BYTES;            // scale tiles of the resident operand (new operand only)
constexpr int STR_OFF = RES_OFF + ATOMS * SF_TILE;      // scale tiles of the streamed operand
constexpr int STAGE_BYTES = STR_OFF + ATOMS * SF_TILE;  // 73728, a multiple of 1024
constexpr int BAR_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;    // barriers + 1024-byte alignment slack
constexpr int NCOPY = 2;       // scale-copier warps: each tcgen05.cp holds its issuing thread, so they share a stage
constexpr int THREADS = 192 + 32 * NCOPY;  // 4 epilogue warps, producer, MMA issuer, scale copiers
constexpr int PREFETCH = 2;         // ring stages pulled into L2 ahead of the ring (measured: 1-2 best, 6 costs 4 %)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 128;  // one accumulator: 128 fp32 columns
constexpr uint32_t SFB_STAGE_COLS = 4 * ATOMS;  // B scales of one ring stage
// TMEM columns: nacc accumulators at [0, 128 nacc); resident scales (4 columns
// per 64-element K atom, all of K) at RES_COL = 128 nacc; streamed scales of
// ring stage s: 32 columns at RES_COL + K/16 + 32 s. nacc is 2 when that fits,
// else 1.
static_assert(STAGE_BYTES % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(SMEM_BYTES + 8 * kMaxExperts + 128 <= 232448, "shared memory budget (dynamic + static)");
constexpr int kMaxResidentK = (TMEM_COLS - ACC_COLS - SFB_STAGE_COLS * STAGES) * 16;  // 4608 with one accumulator

using Params = GemmParams;

// full, empty, tfull (2), tempty (2), drain, sfull, sempty, sready, cdrain, resfree: all in the 256 bytes at
// BAR_OFF
static_assert(8 * (2 * STAGES + 2 + 2 + 1 + 2 * kSchedSlots + STAGES + 1 + 1) <= 256, "barriers fit their area");

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ AMaps tmA, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_poff[kMaxExperts];
  __shared__ int s_cstart[kMaxExperts + 2];  // dynamic schedule: the chunk table (build_chunk_table)
  __shared__ int s_sched[kSchedSlots];

  __shared__ int s_abort;

  // The routing layout is final before this grid starts (each kernel of the chain waits on its predecessor
  // before it lets its successor start), so the set-up below (tile ranges, TMEM, barriers, the chunk table)
  // overlaps the previous kernel, and the wait for it comes after. The schedule counter (dynamic chunks, or
  // the static schedule's pool) is zero at launch; the last CTA to finish zeroes it again.
  const int E = prm.E, NT = prm.NT;
  const int R = min(__ldcg(prm.poff + E - 1), prm.cap);
  const int r128 = R / BM;
  const int pool = (!prm.dyn && prm.steal) ? tail_pool(r128 * NT, (int)gridDim.x) : 0;
  int tau0, tau1;
  cta_range(r128 * NT - pool, tau0, tau1);
  if (tau0 >= tau1 && pool == 0 && !prm.dyn) {  // (with a pool every CTA has at least three tiles of its own)
    if (threadIdx.x == 0) sched_release(prm.sched);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = smem + BAR_OFF;          // STAGES x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * STAGES;   // STAGES x 8 bytes
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;  // 2 x 8 bytes
  const uint32_t bar_tempty = bar_tfull + 16;         // 2 x 8 bytes
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_sfull = bar_drain + 8;            // kSchedSlots x 8 bytes: a chunk id was written
  const uint32_t bar_sempty = bar_sfull + 8 * kSchedSlots;  // kSchedSlots x 8 bytes: it was read
  const uint32_t bar_sready = bar_sempty + 8 * kSchedSlots;  // STAGES x 8 bytes: the stage's scales are in TMEM
  const uint32_t bar_cdrain = bar_sready + 8 * STAGES;       // the copier's last copies completed
  // one phase per change of the fixed operand: every MMA that read the resident scales before it completed
  const uint32_t bar_resfree = bar_cdrain + 8;

  for (int e = threadIdx.x; e < E; e += THREADS) s_poff[e] = __ldcg(prm.poff + e);
  if (prm.dyn) {
    __syncthreads();
    if (warp == 0) build_chunk_table(s_poff, s_cstart, E, NT, r128, (int)gridDim.x, lane);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);  // one arrive per epilogue warp
    }
    mbar_init(bar_drain, 1);
    for (int q = 0; q < kSchedSlots; ++q) {
      mbar_init(bar_sfull + 8 * q, 1);
      mbar_init(bar_sempty + 8 * q, 1 + NCOPY + 4);  // the MMA issuer, the scale copiers and the epilogue warps
    }
    for (int s = 0; s < STAGES; ++s) mbar_init(bar_sready + 8 * s, NCOPY);  // one commit per copier
    mbar_init(bar_cdrain, NCOPY);
    mbar_init(bar_resfree, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  int n_chunks = prm.dyn ? s_cstart[E] : pool;

  const int KB = prm.KB;
  const int katoms_total = prm.K / 64;
  const int nacc = prm.nacc;
  const uint32_t res_col = ACC_COLS * nacc;
  const uint32_t str_col = res_col + 4u * katoms_total;
  pdl_wait();  // the activations and every other result of the previous launch are needed from here on
  pdl_trigger();
  if (threadIdx.x == 0) s_abort = (*(volatile uint32_t*)prm.err & kAbortMask) != 0;
  __syncthreads();
  if (s_abort) {  // an earlier timeout poisons the call: no role takes a tile
    tau1 = tau0;
    n_chunks = 0;
  }

  if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_once = policy_evict_first();  // weights of a one-m-tile expert are read once
    const uint64_t pol_keep = policy_evict_last();   // activations are re-read by every n-tile
    const uint64_t pol_reuse = policy_evict_normal();  // weights re-read by the next m-tiles of the expert
    const int n_stages = (tau1 - tau0) * KB;
    const int wblocks = (prm.K + 255) / 256;      // 16 KB weight blocks per tile
    // L2 prefetch cursor: stage j of this CTA's range is k-stage j % KB of tile tau0 + j / KB
    TileCursor pc;
    pc.seek(tau0, s_poff, E, NT, r128);
    auto prefetch = [&](int j) {
      const int kb = j % KB;
      if (kb == 0 && j > 0) pc.step(s_poff, E, NT, r128);
      const size_t blk = (size_t)(pc.e * NT + pc.nt);
      const int nblk = min(HALVES, wblocks - kb * HALVES);
      bulk_prefetch_l2(prm.b_codes + (blk * wblocks + (size_t)kb * HALVES) * HALF_BYTES, nblk * HALF_BYTES);
      bulk_prefetch_l2(prm.b_sf + (blk * katoms_total + (size_t)kb * ATOMS) * SF_TILE,
                       min(ATOMS, katoms_total - kb * ATOMS) * SF_TILE);
    };
    if (!prm.dyn)  // the dynamic schedule learns its tiles as it goes: no look-ahead prefetch
      for (int j = 0; j < min(PREFETCH, n_stages); ++j) prefetch(j);
    int it = 0, prev_key = INT_MIN, prev_mt = -1, a_box = 3;
    bool ok = true;
    TileSource<kRoleProducer> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    while (ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128)) {
      const bool res_a = (t.me == 1);  // one m-tile: the activations are the fixed operand, else the weights
      const int key = res_a ? t.mt : -1 - (t.e * NT + t.nt);
      const bool new_res = (key != prev_key);  // resident scales go to TMEM once per fixed operand
      prev_key = key;
      const int a_row = t.mt * BM;
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
      const uint32_t a_half = (uint32_t)(16 << a_box) * KBYTES;  // bytes of one activation block
      // one m-tile: weights stream through once and the activation tile is re-read by every n-tile;
      // several: the weight tile is re-read by the next m-tiles, and no tile deserves to outlive the others
      const uint64_t pol_w = res_a ? pol_once : pol_reuse;
      const uint64_t pol_a = res_a ? pol_keep : pol_reuse;
      const uint8_t* bsrc = prm.b_codes + (size_t)(t.e * NT + t.nt) * wblocks * HALF_BYTES;
      const uint8_t* sfa = prm.a_sf + (size_t)t.mt * katoms_total * SF_TILE;
      const uint8_t* sfb = prm.b_sf + ((size_t)t.e * NT + t.nt) * katoms_total * SF_TILE;
      const uint8_t* sf_res = res_a ? sfa : sfb;
      const uint8_t* sf_str = res_a ? sfb : sfa;
      const uint64_t pol_res = res_a ? pol_a : pol_w;
      const uint64_t pol_str = res_a ? pol_w : pol_a;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        if (!prm.dyn && it + PREFETCH < n_stages) prefetch(it + PREFETCH);
        const int s = it % STAGES;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, prm.err)) {
          ok = false;
          break;
        }
        const int atoms = min(ATOMS, katoms_total - kb * ATOMS);
        const int halves = (atoms + 3) / 4;
        const uint32_t st = smem + s * STAGE_BYTES;
        mbar_arrive_expect_tx(bar_full + 8 * s,
                              halves * (HALF_BYTES + a_half) + (new_res ? 2 : 1) * atoms * SF_TILE);
        bulk_load(st + A_BYTES, bsrc + (size_t)kb * B_BYTES, halves * HALF_BYTES, bar_full + 8 * s, pol_w);
        for (int h = 0; h < halves; ++h)
          tma_load_2d(st + h * HALF_BYTES, &tmA.box[a_box], bar_full + 8 * s, (kb * HALVES + h) * KBYTES, a_row,
                      pol_a);
        if (new_res)
          bulk_load(st + RES_OFF, sf_res + (size_t)kb * ATOMS * SF_TILE, atoms * SF_TILE, bar_full + 8 * s, pol_res);
        bulk_load(st + STR_OFF, sf_str + (size_t)kb * ATOMS * SF_TILE, atoms * SF_TILE, bar_full + 8 * s, pol_str);
      }
    }
    sched_release(prm.sched);  // this CTA takes no more chunks
    // on every path, let the copies already issued land before the CTA exits
    for (int j = max(0, it - STAGES); j < it; ++j) drain_wait(bar_full + 8 * (j % STAGES), (uint32_t)(j / STAGES) & 1u);
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // This thread and the scale copier (warp 6) share the per-stage tensor-core instruction stream: every
    // tcgen05 instruction holds its issuing thread for about the same time, so the copier issues the stage's
    // scale copies (and commits them to bar_sready) while this thread issues the MMAs of the stage before.
    // Every shared-memory descriptor is built from its full byte address: the 14-bit address field wraps
    // with the shared window, so adding offsets to an already-masked descriptor could carry into the
    // reserved bits.
    constexpr uint32_t idesc = idesc_nvf4(BM, BN);
    int tl = 0, prev_key = INT_MIN;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    TileSource<kRoleMma> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    for (; ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128);
         ++tl) {
      const bool res_a = (t.me == 1);
      const int key = res_a ? t.mt : -1 - (t.e * NT + t.nt);
      // a new fixed operand: bar_resfree completes once every MMA issued so far (all of them read the old
      // resident scales) has completed, and the copiers wait for that before they overwrite them
      if (tl > 0 && key != prev_key) tc_commit(bar_resfree);
      prev_key = key;
      const int b = tl % nacc;
      const uint32_t use = (uint32_t)(tl / nacc);
      // the epilogue has drained this accumulator buffer
      if (!mbar_wait(bar_tempty + 8 * b, (use & 1u) ^ 1u, prm.err)) {
        ok = false;
        break;
      }
      const uint32_t acc = tmem + ACC_COLS * b;
      for (int kb = 0; kb < KB; ++kb) {
        // the operands are in shared memory and the copier's scale copies for this stage have completed
        if (!mbar_wait(bar_full + 8 * s, ph, prm.err) || !mbar_wait(bar_sready + 8 * s, ph, prm.err)) {
          ok = false;
          break;
        }
        // order the tensor-core reads of this stage after the waits that made the TMA writes and the
        // scale copies visible (without it MMAs can read stale shared memory)
        tc_fence_after();
        const uint32_t st = smem + (uint32_t)s * STAGE_BYTES;
        const uint32_t res_t = tmem + res_col + 4u * ATOMS * kb;
        const uint32_t str_t = tmem + str_col + SFB_STAGE_COLS * s;
        const uint32_t sfa_t = res_a ? res_t : str_t;  // TMEM scales of A and of B for this stage
        const uint32_t sfb_t = res_a ? str_t : res_t;
        const uint32_t acc0 = kb > 0 ? 1u : 0u;
        if (kb * ATOMS + ATOMS <= katoms_total) {  // a full stage: 8 MMAs
#pragma unroll
          for (int a = 0; a < ATOMS; ++a) {
            const uint32_t ko = (a >> 2) * HALF_BYTES + (a & 3) * 32;  // K offset inside the stage
            tc_mma_nvf4(acc, desc_sw128(st + ko), desc_sw128(st + A_BYTES + ko), idesc, sfa_t + 4 * a,
                        sfb_t + 4 * a, a > 0 ? 1u : acc0);
          }
        } else {  // the partial last stage of a K that is not a multiple of 512
          const int atoms = katoms_total - kb * ATOMS;
          for (int a = 0; a < atoms; ++a) {
            const uint32_t ko = (a >> 2) * HALF_BYTES + (a & 3) * 32;
            tc_mma_nvf4(acc, desc_sw128(st + ko), desc_sw128(st + A_BYTES + ko), idesc, sfa_t + 4 * a,
                        sfb_t + 4 * a, (kb > 0 || a > 0) ? 1u : 0u);
          }
        }
        tc_commit(bar_empty + 8 * s);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) tc_commit(bar_tfull + 8 * b);
    }
    // no MMA may still write TMEM when it is freed
    tc_commit(bar_drain);
    drain_wait(bar_drain, 0);
  } else if (warp >= 6 && warp < 6 + NCOPY && lane == 0) {
    // ------------------------------------------------------------ scale copiers
    // Copier c takes the scale atoms a with a % NCOPY == c of every stage.
    const int cpy = warp - 6;
    // Per stage: the 8 streamed scale tiles (and, for a new fixed operand, its 8 resident ones) from the
    // stage's shared memory into TMEM, then one commit to bar_sready. TMEM slot s of the streamed scales
    // is free again once stage s is full: the producer refilled it only after the MMAs of its previous use
    // committed bar_empty. Resident scales are overwritten only after every MMA that read them has
    // completed: the MMA issuer commits bar_resfree once per change of the fixed operand, before the new
    // operand's first MMA. A copier can be several tiles ahead of the MMAs (a tile of one or two ring
    // stages), but never a whole change ahead: it cannot pass a change until the MMAs of the change before
    // have completed, so the parity of its wait always names the right phase. (A wait on the previous
    // tile's accumulator barrier could name a phase two uses back when the copier ran two tiles ahead.)
    int tl = 0, prev_key = INT_MIN, nchg = 0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    TileSource<kRoleCopier> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    for (; ok && src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128);
         ++tl) {
      const bool res_a = (t.me == 1);
      const int key = res_a ? t.mt : -1 - (t.e * NT + t.nt);
      const bool new_res = (key != prev_key);
      prev_key = key;
      if (new_res && tl > 0) {
        if (!mbar_wait(bar_resfree, (uint32_t)nchg & 1u, prm.err)) {
          ok = false;
          break;
        }
        ++nchg;
      }
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(bar_full + 8 * s, ph, prm.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem + (uint32_t)s * STAGE_BYTES;
        const uint32_t res_t = tmem + res_col + 4u * ATOMS * kb;
        const uint32_t str_t = tmem + str_col + SFB_STAGE_COLS * s;
        if (kb * ATOMS + ATOMS <= katoms_total) {  // a full stage: 8 scale atoms, shared by the copiers
          if (new_res) {
#pragma unroll
            for (int a = cpy; a < ATOMS; a += NCOPY)
              tc_cp_scales(res_t + 4 * a, desc_scales(st + RES_OFF + a * SF_TILE));
          }
#pragma unroll
          for (int a = cpy; a < ATOMS; a += NCOPY) tc_cp_scales(str_t + 4 * a, desc_scales(st + STR_OFF + a * SF_TILE));
        } else {  // the partial last stage of a K that is not a multiple of 512
          const int atoms = katoms_total - kb * ATOMS;
          for (int a = cpy; a < atoms; a += NCOPY) {
            if (new_res) tc_cp_scales(res_t + 4 * a, desc_scales(st + RES_OFF + a * SF_TILE));
            tc_cp_scales(str_t + 4 * a, desc_scales(st + STR_OFF + a * SF_TILE));
          }
        }
        tc_commit(bar_sready + 8 * s);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // no copy may still write TMEM when it is freed
    tc_commit(bar_cdrain);
    drain_wait(bar_cdrain, 0);
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    int tl = 0;
    float hrun = 0.0f;  // W1 modes: amax|h| of this thread's rows, NaN if any h was NaN
    TileSource<kRoleEpilogue> src;
    src.init(prm, tau0, tau1, s_poff, E, NT, r128);
    Tile t;
    for (; src.next(t, prm, tau0, s_poff, s_cstart, s_sched, bar_sfull, bar_sempty, n_chunks, E, NT, r128); ++tl) {
      const int r = t.mt * BM + warp * 32 + lane;
      // the row's pair and the expert's alpha are loaded before the accumulator wait, which hides them
      const int p = __ldcg(prm.pair_of_row + r);
      const float alpha = __ldg(prm.alpha + t.e);
      const int b = tl % nacc;
      const uint32_t use = (uint32_t)(tl / nacc);
      // the whole warp takes one decision: tcgen05.ld is warp-collective
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_tfull + 8 * b, use & 1u, prm.err) ? 1 : 0)) break;
      tc_fence_after();
      const bool any_real = __any_sync(0xFFFFFFFFu, p >= 0);
      const uint32_t tacc = tmem + ACC_COLS * b + ((uint32_t)(warp * 32) << 16);
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
      if (lane == 0) mbar_arrive(bar_tempty + 8 * b);  // the accumulator is free for the next tile
      if (p < 0) continue;                     // padding rows carry nothing ("Bug 14")
      epilogue_row<MODE>(prm, v, r, p, t.nt, alpha, hrun);
    }
    epilogue_amax_flush<MODE>(prm, hrun);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

// ------------------------------------------------------------ host side --
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// 2-D uint8 tensor [rows][inner_bytes], 128-byte-swizzled boxes of box_rows x 128 bytes.
bool encode_u8_sw128(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {(cuuint32_t)KBYTES, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
template <int MODE>
bool configure_once() {
  static int ok = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    ok = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) ==
                 cudaSuccess
             ? 1
             : 0;
  });
  return ok == 1;
}

}  // namespace

int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev] = n;
  }
  return counts[dev];
}

size_t tiled_weight_bytes(int32_t rows, int32_t K) { return (size_t)rows * (size_t)((K + 255) / 256) * KBYTES; }

fp4moe_status gemm_launch(GemmMode mode, const fp4moe_config& cfg, int32_t T, const uint8_t* a_codes,
                          const uint8_t* a_sf, const int32_t* poff, const int32_t* pair_of_row,
                          const uint8_t* b_codes, const uint8_t* b_sf, const float* alpha, const float* gs2,
                          uint8_t* out_codes, uint8_t* out_sf, float* amax, uint32_t* status, uint16_t* o_pairs,
                          uint32_t* err, int* sched, cudaStream_t st) {
  if (T == 0) return FP4MOE_OK;
  if (mode != kW2Rows && amax == nullptr) return FP4MOE_INVALID_ARG;
  if (mode == kW1SwiGLU && status == nullptr) return FP4MOE_INVALID_ARG;
  const bool w2 = (mode == kW2Rows);
  const int Kc = w2 ? cfg.inter : cfg.hidden;
  if (Kc > kMaxResidentK) return FP4MOE_UNSUPPORTED;
  Params prm;
  prm.E = local_experts(cfg);
  prm.K = w2 ? cfg.inter : cfg.hidden;
  prm.KB = (prm.K + 64 * ATOMS - 1) / (64 * ATOMS);
  prm.nacc = (2 * (int)ACC_COLS + prm.K / 16 + (int)SFB_STAGE_COLS * STAGES <= (int)TMEM_COLS) ? 2 : 1;
  prm.b_rows = w2 ? cfg.hidden : 2 * cfg.inter;
  prm.NT = prm.b_rows / BN;
  prm.k = cfg.top_k;
  prm.cap = (int)capacity_rows(cfg, T);
  prm.I = cfg.inter;
  prm.H = cfg.hidden;
  prm.limit = cfg.swiglu_limit;
  prm.poff = poff;
  prm.pair_of_row = pair_of_row;
  prm.b_codes = b_codes;
  prm.a_sf = a_sf;
  prm.b_sf = b_sf;
  prm.alpha = alpha;
  prm.gs2 = gs2;
  prm.out_codes = out_codes;
  prm.out_sf = out_sf;
  prm.amax = amax;
  prm.status = status;
  prm.o_pairs = o_pairs;
  prm.o_pairs32 = (reinterpret_cast<uintptr_t>(o_pairs) & 31u) == 0 ? 1 : 0;
  prm.err = err;
  // the dynamic chunk schedule pays off once experts average a whole m-tile (prefill sizes)
  prm.dyn = ((int64_t)T * cfg.top_k >= (int64_t)local_experts(cfg) * BM) ? 1 : 0;
  if (prm.dyn && sched == nullptr) return FP4MOE_INVALID_ARG;
  prm.steal = (!prm.dyn && sched != nullptr) ? 1 : 0;
  prm.sched = sched;  // zero between launches: no memset splits the launch chain
  AMaps tmA;
  for (int b = 0; b < 4; ++b)
    if (!encode_u8_sw128(&tmA.box[b], a_codes, (uint64_t)prm.K / 2, (uint64_t)prm.cap, 16u << b))
      return FP4MOE_CUDA_ERROR;
  // 128 x 256 tiles (gemm_wide.cu) wherever K and the weight rows allow them: they halve the tiles, and with
  // them the per-tile activation reloads, scale copies and epilogues, and they issue fewer MMAs per MAC. On the
  // DeepSeek-V4-Flash shape they are faster at every batch size (decode, T = 64: 430 against 452 us per layer
  // back to back). W1's K (hidden) and rows (2 x intermediate) always allow them; this kernel remains for a
  // W2 whose K (intermediate) is an odd multiple of 128.
  if (gemm_wide_fits(prm.K, prm.b_rows)) return gemm_wide_launch(mode, prm, tmA, st);
  if (mode != kW2Rows) return FP4MOE_UNSUPPORTED;  // (not reached: the configuration check guarantees it)
  const int nsm = sm_count();
  if (nsm <= 0) return FP4MOE_CUDA_ERROR;
  const int max_tiles = (prm.cap / BM) * prm.NT;
  const unsigned grid = (unsigned)(max_tiles < nsm ? max_tiles : nsm);
  if (!configure_once<kW2Rows>()) return FP4MOE_CUDA_ERROR;
  return launch_pdl(grouped_gemm_kernel<kW2Rows>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, tmA, prm) == cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_CUDA_ERROR;
}

}  // namespace fp4moe
