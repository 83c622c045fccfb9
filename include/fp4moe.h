/*
 * fp4moe.h - C ABI of a single-GPU routed mixture-of-experts FFN layer with
 * block-scaled FP4 (NVFP4) experts, for GB300 (sm_103a).
 *
 * The layer is the one on "Current Bug: CuTeDSLMoERunner - Status & Debug
 * History", section "Key Architecture: CuTeDSL NVFP4 MoE / Data Flow":
 *   route -> per-expert counts and offsets -> scatter into 128-row-padded
 *   expert slots -> NVFP4 quantise with per-expert swizzled block scales ->
 *   grouped GEMM W13 (gate | up) -> clamped SwiGLU -> NVFP4 requantise ->
 *   grouped GEMM W2 -> weighted top-k combine.
 * At the DeepSeek-V4-Flash shape ("Lucifer-CUTLASS TP3 virtual-padding
 * audit", section "TP3 shape plan") that is hidden 4096, intermediate 2048,
 * 256 experts, top-k 6 and swiglu_limit 10.
 *
 * Conventions, shared by every call:
 *  - Each call returns fp4moe_status. FP4MOE_OK means the work was ENQUEUED on
 *    `stream`. It does not mean the work has finished.
 *  - The caller owns all device memory. The library never allocates device
 *    memory, never synchronises, and never reads device values on the host
 *    (exceptions: the prep helpers marked so, and fp4moe_read_error).
 *    "CUDA-Graph Safety / GPU-Native Requirements", SECTION B, asks this of
 *    every graph-captured step. The hot-path calls can therefore be captured
 *    into a CUDA graph once they have each been called once outside capture:
 *    the first call configures kernel attributes.
 *  - Pointers are DEVICE pointers unless named *_host. Every device pointer
 *    must be 16-byte aligned, or FP4MOE_MISALIGNED is returned.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - T (tokens) is a host integer, 0 <= T <= cfg->max_tokens. It selects the
 *    launch sizes, so one CUDA graph is captured per T.
 *  - `ws` is a device workspace of fp4moe_workspace_bytes(cfg) bytes. Zero it
 *    once before first use: its header holds counters (the grouped GEMMs'
 *    tile schedules, fp4moe_batch_gs1) that every call leaves at zero again,
 *    so no call needs a memset. Its first 4 bytes are a sticky device error word:
 *    a bitwise OR of FP4MOE_ERR_* values. Kernels set bits there instead of
 *    trapping. Read and clear it with fp4moe_read_error outside any graph.
 *    A second sticky word reports saturated activation block scales
 *    (FP4MOE_SAT_*, fp4moe_read_scale_status), beside the running amax of h
 *    that fp4moe_refresh_gs2 turns into a new L2 scale.
 *    Calls that share a workspace must be ordered on one stream.
 *
 * Padded layout (from "Current Bug", sections "Bug 2", "Bug 4", "Bug 9" and
 * "Bug 14"):
 *  - counts[e]: number of (token, k) pairs routed to expert e.
 *  - offsets[e]: inclusive running sum of counts, with NO leading 0
 *    (counts [4,4,0] -> offsets [4,8,8]).
 *  - P_e = align_up(counts[e], 128). padded_offsets[e] is the inclusive
 *    running sum of P_e, also with no leading 0. Expert e owns rows
 *    [padded_offsets[e] - P_e, padded_offsets[e]). A row's expert is
 *    searchsorted(padded_offsets, row, right=True).
 *  - R = padded_offsets[E-1] <= fp4moe_capacity_rows(cfg, T) = CAP, where
 *    CAP = align_down(T*k + 127*min(E, T*k), 128), at least 128.
 *  - Inside an expert, real rows come first, in ascending pair index
 *    p = t*k + j. Padding rows follow.
 *  - pair_of_row[r] = p for a real row, -1 for a padding row (r < R). Rows
 *    r >= R are not written. The row's token is p / k.
 *  - Activations in slot order: a*_fp4 is [CAP][K/2] bytes, two E2M1 codes
 *    per byte, element 2i in the low nibble. a*_sf holds the E4M3 block
 *    scales (one per 16 elements) in the 128x4 "32_4_4" tile layout
 *    ("Bug 1", "Bug 11"), with C = K/16 scale columns:
 *      byte(r, c) = ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4
 *    Padding rows are never written: their contents are unspecified. The
 *    GEMMs compute them like any other row (the rows of an MMA are
 *    independent) and then drop them, so no real row depends on them.
 *
 * NVFP4 value of code q under block scale sf and global scale g:
 *   decode_e2m1(q) * decode_e4m3(sf) / g.
 * g is the quant-direction global scale RN(2688 / amax) ("Current Bug",
 * sections "Bug 5" and "Bug 6": separate L1 and L2 activation scales, fixed
 * in a warmup pass).
 *
 * Expert weights (written by fp4moe_quantize_weights, K-major):
 *  - Codes are PRE-TILED so that the GEMM streams each stage as one
 *    contiguous 16 KB read. A matrix of R rows (R % 128 == 0) by K elements
 *    is stored as 16384-byte blocks ordered [expert][row tile r/128][k stage
 *    (K index)/256]. Inside a block, row i (0..127) has 128 bytes (256 codes,
 *    element 2c in the low nibble of byte c). Its 16-byte chunk j (bytes
 *    16j .. 16j+15 of that K slice) is stored at offset i*128 + (j ^ (i%8))*16:
 *    the 128-byte swizzle that the tensor cores read from shared memory.
 *    K is zero-padded to a multiple of 256.
 *  - Scales: E4M3, one per 16 elements, in the 128x4 tile layout per expert
 *    (C = K/16 columns): [E][R/128][K/64][512] bytes.
 *  - W1: R = 2I rows, K = H. Rows are in KERNEL order: for each 64-feature
 *    group f = 0 .. I/64-1, rows [128f, 128f+64) are gate features
 *    [64f, 64f+64) and rows [128f+64, 128f+128) are up features
 *    [64f, 64f+64). Logical W13 has the gate in rows [0, I) and up in rows
 *    [I, 2I).
 *  - W2: R = H rows, K = I.
 *  - One fp32 quant-direction global scale per expert per matrix.
 *  - alpha1[e] = 1 / (gs1 * gw1[e]) and alpha2[e] = 1 / (gs2 * gw2[e]),
 *    written by fp4moe_make_alpha.
 *
 * MXFP4 layers (w_format == FP4MOE_W_MXFP4) are the TP3 shard variant of
 * "Lucifer-CUTLASS TP3 virtual-padding audit", section "Remaining kernel
 * assumptions": BF16 activations with MXFP4 weights.
 *  - cfg->inter is the kernel-local width (a multiple of 128).
 *    cfg->inter_logical is the rank's logical width (a multiple of 32, at
 *    most inter). W1 rows and W2 columns past it must be zero ("Required
 *    loader changes", item 5).
 *  - Weights: E2M1 codes with one E8M0 scale per 32 elements along K (OCP
 *    Microscaling v1.0), written by fp4moe_quantize_weights from the fp32
 *    kernel-local shard, in an atom-tiled layout. Blocks of one expert, one
 *    128-row tile and one 64-element K atom are ordered [expert][row
 *    tile][atom]:
 *      codes: 4096 bytes per block, row i at bytes 32i .. 32i+31, element 2c
 *        in the low nibble of byte c;
 *      scales: 256 bytes per block, row i at bytes 2i (elements 0..31 of the
 *        atom) and 2i+1 (elements 32..63).
 *    W1 rows are in the kernel order above. There are no global scales: gw1,
 *    gw2, gs1, gs2 and alpha are unused, and may be NULL in these calls.
 *  - Activations in slot order stay bf16: a1_fp4 is [CAP][H] bf16 and
 *    a2_fp4 is [CAP][I] bf16. a1_sf and a2_sf are unused.
 *  - W1: h = silu(min(g, L)) * clamp(u, -L, L) is rounded to bf16. W2 and
 *    the combine are those of the NVFP4 layer. fp4moe_calibrate returns
 *    FP4MOE_UNSUPPORTED.
 *
 * Expert parallelism ("Current Bug", "Bug 8", "Bug 13" and "EP Configuration"):
 * with ep_count > 0 the layer holds experts [ep_first, ep_first + ep_count)
 * of the router's num_experts.
 *  - The router still scores all num_experts, and topk_ids / topk_w stay
 *    global.
 *  - counts, offsets, padded_offsets, the weights and alpha are per local
 *    expert (ep_count entries); local id = global id - ep_first.
 *  - A pair whose expert is held elsewhere gets slot_of_pair = -1, takes no
 *    row, and is left out of this layer's sum, so y is this rank's part of
 *    the output. Summing the parts of all ranks gives the whole layer.
 *  - CAP uses ep_count in place of E.
 *  - Warm-up calibration sees local ids only (the fix of "Bug 13").
 *  - moe_combine and moe_grouped_gemm_w2_combine cannot tell which pairs are
 *    held elsewhere, so they return FP4MOE_UNSUPPORTED for such layers. Use
 *    moe_forward.
 *
 * Supported shapes: H % 256 == 0, I % 128 == 0, H <= 4608, I <= 4608 (the
 * activation scales of a 128-row tile stay resident in TMEM for all of K),
 * 1 <= k <= 16, k <= E <= 1024, w_format FP4MOE_W_NVFP4 or FP4MOE_W_MXFP4.
 * Anything else returns FP4MOE_UNSUPPORTED.
 */
#ifndef FP4MOE_H_
#define FP4MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fp4moe_stream_t;

typedef enum fp4moe_status {
  FP4MOE_OK = 0,
  FP4MOE_INVALID_ARG = 1,   /* null pointer, T out of range, bad config field */
  FP4MOE_MISALIGNED = 2,    /* a device pointer is not 16-byte aligned */
  FP4MOE_CAPACITY = 3,      /* T > max_tokens, or a buffer bound would be exceeded */
  FP4MOE_UNSUPPORTED = 4,   /* shape or format outside the supported set */
  FP4MOE_CUDA_ERROR = 5     /* a CUDA runtime call or launch failed */
} fp4moe_status;

/* Device error word bits (sticky; see fp4moe_read_error). */
#define FP4MOE_ERR_TIMEOUT   0x1u  /* a bounded wait inside a kernel expired; its tile was skipped */
#define FP4MOE_ERR_EXPERT_ID 0x2u  /* a routed expert id was outside [0, E) */
#define FP4MOE_ERR_CAPACITY  0x4u  /* padded rows R exceeded CAP */
#define FP4MOE_ERR_NAN       0x8u  /* a NaN reached an NVFP4 activation quantiser (x in moe_quantize_scatter,
                                      or h in the W1 epilogue or fp4moe_calibrate); the codes of that block
                                      are unspecified, and so are the outputs of its token */
#define FP4MOE_ERR_SCALE_RANGE 0x10u /* fp4moe_mxfp4_as_nvfp4: an MX scale is NaN, or lies more than 17 binades
                                         below its matrix's largest, and has no exact E4M3 form */

/* Scale-status bits: a second sticky word of the workspace (fp4moe_read_scale_status). They are not
 * errors: a fixed activation global scale that a batch outgrows saturates its E4M3 block scales, which is
 * part of the definition ("Current Bug", "Bug 5"). They tell the caller that a scale has gone stale. */
#define FP4MOE_SAT_L1 0x1u  /* some L1 block scale s = RN(RN(amax/6) * gs1) of x saturated: s > 464, so E4M3
                               rounding takes it above 448, the largest finite value */
#define FP4MOE_SAT_L2 0x2u  /* the same for h under gs2 in the W1 epilogue */

#define FP4MOE_W_NVFP4 0
#define FP4MOE_W_MXFP4 1

typedef struct fp4moe_config {
  int32_t hidden;        /* H */
  int32_t inter;         /* I, kernel-local intermediate width */
  int32_t inter_logical; /* logical intermediate (== inter for NVFP4) */
  int32_t num_experts;   /* E */
  int32_t top_k;         /* k */
  int32_t max_tokens;    /* largest T any call will pass */
  float swiglu_limit;    /* L of the clamped SwiGLU */
  int32_t w_format;      /* FP4MOE_W_NVFP4 or FP4MOE_W_MXFP4 */
  int32_t ep_first;      /* expert parallelism: first expert this layer holds (global id) */
  int32_t ep_count;      /* experts it holds; 0 = all num_experts (no expert parallelism) */
  int32_t shared_inter;  /* Is, the shared expert's kernel-local intermediate width (multiple of 128);
                            0 = the layer has no shared expert */
} fp4moe_config;

/* Version of this ABI (major*100 + minor). */
int32_t fp4moe_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* fp4moe_status_string(fp4moe_status s);

/* CAP(T): rows of every slot-ordered activation buffer for a T-token call. */
size_t fp4moe_capacity_rows(const fp4moe_config* cfg, int32_t T);

/* Bytes of the workspace for any T <= cfg->max_tokens (0 on a bad config). */
size_t fp4moe_workspace_bytes(const fp4moe_config* cfg);

/* Byte sizes of the kernel-ready expert weight buffers (any output may be NULL). */
fp4moe_status fp4moe_weight_bytes(const fp4moe_config* cfg, size_t* w1_codes, size_t* w1_sf,
                                  size_t* w2_codes, size_t* w2_sf);

/*
 * moe_route: router logits, softmax top-k, per-expert counts, offsets and
 * 128-row-padded slots. Hot-path calls launch their kernels with programmatic
 * dependent launch, so consecutive kernels overlap their launch latency.
 * Each of them waits for its predecessor before it lets its own successor
 * start. So when a grouped GEMM starts, the kernel two places before it has
 * finished, and the GEMM reads padded_offsets and pair_of_row during a
 * set-up that overlaps its predecessor. A caller's own kernel placed right
 * before a grouped GEMM must therefore not trigger its dependents before it
 * has written those two arrays (kernels that never trigger early, and
 * copies, are fine).
 *   l[t,e] = RN_f32(sum_h x[t,h]*router_w[e,h]) (+ router_bias[e] in fp32):
 *     the exact sum rounded once, to within an ulp (an fp32 compensated
 *     two-sum reduction in a fixed order).
 *   topk_ids[t,:]: the k largest l[t,:], in descending order; ties go to the
 *     lower expert id.
 *   topk_w[t,j] = exp(l_j - l_max) / sum_selected exp(l - l_max) (fp32).
 *   The logits are found in two passes. A tensor-core pass gives every
 *   l~[t,e] with a bound d[t,e] = 2^-12 |x_t| |w_e| + 2^-21 |l~|. Then every
 *   expert whose interval [l~ - d, l~ + d] reaches the k-th largest lower
 *   end gets the exact l above. So ids and weights are those of the exact
 *   logits. logits_out[t,e] holds l for those candidate experts (always
 *   including the k selected ones) and l~ for the others, and |l~ - l| <= d.
 *   counts, offsets, padded_offsets, slot_of_pair, pair_of_row as above.
 * Slot ranks are integer-deterministic: they do not depend on the order of
 * atomics.
 *   x [T][H] bf16, router_w [E][H] bf16, router_bias [E] fp32 or NULL,
 *   logits_out [T][E] fp32 or NULL, topk_ids [T][k] int32, topk_w [T][k] fp32,
 *   counts/offsets/padded_offsets [E] int32, slot_of_pair [T*k] int32,
 *   pair_of_row [CAP] int32.
 * Source: "Current Bug", "Data Flow" (remap -> sort by expert). "CUDA-Graph
 * Safety", SECTION B (counts by scatter-add into a fixed buffer, no
 * bincount) and SECTION C row 4.
 */
fp4moe_status moe_route(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                        const float* router_bias, float* logits_out, int32_t* topk_ids, float* topk_w,
                        int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* slot_of_pair,
                        int32_t* pair_of_row, void* ws, fp4moe_stream_t stream);

/*
 * moe_route_noalloc: moe_route for callers that cannot hand the library a
 * workspace. None of the source pages describe such a call. It is here for
 * embedders whose device memory is reserved in full up front and that forbid
 * any later device allocation, and for C callers with no allocator of their
 * own to size and own a workspace. cudaMalloc can also synchronise the whole
 * device, which such callers must avoid. The call itself allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Its outputs and their meaning are those of moe_route, computed by the same
 * kernels. What moe_route keeps in `ws` (the per-chunk expert histograms, the
 * squared norms of the router rows and, for T <= 256, the router's partial
 * logit tiles of a split K) lives here in one
 * library-owned scratch array in device memory, a file-scope __device__
 * array of FP4MOE_NOALLOC_SCRATCH_BYTES bytes in the library image. The array
 * bounds the sizes:
 *   T <= FP4MOE_NOALLOC_MAX_TOKENS and num_experts <= FP4MOE_NOALLOC_MAX_EXPERTS,
 * otherwise the call returns FP4MOE_CAPACITY before it enqueues anything.
 * T must also respect cfg->max_tokens, as for moe_route.
 *
 * Differences from moe_route:
 *   - logits_out is required (non-NULL): the scratch has no room for logits.
 *   - err: optional device uint32. If non-NULL, FP4MOE_ERR_* bits are OR-ed
 *     into it; the call never clears it. If NULL, errors go to a word in the
 *     scratch that each call clears, so they are lost.
 *
 * Set-up and sharing:
 *   - Every call looks up the array's device address in the current
 *     device's context with cudaGetSymbolAddress, which allocates nothing. The
 *     address therefore stays right after a context is destroyed and created
 *     again (cudaDeviceReset), when the library's device code is loaded anew.
 *     The call returns FP4MOE_CUDA_ERROR if the lookup fails. Make the first
 *     call on each device before any stream capture begins: that lookup may
 *     load the library's device code.
 *   - Every call on a device shares the one array. Each call clears, on
 *     `stream`, the part that must start at zero (the scratch error word);
 *     every other byte it reads it has written first. Two calls whose work
 *     overlaps on the device
 *     therefore race and corrupt each other's results. This happens with
 *     different streams without an ordering between them, or with different
 *     host threads. Order them on one stream or with events.
 */
#define FP4MOE_NOALLOC_MAX_TOKENS 8192
#define FP4MOE_NOALLOC_MAX_EXPERTS 256
#define FP4MOE_NOALLOC_SCRATCH_BYTES (256 + 4 * 256 + 4 * 256 * (8192 / 64) + 16 * 257 * 4 * 256)
fp4moe_status moe_route_noalloc(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                                const float* router_bias, float* logits_out, int32_t* topk_ids, float* topk_w,
                                int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* slot_of_pair,
                                int32_t* pair_of_row, uint32_t* err, fp4moe_stream_t stream);

/*
 * moe_quantize_scatter: L1 activation quantisation into slot order. Row
 * slot_of_pair[t*k + j] gets NVFP4(x[t]) under the global scale *gs1, for
 * every token t and every j < k. Codes go to a1_fp4 [CAP][H/2] and swizzled
 * scales to a1_sf [CAP*H/16 bytes]. Padding rows are left untouched.
 * Per 16-element block, in IEEE fp32 with RNE:
 *   a = max|v|; s = RN(RN(a/6)*g); sf = E4M3_satfinite(s);
 *   inv = sf ? RN(g/sf) : 0; q = E2M1_satfinite(RN(v*inv)).
 * Source: "Current Bug", "Data Flow" (quantize_activation_nvfp4 and
 * _assemble_scales_cudagraph_safe), "Bug 1" and "Bug 14".
 */
fp4moe_status moe_quantize_scatter(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const float* gs1,
                                   const int32_t* slot_of_pair, uint8_t* a1_fp4, uint8_t* a1_sf, void* ws,
                                   fp4moe_stream_t stream);

/*
 * moe_grouped_gemm_w1_swiglu: for every padded row r of expert e,
 *   [g; u] = alpha1[e] * (A1[r] . W1_e), a block-scaled FP4 MMA with fp32
 *   accumulation,
 *   h = silu(min(g, L)) * clamp(u, -L, L)  (fp32),
 * then NVFP4-requantise h under *gs2 into a2_fp4 [CAP][I/2] and a2_sf
 * (swizzled, C = I/16). Padding rows are left untouched.
 * Source: "Current Bug", "Data Flow" (run_nvfp4_grouped_gemm -> l1_out ->
 * SiLU(gate)*up -> quantise), "Bug 6" and "Bug 7". "Lucifer-CUTLASS TP3
 * virtual-padding audit", "TP3 shape plan" (swiglu_limit).
 */
fp4moe_status moe_grouped_gemm_w1_swiglu(const fp4moe_config* cfg, int32_t T, const uint8_t* a1_fp4,
                                         const uint8_t* a1_sf, const int32_t* padded_offsets,
                                         const int32_t* pair_of_row, const uint8_t* w1_fp4, const uint8_t* w1_sf,
                                         const float* alpha1, const float* gs2, uint8_t* a2_fp4, uint8_t* a2_sf,
                                         void* ws, fp4moe_stream_t stream);

/*
 * moe_grouped_gemm_w2: the second grouped GEMM on its own. For every real
 * row r (pair p = pair_of_row[r]),
 *   o_pairs[p][:] = bf16( alpha2[e] * (A2[r] . W2_e) )  (bf16 [T*k][H]),
 * the fp32 accumulator rounded once to bf16 (round to nearest even).
 * Source: "Current Bug", "Data Flow" (L2 grouped GEMM -> l2_out (BF16)).
 * Rows of pairs that no local expert holds are not written.
 */
fp4moe_status moe_grouped_gemm_w2(const fp4moe_config* cfg, int32_t T, const uint8_t* a2_fp4, const uint8_t* a2_sf,
                                  const int32_t* padded_offsets, const int32_t* pair_of_row, const uint8_t* w2_fp4,
                                  const uint8_t* w2_sf, const float* alpha2, uint16_t* o_pairs, void* ws,
                                  fp4moe_stream_t stream);

/*
 * moe_combine: y[t][:] = bf16( sum_{j=0..k-1} topk_w[t][j] * o_pairs[t*k+j][:] ),
 * o_pairs bf16 [T*k][H] (as moe_grouped_gemm_w2 writes it), accumulated in
 * fp32 in j order. Source: "Current Bug", "Data Flow" (l2_out (BF16) ->
 * scatter_add -> y) and "Bug 14" (padding rows are dropped).
 */
fp4moe_status moe_combine(const fp4moe_config* cfg, int32_t T, const uint16_t* o_pairs, const float* topk_w,
                          uint16_t* y, fp4moe_stream_t stream);

/* moe_grouped_gemm_w2 followed by moe_combine, with o_pairs inside `ws`. */
fp4moe_status moe_grouped_gemm_w2_combine(const fp4moe_config* cfg, int32_t T, const uint8_t* a2_fp4,
                                          const uint8_t* a2_sf, const int32_t* padded_offsets,
                                          const int32_t* pair_of_row, const uint8_t* w2_fp4, const uint8_t* w2_sf,
                                          const float* alpha2, const float* topk_w, uint16_t* y, void* ws,
                                          fp4moe_stream_t stream);

/*
 * moe_forward: the whole layer (route, quantize_scatter, W1+SwiGLU+requant,
 * W2, combine) on one stream, with every intermediate inside `ws`.
 * y [T][H] bf16. topk_ids_out / topk_w_out may be NULL. When they are not,
 * the routing decision is copied there.
 */
fp4moe_status moe_forward(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                          const float* router_bias, const float* gs1, const float* gs2, const uint8_t* w1_fp4,
                          const uint8_t* w1_sf, const float* alpha1, const uint8_t* w2_fp4, const uint8_t* w2_sf,
                          const float* alpha2, uint16_t* y, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                          fp4moe_stream_t stream);

/* --------------------------------------------------------- shared expert --
 * DeepSeek-V4-Flash has one shared expert of intermediate size 2048 beside
 * the routed ones ("Lucifer-CUTLASS TP3 virtual-padding audit", "TP3 shape
 * plan"; align_up(ceil(2048 / 3), 128) = 768 per TP3 rank, rank 2 holding 512
 * real features and 256 zeros). Its weights and scales are block-FP8 ("Paths
 * that already appear compatible"). It runs in the same captured step as the
 * router and the routed MoE ("DSV4 -> vLLM: CUDA-Graph Safety", Graph B).
 *
 * Block-FP8, as read here (the pages name the format only; this is the FP8
 * recipe of the DeepSeek-V3 technical report): E4M3 values with one fp32
 * scale per 128 x 128 weight block and per 1 x 128 activation group along K.
 * For each block or group, in IEEE fp32 with RNE:
 *   s = amax / 448,  code_i = E4M3_satfinite(v_i / s),  and every code is 0
 *   when s == 0.  The value of code q is q * s.
 * The expert (every token, weight 1):
 *   [g | u] = x~ W1~^T,  h = silu(min(g, L)) * clamp(u, -L, L),
 *   o_shared = h~ W2~^T  (fp32 [T][H]),
 * where x~ and h~ are x and h quantised per 1 x 128 group and dequantised,
 * and L is cfg->swiglu_limit. The combine adds o_shared to the routed sum:
 *   y[t] = bf16( sum_j w[t,j] * o[t*k+j] + o_shared[t] ).
 *
 * Weights (written by fp4moe_shared_quantize_weights, K-major, plain
 * row-major bytes; 16-byte aligned):
 *   w1        [2 Is][H] E4M3 in kernel row order: rows 128 j .. 128 j + 63
 *             hold gate features 64 j .. 64 j + 63, and rows 128 j + 64 ..
 *             128 j + 127 the up rows of the same features.
 *   w1_scales [2 Is / 128][H / 128] fp32 in logical block order: rows
 *             [0, Is / 128) are the gate blocks, the rest the up blocks.
 *   w2        [H][Is] E4M3.
 *   w2_scales [H / 128][Is / 128] fp32.
 * Under TP each rank holds its own 128-aligned slice of the features, zero
 * past the end of the expert, and the ranks' o_shared sum to the whole.
 * Requires cfg->shared_inter > 0 (else FP4MOE_INVALID_ARG), and H and Is
 * at most 4096 (else FP4MOE_UNSUPPORTED).
 */
typedef struct fp4moe_shared_weights {
  const uint8_t* w1;
  const float* w1_scales;
  const uint8_t* w2;
  const float* w2_scales;
} fp4moe_shared_weights;

/* Byte sizes of the shared expert's weight buffers (any output may be NULL). */
fp4moe_status fp4moe_shared_weight_bytes(const fp4moe_config* cfg, size_t* w1, size_t* w1_scales, size_t* w2,
                                         size_t* w2_scales);

/*
 * fp4moe_shared_quantize_weights (load-time prep): block-FP8 of one matrix.
 *   which = 1: w [2 Is][H] fp32, logical order (gate rows then up rows);
 *   which = 2: w [H][Is] fp32.
 * codes_out and scales_out get the layouts above.
 */
fp4moe_status fp4moe_shared_quantize_weights(const fp4moe_config* cfg, int32_t which, const float* w,
                                             uint8_t* codes_out, float* scales_out, fp4moe_stream_t stream);

/*
 * moe_shared_expert: o_shared [T][H] fp32 for x [T][H] bf16. Three kernels:
 * the 1 x 128 quantisation of x, W1 with the SwiGLU and the requantisation
 * of h, and W2. Intermediates live in `ws`.
 */
fp4moe_status moe_shared_expert(const fp4moe_config* cfg, int32_t T, const uint16_t* x,
                                const fp4moe_shared_weights* se, float* o_shared, void* ws, fp4moe_stream_t stream);

/*
 * moe_combine_shared: moe_combine with the shared expert's output added,
 *   y[t] = bf16( sum_j w[t,j] * o[t*k+j] + o_shared[t] ),
 * the shared term last. slot_of_pair may be NULL; when given, pairs with
 * slot -1 (held by another rank) are left out, which makes it valid for
 * expert-parallel layers. o_shared may be NULL (no shared term).
 */
fp4moe_status moe_combine_shared(const fp4moe_config* cfg, int32_t T, const uint16_t* o_pairs, const float* topk_w,
                                 const int32_t* slot_of_pair, const float* o_shared, uint16_t* y,
                                 fp4moe_stream_t stream);

/*
 * moe_forward_shared: moe_forward plus the shared expert, every intermediate
 * inside `ws`, then one combine of both. Arguments are those of moe_forward
 * plus `se`. moe_forward itself ignores cfg->shared_inter.
 * The shared expert needs only x, so it runs beside the routing and the
 * routed experts: the call records an event on `stream`, runs the shared
 * expert on a library-owned stream that waits for it, and makes `stream`
 * wait for that branch before the combine. Everything stays ordered after
 * the work already on `stream`, and the combine (and all later work on
 * `stream`) after both branches. Under stream capture the branch joins the
 * graph through the two events. Each host thread has its own side stream and
 * events per device, created on its first call there: make that first call
 * outside stream capture.
 */
fp4moe_status moe_forward_shared(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                                 const float* router_bias, const float* gs1, const float* gs2, const uint8_t* w1_fp4,
                                 const uint8_t* w1_sf, const float* alpha1, const uint8_t* w2_fp4,
                                 const uint8_t* w2_sf, const float* alpha2, const fp4moe_shared_weights* se,
                                 uint16_t* y, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                                 fp4moe_stream_t stream);

/* ------------------------------------------------------------------ prep --
 * Load-time helpers. They run outside the timed hot path and may use
 * cudaMemsetAsync. They still never synchronise.
 */

/*
 * fp4moe_quantize_weights: NVFP4-quantise n_experts experts of one matrix.
 *   which = 1: w [n][2I][H] fp32 logical W13 (gate rows first) -> W1 layout
 *   which = 2: w [n][H][I] fp32 -> W2 layout
 * gs_out[e] = RN(2688 / amax(w_e)) is the quant-direction global scale of
 * expert e. Codes and swizzled scales go to the layouts described above.
 * Experts are independent, so a caller may convert them in chunks by passing
 * offset pointers.
 * MXFP4 layers: w is the rank's kernel-local fp32 shard (I = cfg->inter,
 * zero past inter_logical). Every 32 elements along K share the scale
 * 2^X, X = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 for an
 * all-zero block). The codes are E2M1(v / 2^X) with round-to-nearest-even and
 * saturation. They go to the atom-tiled MXFP4 layout, and gs_out is unused.
 * Because 32-element groups never straddle a shard boundary, quantising the
 * shard gives the same bytes as quantising the full tensor and cutting it
 * ("Packed W2 weight is wrong", "W2 E8M0 scales are wrong").
 * Source: "Current Bug", "vLLM Integration Status" (weight stacking
 * make_b_k_major + assemble_scales_3d_side).
 */
fp4moe_status fp4moe_quantize_weights(const fp4moe_config* cfg, int32_t which, int32_t n_experts, const float* w,
                                      uint8_t* codes_out, uint8_t* sf_out, float* gs_out, fp4moe_stream_t stream);

/*
 * fp4moe_mxfp4_as_nvfp4: MXFP4 weights for the NVFP4 layer's block-scaled
 * FP4 MMA. Load time, not the hot path; it never synchronises.
 * Source: "Lucifer-CUTLASS TP3 virtual-padding audit" ("Remaining kernel
 * assumptions": MXFP4 expert weights, E2M1 codes with one E8M0 scale per 32
 * elements) and "Current Bug" ("Data Flow": the NVFP4 grouped GEMM). An MX
 * scale 2^X is a power of two, and E4M3 holds every power of two from 2^-9
 * to 2^8, so with one factor per expert matrix, G = X_max - 8, the MX value
 * e2m1(q) * 2^X is exactly e2m1(q) * e4m3(sf) / gw for sf = E4M3(2^(X - G))
 * on both 16-element halves of the block and gw = 2^-G. The layer then runs
 * the NVFP4 hot path unchanged (NVFP4 activations with gs1 / gs2 and alpha =
 * 1 / (gs * gw)).
 *   cfg: the target NVFP4 layer (w_format FP4MOE_W_NVFP4; for a TP shard,
 *     inter is the kernel width and inter_logical the logical one).
 *   which = 1: mx_codes / mx_sf are n_experts experts of W1 in the
 *     atom-tiled MXFP4 layout (as fp4moe_quantize_weights or
 *     fp4moe_shard_mxfp4 write it for an MXFP4 layer of the same hidden and
 *     inter); codes_out / sf_out / gw_out receive the W1 layout and gw1.
 *     which = 2: the same for W2 and gw2.
 *   err: device uint32 receiving FP4MOE_ERR_SCALE_RANGE if an E8M0 byte is
 *     NaN, a block with byte 0 has nonzero codes, or a block lies outside
 *     the 18-binade window [X_max - 17, X_max] (its scale is then clamped
 *     into the window and the result is no longer exact).
 * All pointers 16-byte aligned. MXFP4 target layers: FP4MOE_UNSUPPORTED.
 */
fp4moe_status fp4moe_mxfp4_as_nvfp4(const fp4moe_config* cfg, int32_t which, int32_t n_experts, const uint8_t* mx_codes,
                                   const uint8_t* mx_sf, uint8_t* codes_out, uint8_t* sf_out, float* gw_out,
                                   uint32_t* err, fp4moe_stream_t stream);

/*
 * fp4moe_tp_shard_units: where one tensor-parallel rank's slice of an axis
 * lies, counted in that tensor's storage unit. Host arithmetic only; no GPU.
 * Source: "Lucifer-CUTLASS TP3 virtual-padding audit", "TP3 shape plan" (the
 * per-rank width align_up(ceil(width / tp), align) and the kernel width that
 * rounds it up to kernel_align) and "Required loader changes" (offsets taken
 * in logical elements, then divided by the elements per storage unit: 1 for
 * unpacked W13 rows, 2 for packed W2 bytes, 32 for E8M0 groups).
 *   width: logical elements of the full axis (e.g. 2048); tp: ranks; rank in
 *   [0, tp); unit: elements per storage unit.
 *   src_offset: first source unit of the rank's slice; count: units copied
 *   (the last rank may get fewer, or none); zero_tail: destination units
 *   past the slice, up to the kernel width, which must be zero. Any output
 *   pointer may be NULL.
 * For width 2048, tp 3, align 32, kernel_align 128: unit 1 gives offsets
 * 0/704/1408 with tails 64/64/128; unit 2 gives 0/352/704 with tails
 * 32/32/64; unit 32 gives 0/22/44 with tails 2/2/4.
 * Errors: FP4MOE_INVALID_ARG for a non-positive size or a rank outside
 * [0, tp); FP4MOE_UNSUPPORTED when a slice boundary or the kernel width
 * splits a storage unit.
 */
fp4moe_status fp4moe_tp_shard_units(int32_t width, int32_t tp, int32_t align, int32_t kernel_align, int32_t rank,
                                    int32_t unit, int32_t* src_offset, int32_t* count, int32_t* zero_tail);

/*
 * fp4moe_shard_mxfp4: cut tensor-parallel rank tp_rank's kernel-local shard
 * of n_experts experts out of an already quantised, full-width MXFP4
 * checkpoint, straight into the atom-tiled MXFP4 weight layout above. Load
 * time, not the hot path; it never synchronises.
 * Source: "Lucifer-CUTLASS TP3 virtual-padding audit", sections "Packed W2
 * weight is wrong", "W2 E8M0 scales are wrong" and "Required loader
 * changes": the slice of the intermediate axis is counted in logical
 * elements and read in each tensor's storage unit, and every destination
 * element past the rank's logical count is zero (zero codes, zero E8M0
 * bytes).
 *   cfg: an MXFP4 layer whose inter / inter_logical are the kernel and
 *     logical widths of the plan of full_inter over tp ranks (align 32,
 *     kernel align 128), e.g. 768 / 704 for 2048 over 3; otherwise
 *     FP4MOE_INVALID_ARG.
 *   which = 1: ck_codes [n][2 full_inter][H / 2] bytes (gate rows first,
 *     then up; element 2c in the low nibble of byte c), ck_sf
 *     [n][2 full_inter][H / 32] E8M0 bytes. Writes the W1 layout (kernel row
 *     order).
 *   which = 2: ck_codes [n][H][full_inter / 2] bytes (packed along the
 *     intermediate axis), ck_sf [n][H][full_inter / 32]. Writes the W2 layout.
 *   codes_out / sf_out: the layer's W1 or W2 weight buffers (or an offset
 *     into them, for a chunk of experts).
 * Because 32-element groups never straddle a rank boundary, the result equals
 * fp4moe_quantize_weights applied to the rank's fp32 shard, byte for byte.
 * All pointers 16-byte aligned. full_inter must be a multiple of 32
 * (FP4MOE_UNSUPPORTED otherwise); NVFP4 layers: FP4MOE_UNSUPPORTED.
 */
fp4moe_status fp4moe_shard_mxfp4(const fp4moe_config* cfg, int32_t which, int32_t n_experts, int32_t full_inter,
                                 int32_t tp, int32_t tp_rank, const uint8_t* ck_codes, const uint8_t* ck_sf,
                                 uint8_t* codes_out, uint8_t* sf_out, fp4moe_stream_t stream);

/*
 * fp4moe_batch_gs1: the L1 activation global scale taken from the batch in
 * hand rather than from a warm-up pass, with no host synchronisation:
 *   gs1_out[0] = RN(2688 / amax|x[0..T)|) (1 for an all-zero batch),
 *   alpha1_out[e] = RN(1 / RN(gs1_out[0] * gw1[e])) for e < E.
 * Pass gs1_out and alpha1_out to moe_forward (or to moe_quantize_scatter and
 * moe_grouped_gemm_w1_swiglu) on the same stream. Activations beyond a
 * warm-up batch's range would otherwise saturate in E4M3: "Current Bug",
 * "Bug 5", where the wrong input_scale makes block scales saturate at 448.
 * gs2 stays the warm-up value, because the amax of h is known only after the
 * whole W1 GEMM.
 * One launch. It uses two words of the workspace header, which it leaves at
 * zero. Calls that share a workspace must be ordered on one stream.
 */
fp4moe_status fp4moe_batch_gs1(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const float* gw1,
                               float* gs1_out, float* alpha1_out, void* ws, fp4moe_stream_t stream);

/*
 * fp4moe_refresh_gs2: the L2 activation global scale taken from the h of
 * recent calls instead of the warm-up pass, with no host synchronisation.
 * Every W1 epilogue (moe_grouped_gemm_w1_swiglu, moe_forward) folds the
 * amax of the h it quantised into a running maximum in the workspace header.
 * This call, in one launch on `stream`:
 *   if that running amax a > 0:
 *     gs2_inout[0] = RN(2688 / a),
 *     alpha2_out[e] = RN(1 / RN(gs2_inout[0] * gw2[e])) for every local expert e;
 *   (with a == 0, no h since the last refresh, gs2 and alpha2 are left alone)
 * and then clears the running amax.
 * The scale is LAGGED: it covers the calls made before the refresh and
 * applies to the calls made after it. A batch whose h exceeds the range of
 * the gs2 it ran with still saturates in E4M3, and sets FP4MOE_SAT_L2; a
 * refresh then adapts gs2 for the next calls. That is the calibration drift
 * of "Current Bug", "Bug 5" and "Bug 6" (an L2 amax of about 286 against a
 * scale taken from a much smaller range), detected and corrected on the device.
 * gw2 [E] is the W2 weight global-scale table of fp4moe_quantize_weights.
 * MXFP4 layers have no global scales: FP4MOE_UNSUPPORTED.
 */
fp4moe_status fp4moe_refresh_gs2(const fp4moe_config* cfg, void* ws, const float* gw2, float* gs2_inout,
                                 float* alpha2_out, fp4moe_stream_t stream);

/* alpha[e] = RN(1 / RN(gs_act[0] * gs_w[e])) for e < n. */
fp4moe_status fp4moe_make_alpha(int32_t n, const float* gs_act, const float* gs_w, float* alpha,
                                fp4moe_stream_t stream);

/*
 * fp4moe_calibrate: activation global scales from a warmup batch
 * ("Current Bug", sections "Bug 5" and "Bug 6": compute_activation_global_scales
 * runs before capture, separately for L1 and L2).
 *   gs1 = RN(2688 / amax|x_warm|)
 *   gs2 = RN(2688 / amax|h|), where h is the SwiGLU output over every real
 *         slot row of the warmup batch, quantised under gs1.
 * Needs the gw1 table (weight global scales of W1) to form alpha1 internally.
 * Writes gs1_out[0] and gs2_out[0].
 */
fp4moe_status fp4moe_calibrate(const fp4moe_config* cfg, int32_t T, const uint16_t* x_warm, const uint16_t* router_w,
                               const float* router_bias, const uint8_t* w1_fp4, const uint8_t* w1_sf,
                               const float* gw1, float* gs1_out, float* gs2_out, void* ws, fp4moe_stream_t stream);

/*
 * fp4moe_quantize_rows_f32: the NVFP4 block quantiser on its own. It is the
 * same device routine the kernels above use, for tests of the codec and of
 * the requantisation step on identical fp32 input.
 *   in [rows][K] fp32; g[rows] per-row global scales (device);
 *   codes [rows][K/2]; sf swizzled with C = K/16 (rows % 128 == 0, K % 64 == 0).
 */
fp4moe_status fp4moe_quantize_rows_f32(int32_t rows, int32_t K, const float* in, const float* g, uint8_t* codes,
                                       uint8_t* sf, fp4moe_stream_t stream);

/*
 * fp4moe_tensor_peak_probe: a measurement of the dense NVFP4 tensor-core
 * rate, the denominator of the grouped GEMMs' tensor-pipe utilisation. The
 * pages give no peak for the hardware; this replaces a vendor figure by a
 * measured one.
 * One CTA per SM issues iters x 4 back-to-back
 * tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X of shape
 * M = 128, N = n, K = 64 on operands held in shared memory (no global
 * traffic), then waits for them. The caller times the launch on `stream`;
 * it performs (SMs) x iters x 4 x 2 x 128 x n x 64 flops, where SMs is the
 * device's multiprocessor count.
 *   n: 128 or 256; iters in [1, 2^22]; err: device uint32 receiving
 *   FP4MOE_ERR_TIMEOUT if the final bounded wait runs out.
 * Errors: FP4MOE_INVALID_ARG for other sizes or a NULL err, FP4MOE_MISALIGNED
 * for an err not 16-byte aligned.
 */
fp4moe_status fp4moe_tensor_peak_probe(int32_t n, int32_t iters, uint32_t* err, fp4moe_stream_t stream);

/*
 * fp4moe_selftest_wait_timeout: a test of the failure path, with no
 * counterpart in the source pages. Every spin-wait in the library's kernels
 * is bounded: when it runs out it sets FP4MOE_ERR_TIMEOUT in the error word,
 * its kernel returns, and later kernels that see the bit skip their work, so
 * a lost arrival never hangs the GPU. This call launches one kernel that
 * waits, through that same routine, on an mbarrier nothing arrives at, for
 * limit_ns nanoseconds (1 ms .. 50 ms, else FP4MOE_INVALID_ARG).
 *   err    device uint32 error word (a workspace's first 4 bytes, or any
 *          4-byte-aligned word); receives FP4MOE_ERR_TIMEOUT.
 *   result device uint32; receives 0 (the wait gave up) or 1 (it completed,
 *          which would be a fault in the bounded-wait routine).
 * Nothing traps or faults: the context stays usable.
 */
fp4moe_status fp4moe_selftest_wait_timeout(uint32_t* err, int64_t limit_ns, uint32_t* result, fp4moe_stream_t stream);

/*
 * fp4moe_read_error: copy the workspace's device error word to *err_host.
 * If clear != 0, zero it afterwards. This call SYNCHRONISES `stream`: use it
 * outside graphs, between steps.
 */
fp4moe_status fp4moe_read_error(void* ws, uint32_t* err_host, int32_t clear, fp4moe_stream_t stream);

/*
 * fp4moe_read_scale_status: copy the workspace's sticky FP4MOE_SAT_* word to
 * *flags_host and, when amax_h_host is not NULL, the running amax|h| of the
 * W1 epilogues since the last fp4moe_refresh_gs2 (0 if none). If clear != 0,
 * zero the flags word afterwards (the running amax is cleared only by a
 * refresh). SYNCHRONISES `stream`: use it outside graphs, between steps.
 */
fp4moe_status fp4moe_read_scale_status(void* ws, uint32_t* flags_host, float* amax_h_host, int32_t clear,
                                       fp4moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4MOE_H_ */
