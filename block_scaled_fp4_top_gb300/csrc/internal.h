// Internal declarations shared by the translation units of libfp4moe.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fp4moe.h"

namespace fp4moe {

// Launch `kernel` on `st` with programmatic stream serialisation allowed (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

size_t capacity_rows(const fp4moe_config& cfg, int32_t T);

// Experts this layer holds: [ep_first, ep_first + ep_count) of the router's num_experts, or all of them.
inline int local_experts(const fp4moe_config& c) { return c.ep_count > 0 ? c.ep_count : c.num_experts; }

// Byte offsets of the regions of a workspace sized for cfg.max_tokens.
struct WsLayout {
  size_t hist, nw2, rt_part, logits, ids, w, counts, offsets, poff, slot, por, a1, a1sf, a2, a2sf, opairs, alpha_tmp;
  size_t se_qx, se_sx, se_qh, se_sh, se_o;  // shared expert (cfg.shared_inter > 0)
  size_t total;
};
WsLayout ws_layout(const fp4moe_config& cfg);

// Router logits and top-k (router.cu). logits [T][E] receives the approximate logits, then the final ones;
// nw2 [E] receives the squared norms of the router rows. part (part_bytes, may be null) holds the partial
// tiles when K is split over independent CTAs (a single tile of tokens): router_partial_bytes(cfg) is
// enough for any T <= cfg.max_tokens; with less room the split runs over a cluster instead.
fp4moe_status router_topk_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* wr,
                                 const float* bias, float* logits, float* nw2, float* part, size_t part_bytes,
                                 int32_t* ids, float* w, uint32_t* err, cudaStream_t st);
size_t router_partial_bytes(const fp4moe_config& cfg);

// The whole routing step: router_topk_launch, then counts, offsets and slots. hist: per-chunk histograms
// for large T (nchunks x E int32).
fp4moe_status route_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                           const float* bias, float* logits, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* poff, int32_t* slot_of_pair, int32_t* pair_of_row,
                           int32_t* hist, float* nw2, float* part, size_t part_bytes, uint32_t* err,
                           cudaStream_t st);

// status: sticky FP4MOE_SAT_L1 when a block scale saturates; err: FP4MOE_ERR_NAN for a NaN in x
fp4moe_status quant_scatter_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const float* gs1,
                                   const int32_t* slot_of_pair, uint8_t* a1, uint8_t* a1_sf, uint32_t* status,
                                   uint32_t* err, cudaStream_t st);
// gs2 and alpha2 from the running amax|h| of the W1 epilogues (left as they are when it is zero), which is
// then cleared: fp4moe_refresh_gs2
fp4moe_status refresh_gs2_launch(int32_t E, float* amax_run, const float* gw2, float* gs2, float* alpha2,
                                 cudaStream_t st);

// rows [n_rows_total][K] fp32 -> NVFP4; g indexed by row / g_div; optional W1 gate/up row permutation
// (rows_per_group = rows of one expert, inter = I, or 0 for no permutation); tiled != 0 writes the codes in
// the pre-tiled weight layout (16 KB blocks of 128 rows x 128 bytes, 128-byte swizzled).
fp4moe_status quant_rows_launch(int64_t n_rows_total, int32_t K, int32_t rows_per_group, int32_t inter,
                                int32_t tiled, const float* in, const float* g, int32_t g_div, uint8_t* codes,
                                uint8_t* sf, cudaStream_t st);

// bytes of one matrix of `rows` x K in the pre-tiled weight layout (K padded up to a multiple of 256)
size_t tiled_weight_bytes(int32_t rows, int32_t K);

fp4moe_status amax_f32_launch(int32_t n_groups, int64_t per_group, const float* in, float* amax, cudaStream_t st);
fp4moe_status amax_bf16_launch(int64_t n, const uint16_t* in, float* amax, cudaStream_t st);
fp4moe_status gs_from_amax_launch(int32_t n, float* inout, cudaStream_t st);
fp4moe_status make_alpha_launch(int32_t n, const float* gs_act, const float* gs_w, float* alpha, cudaStream_t st);
// gs1 and alpha1 from the batch's own amax, one launch; acc and done are zero words that it leaves zero
fp4moe_status batch_gs1_launch(int32_t T, int32_t H, const uint16_t* x, int32_t E, const float* gw1, float* gs1,
                               float* alpha1, unsigned int* acc, unsigned int* done, cudaStream_t st);

enum GemmMode { kW1SwiGLU = 0, kW1Amax = 1, kW2Rows = 2 };
fp4moe_status gemm_launch(GemmMode mode, const fp4moe_config& cfg, int32_t T, const uint8_t* a_codes,
                          const uint8_t* a_sf, const int32_t* poff, const int32_t* pair_of_row,
                          const uint8_t* b_codes, const uint8_t* b_sf, const float* alpha, const float* gs2,
                          uint8_t* out_codes, uint8_t* out_sf, float* amax, uint32_t* status, uint16_t* o_pairs,
                          uint32_t* err, int* sched, cudaStream_t st);

// SMs of the current device (cached per device), 0 on error
int sm_count();
// probe.cu: dense FP4 tensor-core throughput (fp4moe_tensor_peak_probe)
fp4moe_status tensor_peak_launch(int32_t n, int32_t iters, uint32_t* err, cudaStream_t st);

// selftest.cu: one bounded wait that runs out (see fp4moe_selftest_wait_timeout)
fp4moe_status selftest_wait_launch(uint32_t* err, int64_t limit_ns, uint32_t* result, cudaStream_t st);

// mxgemm.cu: MXFP4 weights x bf16 activations. w2 = false: W1 with SwiGLU into bf16 rows out_bf16 [cap][I];
// w2 = true: W2 into fp32 rows o_pairs [T*k][H]. Weights in the atom-tiled MXFP4 layout (see fp4moe.h).
fp4moe_status mx_gemm_launch(bool w2, const fp4moe_config& cfg, int32_t T, const uint16_t* a_bf16,
                             const int32_t* poff, const int32_t* pair_of_row, const uint8_t* b_codes,
                             const uint8_t* b_sf, uint16_t* out_bf16, uint16_t* o_pairs, uint32_t* err,
                             cudaStream_t st);
fp4moe_status mx_quant_rows_launch(int64_t n_rows, int32_t K, int32_t rows_per_group, int32_t inter, const float* in,
                                   uint8_t* codes, uint8_t* sf, cudaStream_t st);
// one TP rank's shard of a quantised full-width MXFP4 checkpoint into the atom-tiled layout (fp4moe_shard_mxfp4).
// w1: rows = 2 Ik logical W13 rows, Kd = H; else rows = H, Kd = Ik. src_row_elems: elements of one source row
// (H for W13, I_full for W2). first / count: the rank's logical slice of I.
fp4moe_status mx_shard_launch(int32_t n_experts, bool w1, int32_t rows, int32_t Kd, int32_t Ik, int32_t full_inter,
                              int32_t src_row_elems, int32_t first, int32_t count, const uint8_t* src_codes,
                              const uint8_t* src_sf, uint8_t* codes, uint8_t* sf, cudaStream_t st);
// MXFP4 weights (atom-tiled MX layout) -> the NVFP4 weight layout with E4M3 scales 2^(X - G) and gw = 2^-G
// (fp4moe_mxfp4_as_nvfp4). rows = 2 I (W1) or H (W2); K = H (W1) or I (W2).
fp4moe_status mx_as_nvfp4_launch(int32_t n_experts, int32_t rows, int32_t K, const uint8_t* mx_codes,
                                 const uint8_t* mx_sf, uint8_t* codes, uint8_t* sf, float* gw, uint32_t* err,
                                 cudaStream_t st);
fp4moe_status scatter_rows_bf16_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x,
                                       const int32_t* slot_of_pair, uint16_t* a1, cudaStream_t st);

// y[t] = bf16(sum_j w[t,j] o[t*k+j] + o_shared[t]); with slot_of_pair, pairs without a slot (held by no local
// expert) are left out of the sum; o_shared may be null
fp4moe_status combine_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* o_pairs, const float* w,
                             const int32_t* slot_of_pair, const float* o_shared, uint16_t* y, cudaStream_t st);

// segemm.cu: the block-FP8 shared expert. se_tcap: rows of its activation buffers (max_tokens rounded up to
// 128). se_forward_launch: x -> qx/sx, W1 + SwiGLU -> qh/sh, W2 -> out [T][H] fp32.
size_t se_tcap(const fp4moe_config& cfg);
fp4moe_status se_quant_weights_launch(const fp4moe_config& cfg, int32_t which, const float* w, uint8_t* codes,
                                      float* scales, cudaStream_t st);
fp4moe_status se_forward_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const uint8_t* w1,
                                const float* s1, const uint8_t* w2, const float* s2, uint8_t* qx, float* sx,
                                uint8_t* qh, float* sh, float* out, uint32_t* err, cudaStream_t st);

}  // namespace fp4moe
