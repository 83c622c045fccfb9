// C ABI of libfp4moe: argument checks, workspace layout and the composed
// calls (moe_forward, moe_grouped_gemm_w2_combine, fp4moe_calibrate).
//
// Host code here validates host-known integers and pointer alignment, then
// enqueues kernels. It never synchronises and never allocates, apart from
// fp4moe_read_error and the documented prep helpers. It never reads device
// values. "CUDA-Graph Safety / GPU-Native Requirements", SECTION B, lists the
// hidden host syncs, allocations and device-value branches that a captured
// step must not contain.
#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

namespace {

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// "Lucifer-CUTLASS TP3 virtual-padding audit", "TP3 shape plan": the logical width of each rank is
// align_up(ceil(width / tp), align) and the kernel-local width rounds it up to kernel_align.
inline void tp_widths(int64_t width, int64_t tp, int64_t align, int64_t kernel_align, int64_t& local,
                      int64_t& kernel) {
  local = ((width + tp - 1) / tp + align - 1) / align * align;
  kernel = (local + kernel_align - 1) / kernel_align * kernel_align;
}

fp4moe_status check_cfg(const fp4moe_config* c) {
  if (c == nullptr) return FP4MOE_INVALID_ARG;
  if (c->hidden <= 0 || c->inter <= 0 || c->num_experts <= 0 || c->top_k <= 0 || c->max_tokens < 0 ||
      !(c->swiglu_limit > 0.0f))
    return FP4MOE_INVALID_ARG;
  if (c->w_format != FP4MOE_W_NVFP4 && c->w_format != FP4MOE_W_MXFP4) return FP4MOE_UNSUPPORTED;
  if (c->hidden % 256 != 0 || c->inter % 128 != 0) return FP4MOE_UNSUPPORTED;
  if (c->top_k > kMaxTopK || c->num_experts > kMaxExperts || c->top_k > c->num_experts) return FP4MOE_UNSUPPORTED;
  // expert parallelism: the layer holds experts [ep_first, ep_first + ep_count) of the router's num_experts
  if (c->ep_count < 0 || (c->ep_count == 0 && c->ep_first != 0) ||
      (c->ep_count > 0 && (c->ep_first < 0 || c->ep_first + c->ep_count > c->num_experts)))
    return FP4MOE_INVALID_ARG;
  if (c->shared_inter < 0) return FP4MOE_INVALID_ARG;
  if (c->shared_inter % 128 != 0) return FP4MOE_UNSUPPORTED;  // whole 128 x 128 FP8 blocks
  if (c->shared_inter > 0 && (c->hidden > 4096 || c->shared_inter > 4096))
    return FP4MOE_UNSUPPORTED;  // the shared GEMM keeps up to 32 K blocks of scales in shared memory
  if (c->w_format == FP4MOE_W_NVFP4) {  // a TP shard: whole 16-element scale blocks inside the kernel width
    if (c->inter_logical < 0 || c->inter_logical > c->inter || c->inter_logical % 16 != 0) return FP4MOE_UNSUPPORTED;
  } else {  // MXFP4: the logical width is whole 32-element scale groups inside the kernel width
    if (c->inter_logical < 0 || c->inter_logical > c->inter || c->inter_logical % 32 != 0) return FP4MOE_UNSUPPORTED;
  }
  return FP4MOE_OK;
}

inline bool is_mx(const fp4moe_config* c) { return c->w_format == FP4MOE_W_MXFP4; }

fp4moe_status check_T(const fp4moe_config* c, int32_t T) {
  if (T < 0) return FP4MOE_INVALID_ARG;
  if (T > c->max_tokens) return FP4MOE_CAPACITY;
  return FP4MOE_OK;
}

// every pointer non-null and 16-byte aligned
template <typename... P>
fp4moe_status check_ptrs(P... ps) {
  const void* arr[] = {static_cast<const void*>(ps)...};
  for (const void* p : arr)
    if (p == nullptr) return FP4MOE_INVALID_ARG;
  for (const void* p : arr)
    if (!a16(p)) return FP4MOE_MISALIGNED;
  return FP4MOE_OK;
}

inline fp4moe_status check_opt(const void* p) { return (p == nullptr || a16(p)) ? FP4MOE_OK : FP4MOE_MISALIGNED; }

#define FP4_TRY(expr)                          \
  do {                                         \
    const fp4moe_status s_ = (expr);           \
    if (s_ != FP4MOE_OK) return s_;            \
  } while (0)

template <typename Tp>
Tp* at(void* ws, size_t off) {
  return reinterpret_cast<Tp*>(static_cast<uint8_t*>(ws) + off);
}
inline uint32_t* err_word(void* ws) { return at<uint32_t>(ws, kWsErr); }
inline uint32_t* scale_flags(void* ws) { return at<uint32_t>(ws, kWsScaleFlags); }
inline float* amax_h_run(void* ws) { return at<float>(ws, kWsAmaxHRun); }

}  // namespace

size_t capacity_rows(const fp4moe_config& cfg, int32_t T) {
  const int64_t pairs = (int64_t)T * cfg.top_k;
  const int64_t cap = (pairs + 127 * std::min<int64_t>(local_experts(cfg), pairs)) / 128 * 128;
  return (size_t)std::max<int64_t>(cap, 128);
}

WsLayout ws_layout(const fp4moe_config& c) {
  WsLayout L{};
  size_t off = kWsHeader;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1), 256);
    return o;
  };
  const size_t Tm = (size_t)c.max_tokens, E = (size_t)c.num_experts, k = (size_t)c.top_k;
  const size_t cap = capacity_rows(c, c.max_tokens);
  const size_t nchunks = std::max<size_t>(1, (Tm + kRouteChunk - 1) / kRouteChunk);
  L.hist = take(nchunks * E * 4);
  L.nw2 = take(E * 4);
  L.rt_part = take(router_partial_bytes(c));
  L.logits = take(Tm * E * 4);
  L.ids = take(Tm * k * 4);
  L.w = take(Tm * k * 4);
  L.counts = take(E * 4);
  L.offsets = take(E * 4);
  L.poff = take(E * 4);
  L.slot = take(Tm * k * 4);
  L.por = take(cap * 4);
  const bool mx = c.w_format == FP4MOE_W_MXFP4;  // MXFP4 layers keep their slot activations in bf16
  L.a1 = take(mx ? cap * (size_t)c.hidden * 2 : cap * (size_t)c.hidden / 2);
  L.a1sf = take(mx ? 0 : cap * (size_t)c.hidden / 16);
  L.a2 = take(mx ? cap * (size_t)c.inter * 2 : cap * (size_t)c.inter / 2);
  L.a2sf = take(mx ? 0 : cap * (size_t)c.inter / 16);
  L.opairs = take(Tm * k * (size_t)c.hidden * 2);  // bf16 pair rows
  L.alpha_tmp = take(E * 4);
  if (c.shared_inter > 0) {  // the shared expert: FP8 activations, their scales, and its fp32 output
    const size_t tcap = se_tcap(c), Is = (size_t)c.shared_inter, H = (size_t)c.hidden;
    L.se_qx = take(tcap * H);
    L.se_sx = take(H / 128 * tcap * 4);
    L.se_qh = take(tcap * Is);
    L.se_sh = take(Is / 128 * tcap * 4);
    L.se_o = take(Tm * H * 4);
  }
  L.total = off;
  return L;
}

// Scratch of moe_route_noalloc, owned by the library image. Layout:
// [0, 256) error word, then the squared norms of the router rows (the
// router's error bound), then the per-chunk expert histograms of the large-T
// layout, then the router's partial tiles for a single tile of tokens
// (16 K splits of up to 256 tokens and their norm rows).
namespace {
constexpr size_t kScratchErr = 0;
constexpr size_t kScratchNw2 = 256;
constexpr size_t kScratchHist = kScratchNw2 + 4 * (size_t)FP4MOE_NOALLOC_MAX_EXPERTS;
constexpr size_t kScratchPart = kScratchHist + 4 * (size_t)FP4MOE_NOALLOC_MAX_EXPERTS *
                                                   ((FP4MOE_NOALLOC_MAX_TOKENS + kRouteChunk - 1) / kRouteChunk);
constexpr size_t kScratchPartBytes = 16 * (256 + 1) * 4 * (size_t)FP4MOE_NOALLOC_MAX_EXPERTS;
static_assert(kScratchPart + kScratchPartBytes == FP4MOE_NOALLOC_SCRATCH_BYTES,
              "scratch layout and its advertised size disagree");

__device__ __align__(256) uint8_t g_route_scratch[FP4MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch in the current device's context, looked up on every call: the lookup allocates
// nothing, and a fresh lookup stays right after the context is torn down and created again (the module is then
// loaded again, possibly at another address).
fp4moe_status route_scratch(uint8_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return FP4MOE_CUDA_ERROR;
  *out = static_cast<uint8_t*>(p);
  return FP4MOE_OK;
}
}  // namespace

namespace {
// The shared expert runs beside the routing and the routed experts: moe_forward_shared forks it onto a
// library-owned stream and joins it back before the combine, with events. Each host thread gets its own side
// stream and event pair per device (two threads never share an event), created on first use.
constexpr int kMaxDevices = 64;
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  ~SideStream() {
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (s) cudaStreamDestroy(s);
  }
};

fp4moe_status side_stream(SideStream** out) {
  thread_local SideStream per_dev[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4MOE_CUDA_ERROR;
  SideStream& ss = per_dev[dev];
  if (ss.s == nullptr) {
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess)
      return FP4MOE_CUDA_ERROR;
  }
  *out = &ss;
  return FP4MOE_OK;
}

fp4moe_status check_shared(const fp4moe_config* cfg, const fp4moe_shared_weights* se) {
  if (cfg->shared_inter <= 0 || se == nullptr) return FP4MOE_INVALID_ARG;
  return check_ptrs(se->w1, se->w1_scales, se->w2, se->w2_scales);
}

fp4moe_status shared_launch(const fp4moe_config& cfg, int32_t T, const uint16_t* x, const fp4moe_shared_weights& se,
                            float* o_shared, void* ws, cudaStream_t st) {
  const WsLayout L = ws_layout(cfg);
  return se_forward_launch(cfg, T, x, se.w1, se.w1_scales, se.w2, se.w2_scales, at<uint8_t>(ws, L.se_qx),
                           at<float>(ws, L.se_sx), at<uint8_t>(ws, L.se_qh), at<float>(ws, L.se_sh), o_shared,
                           err_word(ws), st);
}

// The routed layer, with the shared expert's output added in the combine when se is not NULL.
fp4moe_status forward_impl(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                           const float* router_bias, const float* gs1, const float* gs2, const uint8_t* w1_fp4,
                           const uint8_t* w1_sf, const float* alpha1, const uint8_t* w2_fp4, const uint8_t* w2_sf,
                           const float* alpha2, const fp4moe_shared_weights* se, uint16_t* y, int32_t* topk_ids_out,
                           float* topk_w_out, void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  const bool mx = is_mx(cfg);  // MXFP4: gs1, gs2, alpha1 and alpha2 are unused and may be NULL
  if (mx) FP4_TRY(check_ptrs(x, router_w, w1_fp4, w1_sf, w2_fp4, w2_sf, y, ws));
  else FP4_TRY(check_ptrs(x, router_w, gs1, gs2, w1_fp4, w1_sf, alpha1, w2_fp4, w2_sf, alpha2, y, ws));
  FP4_TRY(check_opt(router_bias));
  FP4_TRY(check_opt(topk_ids_out));
  FP4_TRY(check_opt(topk_w_out));
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*cfg);
  uint32_t* err = err_word(ws);
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* poff = at<int32_t>(ws, L.poff);
  int32_t* por = at<int32_t>(ws, L.por);
  // the shared expert needs only x: fork it off before the routing, join it back before the combine
  float* o_shared = nullptr;
  SideStream* side = nullptr;
  fp4moe_status rs = FP4MOE_OK;
  if (se != nullptr) {
    FP4_TRY(side_stream(&side));
    o_shared = at<float>(ws, L.se_o);
    if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return FP4MOE_CUDA_ERROR;
    rs = shared_launch(*cfg, T, x, *se, o_shared, ws, side->s);
    if (cudaEventRecord(side->join, side->s) != cudaSuccess && rs == FP4MOE_OK) rs = FP4MOE_CUDA_ERROR;
  }
  auto routed = [&]() -> fp4moe_status {
    FP4_TRY(route_launch(*cfg, T, x, router_w, router_bias, at<float>(ws, L.logits), ids, w,
                         at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets), poff, at<int32_t>(ws, L.slot), por,
                         at<int32_t>(ws, L.hist), at<float>(ws, L.nw2), at<float>(ws, L.rt_part),
                         router_partial_bytes(*cfg), err, st));
    if (mx) {
      uint16_t* a1 = at<uint16_t>(ws, L.a1);
      uint16_t* a2 = at<uint16_t>(ws, L.a2);
      FP4_TRY(scatter_rows_bf16_launch(*cfg, T, x, at<int32_t>(ws, L.slot), a1, st));
      FP4_TRY(mx_gemm_launch(false, *cfg, T, a1, poff, por, w1_fp4, w1_sf, a2, nullptr, err, st));
      return mx_gemm_launch(true, *cfg, T, a2, poff, por, w2_fp4, w2_sf, nullptr, at<uint16_t>(ws, L.opairs), err, st);
    }
    FP4_TRY(quant_scatter_launch(*cfg, T, x, gs1, at<int32_t>(ws, L.slot), at<uint8_t>(ws, L.a1),
                                 at<uint8_t>(ws, L.a1sf), scale_flags(ws), err, st));
    FP4_TRY(gemm_launch(kW1SwiGLU, *cfg, T, at<uint8_t>(ws, L.a1), at<uint8_t>(ws, L.a1sf), poff, por, w1_fp4, w1_sf,
                        alpha1, gs2, at<uint8_t>(ws, L.a2), at<uint8_t>(ws, L.a2sf), amax_h_run(ws), scale_flags(ws),
                        nullptr, err, at<int>(ws, kWsSchedW1), st));
    return gemm_launch(kW2Rows, *cfg, T, at<uint8_t>(ws, L.a2), at<uint8_t>(ws, L.a2sf), poff, por, w2_fp4, w2_sf,
                       alpha2, nullptr, nullptr, nullptr, nullptr, nullptr, at<uint16_t>(ws, L.opairs), err,
                       at<int>(ws, kWsSchedW2), st);
  };
  const fp4moe_status rr = routed();
  // the join is waited on every path, so a stream capture never ends with the side branch open
  if (side != nullptr && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess && rs == FP4MOE_OK)
    rs = FP4MOE_CUDA_ERROR;
  FP4_TRY(rr);
  FP4_TRY(rs);
  FP4_TRY(combine_launch(*cfg, T, at<uint16_t>(ws, L.opairs), w, cfg->ep_count > 0 ? at<int32_t>(ws, L.slot) : nullptr,
                         o_shared, y, st));
  const size_t pk = (size_t)T * cfg->top_k;
  if (topk_ids_out && pk && cudaMemcpyAsync(topk_ids_out, ids, pk * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  if (topk_w_out && pk && cudaMemcpyAsync(topk_w_out, w, pk * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  return FP4MOE_OK;
}
}  // namespace

}  // namespace fp4moe

using namespace fp4moe;

extern "C" {

int32_t fp4moe_abi_version(void) { return 105; }

const char* fp4moe_status_string(fp4moe_status s) {
  switch (s) {
    case FP4MOE_OK: return "FP4MOE_OK";
    case FP4MOE_INVALID_ARG: return "FP4MOE_INVALID_ARG";
    case FP4MOE_MISALIGNED: return "FP4MOE_MISALIGNED";
    case FP4MOE_CAPACITY: return "FP4MOE_CAPACITY";
    case FP4MOE_UNSUPPORTED: return "FP4MOE_UNSUPPORTED";
    case FP4MOE_CUDA_ERROR: return "FP4MOE_CUDA_ERROR";
  }
  return "FP4MOE_UNKNOWN";
}

size_t fp4moe_capacity_rows(const fp4moe_config* cfg, int32_t T) {
  if (check_cfg(cfg) != FP4MOE_OK || T < 0) return 0;
  return capacity_rows(*cfg, T);
}

size_t fp4moe_workspace_bytes(const fp4moe_config* cfg) {
  if (check_cfg(cfg) != FP4MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

fp4moe_status fp4moe_weight_bytes(const fp4moe_config* cfg, size_t* w1_codes, size_t* w1_sf, size_t* w2_codes,
                                  size_t* w2_sf) {
  FP4_TRY(check_cfg(cfg));
  const size_t E = local_experts(*cfg), H = cfg->hidden, I = cfg->inter;
  if (is_mx(cfg)) {  // atom-tiled: two codes per byte, one E8M0 byte per 32 elements
    if (w1_codes) *w1_codes = E * 2 * I * H / 2;
    if (w1_sf) *w1_sf = E * 2 * I * H / 32;
    if (w2_codes) *w2_codes = E * H * I / 2;
    if (w2_sf) *w2_sf = E * H * I / 32;
    return FP4MOE_OK;
  }
  if (w1_codes) *w1_codes = E * tiled_weight_bytes(2 * cfg->inter, cfg->hidden);
  if (w1_sf) *w1_sf = E * 2 * I * H / 16;
  if (w2_codes) *w2_codes = E * tiled_weight_bytes(cfg->hidden, cfg->inter);
  if (w2_sf) *w2_sf = E * H * I / 16;
  return FP4MOE_OK;
}

fp4moe_status moe_route(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                        const float* router_bias, float* logits_out, int32_t* topk_ids, float* topk_w,
                        int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* slot_of_pair,
                        int32_t* pair_of_row, void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  FP4_TRY(check_ptrs(x, router_w, topk_ids, topk_w, counts, offsets, padded_offsets, slot_of_pair, pair_of_row, ws));
  FP4_TRY(check_opt(router_bias));
  FP4_TRY(check_opt(logits_out));
  const WsLayout L = ws_layout(*cfg);
  float* logits = logits_out ? logits_out : at<float>(ws, L.logits);
  return route_launch(*cfg, T, x, router_w, router_bias, logits, topk_ids, topk_w, counts, offsets, padded_offsets,
                      slot_of_pair, pair_of_row, at<int32_t>(ws, L.hist), at<float>(ws, L.nw2),
                      at<float>(ws, L.rt_part), router_partial_bytes(*cfg), err_word(ws), (cudaStream_t)stream);
}

fp4moe_status moe_route_noalloc(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                                const float* router_bias, float* logits_out, int32_t* topk_ids, float* topk_w,
                                int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* slot_of_pair,
                                int32_t* pair_of_row, uint32_t* err, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (T > FP4MOE_NOALLOC_MAX_TOKENS || cfg->num_experts > FP4MOE_NOALLOC_MAX_EXPERTS) return FP4MOE_CAPACITY;
  FP4_TRY(check_ptrs(x, router_w, logits_out, topk_ids, topk_w, counts, offsets, padded_offsets, slot_of_pair,
                     pair_of_row));
  FP4_TRY(check_opt(router_bias));
  if ((reinterpret_cast<uintptr_t>(err) & 3u) != 0) return FP4MOE_MISALIGNED;
  uint8_t* s = nullptr;
  FP4_TRY(route_scratch(&s));
  const cudaStream_t st = (cudaStream_t)stream;
  // the scratch error word starts at zero
  if (cudaMemsetAsync(s + kScratchErr, 0, 4, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  return route_launch(*cfg, T, x, router_w, router_bias, logits_out, topk_ids, topk_w, counts, offsets,
                      padded_offsets, slot_of_pair, pair_of_row, reinterpret_cast<int32_t*>(s + kScratchHist),
                      reinterpret_cast<float*>(s + kScratchNw2), reinterpret_cast<float*>(s + kScratchPart),
                      kScratchPartBytes,
                      err != nullptr ? err : reinterpret_cast<uint32_t*>(s + kScratchErr), st);
}

fp4moe_status moe_quantize_scatter(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const float* gs1,
                                   const int32_t* slot_of_pair, uint8_t* a1_fp4, uint8_t* a1_sf, void* ws,
                                   fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (is_mx(cfg)) {  // bf16 rows into slot order; gs1 and a1_sf are unused
    FP4_TRY(check_ptrs(x, slot_of_pair, a1_fp4, ws));
    return scatter_rows_bf16_launch(*cfg, T, x, slot_of_pair, reinterpret_cast<uint16_t*>(a1_fp4),
                                    (cudaStream_t)stream);
  }
  FP4_TRY(check_ptrs(x, gs1, slot_of_pair, a1_fp4, a1_sf, ws));
  return quant_scatter_launch(*cfg, T, x, gs1, slot_of_pair, a1_fp4, a1_sf, scale_flags(ws), err_word(ws),
                              (cudaStream_t)stream);
}

fp4moe_status moe_grouped_gemm_w1_swiglu(const fp4moe_config* cfg, int32_t T, const uint8_t* a1_fp4,
                                         const uint8_t* a1_sf, const int32_t* padded_offsets,
                                         const int32_t* pair_of_row, const uint8_t* w1_fp4, const uint8_t* w1_sf,
                                         const float* alpha1, const float* gs2, uint8_t* a2_fp4, uint8_t* a2_sf,
                                         void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (is_mx(cfg)) {  // bf16 slot rows in and out; a1_sf, alpha1, gs2 and a2_sf are unused
    FP4_TRY(check_ptrs(a1_fp4, padded_offsets, pair_of_row, w1_fp4, w1_sf, a2_fp4, ws));
    return mx_gemm_launch(false, *cfg, T, reinterpret_cast<const uint16_t*>(a1_fp4), padded_offsets, pair_of_row,
                          w1_fp4, w1_sf, reinterpret_cast<uint16_t*>(a2_fp4), nullptr, err_word(ws),
                          (cudaStream_t)stream);
  }
  FP4_TRY(check_ptrs(a1_fp4, a1_sf, padded_offsets, pair_of_row, w1_fp4, w1_sf, alpha1, gs2, a2_fp4, a2_sf, ws));
  return gemm_launch(kW1SwiGLU, *cfg, T, a1_fp4, a1_sf, padded_offsets, pair_of_row, w1_fp4, w1_sf, alpha1, gs2,
                     a2_fp4, a2_sf, amax_h_run(ws), scale_flags(ws), nullptr, err_word(ws), at<int>(ws, kWsSchedW1),
                     (cudaStream_t)stream);
}

fp4moe_status moe_grouped_gemm_w2(const fp4moe_config* cfg, int32_t T, const uint8_t* a2_fp4, const uint8_t* a2_sf,
                                  const int32_t* padded_offsets, const int32_t* pair_of_row, const uint8_t* w2_fp4,
                                  const uint8_t* w2_sf, const float* alpha2, uint16_t* o_pairs, void* ws,
                                  fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (is_mx(cfg)) {
    FP4_TRY(check_ptrs(a2_fp4, padded_offsets, pair_of_row, w2_fp4, w2_sf, o_pairs, ws));
    return mx_gemm_launch(true, *cfg, T, reinterpret_cast<const uint16_t*>(a2_fp4), padded_offsets, pair_of_row,
                          w2_fp4, w2_sf, nullptr, o_pairs, err_word(ws), (cudaStream_t)stream);
  }
  FP4_TRY(check_ptrs(a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, o_pairs, ws));
  return gemm_launch(kW2Rows, *cfg, T, a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, nullptr,
                     nullptr, nullptr, nullptr, nullptr, o_pairs, err_word(ws), at<int>(ws, kWsSchedW2),
                     (cudaStream_t)stream);
}

fp4moe_status moe_combine(const fp4moe_config* cfg, int32_t T, const uint16_t* o_pairs, const float* topk_w,
                          uint16_t* y, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  FP4_TRY(check_ptrs(o_pairs, topk_w, y));
  if (cfg->ep_count > 0) return FP4MOE_UNSUPPORTED;  // the pairs held elsewhere are known only to moe_forward
  return combine_launch(*cfg, T, o_pairs, topk_w, nullptr, nullptr, y, (cudaStream_t)stream);
}

fp4moe_status moe_grouped_gemm_w2_combine(const fp4moe_config* cfg, int32_t T, const uint8_t* a2_fp4,
                                          const uint8_t* a2_sf, const int32_t* padded_offsets,
                                          const int32_t* pair_of_row, const uint8_t* w2_fp4, const uint8_t* w2_sf,
                                          const float* alpha2, const float* topk_w, uint16_t* y, void* ws,
                                          fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (cfg->ep_count > 0) return FP4MOE_UNSUPPORTED;  // the pairs held elsewhere are known only to moe_forward
  const WsLayout L = ws_layout(*cfg);
  uint16_t* o = at<uint16_t>(ws, L.opairs);
  if (is_mx(cfg)) {
    FP4_TRY(check_ptrs(a2_fp4, padded_offsets, pair_of_row, w2_fp4, w2_sf, topk_w, y, ws));
    FP4_TRY(mx_gemm_launch(true, *cfg, T, reinterpret_cast<const uint16_t*>(a2_fp4), padded_offsets, pair_of_row,
                           w2_fp4, w2_sf, nullptr, o, err_word(ws), (cudaStream_t)stream));
    return combine_launch(*cfg, T, o, topk_w, nullptr, nullptr, y, (cudaStream_t)stream);
  }
  FP4_TRY(check_ptrs(a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, topk_w, y, ws));
  FP4_TRY(gemm_launch(kW2Rows, *cfg, T, a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, nullptr,
                      nullptr, nullptr, nullptr, nullptr, o, err_word(ws), at<int>(ws, kWsSchedW2),
                      (cudaStream_t)stream));
  return combine_launch(*cfg, T, o, topk_w, nullptr, nullptr, y, (cudaStream_t)stream);
}


fp4moe_status moe_forward(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                          const float* router_bias, const float* gs1, const float* gs2, const uint8_t* w1_fp4,
                          const uint8_t* w1_sf, const float* alpha1, const uint8_t* w2_fp4, const uint8_t* w2_sf,
                          const float* alpha2, uint16_t* y, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                          fp4moe_stream_t stream) {
  return forward_impl(cfg, T, x, router_w, router_bias, gs1, gs2, w1_fp4, w1_sf, alpha1, w2_fp4, w2_sf, alpha2,
                      nullptr, y, topk_ids_out, topk_w_out, ws, stream);
}

fp4moe_status moe_forward_shared(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const uint16_t* router_w,
                                 const float* router_bias, const float* gs1, const float* gs2, const uint8_t* w1_fp4,
                                 const uint8_t* w1_sf, const float* alpha1, const uint8_t* w2_fp4,
                                 const uint8_t* w2_sf, const float* alpha2, const fp4moe_shared_weights* se,
                                 uint16_t* y, int32_t* topk_ids_out, float* topk_w_out, void* ws,
                                 fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_shared(cfg, se));
  return forward_impl(cfg, T, x, router_w, router_bias, gs1, gs2, w1_fp4, w1_sf, alpha1, w2_fp4, w2_sf, alpha2, se,
                      y, topk_ids_out, topk_w_out, ws, stream);
}

fp4moe_status moe_shared_expert(const fp4moe_config* cfg, int32_t T, const uint16_t* x,
                                const fp4moe_shared_weights* se, float* o_shared, void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  FP4_TRY(check_shared(cfg, se));
  FP4_TRY(check_ptrs(x, o_shared, ws));
  return shared_launch(*cfg, T, x, *se, o_shared, ws, (cudaStream_t)stream);
}

fp4moe_status moe_combine_shared(const fp4moe_config* cfg, int32_t T, const uint16_t* o_pairs, const float* topk_w,
                                 const int32_t* slot_of_pair, const float* o_shared, uint16_t* y,
                                 fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  FP4_TRY(check_ptrs(o_pairs, topk_w, y));
  FP4_TRY(check_opt(slot_of_pair));
  FP4_TRY(check_opt(o_shared));
  if (cfg->ep_count > 0 && slot_of_pair == nullptr) return FP4MOE_INVALID_ARG;  // which pairs are held here
  return combine_launch(*cfg, T, o_pairs, topk_w, slot_of_pair, o_shared, y, (cudaStream_t)stream);
}

fp4moe_status fp4moe_shared_weight_bytes(const fp4moe_config* cfg, size_t* w1, size_t* w1_scales, size_t* w2,
                                         size_t* w2_scales) {
  FP4_TRY(check_cfg(cfg));
  if (cfg->shared_inter <= 0) return FP4MOE_INVALID_ARG;
  const size_t H = cfg->hidden, Is = cfg->shared_inter;
  if (w1) *w1 = 2 * Is * H;
  if (w1_scales) *w1_scales = (2 * Is / 128) * (H / 128) * 4;
  if (w2) *w2 = H * Is;
  if (w2_scales) *w2_scales = (H / 128) * (Is / 128) * 4;
  return FP4MOE_OK;
}

fp4moe_status fp4moe_shared_quantize_weights(const fp4moe_config* cfg, int32_t which, const float* w,
                                             uint8_t* codes_out, float* scales_out, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  if (cfg->shared_inter <= 0 || (which != 1 && which != 2)) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(w, codes_out, scales_out));
  return se_quant_weights_launch(*cfg, which, w, codes_out, scales_out, (cudaStream_t)stream);
}


fp4moe_status fp4moe_quantize_weights(const fp4moe_config* cfg, int32_t which, int32_t n_experts, const float* w,
                                      uint8_t* codes_out, uint8_t* sf_out, float* gs_out, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  if (which != 1 && which != 2) return FP4MOE_INVALID_ARG;
  if (n_experts < 0 || n_experts > local_experts(*cfg)) return FP4MOE_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  const int32_t rows = which == 1 ? 2 * cfg->inter : cfg->hidden;
  const int32_t K = which == 1 ? cfg->hidden : cfg->inter;
  if (is_mx(cfg)) {  // OCP MX scales per 32 elements; no global scale (gs_out is unused)
    FP4_TRY(check_ptrs(w, codes_out, sf_out));
    return mx_quant_rows_launch((int64_t)n_experts * rows, K, rows, which == 1 ? cfg->inter : 0, w, codes_out,
                                sf_out, st);
  }
  FP4_TRY(check_ptrs(w, codes_out, sf_out, gs_out));
  FP4_TRY(amax_f32_launch(n_experts, (int64_t)rows * K, w, gs_out, st));
  FP4_TRY(gs_from_amax_launch(n_experts, gs_out, st));
  if (K % 256 != 0 &&  // the last k-stage of every block is padded with zero codes
      cudaMemsetAsync(codes_out, 0, (size_t)n_experts * tiled_weight_bytes(rows, K), st) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  return quant_rows_launch((int64_t)n_experts * rows, K, rows, which == 1 ? cfg->inter : 0, 1, w, gs_out, rows,
                           codes_out, sf_out, st);
}

fp4moe_status fp4moe_tp_shard_units(int32_t width, int32_t tp, int32_t align, int32_t kernel_align, int32_t rank,
                                    int32_t unit, int32_t* src_offset, int32_t* count, int32_t* zero_tail) {
  if (width <= 0 || tp <= 0 || align <= 0 || kernel_align <= 0 || unit <= 0 || rank < 0 || rank >= tp)
    return FP4MOE_INVALID_ARG;
  int64_t local = 0, kernel = 0;
  tp_widths(width, tp, align, kernel_align, local, kernel);
  const int64_t start = (int64_t)rank * local;
  const int64_t n = std::max<int64_t>(0, std::min<int64_t>(local, (int64_t)width - start));
  // a slice that splits a storage unit cannot be cut in that unit
  if (start % unit != 0 || n % unit != 0 || kernel % unit != 0 || kernel > INT32_MAX) return FP4MOE_UNSUPPORTED;
  if (src_offset) *src_offset = (int32_t)(start / unit);
  if (count) *count = (int32_t)(n / unit);
  if (zero_tail) *zero_tail = (int32_t)((kernel - n) / unit);
  return FP4MOE_OK;
}

fp4moe_status fp4moe_shard_mxfp4(const fp4moe_config* cfg, int32_t which, int32_t n_experts, int32_t full_inter,
                                 int32_t tp, int32_t tp_rank, const uint8_t* ck_codes, const uint8_t* ck_sf,
                                 uint8_t* codes_out, uint8_t* sf_out, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  if (!is_mx(cfg)) return FP4MOE_UNSUPPORTED;
  if (which != 1 && which != 2) return FP4MOE_INVALID_ARG;
  if (n_experts < 0 || n_experts > local_experts(*cfg)) return FP4MOE_INVALID_ARG;
  if (full_inter <= 0 || full_inter % 32 != 0) return FP4MOE_UNSUPPORTED;  // whole E8M0 groups, whole bytes
  int32_t first = 0, count = 0, tail = 0;
  FP4_TRY(fp4moe_tp_shard_units(full_inter, tp, 32, 128, tp_rank, 1, &first, &count, &tail));
  // the plan's widths must be the layer's: the logical width per rank, and the kernel width it rounds up to
  int64_t local = 0, kernel = 0;
  tp_widths(full_inter, tp, 32, 128, local, kernel);
  if (kernel != cfg->inter || local != cfg->inter_logical) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(ck_codes, ck_sf, codes_out, sf_out));
  const bool w1 = which == 1;
  const int32_t rows = w1 ? 2 * cfg->inter : cfg->hidden;
  const int32_t Kd = w1 ? cfg->hidden : cfg->inter;
  return mx_shard_launch(n_experts, w1, rows, Kd, cfg->inter, full_inter, w1 ? cfg->hidden : full_inter, first, count,
                         ck_codes, ck_sf, codes_out, sf_out, (cudaStream_t)stream);
}

fp4moe_status fp4moe_mxfp4_as_nvfp4(const fp4moe_config* cfg, int32_t which, int32_t n_experts, const uint8_t* mx_codes,
                                   const uint8_t* mx_sf, uint8_t* codes_out, uint8_t* sf_out, float* gw_out,
                                   uint32_t* err, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  if (is_mx(cfg)) return FP4MOE_UNSUPPORTED;  // the target is an NVFP4 layer
  if (which != 1 && which != 2) return FP4MOE_INVALID_ARG;
  if (n_experts < 0 || n_experts > local_experts(*cfg)) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(mx_codes, mx_sf, codes_out, sf_out, gw_out, err));
  const int32_t rows = which == 1 ? 2 * cfg->inter : cfg->hidden;
  const int32_t K = which == 1 ? cfg->hidden : cfg->inter;
  return mx_as_nvfp4_launch(n_experts, rows, K, mx_codes, mx_sf, codes_out, sf_out, gw_out, err,
                            (cudaStream_t)stream);
}

fp4moe_status fp4moe_make_alpha(int32_t n, const float* gs_act, const float* gs_w, float* alpha,
                                fp4moe_stream_t stream) {
  if (n < 0) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(gs_act, gs_w, alpha));
  return make_alpha_launch(n, gs_act, gs_w, alpha, (cudaStream_t)stream);
}

fp4moe_status fp4moe_calibrate(const fp4moe_config* cfg, int32_t T, const uint16_t* x_warm, const uint16_t* router_w,
                               const float* router_bias, const uint8_t* w1_fp4, const uint8_t* w1_sf,
                               const float* gw1, float* gs1_out, float* gs2_out, void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (is_mx(cfg)) return FP4MOE_UNSUPPORTED;  // MXFP4 layers keep bf16 activations: no global scales
  FP4_TRY(check_ptrs(x_warm, router_w, w1_fp4, w1_sf, gw1, gs1_out, gs2_out, ws));
  FP4_TRY(check_opt(router_bias));
  const cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*cfg);
  uint32_t* err = err_word(ws);
  float* amax_x = at<float>(ws, kWsAmaxX);
  float* amax_h = at<float>(ws, kWsAmaxH);
  int32_t* poff = at<int32_t>(ws, L.poff);
  int32_t* por = at<int32_t>(ws, L.por);
  FP4_TRY(amax_bf16_launch((int64_t)T * cfg->hidden, x_warm, amax_x, st));
  if (cudaMemcpyAsync(gs1_out, amax_x, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  FP4_TRY(gs_from_amax_launch(1, gs1_out, st));
  FP4_TRY(route_launch(*cfg, T, x_warm, router_w, router_bias, at<float>(ws, L.logits), at<int32_t>(ws, L.ids),
                       at<float>(ws, L.w), at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets), poff,
                       at<int32_t>(ws, L.slot), por, at<int32_t>(ws, L.hist), at<float>(ws, L.nw2),
                       at<float>(ws, L.rt_part), router_partial_bytes(*cfg), err, st));
  FP4_TRY(quant_scatter_launch(*cfg, T, x_warm, gs1_out, at<int32_t>(ws, L.slot), at<uint8_t>(ws, L.a1),
                               at<uint8_t>(ws, L.a1sf), scale_flags(ws), err, st));
  float* alpha = at<float>(ws, L.alpha_tmp);
  FP4_TRY(make_alpha_launch(local_experts(*cfg), gs1_out, gw1, alpha, st));
  if (cudaMemsetAsync(amax_h, 0, 4, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  FP4_TRY(gemm_launch(kW1Amax, *cfg, T, at<uint8_t>(ws, L.a1), at<uint8_t>(ws, L.a1sf), poff, por, w1_fp4, w1_sf,
                      alpha, nullptr, nullptr, nullptr, amax_h, nullptr, nullptr, err, at<int>(ws, kWsSchedW1), st));
  if (cudaMemcpyAsync(gs2_out, amax_h, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  return gs_from_amax_launch(1, gs2_out, st);
}

fp4moe_status fp4moe_batch_gs1(const fp4moe_config* cfg, int32_t T, const uint16_t* x, const float* gw1,
                               float* gs1_out, float* alpha1_out, void* ws, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  FP4_TRY(check_T(cfg, T));
  if (is_mx(cfg)) return FP4MOE_UNSUPPORTED;  // MXFP4 layers keep bf16 activations: no global scales
  FP4_TRY(check_ptrs(x, gw1, gs1_out, alpha1_out, ws));
  return batch_gs1_launch(T, cfg->hidden, x, local_experts(*cfg), gw1, gs1_out, alpha1_out,
                          at<unsigned int>(ws, kWsBatchAmax), at<unsigned int>(ws, kWsBatchDone),
                          (cudaStream_t)stream);
}

fp4moe_status fp4moe_quantize_rows_f32(int32_t rows, int32_t K, const float* in, const float* g, uint8_t* codes,
                                       uint8_t* sf, fp4moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 64 != 0 || rows % 128 != 0) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(in, g, codes, sf));
  return quant_rows_launch(rows, K, rows > 0 ? rows : 1, 0, 0, in, g, 1, codes, sf, (cudaStream_t)stream);
}

fp4moe_status fp4moe_tensor_peak_probe(int32_t n, int32_t iters, uint32_t* err, fp4moe_stream_t stream) {
  if ((n != 128 && n != 256) || iters < 1 || iters > (1 << 22)) return FP4MOE_INVALID_ARG;
  FP4_TRY(check_ptrs(err));
  return tensor_peak_launch(n, iters, err, (cudaStream_t)stream);
}

fp4moe_status fp4moe_selftest_wait_timeout(uint32_t* err, int64_t limit_ns, uint32_t* result, fp4moe_stream_t stream) {
  if (err == nullptr || result == nullptr) return FP4MOE_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(err) | reinterpret_cast<uintptr_t>(result)) & 3u) != 0) return FP4MOE_MISALIGNED;
  if (limit_ns < 1000000 || limit_ns > 50000000) return FP4MOE_INVALID_ARG;
  return selftest_wait_launch(err, limit_ns, result, (cudaStream_t)stream);
}

fp4moe_status fp4moe_read_error(void* ws, uint32_t* err_host, int32_t clear, fp4moe_stream_t stream) {
  if (ws == nullptr || err_host == nullptr) return FP4MOE_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(err_host, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  if (clear) {
    if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  }
  return FP4MOE_OK;
}

fp4moe_status fp4moe_read_scale_status(void* ws, uint32_t* flags_host, float* amax_h_host, int32_t clear,
                                       fp4moe_stream_t stream) {
  if (ws == nullptr || flags_host == nullptr) return FP4MOE_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  uint32_t words[2] = {0u, 0u};  // the flags word and the running amax|h|, adjacent in the header
  static_assert(kWsAmaxHRun == kWsScaleFlags + 4, "scale words are adjacent");
  if (cudaMemcpyAsync(words, at<uint8_t>(ws, kWsScaleFlags), 8, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FP4MOE_CUDA_ERROR;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  *flags_host = words[0];
  if (amax_h_host != nullptr) memcpy(amax_h_host, &words[1], 4);
  if (clear) {
    if (cudaMemsetAsync(at<uint8_t>(ws, kWsScaleFlags), 0, 4, st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FP4MOE_CUDA_ERROR;
  }
  return FP4MOE_OK;
}

fp4moe_status fp4moe_refresh_gs2(const fp4moe_config* cfg, void* ws, const float* gw2, float* gs2_inout,
                                 float* alpha2_out, fp4moe_stream_t stream) {
  FP4_TRY(check_cfg(cfg));
  if (is_mx(cfg)) return FP4MOE_UNSUPPORTED;  // MXFP4 layers keep bf16 activations: no global scales
  FP4_TRY(check_ptrs(ws, gw2, gs2_inout, alpha2_out));
  return refresh_gs2_launch(local_experts(*cfg), amax_h_run(ws), gw2, gs2_inout, alpha2_out, (cudaStream_t)stream);
}

}  // extern "C"
