"""Python binding of the fp4moe C ABI: torch tensors in, C calls out.

Each function has the name of its C entry point and only marshals arguments:
it takes the device pointers of contiguous CUDA tensors and the current
stream, calls the library and raises Fp4MoeError on a non-OK status. All the
layer's arithmetic runs in the CUDA kernels of libfp4moe.so.

``MoELayer`` is a convenience owner of the buffers (allocated through torch)
for one configuration. It also runs the load-time prep: weight quantisation,
calibration and alpha tables.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import Config


class Fp4MoeError(RuntimeError):
    pass


def config(hidden: int, inter: int, num_experts: int, top_k: int, max_tokens: int, swiglu_limit: float,
           inter_logical: int = 0, w_format: int = _lib.W_NVFP4, ep_first: int = 0, ep_count: int = 0,
           shared_inter: int = 0) -> Config:
    """Layer configuration. ep_count > 0 makes the layer hold experts [ep_first, ep_first + ep_count) only;
    shared_inter > 0 gives it a block-FP8 shared expert of that (kernel-local) intermediate width."""
    return Config(hidden, inter, inter_logical or inter, num_experts, top_k, max_tokens, swiglu_limit, w_format,
                  ep_first, ep_count, shared_inter)


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise Fp4MoeError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != _lib.OK:
        name = _lib.load().fp4moe_status_string(rc).decode()
        raise Fp4MoeError(f"{what}: {name}")


def capacity_rows(cfg: Config, T: int) -> int:
    return _lib.load().fp4moe_capacity_rows(ctypes.byref(cfg), T)


def workspace_bytes(cfg: Config) -> int:
    return _lib.load().fp4moe_workspace_bytes(ctypes.byref(cfg))


def weight_bytes(cfg: Config):
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(_lib.load().fp4moe_weight_bytes(ctypes.byref(cfg), *[ctypes.byref(x) for x in v]), "fp4moe_weight_bytes")
    return tuple(x.value for x in v)


def moe_route(cfg, T, x, router_w, router_bias, logits_out, topk_ids, topk_w, counts, offsets, padded_offsets,
              slot_of_pair, pair_of_row, ws, stream=None):
    _check(_lib.load().moe_route(ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias), _p(logits_out),
                                 _p(topk_ids), _p(topk_w), _p(counts), _p(offsets), _p(padded_offsets),
                                 _p(slot_of_pair), _p(pair_of_row), _p(ws), _s(stream)), "moe_route")


def moe_route_noalloc(cfg, T, x, router_w, router_bias, logits_out, topk_ids, topk_w, counts, offsets,
                      padded_offsets, slot_of_pair, pair_of_row, err=None, stream=None):
    """moe_route without a workspace: for callers that must not allocate device
    memory. The library's own fixed scratch stands in for the workspace, so
    calls on one device must not overlap (see include/fp4moe.h)."""
    _check(_lib.load().moe_route_noalloc(ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias),
                                         _p(logits_out), _p(topk_ids), _p(topk_w), _p(counts), _p(offsets),
                                         _p(padded_offsets), _p(slot_of_pair), _p(pair_of_row), _p(err),
                                         _s(stream)), "moe_route_noalloc")


def moe_quantize_scatter(cfg, T, x, gs1, slot_of_pair, a1_fp4, a1_sf, ws, stream=None):
    _check(_lib.load().moe_quantize_scatter(ctypes.byref(cfg), T, _p(x), _p(gs1), _p(slot_of_pair), _p(a1_fp4),
                                            _p(a1_sf), _p(ws), _s(stream)), "moe_quantize_scatter")


def moe_grouped_gemm_w1_swiglu(cfg, T, a1_fp4, a1_sf, padded_offsets, pair_of_row, w1_fp4, w1_sf, alpha1, gs2,
                               a2_fp4, a2_sf, ws, stream=None):
    _check(_lib.load().moe_grouped_gemm_w1_swiglu(ctypes.byref(cfg), T, _p(a1_fp4), _p(a1_sf), _p(padded_offsets),
                                                  _p(pair_of_row), _p(w1_fp4), _p(w1_sf), _p(alpha1), _p(gs2),
                                                  _p(a2_fp4), _p(a2_sf), _p(ws), _s(stream)),
           "moe_grouped_gemm_w1_swiglu")


def moe_grouped_gemm_w2(cfg, T, a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, o_pairs, ws,
                        stream=None):
    _check(_lib.load().moe_grouped_gemm_w2(ctypes.byref(cfg), T, _p(a2_fp4), _p(a2_sf), _p(padded_offsets),
                                           _p(pair_of_row), _p(w2_fp4), _p(w2_sf), _p(alpha2), _p(o_pairs), _p(ws),
                                           _s(stream)), "moe_grouped_gemm_w2")


def moe_combine(cfg, T, o_pairs, topk_w, y, stream=None):
    _check(_lib.load().moe_combine(ctypes.byref(cfg), T, _p(o_pairs), _p(topk_w), _p(y), _s(stream)), "moe_combine")


def moe_grouped_gemm_w2_combine(cfg, T, a2_fp4, a2_sf, padded_offsets, pair_of_row, w2_fp4, w2_sf, alpha2, topk_w,
                                y, ws, stream=None):
    _check(_lib.load().moe_grouped_gemm_w2_combine(ctypes.byref(cfg), T, _p(a2_fp4), _p(a2_sf), _p(padded_offsets),
                                                   _p(pair_of_row), _p(w2_fp4), _p(w2_sf), _p(alpha2), _p(topk_w),
                                                   _p(y), _p(ws), _s(stream)), "moe_grouped_gemm_w2_combine")


def moe_forward(cfg, T, x, router_w, router_bias, gs1, gs2, w1_fp4, w1_sf, alpha1, w2_fp4, w2_sf, alpha2, y,
                topk_ids_out, topk_w_out, ws, stream=None):
    _check(_lib.load().moe_forward(ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias), _p(gs1), _p(gs2),
                                   _p(w1_fp4), _p(w1_sf), _p(alpha1), _p(w2_fp4), _p(w2_sf), _p(alpha2), _p(y),
                                   _p(topk_ids_out), _p(topk_w_out), _p(ws), _s(stream)), "moe_forward")


def fp4moe_quantize_weights(cfg, which, n_experts, w, codes_out, sf_out, gs_out, stream=None):
    _check(_lib.load().fp4moe_quantize_weights(ctypes.byref(cfg), which, n_experts, _p(w), _p(codes_out),
                                               _p(sf_out), _p(gs_out), _s(stream)), "fp4moe_quantize_weights")


def fp4moe_mxfp4_as_nvfp4(cfg, which, n_experts, mx_codes, mx_sf, codes_out, sf_out, gw_out, err, stream=None):
    _check(_lib.load().fp4moe_mxfp4_as_nvfp4(ctypes.byref(cfg), which, n_experts, _p(mx_codes), _p(mx_sf),
                                             _p(codes_out), _p(sf_out), _p(gw_out), _p(err), _s(stream)),
           "fp4moe_mxfp4_as_nvfp4")


def fp4moe_tp_shard_units(width, tp, align, kernel_align, rank, unit):
    """(source offset, units copied, zero tail) of one rank's slice, in storage units (host arithmetic)."""
    out = [ctypes.c_int32() for _ in range(3)]
    _check(_lib.load().fp4moe_tp_shard_units(width, tp, align, kernel_align, rank, unit,
                                             *[ctypes.byref(v) for v in out]), "fp4moe_tp_shard_units")
    return tuple(v.value for v in out)


def fp4moe_shard_mxfp4(cfg, which, n_experts, full_inter, tp, tp_rank, ck_codes, ck_sf, codes_out, sf_out,
                       stream=None):
    _check(_lib.load().fp4moe_shard_mxfp4(ctypes.byref(cfg), which, n_experts, full_inter, tp, tp_rank, _p(ck_codes),
                                          _p(ck_sf), _p(codes_out), _p(sf_out), _s(stream)), "fp4moe_shard_mxfp4")


def fp4moe_make_alpha(n, gs_act, gs_w, alpha, stream=None):
    _check(_lib.load().fp4moe_make_alpha(n, _p(gs_act), _p(gs_w), _p(alpha), _s(stream)), "fp4moe_make_alpha")


def fp4moe_calibrate(cfg, T, x_warm, router_w, router_bias, w1_fp4, w1_sf, gw1, gs1_out, gs2_out, ws, stream=None):
    _check(_lib.load().fp4moe_calibrate(ctypes.byref(cfg), T, _p(x_warm), _p(router_w), _p(router_bias), _p(w1_fp4),
                                        _p(w1_sf), _p(gw1), _p(gs1_out), _p(gs2_out), _p(ws), _s(stream)),
           "fp4moe_calibrate")


def fp4moe_batch_gs1(cfg, T, x, gw1, gs1_out, alpha1_out, ws, stream=None):
    _check(_lib.load().fp4moe_batch_gs1(ctypes.byref(cfg), T, _p(x), _p(gw1), _p(gs1_out), _p(alpha1_out), _p(ws),
                                        _s(stream)), "fp4moe_batch_gs1")


def fp4moe_quantize_rows_f32(rows, K, inp, g, codes, sf, stream=None):
    _check(_lib.load().fp4moe_quantize_rows_f32(rows, K, _p(inp), _p(g), _p(codes), _p(sf), _s(stream)),
           "fp4moe_quantize_rows_f32")


def fp4moe_tensor_peak_probe(n, iters, err, stream=None):
    """Launch the dense FP4 tensor-core rate probe (see include/fp4moe.h); the caller times it."""
    _check(_lib.load().fp4moe_tensor_peak_probe(n, iters, _p(err), _s(stream)), "fp4moe_tensor_peak_probe")


def fp4moe_selftest_wait_timeout(err, limit_ns, result, stream=None):
    """One bounded wait that runs out on purpose (a test of the failure path; see include/fp4moe.h)."""
    _check(_lib.load().fp4moe_selftest_wait_timeout(_p(err), int(limit_ns), _p(result), _s(stream)),
           "fp4moe_selftest_wait_timeout")


def _sw(se):
    """fp4moe_shared_weights from a SharedWeights holder (device pointers of its four tensors)."""
    return ctypes.byref(_lib.SharedWeights(_p(se.w1), _p(se.w1_scales), _p(se.w2), _p(se.w2_scales)))


def shared_weight_bytes(cfg: Config):
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(_lib.load().fp4moe_shared_weight_bytes(ctypes.byref(cfg), *[ctypes.byref(x) for x in v]),
           "fp4moe_shared_weight_bytes")
    return tuple(x.value for x in v)


def fp4moe_shared_quantize_weights(cfg, which, w, codes_out, scales_out, stream=None):
    _check(_lib.load().fp4moe_shared_quantize_weights(ctypes.byref(cfg), which, _p(w), _p(codes_out),
                                                      _p(scales_out), _s(stream)), "fp4moe_shared_quantize_weights")


def moe_shared_expert(cfg, T, x, se, o_shared, ws, stream=None):
    _check(_lib.load().moe_shared_expert(ctypes.byref(cfg), T, _p(x), _sw(se), _p(o_shared), _p(ws), _s(stream)),
           "moe_shared_expert")


def moe_combine_shared(cfg, T, o_pairs, topk_w, slot_of_pair, o_shared, y, stream=None):
    _check(_lib.load().moe_combine_shared(ctypes.byref(cfg), T, _p(o_pairs), _p(topk_w), _p(slot_of_pair),
                                          _p(o_shared), _p(y), _s(stream)), "moe_combine_shared")


def moe_forward_shared(cfg, T, x, router_w, router_bias, gs1, gs2, w1_fp4, w1_sf, alpha1, w2_fp4, w2_sf, alpha2, se,
                       y, topk_ids_out, topk_w_out, ws, stream=None):
    _check(_lib.load().moe_forward_shared(ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias), _p(gs1),
                                          _p(gs2), _p(w1_fp4), _p(w1_sf), _p(alpha1), _p(w2_fp4), _p(w2_sf),
                                          _p(alpha2), _sw(se), _p(y), _p(topk_ids_out), _p(topk_w_out), _p(ws),
                                          _s(stream)), "moe_forward_shared")


def fp4moe_read_error(ws, clear=True, stream=None) -> int:
    v = ctypes.c_uint32()
    _check(_lib.load().fp4moe_read_error(_p(ws), ctypes.byref(v), 1 if clear else 0, _s(stream)), "fp4moe_read_error")
    return v.value


def fp4moe_read_scale_status(ws, clear=True, stream=None):
    """(FP4MOE_SAT_* flags, running amax|h| since the last gs2 refresh)."""
    v, a = ctypes.c_uint32(), ctypes.c_float()
    _check(_lib.load().fp4moe_read_scale_status(_p(ws), ctypes.byref(v), ctypes.byref(a), 1 if clear else 0,
                                                _s(stream)), "fp4moe_read_scale_status")
    return v.value, a.value


def fp4moe_refresh_gs2(cfg, ws, gw2, gs2_inout, alpha2_out, stream=None):
    _check(_lib.load().fp4moe_refresh_gs2(ctypes.byref(cfg), _p(ws), _p(gw2), _p(gs2_inout), _p(alpha2_out),
                                          _s(stream)), "fp4moe_refresh_gs2")


# --------------------------------------------------------------------------
@dataclass
class Weights:
    w1_fp4: torch.Tensor
    w1_sf: torch.Tensor
    gw1: torch.Tensor
    w2_fp4: torch.Tensor
    w2_sf: torch.Tensor
    gw2: torch.Tensor


@dataclass
class SharedWeights:
    """The shared expert's block-FP8 weights in the layout of include/fp4moe.h."""
    w1: torch.Tensor         # [2 Is][H] E4M3 bytes, kernel row order
    w1_scales: torch.Tensor  # [2 Is / 128][H / 128] fp32
    w2: torch.Tensor         # [H][Is]
    w2_scales: torch.Tensor  # [H / 128][Is / 128]


class MoELayer:
    """Owns the device buffers of one layer configuration and calls the C ABI on them."""

    def __init__(self, cfg: Config, device: str = "cuda"):
        self.cfg = cfg
        self.device = device
        E, H, I = (cfg.ep_count or cfg.num_experts), cfg.hidden, cfg.inter
        b1, s1, b2, s2 = weight_bytes(cfg)
        u8 = dict(dtype=torch.uint8, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.weights = Weights(torch.empty(b1, **u8), torch.empty(s1, **u8), torch.empty(E, **f32),
                               torch.empty(b2, **u8), torch.empty(s2, **u8), torch.empty(E, **f32))
        self.ws = torch.zeros(workspace_bytes(cfg), **u8)
        self.gs1 = torch.ones(1, **f32)
        self.gs2 = torch.ones(1, **f32)
        self.alpha1 = torch.empty(E, **f32)
        self.alpha2 = torch.empty(E, **f32)
        self.router_w = None
        self.router_bias = None
        self.shared = None
        if cfg.shared_inter > 0:
            sb = shared_weight_bytes(cfg)
            self.shared = SharedWeights(torch.empty(sb[0], **u8), torch.empty(sb[1] // 4, **f32),
                                        torch.empty(sb[2], **u8), torch.empty(sb[3] // 4, **f32))

    # ---- load-time prep
    def quantize_weights(self, which: int, e0: int, w: torch.Tensor):
        """Quantise experts [e0, e0 + w.shape[0]) of W1 (which=1, [n, 2I, H]) or W2 (which=2, [n, H, I]).

        NVFP4 layers quantise to E2M1 with E4M3 scales per 16 and a global scale per expert. MXFP4 layers
        (w_format MXFP4) quantise to E2M1 with E8M0 scales per 32; their rows are the rank's kernel-local
        shard, zero past the logical width.
        """
        cfg, W = self.cfg, self.weights
        n = w.shape[0]
        E = cfg.ep_count or cfg.num_experts
        b1, s1, b2, s2 = weight_bytes(cfg)
        if which == 1:
            per_c, per_s = b1 // E, s1 // E
            codes, sf, gs = W.w1_fp4, W.w1_sf, W.gw1
        else:
            per_c, per_s = b2 // E, s2 // E
            codes, sf, gs = W.w2_fp4, W.w2_sf, W.gw2
        fp4moe_quantize_weights(cfg, which, n, w.contiguous(), codes[e0 * per_c:(e0 + n) * per_c],
                                sf[e0 * per_s:(e0 + n) * per_s], gs[e0:e0 + n])

    def shard_mxfp4_weights(self, which: int, e0: int, ck_codes: torch.Tensor, ck_sf: torch.Tensor,
                            full_inter: int, tp: int, tp_rank: int):
        """Cut rank tp_rank's shard of experts [e0, e0 + n) from a quantised full-width MXFP4 checkpoint.

        which=1: ck_codes [n, 2 full_inter, H / 2] bytes (gate rows first), ck_sf [n, 2 full_inter, H / 32];
        which=2: ck_codes [n, H, full_inter / 2], ck_sf [n, H, full_inter / 32] (see fp4moe_shard_mxfp4).
        """
        cfg, W = self.cfg, self.weights
        n = ck_codes.shape[0]
        E = cfg.ep_count or cfg.num_experts
        b1, s1, b2, s2 = weight_bytes(cfg)
        per_c, per_s = (b1 // E, s1 // E) if which == 1 else (b2 // E, s2 // E)
        codes, sf = (W.w1_fp4, W.w1_sf) if which == 1 else (W.w2_fp4, W.w2_sf)
        fp4moe_shard_mxfp4(cfg, which, n, full_inter, tp, tp_rank, ck_codes.contiguous(), ck_sf.contiguous(),
                           codes[e0 * per_c:(e0 + n) * per_c], sf[e0 * per_s:(e0 + n) * per_s])

    def load_mxfp4_weights(self, which: int, e0: int, mx_codes: torch.Tensor, mx_sf: torch.Tensor,
                           err: torch.Tensor):
        """NVFP4 layers: take experts [e0, e0 + n) of W1 (which=1) or W2 (which=2) from MXFP4 weights in the
        atom-tiled MX layout (fp4moe_mxfp4_as_nvfp4); n follows from the buffer sizes of an MXFP4 layer of the
        same hidden and inter. err receives FP4MOE_ERR_SCALE_RANGE for a scale without an exact form."""
        cfg, W = self.cfg, self.weights
        E = cfg.ep_count or cfg.num_experts
        b1, s1, b2, s2 = weight_bytes(cfg)
        rows, K = (2 * cfg.inter, cfg.hidden) if which == 1 else (cfg.hidden, cfg.inter)
        n = mx_codes.numel() // (rows * K // 2)
        per_c, per_s = (b1 // E, s1 // E) if which == 1 else (b2 // E, s2 // E)
        codes, sf, gw = (W.w1_fp4, W.w1_sf, W.gw1) if which == 1 else (W.w2_fp4, W.w2_sf, W.gw2)
        fp4moe_mxfp4_as_nvfp4(cfg, which, n, mx_codes.contiguous(), mx_sf.contiguous(),
                              codes[e0 * per_c:(e0 + n) * per_c], sf[e0 * per_s:(e0 + n) * per_s], gw[e0:e0 + n], err)

    def quantize_shared_weights(self, which: int, w: torch.Tensor):
        """Block-FP8 of the shared expert's W1 (which=1, [2 Is, H], gate rows then up) or W2 (which=2, [H, Is])."""
        se = self.shared
        codes, scales = (se.w1, se.w1_scales) if which == 1 else (se.w2, se.w2_scales)
        fp4moe_shared_quantize_weights(self.cfg, which, w.contiguous(), codes, scales)

    def set_router(self, router_w: torch.Tensor, router_bias: torch.Tensor | None = None):
        self.router_w = router_w.contiguous()
        self.router_bias = None if router_bias is None else router_bias.contiguous()

    def calibrate(self, x_warm: torch.Tensor):
        T = x_warm.shape[0]
        W = self.weights
        fp4moe_calibrate(self.cfg, T, x_warm, self.router_w, self.router_bias, W.w1_fp4, W.w1_sf, W.gw1, self.gs1,
                         self.gs2, self.ws)
        self.update_alpha()

    def set_global_scales(self, gs1: float, gs2: float):
        self.gs1.fill_(gs1)
        self.gs2.fill_(gs2)
        self.update_alpha()

    def batch_gs1(self, x: torch.Tensor, stream=None):
        """Take gs1 (and alpha1) from this batch's own amax, on the device (see fp4moe_batch_gs1)."""
        fp4moe_batch_gs1(self.cfg, x.shape[0], x, self.weights.gw1, self.gs1, self.alpha1, self.ws, stream)

    def update_alpha(self):
        E = self.cfg.ep_count or self.cfg.num_experts
        fp4moe_make_alpha(E, self.gs1, self.weights.gw1, self.alpha1)
        fp4moe_make_alpha(E, self.gs2, self.weights.gw2, self.alpha2)

    # ---- hot path
    def forward(self, x: torch.Tensor, y: torch.Tensor, topk_ids: torch.Tensor | None = None,
                topk_w: torch.Tensor | None = None, stream=None):
        W = self.weights
        if self.shared is not None:  # routed experts plus the shared expert, one combine
            moe_forward_shared(self.cfg, x.shape[0], x, self.router_w, self.router_bias, self.gs1, self.gs2,
                               W.w1_fp4, W.w1_sf, self.alpha1, W.w2_fp4, W.w2_sf, self.alpha2, self.shared, y,
                               topk_ids, topk_w, self.ws, stream)
            return
        moe_forward(self.cfg, x.shape[0], x, self.router_w, self.router_bias, self.gs1, self.gs2, W.w1_fp4, W.w1_sf,
                    self.alpha1, W.w2_fp4, W.w2_sf, self.alpha2, y, topk_ids, topk_w, self.ws, stream)

    def read_error(self, clear=True) -> int:
        return fp4moe_read_error(self.ws, clear)

    def read_scale_status(self, clear=True):
        """(FP4MOE_SAT_* flags, running amax|h|) of this layer's workspace."""
        return fp4moe_read_scale_status(self.ws, clear)

    def refresh_gs2(self, stream=None):
        """gs2 and alpha2 from the amax|h| of the calls since the last refresh (lagged, on the device)."""
        fp4moe_refresh_gs2(self.cfg, self.ws, self.weights.gw2, self.gs2, self.alpha2, stream)
