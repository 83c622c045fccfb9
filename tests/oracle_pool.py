"""The oracle's per-expert work spread over worker processes, for full-size parity tests.

The oracle is per token and per expert, and each expert's weights must be
generated and quantised once for all of its rows. At the DeepSeek-V4-Flash
shape that is a few seconds of numpy per expert, for up to 256 experts. So the
tests hand every expert's rows to a pool of worker processes:

* the workers are started with ``spawn`` (the test process holds a CUDA
  context, and a forked child of it can hang);
* expert e always goes to worker e % n, which keeps that expert's quantised
  weights (codes packed two per byte) for later calls in the same session, so
  the workloads that share the DSV4 weights quantise each expert once;
* BLAS runs single-threaded in each worker, one worker per core.

Nothing here computes a value of its own: routing, quantisation, the experts
and the combine are the oracle's functions (``oracle.moe``, ``oracle.mxfp4``).
This module only groups rows by expert, ships them and puts the results back
in pair order.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

import synthgen as sg
from oracle import moe, mxfp4, nvfp4

# ----------------------------------------------------------------- workers --

_CACHE: dict = {}


def _weights_key(wl: sg.Workload):
    return (wl.H, wl.I_log, wl.E, wl.model_seed, wl.w_sigma)


def _nv_expert(wl: sg.Workload, e: int) -> moe.QuantExpert:
    key = ("nv", _weights_key(wl), e)
    packed = _CACHE.get(key)
    if packed is None:
        qe = moe.quantize_expert(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e))
        _CACHE[key] = qe._replace(w1_q=nvfp4.pack_codes(qe.w1_q), w2_q=nvfp4.pack_codes(qe.w2_q))
        return qe
    return packed._replace(w1_q=nvfp4.unpack_codes(packed.w1_q), w2_q=nvfp4.unpack_codes(packed.w2_q))


def _mx_checkpoint(wl_full: sg.Workload, e: int) -> mxfp4.MxCheckpoint:
    key = ("mx", _weights_key(wl_full), e)
    ck = _CACHE.get(key)
    if ck is None:
        ck = mxfp4.mx_checkpoint(sg.expert_w1_f32(wl_full, e), sg.expert_w2_f32(wl_full, e))
        _CACHE[key] = ck
    return ck


def _mxnv_expert(wl_full: sg.Workload, e: int, plan, rank) -> moe.QuantExpert:
    """Rank `rank`'s MXFP4 shard of expert e in the NVFP4 operand form (mxfp4.mx_as_nvfp4 per matrix)."""
    sh = mxfp4.mx_shard_checkpoint(_mx_checkpoint(wl_full, e), plan, rank)
    q1, s1, g1 = mxfp4.mx_as_nvfp4(sh.w1_q, sh.w1_s)
    q2, s2, g2 = mxfp4.mx_as_nvfp4(sh.w2_q, sh.w2_s)
    return moe.QuantExpert(q1, s1, g1, q2, s2, g2)


def _expert_jobs(wl: sg.Workload, e: int, requests: list) -> list:
    """Run one expert's requests. Each request is a tuple whose first item names it:

    ("amax", x_bits, gs1)            -> moe.hidden_amax of the rows, quantised under gs1
    ("rows", x_bits, gs1, gs2)       -> moe.pair_rows of the rows (fp64 [n, H])
    ("mx_rows", x_bits, plan, rank)  -> mxfp4.mx_expert_out of rank's shard (wl is the full-width workload)
    ("mxnv_amax", x_bits, gs1, plan, rank)        -> moe.hidden_amax of rank's shard in the NVFP4 operand form
    ("mxnv_rows", x_bits, gs1, gs2, plan, rank)   -> moe.pair_rows of the same
    """
    out = []
    for req in requests:
        kind = req[0]
        if kind == "amax":
            _, x_bits, gs1 = req
            out.append(moe.hidden_amax(_nv_expert(wl, e), moe.dequantized_activations(x_bits, gs1), wl.swiglu_limit))
        elif kind == "rows":
            _, x_bits, gs1, gs2 = req
            out.append(moe.pair_rows(_nv_expert(wl, e), moe.dequantized_activations(x_bits, gs1), gs2,
                                     wl.swiglu_limit))
        elif kind == "mxnv_amax":
            _, x_bits, gs1, plan, rank = req
            out.append(moe.hidden_amax(_mxnv_expert(wl, e, plan, rank), moe.dequantized_activations(x_bits, gs1),
                                       wl.swiglu_limit))
        elif kind == "mxnv_rows":
            _, x_bits, gs1, gs2, plan, rank = req
            out.append(moe.pair_rows(_mxnv_expert(wl, e, plan, rank), moe.dequantized_activations(x_bits, gs1), gs2,
                                     wl.swiglu_limit))
        elif kind == "mx_rows":
            _, x_bits, plan, rank = req
            shard = mxfp4.mx_shard_checkpoint(_mx_checkpoint(wl, e), plan, rank)
            out.append(mxfp4.mx_expert_out(shard, moe.bf16_to_f64(x_bits), wl.swiglu_limit))
        else:
            raise ValueError(kind)
    return out


def _ping() -> int:
    return os.getpid()


# ----------------------------------------------------------------- service --

def _default_workers() -> int:
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    avail_gb = 8.0
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail_gb = int(line.split()[1]) / 2**20
    except OSError:
        pass
    # a DSV4 expert's quantisation peaks near 2 GB of numpy temporaries per worker
    return max(1, min(16, cores, int(avail_gb // 3)))


class OracleService:
    """n single-process executors; expert e always runs on executor e % n."""

    def __init__(self, n_workers: int | None = None):
        self.n = n_workers or _default_workers()
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pools = [cf.ProcessPoolExecutor(1, mp_context=ctx) for _ in range(self.n)]
            for f in [p.submit(_ping) for p in self.pools]:   # start every worker under the 1-thread BLAS setting
                f.result()
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.scales: dict = {}

    def close(self):
        for p in self.pools:
            p.shutdown(wait=True, cancel_futures=True)

    def run(self, wl: sg.Workload, per_expert: dict) -> dict:
        """{e: [request, ...]} -> {e: [result, ...]}, each expert's requests run in order on its own worker."""
        futs = {e: self.pools[e % self.n].submit(_expert_jobs, wl, e, reqs) for e, reqs in per_expert.items() if reqs}
        return {e: f.result() for e, f in futs.items()}

    # ------------------------------------------------------------ NVFP4 layer --

    def calibrate(self, wl: sg.Workload, xw_bits: np.ndarray):
        """The oracle's own warm-up scales (moe.calibrate, with its expert loop on the workers)."""
        key = (wl.name, _weights_key(wl), xw_bits.shape, hash(xw_bits.tobytes()))
        if key not in self.scales:
            gs1 = moe.activation_scale(xw_bits)
            ids, _ = moe.topk_softmax(moe.router_logits(xw_bits, sg.router_bf16(wl), sg.router_bias_f32(wl)), wl.k)
            reqs = {e: [("amax", xw_bits[tt], gs1)] for e, (tt, _) in moe.routed_rows(ids).items()}
            amax = max([r[0] for r in self.run(wl, reqs).values()], default=0.0)
            self.scales[key] = (gs1, nvfp4.global_scale(np.float32(amax)))
        return self.scales[key]

    def layer(self, wl: sg.Workload, batches: list, gs1, gs2) -> list:
        """moe.moe_tokens for several token batches at once, with the router of the workload.

        batches: list of x_bits [n_b, H]. Returns a list of (y_bits [n_b, H], ids [n_b, k], w [n_b, k]).
        """
        wr, bias = sg.router_bf16(wl), sg.router_bias_f32(wl)
        routed, per_expert = [], {}
        for b, x_bits in enumerate(batches):
            ids, w = moe.topk_softmax(moe.router_logits(x_bits, wr, bias), wl.k)
            rr = moe.routed_rows(ids)
            routed.append((ids, w, rr))
            for e, (tt, _) in rr.items():
                per_expert.setdefault(e, []).append(("rows", x_bits[tt], gs1, gs2))
        res = self.run(wl, per_expert)
        cursor = {e: 0 for e in res}
        out = []
        for x_bits, (ids, w, rr) in zip(batches, routed):
            outs = np.zeros((x_bits.shape[0], wl.k, wl.H))
            for e, (tt, jj) in rr.items():
                outs[tt, jj] = res[e][cursor[e]]
                cursor[e] += 1
            out.append((moe.combine(ids, w, outs), ids, w))
        return out

    # ------------------------------------------------------------ MXFP4 layer --

    def mx_partials(self, wl_full: sg.Workload, x_bits: np.ndarray, ids: np.ndarray, plans: list) -> list:
        """mxfp4.mx_moe_partials of the same routed tokens for several (plan, rank) shards.

        wl_full is the generator's full-width view of the experts. Returns one [n, k, H] fp64 array per shard.
        """
        rr = moe.routed_rows(ids)
        per_expert = {e: [("mx_rows", x_bits[tt], plan, rank) for plan, rank in plans] for e, (tt, _) in rr.items()}
        res = self.run(wl_full, per_expert)
        outs = []
        for i in range(len(plans)):
            o = np.zeros((x_bits.shape[0], ids.shape[1], wl_full.H))
            for e, (tt, jj) in rr.items():
                o[tt, jj] = res[e][i]
            outs.append(o)
        return outs

    # ---------------------------------- MXFP4 weights on the NVFP4 path (mxfp4.mx_as_nvfp4) --

    def mxnv_calibrate(self, wl_full: sg.Workload, xw_bits: np.ndarray, plan, rank):
        """moe.calibrate of rank's NVFP4-form shard on a warm-up batch."""
        gs1 = moe.activation_scale(xw_bits)
        ids, _ = moe.topk_softmax(moe.router_logits(xw_bits, sg.router_bf16(wl_full), sg.router_bias_f32(wl_full)),
                                  wl_full.k)
        reqs = {e: [("mxnv_amax", xw_bits[tt], gs1, plan, rank)] for e, (tt, _) in moe.routed_rows(ids).items()}
        amax = max([r[0] for r in self.run(wl_full, reqs).values()], default=0.0)
        return gs1, nvfp4.global_scale(np.float32(amax))

    def mxnv_partials(self, wl_full: sg.Workload, x_bits: np.ndarray, ids: np.ndarray, gs1, gs2, plans: list) -> list:
        """Per-(token, j) partial rows [n, k, H] of the NVFP4-form shards (plan, rank), under gs1 and gs2."""
        rr = moe.routed_rows(ids)
        per_expert = {e: [("mxnv_rows", x_bits[tt], gs1, gs2, plan, rank) for plan, rank in plans]
                      for e, (tt, _) in rr.items()}
        res = self.run(wl_full, per_expert)
        outs = []
        for i in range(len(plans)):
            o = np.zeros((x_bits.shape[0], ids.shape[1], wl_full.H))
            for e, (tt, jj) in rr.items():
                o[tt, jj] = res[e][i]
            outs.append(o)
        return outs
