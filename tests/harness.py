"""Test harness: runs the CUDA path through the C ABI and the CPU oracle on the same seeded inputs,
and compares them. Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import routing_dispatch_expert_gb300 as rde

BF16_TOL = 2e-2  # per-token max relative error of the layer output (bf16 path)
FP8_TOL = 5e-2
# route weights: the selection is bit-exact, the weights themselves only enter the combine; the sigmoid
# layers evaluate them with the fp32 sigmoid (at most ~4e-7 relative each, twice that for the ratio)
WEIGHT_RTOL = 2e-6
MARGIN = 1e-3  # tokens whose selection margin is below this are excluded when routes may differ


def cfg_of(wl: synth.Workload) -> rde.MoeConfig:
    return rde.make_config(T=wl.T, h=wl.h, E=wl.E, k=wl.k, I=wl.I, I_shared=wl.I_shared, n_group=wl.n_group,
                           topk_group=wl.topk_group, score=wl.score, renorm=wl.renorm, routed_scale=wl.routed_scale,
                           dtype=wl.dtype, capacity_factor=wl.capacity_factor)


def config_capacity_factor(wl: synth.Workload) -> float:
    """The capacity factor as the layer config holds it (fp32): the oracle must see the same number."""
    return float(np.float32(wl.capacity_factor))


def route_kwargs(wl: synth.Workload) -> dict:
    return dict(k=wl.k, n_group=wl.n_group, topk_group=wl.topk_group,
                score=oracle.SOFTMAX if wl.score == "softmax" else oracle.SIGMOID, renorm=wl.renorm,
                routed_scale=wl.routed_scale)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns"""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


U32 = 2.0 ** -24  # unit roundoff of fp32 (round to nearest)


def router_error_units(wl: synth.Workload) -> float:
    """Worst-case error of the library's fp32 router GEMM, in units of U32 * sum_d |x_d w_d|.

    Every product is exact: x is bf16 and the fp32 weight enters either as an fp32 FMA operand
    (CUDA-core router) or split exactly into three bf16 terms (tensor-core router), and a bf16 x bf16
    product has at most 16 significant bits. So all error comes from the additions, and by the
    standard bound for summation (Higham, Accuracy and Stability of Numerical Algorithms, ch. 4) it is
    at most D * delta * sum |terms|, where D is the longest chain of rounded additions a product passes
    through and delta the relative error of one addition.

    * CUDA-core router (E < 128, or E not a multiple of 32): delta = U32 (IEEE round to nearest). A
      lane takes 8 elements of each 256-element K chunk of its warp's share, chunks split over kw
      warps (kw = 8 when h / 256 >= 8, else 4, 2, 1), accumulated by fused multiply-adds: 8 *
      ceil(chunks / kw) roundings; then a 5-level butterfly over the lanes and kw - 1 additions of
      the warps' partial sums.
    * Tensor-core router: the accumulator's internal rounding is not documented, so take the
      pessimistic delta = 2 U32 (truncation) for every product added, as if the 512 products of a
      TMEM chunk (8 K blocks of 64) were added one by one; the chunks (at most ceil(3 h / 512) per
      tile) are summed in fp32 registers (round to nearest), and a split K range adds at most 128
      partial sums in a fixed order.
    """
    if wl.E >= 128 and wl.E % 32 == 0:
        return 2.0 * 512 + -(-3 * wl.h // 512) + 128
    chunks = wl.h // 256
    kw = 8 if chunks >= 8 else 4 if chunks >= 4 else 2 if chunks >= 2 else 1
    return 8.0 * -(-chunks // kw) + 5 + (kw - 1)


def router_abs_sum(x_bits: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """sum_d |x_d w_d| per (token, expert), by the oracle on the absolute values."""
    return oracle.router_logits(x_bits & np.uint16(0x7FFF), np.abs(w_r)).astype(np.float64)


def logit_tolerance(wl: synth.Workload, x_bits: np.ndarray, w_r: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Allowed |GPU logit - oracle logit| per (token, expert): the router's worst-case error bound
    (router_error_units) plus the half unit in the last place by which the oracle's own fp32 logit
    (the exact sum, rounded once) can sit from the exact sum."""
    return router_error_units(wl) * U32 * router_abs_sum(x_bits, w_r) + 0.5 * U32 * np.abs(ref) + 1e-30


def rel_err_per_token(y_bits: np.ndarray, ref_bits_or_double: np.ndarray) -> np.ndarray:
    y = oracle.bf16_to_double(y_bits)
    ref = (oracle.bf16_to_double(ref_bits_or_double) if ref_bits_or_double.dtype == np.uint16
           else ref_bits_or_double)
    num = np.abs(y - ref).max(axis=1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return num / den


class GpuLayer:
    """Device inputs of a workload, the layer's weights, one moe_forward, and typed views of the
    intermediates in its workspace."""

    def __init__(self, wl: synth.Workload, device="cuda"):
        self.wl = wl
        self.cfg = cfg_of(wl)
        self.inp = synth.device_inputs(wl, torch, device=device)
        ws = {}
        if wl.dtype == "fp8":
            ws["w_gu"], ws["s_gu"] = rde.quantize_weights_fp8(self.inp["w_gu"])
            ws["w_d"], ws["s_d"] = rde.quantize_weights_fp8(self.inp["w_d"])
            if wl.has_shared:
                ws["w_gu_shared"], ws["s_gu_shared"] = rde.quantize_weights_fp8(self.inp["w_gu_shared"])
                ws["w_d_shared"], ws["s_d_shared"] = rde.quantize_weights_fp8(self.inp["w_d_shared"])
        elif wl.dtype == "nvfp4":
            for n in ("gu", "d") + (("gu_shared", "d_shared") if wl.has_shared else ()):
                ws["w_" + n], ws["s_" + n], ws["g_" + n] = rde.quantize_weights_nvfp4(self.inp["w_" + n])
        else:
            for n in ("w_gu", "w_d", "w_gu_shared", "w_d_shared"):
                ws[n] = self.inp[n]
        self.weights = rde.Weights(w_router=self.inp["w_router"], bias=self.inp["bias"], **ws)
        self.ws = rde.alloc_workspace(self.cfg, device)
        rde.device_status(self.cfg, self.ws)
        self.y = torch.empty_like(self.inp["x"])

    def forward(self):
        rde.forward(self.cfg, self.inp["x"], self.weights, self.y, self.ws)
        torch.cuda.synchronize()
        return self.y

    def view(self, name, dtype, shape):
        return rde.ws_view(self.ws, self.cfg, name, dtype, shape)

    def intermediates(self) -> dict:
        wl = self.wl
        R = wl.T * wl.k
        R_tot = R + (wl.T if wl.has_shared else 0)
        xd_dtype = torch.uint8 if wl.dtype == "fp8" else torch.bfloat16
        out = dict(
            logits=self.view("logits", torch.float32, (wl.T, wl.E)),
            topk_idx=self.view("topk_idx", torch.int32, (wl.T, wl.k)),
            topk_w=self.view("topk_w", torch.float32, (wl.T, wl.k)),
            counts=self.view("counts", torch.int32, (wl.E,)),
            offsets=self.view("offsets", torch.int32, (wl.E + 1,)),
            inv_pos=self.view("inv_pos", torch.int32, (wl.T, wl.k)),
            row_token=self.view("row_token", torch.int32, (R,)),
            row_weight=self.view("row_weight", torch.float32, (R,)),
            xd=self.view("xd", xd_dtype, (R_tot, wl.h)),
            yd=self.view("yd", torch.bfloat16, (R_tot, wl.h)),
        )
        if wl.dtype == "fp8":
            out["xd_scales"] = self.view("xd_scales", torch.float32, (R_tot, wl.h // 128))
        return out

    def expert_weights_host(self, e):
        """bf16 bit patterns of one expert's weights as generated on the device"""
        if e == "shared":
            return bits(self.inp["w_gu_shared"]), bits(self.inp["w_d_shared"])
        return bits(self.inp["w_gu"][e]), bits(self.inp["w_d"][e])


def oracle_tokens(layer: GpuLayer, tokens: np.ndarray, idx: np.ndarray, w: np.ndarray, x_bits: np.ndarray):
    """Oracle layer output for the given tokens with the given routes: one expert at a time (weights
    are read back from the device generator one expert at a time to bound host memory).
    Returns (y_ref bf16 bits [n, h], o [n, k, h] fp64 expert outputs, shared [n, h] or None)."""
    wl = layer.wl
    n = len(tokens)
    o = np.zeros((n, wl.k, wl.h), np.float64)
    xs = x_bits[tokens]
    fp8 = wl.dtype == "fp8"
    if fp8:
        xq, xsc = oracle.quant_1x128(oracle.bf16_to_double(xs))

    def ffn(rows, e):
        gu, d = layer.expert_weights_host(e)
        if fp8:
            (gq, gs), (dq, ds) = oracle.quant_weight_128x128(gu), oracle.quant_weight_128x128(d)
            return oracle.expert_ffn_fp8(xq[rows], xsc[rows], gq, gs, dq, ds)
        if wl.dtype == "nvfp4":
            return oracle.expert_ffn_nvfp4(xs[rows], oracle.quant_weight_nvfp4(gu), oracle.quant_weight_nvfp4(d))
        return oracle.expert_ffn_bf16(xs[rows], gu, d)

    sel = idx[tokens]
    for e in np.unique(sel):
        ti, tj = np.nonzero(sel == e)
        o[ti, tj] = ffn(ti, int(e))
    shared = ffn(np.arange(n), "shared") if wl.has_shared else None
    y = oracle.combine(o, w[tokens], shared)
    return y, o, shared


def selection_margin(wl: synth.Workload, logits: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """Per token: gap between the k-th and (k+1)-th selection keys among the experts of the kept
    groups, and for grouped routing also between the topk_group-th and next group score (the
    smaller of the two). Used only to exclude near-ties when two sides route on different logits."""
    if wl.score == "softmax":
        key = logits.astype(np.float64)
    else:
        s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
        key = (s + (bias if bias is not None else np.float32(0))).astype(np.float64)
    m = np.full(key.shape[0], np.inf)
    if wl.n_group > 1:
        g = key.reshape(key.shape[0], wl.n_group, -1)
        g2 = -np.sort(-g, axis=2)[:, :, :2].sum(axis=2)
        order = np.argsort(-g2, axis=1, kind="stable")
        gs = np.take_along_axis(g2, order, axis=1)
        m = gs[:, wl.topk_group - 1] - gs[:, wl.topk_group]
        kept = np.zeros_like(g2, dtype=bool)
        np.put_along_axis(kept, order[:, :wl.topk_group], True, axis=1)
        key = np.where(np.repeat(kept, key.shape[1] // wl.n_group, axis=1), key, -np.inf)
    srt = -np.sort(-key, axis=1)
    return np.minimum(m, srt[:, wl.k - 1] - srt[:, wl.k])
