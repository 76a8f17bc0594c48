"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws numbers (see ``synth.h`` for the generator's definition); it holds none
of the MoE method's arithmetic. Both the CPU oracle's callers and the GPU path's callers take
their inputs from here, so the two sides see bit-identical inputs.

Workloads follow the five configurations the layer is measured on: a tiny layer, a
Mixtral-shaped layer, and DeepSeek-V3-shaped prefill, decode (Zipf-skewed) and FP8 (Zipf-skewed)
layers.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libsynth_host.so")
_DEV_SO = os.path.join(_BUILD, "libsynth_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

# stream ids of the tensors of one workload
STREAM_X, STREAM_WR, STREAM_BIAS, STREAM_WGU, STREAM_WD, STREAM_WGU_SHARED, STREAM_WD_SHARED = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    k: int
    I: int
    I_shared: int
    n_group: int
    topk_group: int
    score: str  # "softmax" | "sigmoid"
    renorm: bool
    routed_scale: float
    dtype: str  # "bf16" | "fp8" | "nvfp4" (the expert weights' storage type; generated as bf16)
    seed: int
    bias_range: float | None = None  # bias ~ U(-b, b)
    zipf_s: float | None = None  # popularity skew of the router logits
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    wr_sigma: float = 0.02
    capacity_factor: float = 0.0  # 0: dropless

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def has_shared(self) -> bool:
        return self.I_shared > 0

    @property
    def rows(self) -> int:
        """routed (token, slot) rows"""
        return self.T * self.k


_DSV3 = dict(h=7168, E=256, k=8, I=2048, I_shared=2048, n_group=8, topk_group=4, score="sigmoid", renorm=True,
             routed_scale=2.5, bias_range=0.1)

WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", T=4096, h=512, E=8, k=2, I=256, I_shared=0, n_group=1, topk_group=1, score="softmax",
                     renorm=False, routed_scale=1.0, dtype="bf16", seed=0),
    "mixtral": Workload("mixtral", T=8192, h=4096, E=8, k=2, I=14336, I_shared=0, n_group=1, topk_group=1,
                        score="softmax", renorm=True, routed_scale=1.0, dtype="bf16", seed=1),
    "dsv3_prefill": Workload("dsv3_prefill", T=16384, dtype="bf16", seed=2, **_DSV3),
    "dsv3_decode": Workload("dsv3_decode", T=256, dtype="bf16", seed=3, zipf_s=1.2, **_DSV3),
    "dsv3_fp8": Workload("dsv3_fp8", T=32768, dtype="fp8", seed=4, zipf_s=1.0, **_DSV3),
    # the decode layer with NVFP4 expert weights (FP4 MoE weights of the Blackwell deployment)
    "dsv3_decode_fp4": Workload("dsv3_decode_fp4", T=256, dtype="nvfp4", seed=3, zipf_s=1.2, **_DSV3),
}


# ------------------------------------------------------------------------------------------
# build / load
# ------------------------------------------------------------------------------------------
def build(device: bool = True, force: bool = False) -> None:
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_HOST_SO) or os.path.getmtime(_HOST_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", _HOST_SO,
                               src])
    if device:
        src = os.path.join(_HERE, "synth_dev.cu")
        if force or not os.path.exists(_DEV_SO) or os.path.getmtime(_DEV_SO) < os.path.getmtime(src):
            subprocess.check_call(["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler",
                                   "-fPIC", "-shared", "-fmad=false", "-o", _DEV_SO, src])


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            build(device=False)
            lib = ctypes.CDLL(_HOST_SO)
            u64, u32, i64, f32, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_float,
                                      ctypes.c_void_p)
            lib.syn_normal_bf16.argtypes = [u64, u32, i64, i64, f32, vp, i64, vp]
            lib.syn_normal_f32.argtypes = [u64, u32, i64, i64, f32, vp]
            lib.syn_uniform_f32.argtypes = [u64, u32, i64, i64, f32, f32, vp]
            _host = lib
    return _host


def _dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(_DEV_SO):
                build(device=True)
            lib = ctypes.CDLL(_DEV_SO)
            u64, u32, i64, f32, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_float,
                                      ctypes.c_void_p)
            lib.syn_normal_bf16_dev.argtypes = [u64, u32, i64, i64, f32, vp, i64, vp, vp]
            lib.syn_normal_f32_dev.argtypes = [u64, u32, i64, i64, f32, vp, vp]
            lib.syn_uniform_f32_dev.argtypes = [u64, u32, i64, i64, f32, f32, vp, vp]
            for f in (lib.syn_normal_bf16_dev, lib.syn_normal_f32_dev, lib.syn_uniform_f32_dev):
                f.restype = ctypes.c_int
            _dev = lib
    return _dev


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------------------------------
# host draws
# ------------------------------------------------------------------------------------------
def normal_bf16(seed, stream, offset, n, sigma, mu=None) -> np.ndarray:
    out = np.empty(n, np.uint16)
    mu_arr = None if mu is None else np.ascontiguousarray(mu, np.float32)
    _host_lib().syn_normal_bf16(seed, stream, offset, n, sigma, None if mu_arr is None else _ptr(mu_arr),
                                0 if mu_arr is None else mu_arr.size, _ptr(out))
    return out


def normal_f32(seed, stream, offset, n, sigma) -> np.ndarray:
    out = np.empty(n, np.float32)
    _host_lib().syn_normal_f32(seed, stream, offset, n, sigma, _ptr(out))
    return out


def uniform_f32(seed, stream, offset, n, lo, hi) -> np.ndarray:
    out = np.empty(n, np.float32)
    _host_lib().syn_uniform_f32(seed, stream, offset, n, lo, hi, _ptr(out))
    return out


def router_weight(wl: Workload) -> np.ndarray:
    """W_r [E, h] fp32 ~ N(0, wr_sigma)"""
    return normal_f32(wl.seed, STREAM_WR, 0, wl.E * wl.h, wl.wr_sigma).reshape(wl.E, wl.h)


def bias(wl: Workload) -> np.ndarray | None:
    """per-expert selection bias [E] fp32 ~ U(-b, b), or None"""
    if wl.bias_range is None:
        return None
    return uniform_f32(wl.seed, STREAM_BIAS, 0, wl.E, -wl.bias_range, wl.bias_range)


def skew_shift(wl: Workload, w_r: np.ndarray | None = None) -> np.ndarray | None:
    """Per-column shift mu [h] of the activations that skews expert popularity.

    Expert popularity p_r ~ 1/r^s is laid over a seeded random permutation pi of the experts;
    mu is the minimum-norm solution of W_r mu = log p_pi(e), so every token's router logits
    move by log p of the expert (router GEMM and scoring run unchanged on the shifted input).
    """
    if wl.zipf_s is None:
        return None
    if w_r is None:
        w_r = router_weight(wl)
    perm = np.random.default_rng(wl.seed).permutation(wl.E)
    target = np.empty(wl.E, np.float64)
    target[perm] = -wl.zipf_s * np.log(np.arange(1, wl.E + 1, dtype=np.float64))
    a = w_r.astype(np.float64)
    mu = a.T @ np.linalg.solve(a @ a.T, target)
    return mu.astype(np.float32)


def activations(wl: Workload, mu: np.ndarray | None = None, t0: int = 0, n_tok: int | None = None) -> np.ndarray:
    """x [n_tok, h] bf16 bits (uint16) for tokens [t0, t0 + n_tok)"""
    n_tok = wl.T - t0 if n_tok is None else n_tok
    return normal_bf16(wl.seed, STREAM_X, t0 * wl.h, n_tok * wl.h, wl.x_sigma, mu).reshape(n_tok, wl.h)


def expert_weights(wl: Workload, e: int | str) -> tuple[np.ndarray, np.ndarray]:
    """bf16 bits of one expert: (w_gu [2I, h] with gate rows first, w_d [h, I]); e = 'shared' for the
    shared expert."""
    if e == "shared":
        I = wl.I_shared
        gu = normal_bf16(wl.seed, STREAM_WGU_SHARED, 0, 2 * I * wl.h, wl.w_sigma)
        d = normal_bf16(wl.seed, STREAM_WD_SHARED, 0, wl.h * I, wl.w_sigma)
    else:
        I = wl.I
        gu = normal_bf16(wl.seed, STREAM_WGU, e * 2 * I * wl.h, 2 * I * wl.h, wl.w_sigma)
        d = normal_bf16(wl.seed, STREAM_WD, e * wl.h * I, wl.h * I, wl.w_sigma)
    return gu.reshape(2 * I, wl.h), d.reshape(wl.h, I)


# ------------------------------------------------------------------------------------------
# device draws (torch tensors on a CUDA device; generation runs as CUDA kernels)
# ------------------------------------------------------------------------------------------
def _stream_ptr(torch):
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"synthetic input generation failed with CUDA error {rc}")


def device_normal_bf16(torch, shape, seed, stream, sigma, offset=0, mu=None, device="cuda"):
    n = int(np.prod(shape))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    mu_t = None if mu is None else torch.as_tensor(np.ascontiguousarray(mu, np.float32)).to(device)
    _check(_dev_lib().syn_normal_bf16_dev(seed, stream, offset, n, sigma,
                                          None if mu_t is None else ctypes.c_void_p(mu_t.data_ptr()),
                                          0 if mu_t is None else mu_t.numel(), ctypes.c_void_p(out.data_ptr()),
                                          _stream_ptr(torch)))
    return out


def device_inputs(wl: Workload, torch, device="cuda", with_weights=True):
    """All inputs of a workload on the device: x, w_router, bias, w_gu, w_d, w_gu_shared, w_d_shared
    (bf16 expert weights; FP8 weights are derived from these by the library's static quantiser)."""
    w_r = router_weight(wl)
    mu = skew_shift(wl, w_r)
    out = {
        "x": device_normal_bf16(torch, (wl.T, wl.h), wl.seed, STREAM_X, wl.x_sigma, mu=mu, device=device),
        "w_router": torch.from_numpy(w_r).to(device),
        "bias": None if wl.bias_range is None else torch.from_numpy(bias(wl)).to(device),
        "mu": mu,
    }
    if with_weights:
        out["w_gu"] = device_normal_bf16(torch, (wl.E, 2 * wl.I, wl.h), wl.seed, STREAM_WGU, wl.w_sigma, device=device)
        out["w_d"] = device_normal_bf16(torch, (wl.E, wl.h, wl.I), wl.seed, STREAM_WD, wl.w_sigma, device=device)
        if wl.has_shared:
            out["w_gu_shared"] = device_normal_bf16(torch, (2 * wl.I_shared, wl.h), wl.seed, STREAM_WGU_SHARED,
                                                    wl.w_sigma, device=device)
            out["w_d_shared"] = device_normal_bf16(torch, (wl.h, wl.I_shared), wl.seed, STREAM_WD_SHARED, wl.w_sigma,
                                                   device=device)
        else:
            out["w_gu_shared"] = None
            out["w_d_shared"] = None
    return out
