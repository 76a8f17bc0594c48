"""The expert FFN at every tile boundary.

Expert-major rows are laid out by hand so that the groups hold 0, 1, 63, 64, 65, 127, 128, 129, ... rows:
the edges where a single-CTA tile switches from an M = 64 to an M = 128 MMA, where a group takes a
second tile, and where a CTA-pair group's tail becomes a 128-row pair tile. They go through
`moe_expert_ffn` (the step entry point of S5-S6) in bf16, FP8 and NVFP4, and every output row is
compared with the oracle's expert FFN times its route weight (R8: yd is stored already weighted).
The routing steps are not involved, so the counts are exact rather than whatever a router produces.
"""
import numpy as np
import pytest
import torch

import oracle
import routing_dispatch_expert_gb300 as rde
import synth
from harness import BF16_TOL, FP8_TOL, bits

pytestmark = pytest.mark.gpu

# single-CTA tiles: an average below 128 rows per group keeps the bf16 layer off CTA pairs
SINGLE = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257]
# CTA pairs: 320 rows per group on average and 150 full pair tiles of the gate/up launch (I 1280)
PAIR = [127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 513]

SEED = 20261202


def _normal_bits(stream, n, sigma):
    return synth.normal_bf16(SEED, stream, 0, n, sigma)


def _layer(counts, h, I, dtype):
    E = len(counts)
    R = int(sum(counts))
    cfg = rde.make_config(T=R, h=h, E=E, k=1, I=I, I_shared=0, dtype=dtype)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = _normal_bits(901, R * h, 1.0).reshape(R, h)
    gu = _normal_bits(902, E * 2 * I * h, h ** -0.5).reshape(E, 2 * I, h)
    dn = _normal_bits(903, E * h * I, I ** -0.5).reshape(E, h, I)
    rw = synth.uniform_f32(SEED, 904, 0, R, 0.1, 1.0)
    return cfg, offsets, x, gu, dn, rw


def _to_dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).view(dtype).cuda()


def _run(counts, h, I, dtype):
    cfg, offsets, x, gu, dn, rw = _layer(counts, h, I, dtype)
    R = x.shape[0]
    gu_d, dn_d = _to_dev(gu, torch.bfloat16), _to_dev(dn, torch.bfloat16)
    if dtype == "fp8":
        xq, xs = oracle.quant_1x128(oracle.bf16_to_double(x))
        xd, xd_scales = _to_dev(xq, torch.uint8), _to_dev(xs.astype(np.float32), torch.float32)
        (gq, gs), (dq, ds) = rde.quantize_weights_fp8(gu_d), rde.quantize_weights_fp8(dn_d)
        weights = rde.Weights(None, w_gu=gq, s_gu=gs, w_d=dq, s_d=ds)
    elif dtype == "nvfp4":
        xd, xd_scales = _to_dev(x, torch.bfloat16), None
        (gq, gs, gg), (dq, ds, dg) = rde.quantize_weights_nvfp4(gu_d), rde.quantize_weights_nvfp4(dn_d)
        weights = rde.Weights(None, w_gu=gq, s_gu=gs, g_gu=gg, w_d=dq, s_d=ds, g_d=dg)
    else:
        xd, xd_scales = _to_dev(x, torch.bfloat16), None
        weights = rde.Weights(None, w_gu=gu_d, w_d=dn_d)
    yd = torch.full((R, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)  # a new workspace's status word holds whatever was there: clear it
    rde.expert_ffn(cfg, weights, xd, xd_scales, _to_dev(offsets, torch.int32), _to_dev(rw, torch.float32), yd, ws)
    torch.cuda.synchronize()
    assert rde.device_status(cfg, ws) == 0
    got = oracle.bf16_to_double(bits(yd))
    tol = FP8_TOL if dtype == "fp8" else BF16_TOL
    for e, n in enumerate(counts):
        if n == 0:
            continue
        rows = slice(int(offsets[e]), int(offsets[e + 1]))
        if dtype == "fp8":
            ref = oracle.expert_ffn_fp8(xq[rows], xs[rows], *oracle.quant_weight_128x128(gu[e]),
                                        *oracle.quant_weight_128x128(dn[e]))
        elif dtype == "nvfp4":
            ref = oracle.expert_ffn_nvfp4(x[rows], oracle.quant_weight_nvfp4(gu[e]), oracle.quant_weight_nvfp4(dn[e]))
        else:
            ref = oracle.expert_ffn_bf16(x[rows], gu[e], dn[e])
        ref = ref * rw[rows, None].astype(np.float64)
        err = np.abs(got[rows] - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)
        assert err.max() <= tol, f"{dtype}: group {e} ({n} rows): max rel err {err.max():.3e} at row {int(err.argmax())}"


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "nvfp4"])
def test_single_cta_tile_edges(dtype):
    _run(SINGLE, h=256, I=256, dtype=dtype)


def test_pair_tile_edges():
    _run(PAIR, h=256, I=1280, dtype="bf16")
