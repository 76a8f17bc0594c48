"""CUDA path vs the CPU oracle, element by element, on seeded inputs at sizes the oracle finishes in
seconds (several tiles and ragged tails). Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import (BF16_TOL, FP8_TOL, MARGIN, WEIGHT_RTOL, GpuLayer, bits, cfg_of, config_capacity_factor,
                     logit_tolerance, oracle_tokens, rel_err_per_token, route_kwargs, selection_margin)

pytestmark = pytest.mark.gpu

_W = synth.WORKLOADS
SMALL = {
    "tiny": _W["tiny"],  # the full tiny layer: 4096 tokens, h 512, 8 experts, top-2
    "mixtral_small": _W["mixtral"].replace(name="mixtral_small", T=300, h=512, I=384),
    "dsv3_small": _W["dsv3_prefill"].replace(name="dsv3_small", T=500, h=512, E=64, I=256, I_shared=256),
    "dsv3_small_noshared": _W["dsv3_prefill"].replace(name="dsv3_small_noshared", T=129, h=256, E=32, I=128,
                                                      I_shared=0),
    "dsv3_skew": _W["dsv3_decode"].replace(name="dsv3_skew", T=77, h=512, E=64, I=256, I_shared=256),
    "dsv3_hot": _W["dsv3_decode"].replace(name="dsv3_hot", T=400, h=256, E=64, I=128, I_shared=128, zipf_s=6.0),
    "single_token": _W["dsv3_prefill"].replace(name="single_token", T=1, h=256, E=64, I=128, I_shared=128),
    # E >= 128: the router GEMM runs on the tensor cores (fp32 weight as three bf16 terms)
    "dsv3_e256": _W["dsv3_prefill"].replace(name="dsv3_e256", T=300, h=512, E=256, I=128, I_shared=128),
    "dsv3_e128_skew": _W["dsv3_decode"].replace(name="dsv3_e128_skew", T=130, h=256, E=128, I=128, I_shared=128),
    # E = 200 (not a multiple of 32): CUDA-core router with four expert blocks, fused small-batch path
    "e200_fused": _W["dsv3_prefill"].replace(name="e200_fused", T=512, h=256, E=200, k=6, n_group=1, topk_group=1,
                                             I=128, I_shared=0),
    # the FP8 layer: e4m3 experts with 128x128 scales, 1x128 activations, SiLU output requantised
    "fp8_small": _W["dsv3_fp8"].replace(name="fp8_small", T=300, h=512, E=64, I=256, I_shared=256),
    "fp8_e256_skew": _W["dsv3_fp8"].replace(name="fp8_e256_skew", T=257, h=256, E=256, I=128, I_shared=128),
    "fp8_noshared": _W["dsv3_fp8"].replace(name="fp8_noshared", T=129, h=512, E=32, I=384, I_shared=0),
    # capacity factor: overflowing experts keep their earliest tokens, the rest skip them
    "cap_skew": _W["dsv3_decode"].replace(name="cap_skew", T=300, h=512, E=64, I=256, I_shared=256,
                                          capacity_factor=1.25),
    "cap_mixtral": _W["mixtral"].replace(name="cap_mixtral", T=500, h=512, I=256, capacity_factor=1.0),
    "cap_fp8": _W["dsv3_fp8"].replace(name="cap_fp8", T=200, h=256, E=32, I=128, I_shared=128, capacity_factor=1.1),
    # NVFP4 expert weights (e2m1 codes, e4m3 scales per 16, fp32 per matrix), bf16 activations
    "fp4_small": _W["dsv3_decode_fp4"].replace(name="fp4_small", T=300, h=512, E=64, I=256, I_shared=256),
    "fp4_mixtral": _W["mixtral"].replace(name="fp4_mixtral", T=333, h=512, I=512, dtype="nvfp4"),
    "fp4_e256": _W["dsv3_decode_fp4"].replace(name="fp4_e256", T=130, h=256, E=256, I=256, I_shared=256),
    "cap_fp4": _W["dsv3_decode_fp4"].replace(name="cap_fp4", T=200, h=256, E=32, I=256, I_shared=0,
                                             capacity_factor=1.2),
    # large expert groups (several 128-row tiles per expert)
    "fp4_large_groups": _W["dsv3_decode_fp4"].replace(name="fp4_large_groups", T=2200, h=512, E=8, k=4,
                                                      n_group=2, topk_group=1, I=256, I_shared=256),
    "fp4_mixtral_large": _W["mixtral"].replace(name="fp4_mixtral_large", T=1100, h=256, I=256, dtype="nvfp4"),
    # at least 128 rows per expert on average and more full pair tiles than pairs: the bf16 expert GEMMs
    # run on CTA pairs (256-row tiles; a tail of at most 128 rows as a 128-row pair tile)
    "pair_half_tiles": _W["dsv3_prefill"].replace(name="pair_half_tiles", T=600, h=512, E=16, k=4, n_group=4,
                                                  topk_group=2, I=1280, I_shared=1280),
    "pair_mixtral": _W["mixtral"].replace(name="pair_mixtral", T=4500, h=512, I=384),
    "pair_dsv3": _W["dsv3_prefill"].replace(name="pair_dsv3", T=2600, h=512, E=8, k=4, n_group=2, topk_group=1,
                                            I=256, I_shared=256),
    "fp8_large_groups": _W["dsv3_fp8"].replace(name="fp8_large_groups", T=2200, h=512, E=8, k=4, n_group=2,
                                               topk_group=1, I=256, I_shared=256),
    "pair_cap": _W["mixtral"].replace(name="pair_cap", T=4500, h=256, I=512, capacity_factor=1.0),
    # pairs with a shared expert and dropped slots
    "pair_cap_shared": _W["dsv3_prefill"].replace(name="pair_cap_shared", T=1500, h=256, E=8, k=4, n_group=2,
                                                  topk_group=1, I=512, I_shared=512, capacity_factor=1.0),
    # experts of more than 8 pair tiles (2250 rows): the tile order walks them in bands of 8 row tiles
    "pair_bands": _W["mixtral"].replace(name="pair_bands", T=4500, h=256, E=4, I=512),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


def test_device_generator_matches_host_generator():
    t = synth.device_normal_bf16(torch, (1000, 37), 5, synth.STREAM_WGU, 0.02, offset=123)
    np.testing.assert_array_equal(bits(t).ravel(), synth.normal_bf16(5, synth.STREAM_WGU, 123, 37000, 0.02))
    mu = np.linspace(-1, 1, 37).astype(np.float32)
    t = synth.device_normal_bf16(torch, (50, 37), 9, synth.STREAM_X, 1.0, mu=mu)
    np.testing.assert_array_equal(bits(t).ravel(), synth.normal_bf16(9, synth.STREAM_X, 0, 1850, 1.0, mu))


def _check_layer_against_oracle(wl, L: GpuLayer, min_clear=0.5):
    y = L.forward()
    assert rde.device_status(L.cfg, L.ws) == 0
    it = L.intermediates()
    x = bits(L.inp["x"])
    w_r = L.inp["w_router"].cpu().numpy()
    bias = None if L.inp["bias"] is None else L.inp["bias"].cpu().numpy()
    experts = [L.expert_weights_host(e) for e in range(wl.E)]
    shared = L.expert_weights_host("shared") if wl.has_shared else None
    logits = it["logits"].cpu().numpy()

    # step 1a: router GEMM against the fp64 oracle
    lo = oracle.router_logits(x, w_r)
    assert np.all(np.abs(logits.astype(np.float64) - lo) <= logit_tolerance(wl, x, w_r, lo))

    # the whole layer on identical logits
    ref = oracle.forward(x, w_r, bias, experts, shared, logits=logits, fp8=wl.dtype == "fp8",
                         nvfp4=wl.dtype == "nvfp4", capacity_factor=config_capacity_factor(wl),
                         **route_kwargs(wl))
    np.testing.assert_array_equal(it["topk_idx"].cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(it["topk_w"].cpu().numpy(), ref["topk_w"], rtol=WEIGHT_RTOL, atol=1e-7)
    np.testing.assert_array_equal(it["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(it["offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(it["inv_pos"].cpu().numpy(), ref["inv_pos"])
    Rk = int(ref["offsets"][-1])  # kept routed rows (T*k when dropless)
    np.testing.assert_array_equal(it["row_token"].cpu().numpy()[:Rk], ref["row_token"][:Rk])
    rw = it["row_weight"].cpu().numpy()
    kept = ref["inv_pos"].ravel() >= 0
    np.testing.assert_array_equal(rw[ref["inv_pos"].ravel()[kept]], it["topk_w"].cpu().numpy().ravel()[kept])
    R = wl.T * wl.k
    fp8 = wl.dtype == "fp8"
    tol = FP8_TOL if fp8 else BF16_TOL
    if fp8:  # codes and 1x128 scales of the dispatched rows are decided identically: bit-exact
        xd = it["xd"].cpu().numpy()
        xs = it["xd_scales"].cpu().numpy()
        np.testing.assert_array_equal(xd[:Rk], ref["xd"])
        np.testing.assert_array_equal(xs[:Rk], ref["xd_scales"])
        if wl.has_shared:
            np.testing.assert_array_equal(xd[R:], ref["xq"])
            np.testing.assert_array_equal(xs[R:], ref["xs"])
    else:
        xd = bits(it["xd"])
        np.testing.assert_array_equal(xd[:Rk], ref["xd"])
        if wl.has_shared and wl.dtype != "bf16":  # bf16: the shared expert reads x itself
            np.testing.assert_array_equal(xd[R:], x)

    # expert outputs per row (route-weighted), and the shared expert's rows
    yd = oracle.bf16_to_double(bits(it["yd"]))
    o_w = ref["o_rows"] * rw[:Rk, None].astype(np.float64)
    err = np.abs(yd[:Rk] - o_w).max(axis=1) / np.maximum(np.abs(o_w).max(axis=1), 1e-30)
    assert err.max() <= tol, f"routed rows: max rel err {err.max()}"
    if wl.has_shared:
        s = ref["shared_out"]
        err = np.abs(yd[R:] - s).max(axis=1) / np.maximum(np.abs(s).max(axis=1), 1e-30)
        assert err.max() <= tol, f"shared rows: max rel err {err.max()}"

    # layer output, every token
    e = rel_err_per_token(bits(y), ref["y"])
    assert e.max() <= tol, f"y: max rel err {e.max()} at token {e.argmax()}"

    # routing on the oracle's own fp64 logits agrees wherever the decision is not a near-tie
    idx2, _ = oracle.route(lo, bias, **route_kwargs(wl))
    keep = selection_margin(wl, lo, bias) >= MARGIN
    assert keep.mean() >= min_clear
    np.testing.assert_array_equal(np.sort(idx2[keep], axis=1), np.sort(ref["topk_idx"][keep], axis=1))
    return ref


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_matches_oracle(name):
    wl = SMALL[name]
    L = GpuLayer(wl)
    # with Zipf(6) nearly every sigmoid saturates, the group scores no longer depend on the token and
    # every token can sit on the same group-level near-tie: no share of clear tokens is required there
    _check_layer_against_oracle(wl, L, min_clear=0.0 if name == "dsv3_hot" else 0.5)


# dsv3_small: single-CTA tiles; pair_dsv3: CTA pairs (both with the shared expert on the second stream)
@pytest.mark.parametrize("name", ["dsv3_small", "pair_dsv3"])
def test_forward_is_deterministic(name):
    wl = SMALL[name]
    L = GpuLayer(wl)
    y1 = L.forward().clone()
    yd1 = L.intermediates()["yd"].clone()
    y2 = L.forward()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(yd1.view(torch.int16), L.intermediates()["yd"].view(torch.int16))


@pytest.mark.parametrize("name", ["dsv3_small", "pair_dsv3"])
def test_steps_through_their_own_entry_points(name):
    """moe_route (with and without given logits), moe_dispatch, moe_expert_ffn and moe_combine called
    one by one give what moe_forward gives."""
    wl = SMALL[name]
    L = GpuLayer(wl)
    y_fwd = L.forward().clone()
    it = L.intermediates()
    dev = "cuda"
    T, k, E, h = wl.T, wl.k, wl.E, wl.h
    R_tot = T * k + T
    cfg = L.cfg
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    rde.route(cfg, L.inp["x"], L.weights, idx, w, logits=logits, ws=ws)
    assert torch.equal(logits, it["logits"]) and torch.equal(idx, it["topk_idx"]) and torch.equal(w, it["topk_w"])
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    rde.route(cfg, None, L.weights, idx2, w2, logits=logits, logits_given=True)
    assert torch.equal(idx2, idx) and torch.equal(w2, w)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(T, k, dtype=torch.int32, device=dev)
    row_token = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_weight = torch.empty(T * k, dtype=torch.float32, device=dev)
    xd = torch.empty(R_tot, h, dtype=torch.bfloat16, device=dev)
    rde.dispatch(cfg, L.inp["x"], idx, w, counts, offsets, inv_pos, row_token, row_weight, xd, None, ws)
    for a, b in ((counts, "counts"), (offsets, "offsets"), (inv_pos, "inv_pos"), (row_token, "row_token"),
                 (row_weight, "row_weight")):
        assert torch.equal(a, it[b]), b
    R = T * k
    assert torch.equal(xd[:R].view(torch.int16), it["xd"][:R].view(torch.int16))
    # the step entry point copies the shared expert's rows; moe_forward's shared expert reads x itself
    assert torch.equal(xd[R:].view(torch.int16), L.inp["x"].view(torch.int16))
    yd = torch.empty(R_tot, h, dtype=torch.bfloat16, device=dev)
    rde.expert_ffn(cfg, L.weights, xd, None, offsets, row_weight, yd, ws)
    assert torch.equal(yd.view(torch.int16), it["yd"].view(torch.int16))
    y = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
    rde.combine(cfg, yd, inv_pos, y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_fwd.view(torch.int16))
    assert rde.device_status(cfg, ws) == 0


def test_combine_identity_experts_closed_form():
    """With identity experts (yd = route weight x token row, shared row = the token row) combine
    returns x * (sum of the token's weights + 1)."""
    wl = SMALL["dsv3_small"]
    L = GpuLayer(wl)
    L.forward()
    it = L.intermediates()
    R = wl.T * wl.k
    xd = it["xd"].float()
    yd = torch.empty_like(it["yd"])
    yd[:R] = (xd[:R] * it["row_weight"][:, None]).to(torch.bfloat16)
    yd[R:] = L.inp["x"]
    y = torch.empty_like(L.inp["x"])
    rde.combine(L.cfg, yd, it["inv_pos"], y)
    torch.cuda.synchronize()
    x = oracle.bf16_to_double(bits(L.inp["x"]))
    wsum = it["topk_w"].double().sum(dim=1).cpu().numpy()
    ref = x * (wsum[:, None] + 1.0)
    e = rel_err_per_token(bits(y), ref)
    assert e.max() <= 2 ** -7
    assert abs(wsum.mean() - wl.routed_scale) < 1e-5  # renormalised weights sum to the scaling factor


def test_zero_tokens_is_a_no_op():
    wl = SMALL["dsv3_small"].replace(T=0)
    cfg = cfg_of(wl)
    L = GpuLayer(SMALL["dsv3_small"])
    ws = rde.alloc_workspace(cfg)
    y = torch.full((1, wl.h), 7.0, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((1, wl.h), dtype=torch.bfloat16, device="cuda")
    rde.forward(cfg, x, L.weights, y, ws)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_bad_expert_index_is_skipped_and_reported():
    wl = SMALL["dsv3_small"]
    L = GpuLayer(wl)
    L.forward()
    it = L.intermediates()
    cfg = L.cfg
    T, k, E = wl.T, wl.k, wl.E
    idx = it["topk_idx"].clone()
    idx[3, 0] = E
    idx[10, 5] = -7
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)  # a new workspace holds arbitrary bits: read and clear them first
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    inv_pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    row_token = torch.empty(T * k, dtype=torch.int32, device="cuda")
    row_weight = torch.empty(T * k, dtype=torch.float32, device="cuda")
    xd = torch.empty(T * k + T, wl.h, dtype=torch.bfloat16, device="cuda")
    rde.dispatch(cfg, L.inp["x"], idx, it["topk_w"], counts, offsets, inv_pos, row_token, row_weight, xd, None, ws)
    assert rde.device_status(cfg, ws) == rde.moe.MOE_STATUS_BAD_EXPERT_INDEX
    ip = inv_pos.cpu().numpy()
    assert ip[3, 0] == -1 and ip[10, 5] == -1
    good = idx.cpu().numpy()
    valid = (good >= 0) & (good < E)
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(good[valid], minlength=E))
    rows = ip[valid]
    assert sorted(rows.tolist()) == list(range(int(valid.sum())))


def test_timed_out_wait_is_reported_and_the_context_survives():
    """Failure detection without a fault: a bounded mbarrier wait that nothing completes gives up after
    its limit, records MOE_STATUS_WAIT_TIMEOUT, and the next layer call on the same GPU is correct."""
    wl = SMALL["dsv3_small"]
    L = GpuLayer(wl)
    rde.device_status(L.cfg, L.ws)  # clear
    rde.selftest_wait_timeout(L.cfg, L.ws, 2_000_000)  # about a millisecond of SM clock
    torch.cuda.synchronize()
    assert rde.device_status(L.cfg, L.ws) == rde.moe.MOE_STATUS_WAIT_TIMEOUT
    assert rde.device_status(L.cfg, L.ws) == 0  # read and cleared
    y = L.forward()
    assert rde.device_status(L.cfg, L.ws) == 0
    ref = oracle.bf16_to_double(bits(y))
    assert np.isfinite(ref).all()
    _check_layer_against_oracle(wl, L)


def test_fp8_dispatch_is_bit_exact():
    wl = SMALL["dsv3_small"].replace(dtype="fp8")
    cfg = cfg_of(wl)
    inp = synth.device_inputs(wl, torch, with_weights=False)
    T, k, E, h = wl.T, wl.k, wl.E, wl.h
    dev = "cuda"
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    w_only = rde.Weights(w_router=inp["w_router"], bias=inp["bias"])
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    rde.route(cfg, inp["x"], w_only, idx, w, ws=ws)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(T, k, dtype=torch.int32, device=dev)
    row_token = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_weight = torch.empty(T * k, dtype=torch.float32, device=dev)
    xd = torch.empty(T * k + T, h, dtype=torch.uint8, device=dev)
    xs = torch.empty(T * k + T, h // 128, dtype=torch.float32, device=dev)
    rde.dispatch(cfg, inp["x"], idx, w, counts, offsets, inv_pos, row_token, row_weight, xd, xs, ws)
    torch.cuda.synchronize()
    xq, xsc = oracle.quant_1x128(oracle.bf16_to_double(bits(inp["x"])))
    rt = row_token.cpu().numpy()
    np.testing.assert_array_equal(xd[:T * k].cpu().numpy(), xq[rt])
    np.testing.assert_array_equal(xs[:T * k].cpu().numpy(), xsc[rt])
    np.testing.assert_array_equal(xd[T * k:].cpu().numpy(), xq)
    np.testing.assert_array_equal(xs[T * k:].cpu().numpy(), xsc)


def test_nvfp4_weight_quantiser_is_bit_exact():
    g = torch.Generator(device="cpu").manual_seed(4)
    w = torch.randn(3, 64, 512, generator=g) * 0.02 * torch.exp(torch.randn(3, 64, 1, generator=g))
    w[1] = 0.0  # an all-zero matrix -> matrix scale 1, all codes and scales zero
    w[2, :, :16] = 0.0  # a zero block inside a nonzero matrix
    w[2, 3, 100] = 7.0  # an outlier: every other block of the matrix gets a small e4m3 scale
    wb = w.to(torch.bfloat16).cuda()
    q, sc, gs = rde.quantize_weights_nvfp4(wb)
    torch.cuda.synchronize()
    wbits = bits(wb)
    for b in range(3):
        rq, rs, rg = oracle.quant_weight_nvfp4(wbits[b])
        np.testing.assert_array_equal(q[b].cpu().numpy(), rq)
        np.testing.assert_array_equal(sc[b].cpu().numpy(), rs)
        assert gs[b].item() == rg
    assert gs[1].item() == 1.0


def test_fp8_weight_quantiser_is_bit_exact():
    g = torch.Generator(device="cpu").manual_seed(3)
    w = (torch.randn(3, 256, 384, generator=g) * 0.02)
    w[1, :128, :128] = 0.0  # an all-zero tile -> scale 1
    w[2, 5, 7] = 30.0  # an outlier in one tile
    wb = w.to(torch.bfloat16).cuda()
    q, s = rde.quantize_weights_fp8(wb)
    torch.cuda.synchronize()
    wbits = bits(wb)
    for b in range(3):
        rq, rs = oracle.quant_weight_128x128(wbits[b])
        np.testing.assert_array_equal(q[b].cpu().numpy(), rq)
        np.testing.assert_array_equal(s[b].cpu().numpy(), rs)
    assert s[1, 0, 0].item() == 1.0


@pytest.mark.parametrize("score,E,G,Gk,k", [
    ("sigmoid", 256, 8, 4, 8),  # groups of whole lanes (4 lanes of 8 experts)
    ("sigmoid", 64, 4, 2, 8),  # 8 lanes of 2 experts per group
    ("sigmoid", 96, 8, 3, 8),  # 3 experts per lane, 4 lanes per group
    ("sigmoid", 160, 5, 2, 8),  # groups that split a lane: the general group stage
    ("sigmoid", 32, 4, 2, 4),  # one expert per lane
    ("softmax", 256, 1, 1, 8),
    ("softmax", 8, 1, 1, 2),
])
def test_routing_near_ties_bit_exact(score, E, G, Gk, k):
    """Logits built to sit on decision boundaries (exact duplicates, neighbouring fp32 values, nearly
    equal group scores) route exactly as the oracle routes them."""
    rng = np.random.default_rng(21)
    T = 4096
    logits = rng.standard_normal((T, E)).astype(np.float32) * 2
    for t in range(T):
        kind = t % 4
        a = rng.choice(E, min(12, E), replace=False)
        if kind == 0:  # exact duplicates around the selection boundary
            logits[t, a] = logits[t, a[0]]
        elif kind == 1:  # neighbouring fp32 values
            v = np.float32(rng.uniform(0, 3))
            for i, e in enumerate(a):
                logits[t, e] = v
                v = np.nextafter(v, np.float32(10))
        elif kind == 2:  # two groups with nearly the same two best keys
            g0, g1 = rng.choice(G, 2, replace=False) if G > 1 else (0, 0)
            gsz = E // G
            logits[t, g0 * gsz:g0 * gsz + 2] = 4.0
            logits[t, g1 * gsz:g1 * gsz + 2] = np.nextafter(np.float32(4.0), np.float32(0))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if score == "sigmoid" else None
    wl = synth.WORKLOADS["dsv3_prefill"].replace(T=T, h=256, E=E, k=k, I=128, I_shared=0, n_group=G, topk_group=Gk,
                                                 score=score, renorm=True)
    cfg = cfg_of(wl)
    lg = torch.from_numpy(logits).cuda()
    b = None if bias is None else torch.from_numpy(bias).cuda()
    dummy_w = torch.zeros(E, 256, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    rde.route(cfg, None, rde.Weights(w_router=dummy_w, bias=b), idx, w, logits=lg, logits_given=True)
    torch.cuda.synchronize()
    ri, rw = oracle.route(logits, bias, **route_kwargs(wl))
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.parametrize("dtype,cf,pairs", [("bf16", 0.0, False), ("fp8", 0.0, False), ("bf16", 1.1, False),
                                            ("nvfp4", 0.0, False), ("bf16", 0.0, True), ("fp8", 0.0, True)])
def test_eplb_placement_matches_unplaced_layer(dtype, cf, pairs):
    """An EPLB placement (redundant replicas, card-major slots) only reorders the expert-major rows:
    the per-slot permutation matches the oracle and the layer output is bit-identical. With `pairs`
    both layouts average over 128 rows per slot, so the bf16 layers run the CTA-pair GEMMs."""
    if pairs:
        base = synth.WORKLOADS["dsv3_decode"].replace(T=2600, h=512, E=8, k=4, n_group=2, topk_group=1, I=256,
                                                      I_shared=256, zipf_s=1.2, dtype=dtype, capacity_factor=cf)
        n_cards, n_redundant = 2, 2
    else:
        base = synth.WORKLOADS["dsv3_decode"].replace(T=400, h=512, E=64, I=256, I_shared=256, zipf_s=1.2,
                                                      dtype=dtype, capacity_factor=cf)
        n_cards, n_redundant = 8, 8
    L = GpuLayer(base)
    y0 = L.forward().clone()
    it0 = L.intermediates()
    idx = it0["topk_idx"].cpu().numpy()
    load = np.bincount(idx.ravel(), minlength=base.E)
    plan = rde.eplb_plan(load, n_cards=n_cards, n_redundant=n_redundant)
    pl = rde.Placement(plan)
    cfg = rde.make_config(T=base.T, h=base.h, E=base.E, k=base.k, I=base.I, I_shared=base.I_shared,
                          n_group=base.n_group, topk_group=base.topk_group, score=base.score, renorm=base.renorm,
                          routed_scale=base.routed_scale, dtype=dtype, capacity_factor=cf, placement=pl)
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    y = torch.empty_like(y0)
    rde.forward(cfg, L.inp["x"], L.weights, y, ws)
    torch.cuda.synchronize()
    assert rde.device_status(cfg, ws) == 0
    S = pl.n_slots
    counts = rde.ws_view(ws, cfg, "counts", torch.int32, (S,)).cpu().numpy()
    offsets = rde.ws_view(ws, cfg, "offsets", torch.int32, (S + 1,)).cpu().numpy()
    inv_pos = rde.ws_view(ws, cfg, "inv_pos", torch.int32, (base.T, base.k)).cpu().numpy()
    cap = oracle.capacity(config_capacity_factor(base), base.T, base.k, base.E)
    rc, ro, ri, rt = oracle.permute_placed(idx, base.E, plan["slot_expert"], plan["slot_replica"], plan["replicas"],
                                           cap)
    np.testing.assert_array_equal(counts, rc)
    np.testing.assert_array_equal(offsets, ro)
    np.testing.assert_array_equal(inv_pos, ri)
    row_token = rde.ws_view(ws, cfg, "row_token", torch.int32, (base.T * base.k,)).cpu().numpy()
    np.testing.assert_array_equal(row_token[:ro[-1]], rt)
    assert plan["replicas"].max() > 1  # the hot experts really got replicas
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("cf", [0.0, 1.25])
def test_balance_stats_match_the_oracle_counts(cf):
    """Per-step balance read back from the workspace: rows per expert, busiest / mean, experts with
    rows and the assignments a capacity limit dropped, against the oracle's permutation of the same
    expert indices."""
    wl = SMALL["cap_skew"].replace(capacity_factor=cf)
    L = GpuLayer(wl)
    L.forward()
    idx = L.intermediates()["topk_idx"].cpu().numpy()
    b = rde.balance(L.cfg, L.ws)
    cap = oracle.capacity(config_capacity_factor(wl), wl.T, wl.k, wl.E)
    counts, offsets, _, _ = oracle.permute_capacity(idx, wl.E, cap)
    assert b["counts"] == counts.tolist()
    assert b["dropped"] == wl.T * wl.k - int(offsets[-1])
    assert b["active"] == int((counts > 0).sum())
    assert b["max_rows"] == int(counts.max())
    assert b["kept"] == int(offsets[-1])
    # busiest / mean, rounded once to fp32 by the library
    assert b["max_over_mean"] == pytest.approx(counts.max() / (offsets[-1] / wl.E), rel=2.0 ** -24)
    if cf > 0:
        assert b["dropped"] > 0 and max(b["counts"]) <= cap  # the skewed router really overflows
