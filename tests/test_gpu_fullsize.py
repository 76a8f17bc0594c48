"""CUDA path vs the oracle at the full sizes of the measured workloads, in the launch configuration
the bench times (moe_forward): full routing and permutation bit-exact, sampled dispatch rows
bit-exact, the router GEMM of every token within its derived error bound, and the expert rows,
shared-expert rows and layer outputs of a large token sample within tolerance.

The sample (at least 2048 seeded tokens for the expert FFN and the combine) holds 2048
seeded random tokens plus forced ones: for every expert with rows, the tokens of the first and last
row of its last 128-row tile (the ragged tail a grouped GEMM tile covers only partly, which the
CTA-pair kernel runs as a half tile), and for the four busiest experts 64 tokens spread over their
rows (the long groups the tile scheduler walks in bands). The tiny layer (4096 tokens) and the decode
layers (256 tokens) are checked on every token."""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import (BF16_TOL, FP8_TOL, U32, WEIGHT_RTOL, GpuLayer, bits, cfg_of, logit_tolerance, oracle_tokens,
                     rel_err_per_token, route_kwargs, router_abs_sum)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _sample(n, count, seed):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    s.update({0, n - 1})
    return np.array(sorted(s))


def _forced_tokens(counts, offsets, row_token, n_hot=4, per_hot=64):
    """Tokens of each expert's last 128-row tile (its first and last row) and, for the n_hot busiest
    experts, per_hot tokens spread evenly over their rows."""
    toks = set()
    for e in np.nonzero(counts)[0]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        last_tile = lo + 128 * ((hi - lo - 1) // 128)
        toks.update((int(row_token[last_tile]), int(row_token[hi - 1])))
    for e in np.argsort(-counts, kind="stable")[:n_hot]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for r in np.linspace(lo, hi - 1, num=min(per_hot, hi - lo)).astype(np.int64):
            toks.add(int(row_token[r]))
    return toks


def _rel_rows(got, ref):
    return np.abs(got - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)


@pytest.mark.parametrize("name,n_tok", [("tiny", None), ("mixtral", 2048), ("dsv3_prefill", 2048), ("dsv3_decode", None),
                                        ("dsv3_fp8", 2048), ("dsv3_decode_fp4", None)])
def test_full_size_layer(name, n_tok):
    wl = synth.WORKLOADS[name]
    L = GpuLayer(wl)
    y = L.forward()
    assert rde.device_status(L.cfg, L.ws) == 0
    it = L.intermediates()
    x = bits(L.inp["x"])
    bias = None if L.inp["bias"] is None else L.inp["bias"].cpu().numpy()
    logits = it["logits"].cpu().numpy()
    # routing of every token, from the same logits: bit-exact indices
    idx, w = oracle.route(logits, bias, **route_kwargs(wl))
    np.testing.assert_array_equal(it["topk_idx"].cpu().numpy(), idx)
    np.testing.assert_allclose(it["topk_w"].cpu().numpy(), w, rtol=WEIGHT_RTOL, atol=1e-7)
    # aggregation and permutation of every row: bit-exact
    counts, offsets, inv_pos, row_token = oracle.permute(idx, wl.E)
    np.testing.assert_array_equal(it["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(it["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(it["inv_pos"].cpu().numpy(), inv_pos)
    np.testing.assert_array_equal(it["row_token"].cpu().numpy(), row_token)
    # dispatch copies of sampled rows: bit-exact
    R = wl.T * wl.k
    fp8 = wl.dtype == "fp8"
    tol = FP8_TOL if fp8 else BF16_TOL
    rows = _sample(R, 512, 1)
    sel = torch.as_tensor(rows, device="cuda")
    if fp8:
        xq, xsc = oracle.quant_1x128(oracle.bf16_to_double(x[row_token[rows]]))
        np.testing.assert_array_equal(it["xd"][sel].cpu().numpy(), xq)
        np.testing.assert_array_equal(it["xd_scales"][sel].cpu().numpy(), xsc)
    else:
        np.testing.assert_array_equal(bits(it["xd"][sel]), x[row_token[rows]])
    # router GEMM of every token vs the fp64 oracle, within the derived bound
    w_r = L.inp["w_router"].cpu().numpy()
    lo = oracle.router_logits(x, w_r)
    dev = np.abs(logits.astype(np.float64) - lo)
    assert np.all(dev <= logit_tolerance(wl, x, w_r, lo))
    ratio = (dev / np.maximum(router_abs_sum(x, w_r), 1e-30)).max() / U32
    print(f"\n{name}: router logits, max |GPU - oracle| / sum|x w| = {ratio:.2f} U32 (every token)")

    # layer output, expert rows and shared rows of the token sample
    if n_tok is None:
        toks = np.arange(wl.T)
    else:
        toks = np.array(sorted(set(_sample(wl.T, n_tok, 3).tolist()) | _forced_tokens(counts, offsets, row_token)))
    y_ref, o, shared = oracle_tokens(L, toks, idx, w, x)
    tsel = torch.as_tensor(toks, device="cuda")
    e = rel_err_per_token(bits(y[tsel]), y_ref)
    assert e.max() <= tol, f"layer output: max rel err {e.max()}"
    # every (token, slot) row of yd: route-weighted expert output
    yd = oracle.bf16_to_double(bits(it["yd"][torch.as_tensor(inv_pos[toks].ravel(), device="cuda")]))
    ref = (o * w[toks][:, :, None].astype(np.float64)).reshape(-1, wl.h)
    er = _rel_rows(yd, ref)
    assert er.max() <= tol, f"expert rows: max rel err {er.max()}"
    if wl.has_shared:
        ys = oracle.bf16_to_double(bits(it["yd"][torch.as_tensor(R + toks, device="cuda")]))
        es = _rel_rows(ys, shared)
        assert es.max() <= tol, f"shared rows: max rel err {es.max()}"
    print(f"{name}: {len(toks)} tokens, {len(toks) * wl.k} expert rows; max rel err: output {e.max():.2e}, "
          f"expert rows {er.max():.2e}" + (f", shared rows {es.max():.2e}" if wl.has_shared else ""))
    del L
    gc.collect()
    torch.cuda.empty_cache()


def test_full_size_fp8_routing_and_dispatch():
    """The FP8 layer's routing, permutation and 1x128 activation quantisation at full size."""
    wl = synth.WORKLOADS["dsv3_fp8"]
    cfg = cfg_of(wl)
    inp = synth.device_inputs(wl, torch, with_weights=False)
    T, k, E, h = wl.T, wl.k, wl.E, wl.h
    dev = "cuda"
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    w_only = rde.Weights(w_router=inp["w_router"], bias=inp["bias"])
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    rde.route(cfg, inp["x"], w_only, idx, w, logits=logits, ws=ws)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(T, k, dtype=torch.int32, device=dev)
    row_token = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_weight = torch.empty(T * k, dtype=torch.float32, device=dev)
    xd = torch.empty(T * k + T, h, dtype=torch.uint8, device=dev)
    xs = torch.empty(T * k + T, h // 128, dtype=torch.float32, device=dev)
    rde.dispatch(cfg, inp["x"], idx, w, counts, offsets, inv_pos, row_token, row_weight, xd, xs, ws)
    assert rde.device_status(cfg, ws) == 0
    ri, rw = oracle.route(logits.cpu().numpy(), inp["bias"].cpu().numpy(), **route_kwargs(wl))
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=WEIGHT_RTOL, atol=1e-7)
    c, off, ip, rt = oracle.permute(ri, E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), off)
    np.testing.assert_array_equal(inv_pos.cpu().numpy(), ip)
    # Zipf(1.0) skew: the hottest expert takes far more than the mean
    assert c.max() > 4 * c.mean()
    rows = _sample(T * k, 256, 4)
    x = bits(inp["x"])
    xq, xsc = oracle.quant_1x128(oracle.bf16_to_double(x[rt[rows]]))
    sel = torch.as_tensor(rows, device=dev)
    np.testing.assert_array_equal(xd[sel].cpu().numpy(), xq)
    np.testing.assert_array_equal(xs[sel].cpu().numpy(), xsc)
