"""The layer captured as a CUDA graph (moe_graph_*) and the per-batch-size graph cache with padding
(Perplexity blog, "CUDA Graph"; TensorRT-LLM "DeepSeek R1 throughput on Blackwell", runtime
optimisations: graphs per batch size, padded to the nearest captured size). Replays are checked
against the oracle (routing bit-exact on the replay's own logits, outputs within tolerance), and
against the eager moe_forward bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import BF16_TOL, GpuLayer, bits, cfg_of, rel_err_per_token, route_kwargs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _check_with_oracle(L: GpuLayer, x: torch.Tensor, y: torch.Tensor, ws, cfg, T: int):
    """Routing of the first T tokens (bit-exact, from the logits the replay left in ws) and their
    outputs (per-token relative error) against the oracle's layer."""
    wl = L.wl
    xb = bits(x[:T])
    logits = rde.ws_view(ws, cfg, "logits", torch.float32, (cfg.T, wl.E))[:T].cpu().numpy()
    idx = rde.ws_view(ws, cfg, "topk_idx", torch.int32, (cfg.T, wl.k))[:T].cpu().numpy()
    experts = [L.expert_weights_host(e) for e in range(wl.E)]
    shared = L.expert_weights_host("shared") if wl.has_shared else None
    bias = None if L.inp["bias"] is None else L.inp["bias"].cpu().numpy()
    ref = oracle.forward(xb, L.inp["w_router"].cpu().numpy(), bias, experts, shared, logits=logits,
                         **route_kwargs(wl))
    np.testing.assert_array_equal(idx, ref["topk_idx"])
    e = rel_err_per_token(bits(y[:T]), ref["y"])
    assert e.max() <= BF16_TOL, f"T={T}: max rel err {e.max()}"


@pytest.mark.parametrize("name", ["dsv3", "tiny"])
def test_graph_replay_matches_eager(name):
    W = synth.WORKLOADS
    wl = (W["dsv3_prefill"].replace(T=300, h=512, E=64, I=256, I_shared=256) if name == "dsv3"
          else W["tiny"].replace(T=1000))
    L = GpuLayer(wl)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        y_eager = L.forward().clone()
        x_static = L.inp["x"].clone()
        y_static = torch.empty_like(y_eager)
        ws = rde.alloc_workspace(L.cfg)
        rde.device_status(L.cfg, ws)
        g = rde.Graph(L.cfg, x_static, L.weights, y_static, ws, stream)
        y_static.zero_()
        g.launch()
        stream.synchronize()
        assert _same(y_static, y_eager)
        _check_with_oracle(L, x_static, y_static, ws, L.cfg, wl.T)
        # new inputs in the same buffer: the replay follows them
        x2 = synth.device_normal_bf16(torch, tuple(x_static.shape), 99, synth.STREAM_X, 1.0)
        x_static.copy_(x2)
        g.launch()
        stream.synchronize()
        _check_with_oracle(L, x_static, y_static, ws, L.cfg, wl.T)
        L.inp["x"].copy_(x2)
        y2 = L.forward()
        stream.synchronize()
        assert _same(y_static, y2)
        assert rde.device_status(L.cfg, ws) == 0
    del g


def test_graph_cache_pads_to_captured_sizes():
    wl = synth.WORKLOADS["dsv3_decode"].replace(T=64, h=512, E=64, I=256, I_shared=256)
    L = GpuLayer(wl)
    make_cfg = lambda t: cfg_of(wl.replace(T=t))  # noqa: E731
    G = rde.GraphedMoeLayer(make_cfg, L.weights, sizes=[1, 2, 4, 8, 16, 32, 64], h=wl.h)
    for T in (1, 3, 17, 64):
        x = L.inp["x"][:T].contiguous()
        out = G(x)
        torch.cuda.synchronize()
        t_pad = G.padded_size(T)
        assert t_pad == {1: 1, 3: 4, 17: 32, 64: 64}[T]
        # the padded replay against the oracle on the real tokens
        _check_with_oracle(L, x, out, G.ws, make_cfg(t_pad), T)
        # and against an eager call of the unpadded size, bit for bit
        ref = torch.empty_like(x)
        cfg = make_cfg(T)
        ws = rde.alloc_workspace(cfg)
        rde.forward(cfg, x, L.weights, ref, ws)
        torch.cuda.synchronize()
        assert _same(out, ref), T
    with pytest.raises(ValueError):
        G.padded_size(65)
