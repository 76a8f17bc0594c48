"""The layer captured as a CUDA graph (moe_graph_*) and the per-batch-size graph cache with padding:
replays give bit-for-bit the eager moe_forward result."""
import pytest
import torch

import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import GpuLayer, cfg_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


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
        # new inputs in the same buffer: the replay follows them
        x2 = synth.device_normal_bf16(torch, tuple(x_static.shape), 99, synth.STREAM_X, 1.0)
        x_static.copy_(x2)
        g.launch()
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
        ref = torch.empty_like(x)
        cfg = make_cfg(T)
        ws = rde.alloc_workspace(cfg)
        rde.forward(cfg, x, L.weights, ref, ws)
        torch.cuda.synchronize()
        assert G.padded_size(T) == {1: 1, 3: 4, 17: 32, 64: 64}[T]
        assert _same(out, ref), T
    with pytest.raises(ValueError):
        G.padded_size(65)
