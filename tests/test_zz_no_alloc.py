"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate device memory (an engine
whose memory pool owns the whole device, a plug-in hook that only sees the layer's inputs and
outputs). It takes its scratch from a static array inside the library instead of a workspace; its
outputs must equal moe_dispatch's, call after call, although every call reuses the same array.

Collected last on purpose (file name), so a run that stops at the first failure has run every other
test before this one; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from routing_dispatch_expert_gb300 import moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


def _cfg(wl):
    return rde.make_config(T=wl.T, h=wl.h, E=wl.E, k=wl.k, I=wl.I, I_shared=wl.I_shared, n_group=wl.n_group,
                           topk_group=wl.topk_group, score=wl.score, renorm=wl.renorm, routed_scale=wl.routed_scale,
                           dtype=wl.dtype)


def _outputs(wl):
    dev = "cuda"
    T, k, E, h = wl.T, wl.k, wl.E, wl.h
    R_tot = T * k + (T if wl.has_shared else 0)
    fp8 = wl.dtype == "fp8"
    return dict(counts=torch.full((E,), -1, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -1, dtype=torch.int32, device=dev),
                inv_pos=torch.full((T, k), -2, dtype=torch.int32, device=dev),
                row_token=torch.full((T * k,), -1, dtype=torch.int32, device=dev),
                row_weight=torch.full((T * k,), -1.0, dtype=torch.float32, device=dev),
                xd=torch.zeros((R_tot, h), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
                xd_scales=torch.zeros((R_tot, h // 128), dtype=torch.float32, device=dev) if fp8 else None)


def _dispatch_both_ways(wl):
    cfg = _cfg(wl)
    inp = synth.device_inputs(wl, torch, with_weights=False)
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    rde.route(cfg, inp["x"], rde.Weights(w_router=inp["w_router"], bias=inp["bias"]), idx, w, ws=ws)
    a, b = _outputs(wl), _outputs(wl)
    rde.dispatch(cfg, inp["x"], idx, w, a["counts"], a["offsets"], a["inv_pos"], a["row_token"], a["row_weight"],
                 a["xd"], a["xd_scales"], ws)
    rde.dispatch_noalloc(cfg, inp["x"], idx, w, b["counts"], b["offsets"], b["inv_pos"], b["row_token"],
                         b["row_weight"], b["xd"], b["xd_scales"])
    torch.cuda.synchronize()
    for name in a:
        if a[name] is None:
            continue
        x, y = a[name], b[name]
        if x.dtype in (torch.bfloat16, torch.float32):
            x, y = x.view(torch.int32 if x.dtype == torch.float32 else torch.int16), \
                y.view(torch.int32 if y.dtype == torch.float32 else torch.int16)
        assert torch.equal(x, y), f"{wl.name}: {name} differs from moe_dispatch"
    assert int(b["offsets"][-1]) == wl.T * wl.k


def test_matches_workspace_dispatch_on_calls_in_a_row():
    W = synth.WORKLOADS
    first = W["dsv3_prefill"].replace(name="noalloc_a", T=500, h=512, E=64, I=256, I_shared=256)
    second = W["dsv3_fp8"].replace(name="noalloc_b", T=333, h=512, E=32, I=256, I_shared=256, seed=11)
    _dispatch_both_ways(first)
    _dispatch_both_ways(second)  # same static array, other sizes and dtype
    _dispatch_both_ways(first)  # and back: nothing left over from the previous call may leak in


def test_sizes_beyond_the_static_scratch_are_rejected():
    lib = rde.load()
    wl = synth.WORKLOADS["dsv3_prefill"].replace(T=300000)  # ceil(300000 / 512) * 256 > 131072
    cfg = _cfg(wl)
    p = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    rc = lib.moe_dispatch_noalloc(ctypes.byref(cfg), p, p, p, p, p, p, p, p, p, p, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert "static scratch" in lib.moe_last_error().decode()
