"""The layer from two host threads at once, each with its own workspace, output and stream: the
library's per-device state (launch attributes, SM count, the side stream of the shared expert) is set
up once and shared safely, and both threads get the oracle's result (routing bit-exact on their own
logits, outputs within tolerance) and the same bits as a single-threaded call."""
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import BF16_TOL, GpuLayer, bits, rel_err_per_token, route_kwargs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


@pytest.mark.parametrize("name", ["dsv3", "pairs"])
def test_two_host_threads_two_workspaces(name):
    W = synth.WORKLOADS
    # dsv3: single-CTA tiles, tensor-core router, shared expert on the side stream; pairs: CTA-pair tiles
    wl = (W["dsv3_prefill"].replace(name="threads_dsv3", T=300, h=512, E=128, I=256, I_shared=256) if name == "dsv3"
          else W["mixtral"].replace(name="threads_pairs", T=4500, h=512, I=384))
    L = GpuLayer(wl)
    y_ref = L.forward().clone()  # single-threaded reference
    results, errors = {}, []
    barrier = threading.Barrier(2)

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ws = rde.alloc_workspace(L.cfg)
                rde.device_status(L.cfg, ws)
                y = torch.empty_like(L.inp["x"])
                barrier.wait()
                for _ in range(5):
                    rde.forward(L.cfg, L.inp["x"], L.weights, y, ws)
                s.synchronize()
                status = rde.device_status(L.cfg, ws)
                logits = rde.ws_view(ws, L.cfg, "logits", torch.float32, (wl.T, wl.E)).cpu().numpy()
                idx = rde.ws_view(ws, L.cfg, "topk_idx", torch.int32, (wl.T, wl.k)).cpu().numpy()
            results[i] = (y.clone(), status, logits, idx)
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    x = bits(L.inp["x"])
    experts = [L.expert_weights_host(e) for e in range(wl.E)]
    shared = L.expert_weights_host("shared") if wl.has_shared else None
    bias = None if L.inp["bias"] is None else L.inp["bias"].cpu().numpy()
    for i in range(2):
        y, status, logits, idx = results[i]
        assert status == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), i
        ref = oracle.forward(x, L.inp["w_router"].cpu().numpy(), bias, experts, shared, logits=logits,
                             **route_kwargs(wl))
        np.testing.assert_array_equal(idx, ref["topk_idx"])
        assert rel_err_per_token(bits(y), ref["y"]).max() <= BF16_TOL
