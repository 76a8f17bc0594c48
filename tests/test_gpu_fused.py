"""The small-batch path of moe_forward: for T <= 4096 (dropless, one slot per expert, router on the CUDA
cores: E < 128 or not a multiple of 32) the router, top-k, counts, offsets, rows and the dispatch copy
run as one cooperative kernel. Its
results must be bit for bit those of the step entry points (moe_route + moe_dispatch, the six
standalone kernels), and the step must launch fewer kernels. The layer outputs of these shapes are
checked against the oracle in test_gpu_parity.py and test_gpu_fullsize.py."""
import pytest
import torch

import synth
import routing_dispatch_expert_gb300 as rde
from routing_dispatch_expert_gb300 import build as pkg_build
from harness import GpuLayer

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = {
    # E = 8, the largest fused batch
    "tiny": W["tiny"],
    # one token; E = 64 (one router expert block of 64), shared expert on the side stream
    "one_token": W["dsv3_prefill"].replace(name="one_token", T=1, h=256, E=64, I=128, I_shared=128),
    # E = 96: two router expert blocks (64 + 32), k = 6
    "e96": W["mixtral"].replace(name="e96", T=600, h=256, E=96, k=6, I=128),
    # E = 40 (not a multiple of 32): CUDA-core router with a partial lane group in the top-k
    "e40": W["dsv3_prefill"].replace(name="e40", T=333, h=256, E=40, k=4, n_group=4, topk_group=2, I=128,
                                     I_shared=128),
    # E = 200 (not a multiple of 32): four router expert blocks of 64 in the fused router phase, a partial
    # lane group in the top-k, sigmoid scoring without groups
    "e200": W["dsv3_prefill"].replace(name="e200", T=512, h=256, E=200, k=6, n_group=1, topk_group=1, I=128,
                                      I_shared=0),
    # FP8: the shared expert's rows are quantised by the fused copy
    "fp8": W["dsv3_fp8"].replace(name="fp8_fused", T=300, h=512, E=64, I=256, I_shared=256),
    # NVFP4 weights: bf16 copy, shared rows included
    "fp4": W["dsv3_decode_fp4"].replace(name="fp4_fused", T=130, h=256, E=64, I=256, I_shared=256),
}

@pytest.fixture(scope="module", autouse=True)
def built():
    pkg_build.build()
    synth.build()
    rde.load()


def _eq(a, b):
    if a.dtype in (torch.bfloat16, torch.float32):
        return torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))
    return torch.equal(a, b)


@pytest.mark.parametrize("name", list(CASES))
def test_fused_route_and_dispatch_equal_the_step_entry_points(name):
    wl = CASES[name]
    L = GpuLayer(wl)
    L.forward()
    assert rde.device_status(L.cfg, L.ws) == 0
    it = L.intermediates()
    T, k, E, h = wl.T, wl.k, wl.E, wl.h
    dev = "cuda"
    cfg = L.cfg
    ws = rde.alloc_workspace(cfg)
    rde.device_status(cfg, ws)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    rde.route(cfg, L.inp["x"], L.weights, idx, w, logits=logits, ws=ws)
    for a, b in ((logits, "logits"), (idx, "topk_idx"), (w, "topk_w")):
        assert _eq(a, it[b]), b
    R = T * k
    R_tot = R + (T if wl.has_shared else 0)
    fp8 = wl.dtype == "fp8"
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(T, k, dtype=torch.int32, device=dev)
    row_token = torch.empty(R, dtype=torch.int32, device=dev)
    row_weight = torch.empty(R, dtype=torch.float32, device=dev)
    xd = torch.empty(R_tot, h, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xs = torch.empty(R_tot, h // 128, dtype=torch.float32, device=dev) if fp8 else None
    rde.dispatch(cfg, L.inp["x"], idx, w, counts, offsets, inv_pos, row_token, row_weight, xd, xs, ws)
    torch.cuda.synchronize()
    for a, b in ((counts, "counts"), (offsets, "offsets"), (inv_pos, "inv_pos"), (row_token, "row_token"),
                 (row_weight, "row_weight")):
        assert _eq(a, it[b]), b
    # routed rows always; the shared expert's rows where moe_forward's dispatch writes them (FP8 and
    # NVFP4 layers; a bf16 layer's shared expert reads x on its own stream)
    n = R_tot if (wl.has_shared and wl.dtype != "bf16") else R
    assert _eq(xd[:n], it["xd"][:n])
    if fp8:
        assert _eq(xs[:n], it["xd_scales"][:n])
    assert rde.device_status(cfg, ws) == 0


@pytest.mark.parametrize("T,h,fused", [(1, 512, True), (4096, 512, True), (4097, 512, False), (2048, 4096, False)])
def test_small_batch_step_launches_fewer_kernels(T, h, fused):
    """The tiny layer (E 8, no shared expert): fused, a step is 4 launches (route-and-dispatch, gate/up,
    down, combine) instead of 9 (router, top-k, histogram, scan, rank, copy, gate/up, down, combine).
    Above 4096 tokens, or with more router and copy work than the fused kernel pays for (here h 4096), the standalone
    kernels run."""
    wl = W["tiny"].replace(T=T, h=h)
    L = GpuLayer(wl)
    L.forward()
    n0 = rde.launch_count()
    L.forward()
    n1 = rde.launch_count()
    assert n1 - n0 == (4 if fused else 9)
    assert rde.device_status(L.cfg, L.ws) == 0
