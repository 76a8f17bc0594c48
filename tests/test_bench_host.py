"""Host-side arithmetic of the measurement (no GPU): the algorithmic FLOPs and bytes the roofline
fractions divide by, the split of the expert-GEMM bytes between the two launches, the scaling of the
committed small-case DRAM capture to a full workload, and the L2 rule of the timing."""
import json
import os

import pytest

import bench
import synth


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_gemm_bytes_split_between_the_two_launches(name):
    """gate/up + down bytes are exactly the step's expert-GEMM bytes (the shared expert, when there is
    one, has I_shared = I and counts as one more group)."""
    wl = synth.WORKLOADS[name]
    for active in (1, wl.E // 2, wl.E):
        gu, dn = bench.gemm_split_bytes(wl, active)
        assert gu + dn == pytest.approx(bench.gemm_bytes(wl, active), rel=1e-12)
        assert gu > 0 and dn > 0


def test_layer_counts_closed_form():
    """DeepSeek-V3 prefill: router 2·T·h·E, expert GEMMs 6·T·k·h·I + 6·T·h·I_shared (three h x I
    matrices per expert, two FLOPs per multiply-add); bytes: x in and y out in bf16, the fp32 router
    weight and bias, and every active expert's three bf16 matrices once."""
    wl = synth.WORKLOADS["dsv3_prefill"]
    T, h, E, k, I = 16384, 7168, 256, 8, 2048
    flops, gemm_flops, nbytes = bench.layer_counts(wl, 223)
    assert gemm_flops == 6.0 * T * k * h * I + 6.0 * T * h * I
    assert flops == 2.0 * T * h * E + gemm_flops
    assert nbytes == 4.0 * T * h + 4.0 * E * h + 4.0 * E + (223 + 1) * 3.0 * h * I * 2.0


def test_weight_bytes_per_element():
    w = {n: bench.weight_bytes(synth.WORKLOADS[n]) for n in ("dsv3_prefill", "dsv3_fp8", "dsv3_decode_fp4")}
    assert w["dsv3_prefill"] == 2.0
    assert w["dsv3_fp8"] == 1.0 + 4.0 / (128 * 128)  # e4m3 + an fp32 scale per 128 x 128 block
    assert w["dsv3_decode_fp4"] == 0.5 + 1.0 / 16  # two e2m1 codes per byte + an e4m3 scale per 16


def test_traffic_scaling_and_staleness(monkeypatch):
    """The committed capture is scaled by full / small-case algorithmic bytes; a capture taken on other
    sources than the kernel's current ones gives no traffic figure."""
    path = os.path.join(bench.ROOT, "profiles", "grouped_gemm_traffic.json")
    d = json.load(open(path))
    name, entry = next(iter(d["workloads"].items()))
    wl = synth.WORKLOADS[name]
    monkeypatch.setattr(bench, "gemm_source_sha", lambda kernel: entry["kernel_source_sha256"])
    got = bench.gemm_traffic_from_profile(wl, wl.E)
    ratio = sum(entry["measured_bytes"]) / sum(entry["small_case_algorithmic_bytes"])
    assert got == pytest.approx(ratio * sum(bench.gemm_split_bytes(wl, wl.E)) / 2.0, rel=1e-12)
    monkeypatch.setattr(bench, "gemm_source_sha", lambda kernel: "0" * 64)
    assert bench.gemm_traffic_from_profile(wl, wl.E) is None


def test_every_captured_workload_names_a_known_kernel():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "grouped_gemm_traffic.json")))
    for name, entry in d["workloads"].items():
        assert name in synth.WORKLOADS
        assert entry["kernel"] in bench.GEMM_KERNEL_SOURCES
        assert len(entry["measured_bytes"]) == len(entry["small_case_algorithmic_bytes"]) == 2


def test_l2_rule():
    """Only the tiny layer (15 MB of weights and activations) could stay in L2 between steps, so only
    it is timed with L2 flushed; the others read GBs of weights per step."""
    small = {n for n, wl in synth.WORKLOADS.items() if bench.fits_in_l2(wl)}
    assert small == {"tiny"}
    assert bench.config_of(synth.WORKLOADS["tiny"], 1)["l2"] == bench.L2_FLUSHED
    assert bench.config_of(synth.WORKLOADS["dsv3_prefill"], 1)["l2"] == bench.L2_LARGER
