"""Seeded input generator: determinism, sub-range consistency and distribution moments (CPU)."""
import numpy as np

import oracle
import synth


def test_subranges_agree_with_full_stream():
    full = synth.normal_bf16(7, synth.STREAM_WGU, 0, 5000, 0.02)
    part = synth.normal_bf16(7, synth.STREAM_WGU, 1234, 777, 0.02)
    np.testing.assert_array_equal(full[1234:1234 + 777], part)
    a = synth.uniform_f32(3, synth.STREAM_BIAS, 0, 300, -0.1, 0.1)
    np.testing.assert_array_equal(a[100:200], synth.uniform_f32(3, synth.STREAM_BIAS, 100, 100, -0.1, 0.1))


def test_streams_and_seeds_differ():
    a = synth.normal_f32(0, 1, 0, 1000, 1.0)
    assert not np.array_equal(a, synth.normal_f32(1, 1, 0, 1000, 1.0))
    assert not np.array_equal(a, synth.normal_f32(0, 2, 0, 1000, 1.0))
    np.testing.assert_array_equal(a, synth.normal_f32(0, 1, 0, 1000, 1.0))


def test_normal_and_uniform_moments():
    v = synth.normal_f32(11, 1, 0, 400000, 0.02).astype(np.float64)
    assert abs(v.mean()) < 1e-4 and abs(v.std() - 0.02) < 2e-4
    assert np.abs(v).max() < 0.02 * 6.01  # Irwin-Hall(12) support is +-6 sigma
    u = synth.uniform_f32(11, 3, 0, 200000, -0.1, 0.1).astype(np.float64)
    assert u.min() >= -0.1 and u.max() < 0.1 and abs(u.mean()) < 1e-3
    b = oracle.bf16_to_double(synth.normal_bf16(11, 1, 0, 200000, 1.0))
    assert abs(b.std() - 1.0) < 1e-2


def test_bf16_draws_are_rounded_fp32_draws():
    f = synth.normal_f32(5, 1, 0, 10000, 0.02)
    b = synth.normal_bf16(5, 1, 0, 10000, 0.02)
    np.testing.assert_array_equal(b, oracle.bf16_from_double(f.astype(np.float64)))


def test_skew_shift_moves_logits_by_log_popularity():
    wl = synth.WORKLOADS["dsv3_decode"]
    w_r = synth.router_weight(wl)
    mu = synth.skew_shift(wl, w_r)
    shift = w_r.astype(np.float64) @ mu.astype(np.float64)
    perm = np.random.default_rng(wl.seed).permutation(wl.E)
    target = np.empty(wl.E)
    target[perm] = -wl.zipf_s * np.log(np.arange(1, wl.E + 1))
    np.testing.assert_allclose(shift, target, atol=1e-3)


def test_workload_presets():
    w = synth.WORKLOADS
    assert (w["tiny"].T, w["tiny"].h, w["tiny"].E, w["tiny"].k, w["tiny"].I) == (4096, 512, 8, 2, 256)
    assert (w["mixtral"].h, w["mixtral"].I, w["mixtral"].renorm) == (4096, 14336, True)
    d = w["dsv3_prefill"]
    assert (d.T, d.h, d.E, d.k, d.I, d.I_shared, d.n_group, d.topk_group, d.routed_scale) == (
        16384, 7168, 256, 8, 2048, 2048, 8, 4, 2.5)
    assert w["dsv3_decode"].zipf_s == 1.2 and w["dsv3_fp8"].zipf_s == 1.0 and w["dsv3_fp8"].dtype == "fp8"
