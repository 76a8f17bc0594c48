"""Pins of the CPU oracle against things other than itself: values the pages print for worked
examples, library routines (torch / numpy on CPU), closed forms, invariants and brute force."""
import itertools
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------------------------------ bf16
def test_bf16_matches_torch_on_float_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-41]]).astype(np.float32)
    ours = oracle.bf16_from_double(v.astype(np.float64))
    ref = _bf16_bits(torch.from_numpy(v))
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(oracle.bf16_to_double(ours), _from_bits(ref).to(torch.float64).numpy())


def test_bf16_ties_and_single_rounding_from_double():
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,  # midpoint 1 | 1+2^-7: tie to even (down)
        1.0 + 3 * 2.0 ** -8: 0x3F82,  # midpoint 1+2^-7 | 1+2^-6: tie to even (up)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above the midpoint: a float detour would tie down
        -(1.0 + 2.0 ** -8 + 2.0 ** -30): 0xBF81,
    }
    for v, bits in cases.items():
        assert int(oracle.bf16_from_double([v])[0]) == bits, v


def test_bf16_is_nearest_of_neighbours():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(50000) * 3.0
    b = oracle.bf16_from_double(v)
    r = oracle.bf16_to_double(b)
    up = oracle.bf16_to_double((b.astype(np.int32) + 1).astype(np.uint16))
    dn = oracle.bf16_to_double((b.astype(np.int32) - 1).astype(np.uint16))
    assert np.all(np.abs(v - r) <= np.abs(v - up))
    assert np.all(np.abs(v - r) <= np.abs(v - dn))


# ------------------------------------------------------------------------------------ e4m3
def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # finite positive grid
    mids = (vals[:-1] + vals[1:]) / 2
    probes = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                             np.nextafter(mids.astype(np.float32), np.float32(1e9))]).astype(np.float32)
    rng = np.random.default_rng(3)
    probes = np.concatenate([probes, (rng.standard_normal(20000) * 50).astype(np.float32)])
    probes = np.concatenate([probes, -probes])
    probes = probes[np.abs(probes) < 464.0]  # torch turns larger magnitudes into NaN; we saturate
    ours = oracle.e4m3_encode(probes)
    ref = torch.from_numpy(probes).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_saturates():
    c = oracle.e4m3_encode(np.array([464.0, 500.0, 1e30, -1e30], np.float32))
    np.testing.assert_array_equal(c, [0x7E, 0x7E, 0x7E, 0xFE])


def test_quant_1x128_error_bound_and_zero_block():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((7, 384)) * np.exp(rng.standard_normal((7, 1)) * 3)
    v[3, 128:256] = 0.0
    q, s = oracle.quant_1x128(v)
    assert s[3, 1] == 1.0 and np.all(q[3, 128:256] == 0)
    deq = oracle.e4m3_decode(q) * np.repeat(s, 128, axis=1)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, np.repeat(s, 128, axis=1) * 2.0 ** -10)
    assert np.all(np.abs(v - deq) <= bound * (1 + 1e-6))
    # the block maximum lands on the largest code
    for r in range(7):
        for b in range(3):
            if r == 3 and b == 1:
                continue
            blk = v[r, b * 128:(b + 1) * 128]
            i = int(np.argmax(np.abs(blk)))
            assert (q[r, b * 128 + i] & 0x7F) == 0x7E
            assert s[r, b] == np.float32(np.abs(blk).max() / 448.0)


def test_quant_weight_128x128_matches_row_rule():
    rng = np.random.default_rng(5)
    w = oracle.bf16_from_double(rng.standard_normal((256, 384)) * 0.02)
    q, s = oracle.quant_weight_128x128(w)
    wd = oracle.bf16_to_double(w)
    for br in range(2):
        for bc in range(3):
            blk = wd[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128]
            sc = np.float32(np.abs(blk).max() / 448.0)
            assert s[br, bc] == sc
            ref = torch.from_numpy((blk / np.float64(sc)).astype(np.float32)).to(torch.float8_e4m3fn)
            np.testing.assert_array_equal(q[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128],
                                          ref.view(torch.uint8).numpy())


# ------------------------------------------------------------------------------------ logits
def test_router_logits_match_torch_fp64_matmul():
    rng = np.random.default_rng(6)
    x = oracle.bf16_from_double(rng.standard_normal((33, 200)))
    w = (rng.standard_normal((12, 200)) * 0.02).astype(np.float32)
    ours = oracle.router_logits(x, w)
    ref = (torch.from_numpy(oracle.bf16_to_double(x)) @ torch.from_numpy(w.astype(np.float64)).T).numpy()
    np.testing.assert_allclose(ours, ref.astype(np.float32), rtol=1e-6, atol=1e-7)


# ------------------------------------------------------------------------------------ routing
def _brute_topk(key, allowed, k):
    """k-subset of the allowed entries with the largest key sum, sorted by key descending"""
    best, best_sum = None, -math.inf
    for sub in itertools.combinations([i for i in range(len(key)) if allowed[i]], k):
        s = sum(float(key[i]) for i in sub)
        if s > best_sum:
            best, best_sum = sub, s
    return sorted(best, key=lambda i: (-float(key[i]), i))


def test_softmax_topk_brute_force_and_torch_weights():
    rng = np.random.default_rng(7)
    T, E, k = 200, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    for renorm in (False, True):
        idx, w = oracle.route(logits, None, k, score=oracle.SOFTMAX, renorm=renorm)
        p = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=-1).numpy()
        for t in range(T):
            assert list(idx[t]) == _brute_topk(logits[t], [1] * E, k)
            ref = p[t, idx[t]]
            if renorm:
                ref = ref / ref.sum()
            np.testing.assert_allclose(w[t], ref, rtol=1e-6)
        tv, ti = torch.from_numpy(logits).topk(k, dim=-1)
        np.testing.assert_array_equal(idx, ti.numpy())


def _sigmoid_f32(l):
    return (1.0 / (1.0 + np.exp(-l.astype(np.float64)))).astype(np.float32)


def test_grouped_sigmoid_topk_brute_force():
    rng = np.random.default_rng(8)
    T, E, G, Gk, k = 60, 16, 8, 4, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    idx, w = oracle.route(logits, bias, k, G, Gk, oracle.SIGMOID, True, 2.5)
    gs = E // G
    for t in range(T):
        s = _sigmoid_f32(logits[t])
        key = s + bias
        gscore = [float(np.sort(key[g * gs:(g + 1) * gs])[-2:].astype(np.float32).sum(dtype=np.float32))
                  for g in range(G)]
        best_groups, best = None, -math.inf
        for sub in itertools.combinations(range(G), Gk):
            tot = sum(gscore[g] for g in sub)
            if tot > best:
                best_groups, best = sub, tot
        allowed = [1 if (e // gs) in best_groups else 0 for e in range(E)]
        sel = _brute_topk(key, allowed, k)
        assert list(idx[t]) == sel
        ref = s[sel].astype(np.float64)
        np.testing.assert_allclose(w[t], ref / ref.sum() * 2.5, rtol=1e-6)
        assert abs(float(w[t].sum()) - 2.5) < 1e-5


def test_group_score_is_top2_sum_not_max():
    E, G = 8, 4  # groups of two experts
    logits = np.full((1, E), -10.0, np.float32)
    logits[0, 0] = 3.0  # group 0: one strong expert, one weak -> max wins, top-2 sum loses
    logits[0, 2] = logits[0, 3] = 1.0  # group 1: two good experts
    idx, _ = oracle.route(logits, None, 2, G, 1, oracle.SIGMOID, True, 1.0)
    assert sorted(idx[0]) == [2, 3]


def test_bias_selects_but_does_not_weigh():
    E = 4
    logits = np.array([[0.5, 0.4, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 0.0, 0.5, 0.0], np.float32)
    idx, w = oracle.route(logits, bias, 2, 1, 1, oracle.SIGMOID, False, 1.0)
    assert list(idx[0]) == [2, 0]  # s+bias: 0.5+0.5 beats sigmoid(0.5)
    np.testing.assert_allclose(w[0], _sigmoid_f32(logits[0])[[2, 0]], rtol=1e-7)


def test_ties_break_to_lower_index():
    logits = np.zeros((3, 256), np.float32)
    idx, _ = oracle.route(logits, None, 8, 8, 4, oracle.SIGMOID, True, 2.5)
    np.testing.assert_array_equal(idx, np.tile(np.arange(8), (3, 1)))
    idx, _ = oracle.route(logits[:, :8], None, 2, score=oracle.SOFTMAX)
    np.testing.assert_array_equal(idx, np.tile(np.arange(2), (3, 1)))
    # a tie among groups only: groups 1..3 tie, group 0 is worse -> groups 1, 2 kept
    l = np.zeros((1, 16), np.float32)
    l[0, 0:4] = -1.0
    idx, _ = oracle.route(l, None, 8, 4, 2, oracle.SIGMOID, True, 1.0)
    assert sorted(idx[0]) == list(range(4, 12))


def test_p3_worked_example_histogram():
    """The page's seeded routing snippet: recomputed logits routed by the oracle give the printed
    per-expert and per-GPU counts."""
    g = json.load(open(os.path.join(GOLDEN, "p3_routing_histogram.json")))
    torch.manual_seed(g["seed"])
    tokens = torch.randn(g["tokens"], g["hidden"])
    lin = torch.nn.Linear(g["hidden"], g["experts"])
    with torch.no_grad():
        logits = lin(tokens).numpy()
    idx, _ = oracle.route(logits, None, g["top_k"], score=oracle.SOFTMAX)
    counts, offsets, _, _ = oracle.permute(idx, g["experts"])
    assert counts.min() == g["expert_count_min"] and counts.max() == g["expert_count_max"]
    assert counts.sum() == g["assignments"] == offsets[-1]
    per_gpu = counts.reshape(g["gpus"], -1).sum(axis=1)
    assert per_gpu.min() == g["gpu_count_min"] and per_gpu.max() == g["gpu_count_max"]
    _, ti = torch.from_numpy(logits).topk(g["top_k"], dim=-1)
    np.testing.assert_array_equal(idx, ti.numpy())


# ------------------------------------------------------------------------------------ permute
def test_permute_invariants_and_stable_sort():
    rng = np.random.default_rng(9)
    T, E, k = 500, 16, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, inv_pos, row_token = oracle.permute(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    np.testing.assert_array_equal(np.diff(offsets), counts)
    # bijection: every row used once, and it holds the right token
    assert sorted(inv_pos.ravel().tolist()) == list(range(T * k))
    np.testing.assert_array_equal(row_token[inv_pos], np.repeat(np.arange(T), k).reshape(T, k))
    # expert-major, ascending token: the stable sort of the flattened (token, slot) list by expert
    order = np.argsort(idx.ravel(), kind="stable")
    np.testing.assert_array_equal(row_token, order // k)


def test_gather_rows_matches_fancy_indexing():
    rng = np.random.default_rng(10)
    x = rng.integers(0, 65535, (40, 24), dtype=np.uint16)
    rt = rng.integers(0, 40, 100).astype(np.int32)
    np.testing.assert_array_equal(oracle.gather_rows(x, rt), x[rt])


# ------------------------------------------------------------------------------------ experts
def _torch_swiglu(x_bf16, w_gu, w_d, I):
    x = torch.from_numpy(oracle.bf16_to_double(x_bf16))
    gu = torch.from_numpy(oracle.bf16_to_double(w_gu))
    d = torch.from_numpy(oracle.bf16_to_double(w_d))
    g = x @ gu[:I].T
    u = x @ gu[I:].T
    a = (torch.nn.functional.silu(g) * u).to(torch.float32).to(torch.bfloat16).to(torch.float64)
    return (a @ d.T).numpy()


def test_expert_ffn_bf16_matches_torch_swiglu():
    rng = np.random.default_rng(11)
    m, h, I = 9, 256, 128
    x = oracle.bf16_from_double(rng.standard_normal((m, h)))
    w_gu = oracle.bf16_from_double(rng.standard_normal((2 * I, h)) * 0.02)
    w_d = oracle.bf16_from_double(rng.standard_normal((h, I)) * 0.02)
    ours = oracle.expert_ffn_bf16(x, w_gu, w_d)
    ref = _torch_swiglu(x, w_gu, w_d, I)
    assert np.abs(ours - ref).max() <= 1e-3 * np.abs(ref).max()
    # swapping gate and up is a different function: the pin must be able to see it
    swapped = np.concatenate([w_gu[I:], w_gu[:I]])
    assert np.abs(_torch_swiglu(x, swapped, w_d, I) - ours).max() > 1e-2 * np.abs(ref).max()


def test_expert_ffn_fp8_matches_torch_dequantised():
    rng = np.random.default_rng(12)
    m, h, I = 5, 256, 256
    x = oracle.bf16_from_double(rng.standard_normal((m, h)))
    w_gu = oracle.bf16_from_double(rng.standard_normal((2 * I, h)) * 0.02)
    w_d = oracle.bf16_from_double(rng.standard_normal((h, I)) * 0.02)
    xq, xs = oracle.quant_1x128(oracle.bf16_to_double(x))
    gq, gs = oracle.quant_weight_128x128(w_gu)
    dq, ds = oracle.quant_weight_128x128(w_d)
    ours = oracle.expert_ffn_fp8(xq, xs, gq, gs, dq, ds)

    def deq(q, s, bm, bn):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64)
        return v * torch.from_numpy(s.astype(np.float64)).repeat_interleave(bm, 0).repeat_interleave(bn, 1)

    xdq = deq(xq, xs, 1, 128)
    g = xdq @ deq(gq, gs, 128, 128)[:I].T
    u = xdq @ deq(gq, gs, 128, 128)[I:].T
    a = (torch.nn.functional.silu(g) * u).numpy()
    aq, as_ = oracle.quant_1x128(a)
    ref = (deq(aq, as_, 1, 128) @ deq(dq, ds, 128, 128).T).numpy()
    assert np.abs(ours - ref).max() <= 1e-4 * np.abs(ref).max()


# ------------------------------------------------------------------------------------ NVFP4 (e2m1)
# OCP Microscaling formats specification, FP4 E2M1 element: the 8 magnitudes of codes 0..7
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_all_codes_match_the_format_table():
    for c in range(16):
        v = float(oracle.e2m1_decode(c))
        assert v == (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)  # -0 keeps its sign


def test_e2m1_encode_is_nearest_with_ties_to_even_code():
    # brute force: argmin distance over the table, ties to the code whose mantissa bit is 0
    def ref(f):
        a = min(abs(f), 6.0)
        d = [abs(a - v) for v in E2M1_TABLE]
        best = min(d)
        cands = [c for c in range(8) if d[c] == best]
        code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        return code | (8 if math.copysign(1.0, f) < 0 else 0)

    rng = np.random.default_rng(21)
    xs = np.concatenate([np.linspace(-8, 8, 3201), rng.standard_normal(2000) * 3,
                         [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 1e9, -1e9, 0.0, -0.0]])
    xs = xs.astype(np.float32)
    ours = oracle.e2m1_encode(xs)
    want = np.array([ref(float(f)) for f in xs], np.uint8)
    np.testing.assert_array_equal(ours, want)


def _nvfp4_gap(a):
    """spacing of the e2m1 grid around magnitude a (in units of the block's value scale)"""
    return np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))


def test_quant_weight_nvfp4_error_bound_block_max_and_packing():
    rng = np.random.default_rng(22)
    rows, cols = 64, 256
    w = oracle.bf16_from_double(rng.standard_normal((rows, cols)) * 0.02 * np.exp(rng.standard_normal((rows, 1))))
    wv = oracle.bf16_to_double(w)
    q, sc, g = oracle.quant_weight_nvfp4(w)
    amax = np.abs(wv).max()
    assert g == float(np.float32(amax) / np.float32(2688.0))  # the matrix maps onto 6 x 448
    deq = oracle.dequant_nvfp4(q, sc, g)
    p = (oracle.e4m3_decode(sc) * g).repeat(16, axis=1)  # value of one e2m1 step 1.0, per element
    # round to nearest on the e2m1 grid: within half a grid step (saturation at 6 included: the
    # block scale is rounded to e4m3, at most 1/16 relative, so a block max lands in [5.6, 6.4])
    err = np.abs(deq - wv)
    assert np.all(err <= p * _nvfp4_gap(np.abs(wv) / p) / 2 * (1 + 1e-6) + 1e-30)
    # the largest element of every block with a normal (not subnormal) e4m3 scale sits at the top of
    # the grid: code magnitude 7 (value 6)
    codes = np.empty((rows, cols), np.uint8)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    blk = np.abs(wv).reshape(rows, cols // 16, 16).argmax(axis=2)
    top = np.take_along_axis(codes.reshape(rows, cols // 16, 16), blk[..., None], axis=2)[..., 0]
    normal = ((sc >> 3) & 15) > 0
    assert normal.mean() > 0.9 and np.all((top[normal] & 7) == 7)
    # element 2i is the low nibble: a single nonzero element 1 lands in the high nibble of byte 0
    one = np.zeros((1, 16), np.uint16)
    one[0, 1] = oracle.bf16_from_double(np.array([0.5]))[0]
    q1, s1, g1 = oracle.quant_weight_nvfp4(one)
    assert q1[0, 0] == 0x70 and np.all(q1[0, 1:] == 0)
    assert float(oracle.dequant_nvfp4(q1, s1, g1)[0, 1]) == pytest.approx(0.5, rel=1e-6)


def test_quant_weight_nvfp4_zero_matrix_and_zero_block():
    q, sc, g = oracle.quant_weight_nvfp4(np.zeros((4, 32), np.uint16))
    assert g == 1.0 and np.all(q == 0) and np.all(sc == 0)
    w = np.zeros((2, 32), np.uint16)
    w[:, 16:] = oracle.bf16_from_double(np.linspace(-1, 1, 32).reshape(2, 16))
    q, sc, g = oracle.quant_weight_nvfp4(w)
    assert np.all(sc[:, 0] == 0) and np.all(q[:, :8] == 0) and np.all(sc[:, 1] != 0)


def test_quant_weight_nvfp4_grid_values_round_trip():
    # a matrix whose entries are e2m1 grid values times a power of two (each block holding a 6)
    rng = np.random.default_rng(23)
    v = np.array(E2M1_TABLE)[rng.integers(0, 8, (8, 64))] * np.where(rng.random((8, 64)) < 0.5, -1, 1)
    v[:, ::16] = 6.0
    w = oracle.bf16_from_double(v * 2.0 ** -5)
    q, sc, g = oracle.quant_weight_nvfp4(w)
    np.testing.assert_allclose(oracle.dequant_nvfp4(q, sc, g), v * 2.0 ** -5, rtol=1e-6, atol=0)


def test_expert_ffn_nvfp4_matches_torch_swiglu_on_dequantised_weights():
    rng = np.random.default_rng(24)
    m, h, I = 7, 256, 128
    x = oracle.bf16_from_double(rng.standard_normal((m, h)))
    w_gu = oracle.bf16_from_double(rng.standard_normal((2 * I, h)) * 0.02)
    w_d = oracle.bf16_from_double(rng.standard_normal((h, I)) * 0.02)
    gu4, d4 = oracle.quant_weight_nvfp4(w_gu), oracle.quant_weight_nvfp4(w_d)
    ours = oracle.expert_ffn_nvfp4(x, gu4, d4)
    xs = torch.from_numpy(oracle.bf16_to_double(x))
    wg = torch.from_numpy(oracle.dequant_nvfp4(*gu4))
    wd = torch.from_numpy(oracle.dequant_nvfp4(*d4))
    a = torch.nn.functional.silu(xs @ wg[:I].T) * (xs @ wg[I:].T)
    a = a.to(torch.bfloat16).to(torch.float64)  # the SwiGLU product is stored in bf16
    ref = (a @ wd.T).numpy()
    assert np.abs(ours - ref).max() <= 1e-6 * np.abs(ref).max()


# ------------------------------------------------------------------------------------ combine
def test_combine_identity_experts_closed_form():
    """Identity experts: y = x * sum_j w_j (+ x with an identity shared expert)."""
    rng = np.random.default_rng(13)
    T, k, h = 50, 8, 64
    x = oracle.bf16_from_double(rng.standard_normal((T, h)))
    xd = oracle.bf16_to_double(x)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    o = np.repeat(xd[:, None, :], k, axis=1)
    y = oracle.combine(o, w, None)
    ref = oracle.bf16_from_double(xd * w.astype(np.float64).sum(axis=1, keepdims=True))
    np.testing.assert_array_equal(y, ref)
    y2 = oracle.combine(o, w, xd)
    ref2 = oracle.bf16_from_double(xd * (w.astype(np.float64).sum(axis=1, keepdims=True) + 1.0))
    np.testing.assert_array_equal(y2, ref2)
    # renormalised softmax weights sum to one: identity experts return x itself
    _, wr = oracle.route(rng.standard_normal((T, 8)).astype(np.float32), None, 2, score=oracle.SOFTMAX, renorm=True)
    np.testing.assert_array_equal(oracle.combine(o[:, :2], wr, None), x)


def test_forward_single_expert_is_dense_mlp():
    """E = 1, k = 1, softmax: every token goes to expert 0 with weight 1 -> a dense SwiGLU MLP."""
    rng = np.random.default_rng(14)
    T, h, I = 20, 128, 128
    x = oracle.bf16_from_double(rng.standard_normal((T, h)))
    w_r = (rng.standard_normal((1, h)) * 0.02).astype(np.float32)
    w_gu = oracle.bf16_from_double(rng.standard_normal((2 * I, h)) * 0.02)
    w_d = oracle.bf16_from_double(rng.standard_normal((h, I)) * 0.02)
    out = oracle.forward(x, w_r, None, [(w_gu, w_d)], None, k=1, renorm=False)
    np.testing.assert_array_equal(out["topk_idx"], 0)
    np.testing.assert_allclose(out["topk_w"], 1.0)
    ref = _torch_swiglu(x, w_gu, w_d, I)
    y = oracle.bf16_to_double(out["y"])
    assert np.abs(y - ref).max() <= 2 ** -8 * np.abs(ref).max()


# ------------------------------------------------------------------------------------ imbalance
def _p5_sampler(n_experts, top_k, n_tokens, skew, seed):
    """Token-to-expert counts under a shuffled power-law popularity, drawn in the same order as the
    page's simulation so the printed numbers reproduce."""
    rng = random.Random(seed)
    popularity = [(r + 1) ** (-skew) for r in range(n_experts)]
    rng.shuffle(popularity)
    experts = list(range(n_experts))
    counts = [0] * n_experts
    for _ in range(n_tokens):
        picked = set()
        while len(picked) < top_k:
            picked.add(rng.choices(experts, weights=popularity)[0])
        for e in picked:
            counts[e] += 1
    return counts


def test_p5_imbalance_table():
    g = json.load(open(os.path.join(GOLDEN, "p5_imbalance.json")))
    c = _p5_sampler(g["experts"], g["top_k"], g["tokens"], g["skew"], g["seed"])
    assert max(c) == g["hottest"] and min(c) == g["coldest"]
    assert sum(c) / len(c) == g["average"]
    for ep, val in g["contiguous_imbalance"].items():
        assert round(oracle.imbalance(c, int(ep)), 2) == pytest.approx(val)


# ------------------------------------------------------------------------------------ capacity
def test_capacity_keeps_the_earliest_tokens():
    rng = np.random.default_rng(15)
    T, E, k = 300, 8, 2
    pop = np.array([8, 4, 2, 1, 1, 1, 1, 1], np.float64)
    idx = np.stack([rng.choice(E, k, replace=False, p=pop / pop.sum()) for _ in range(T)]).astype(np.int32)
    cap = oracle.capacity(1.25, T, k, E)
    assert cap == int(np.ceil(1.25 * T * k / E))
    counts, offsets, inv_pos, row_token = oracle.permute_capacity(idx, E, cap)
    full = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(counts, np.minimum(full, cap))
    assert full.max() > cap  # the skew really overflows some expert
    for e in range(E):
        toks = np.nonzero((idx == e).any(axis=1))[0]  # tokens choosing e, ascending
        kept = toks[:cap]
        np.testing.assert_array_equal(row_token[offsets[e]:offsets[e + 1]], kept)
        for t in toks[cap:]:
            assert inv_pos[t, list(idx[t]).index(e)] == -1
    # rows of kept entries point back at their token
    ok = inv_pos >= 0
    np.testing.assert_array_equal(row_token[inv_pos[ok]], np.nonzero(ok)[0])


def test_capacity_above_the_largest_load_is_dropless():
    rng = np.random.default_rng(16)
    idx = np.stack([rng.choice(16, 4, replace=False) for _ in range(200)]).astype(np.int32)
    a = oracle.permute(idx, 16)
    b = oracle.permute_capacity(idx, 16, 10 ** 6)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


# ------------------------------------------------------------------------------------ placement
def test_p5_placement_table():
    """The page's table: busiest card / mean after rebalancing, and with one redundant expert per
    card, reproduced by the oracle's planner on the seeded loads."""
    g = json.load(open(os.path.join(GOLDEN, "p5_imbalance.json")))
    c = _p5_sampler(g["experts"], g["top_k"], g["tokens"], g["skew"], g["seed"])
    for ep, val in g["rebalance_imbalance"].items():
        _, _, _, card = oracle.eplb_plan(c, int(ep), 0)
        assert round(oracle.placement_imbalance(card), 2) == pytest.approx(val), ep
    for ep, val in g["redundant_imbalance"].items():
        reps, slot_expert, _, card = oracle.eplb_plan(c, int(ep), int(ep))
        assert reps.sum() == g["experts"] + int(ep)
        assert round(oracle.placement_imbalance(card), 2) == pytest.approx(val), ep


def test_placed_permutation_round_robin():
    rng = np.random.default_rng(17)
    T, E, k = 120, 8, 2
    idx = np.stack([rng.choice(E, k, replace=False, p=[.5, .2, .1, .05, .05, .04, .03, .03])
                    for _ in range(T)]).astype(np.int32)
    load = np.bincount(idx.ravel(), minlength=E)
    reps, slot_expert, slot_replica, _ = oracle.eplb_plan(load, 2, 2)
    counts, offsets, inv_pos, row_token = oracle.permute_placed(idx, E, slot_expert, slot_replica, reps)
    assert counts.sum() == T * k and sorted(inv_pos.ravel()) == list(range(T * k))
    np.testing.assert_array_equal(row_token[inv_pos], np.repeat(np.arange(T), k).reshape(T, k))
    for s in range(len(slot_expert)):  # slot s holds every reps-th token of its expert, in order
        e, i = slot_expert[s], slot_replica[s]
        toks = np.nonzero((idx == e).any(axis=1))[0]
        np.testing.assert_array_equal(row_token[offsets[s]:offsets[s + 1]], toks[i::reps[e]])
    # without redundancy and in expert order, the placed permutation is the plain one
    ident = np.arange(E, dtype=np.int32)
    a = oracle.permute_placed(idx, E, ident, np.zeros(E, np.int32), np.ones(E, np.int32))
    b = oracle.permute(idx, E)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
