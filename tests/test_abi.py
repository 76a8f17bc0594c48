"""The C ABI library: it builds for sm_103a, exports every entry point include/moe.h declares, and
rejects bad arguments before touching a GPU (these calls return before any CUDA call)."""
import ctypes
import os
import re

import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

from routing_dispatch_expert_gb300 import build as pkg_build
from routing_dispatch_expert_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_steps():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward", "moe_workspace_size",
              "moe_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_sizes_match_header_layout():
    assert ctypes.sizeof(moe.MoeConfig) == 13 * 4 + 4 + 8  # 13 scalars, padding, placement pointer
    assert ctypes.sizeof(moe.MoePlacement) == 2 * 4 + 4 * 8
    assert ctypes.sizeof(moe.MoeWeightsStruct) == 14 * 8
    assert ctypes.sizeof(moe.MoeWsLayout) == 16 * 8


def _cfg(**kw):
    base = dict(T=64, h=256, E=8, k=2, I=128)
    base.update(kw)
    return moe.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=0), moe.MOE_ERR_INVALID),
    (dict(k=9), moe.MOE_ERR_INVALID),
    (dict(E=12, n_group=5, topk_group=1), moe.MOE_ERR_INVALID),
    (dict(E=16, n_group=4, topk_group=5), moe.MOE_ERR_INVALID),
    (dict(E=16, k=8, n_group=8, topk_group=2), moe.MOE_ERR_INVALID),  # 2 groups of 2 hold < 8 experts
    (dict(h=200), moe.MOE_ERR_UNSUPPORTED),
    (dict(I=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(I_shared=256), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=2048, k=2), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_INVALID),
    (dict(dtype="nvfp4", I=128), moe.MOE_ERR_UNSUPPORTED),  # NVFP4 block scales need I % 256 == 0
])
def test_config_validation(lib, kw, code):
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(_cfg(**kw)), ctypes.byref(n)) == code
    assert lib.moe_last_error().decode() != ""


def test_workspace_layout_is_ordered_and_aligned(lib):
    for score, shared, dtype in (("softmax", 0, "bf16"), ("sigmoid", 128, "bf16"), ("sigmoid", 128, "fp8")):
        cfg = _cfg(E=16, k=4, n_group=4, topk_group=2, score=score, I_shared=shared, dtype=dtype)
        lay = moe.workspace_layout(cfg)
        offs = [lay[n] for n, _ in moe.MoeWsLayout._fields_]
        assert offs == sorted(offs)
        assert all(o % 256 == 0 for o in offs)
        R_tot = 64 * 4 + (64 if shared else 0)
        assert lay["yd"] - lay["hbuf"] >= (1 if dtype == "fp8" else 2) * R_tot * 128
        assert lay["total"] == moe.workspace_size(cfg)


def test_scratch_holds_the_router_partial_sums_of_small_batches(lib):
    """The tensor-core router (E >= 128) splits the K range of each 128 x 128 output tile over several
    CTAs when a batch has fewer than 64 tiles; their fp32 partial sums live at the end of the scratch
    region. A large batch needs none, so its scratch is the fixed part only."""
    def scratch_bytes(T, E, h):
        lay = moe.workspace_layout(_cfg(T=T, E=E, h=h, k=8, n_group=8, topk_group=4, score="sigmoid"))
        return lay["total"] - lay["scratch"]

    T, E, h = 256, 256, 7168  # decode: 2 x 2 tiles, 112 K blocks of 64 -> 28 splits of 4
    big = scratch_bytes(16384, E, h)  # 128 x 2 tiles: no split
    small = scratch_bytes(T, E, h)
    assert small >= 28 * T * E * 4
    assert small - 28 * T * E * 4 < big  # the rest is the status word and the histograms
    assert scratch_bytes(T, 64, h) < 28 * T * 64 * 4  # E < 128: CUDA-core router, no partial sums


def test_wait_timeout_selftest_checks_its_arguments(lib):
    """The failure-detection self-test rejects a limit outside [1, 4e9] before any CUDA call."""
    cfg = _cfg()
    fake_ws = ctypes.c_void_p(1 << 20)  # never dereferenced: the call fails on the limit first
    big = ctypes.c_size_t(1 << 40)
    for bad in (0, -5, 5_000_000_000):
        assert lib.moe_selftest_wait_timeout(ctypes.byref(cfg), fake_ws, big, bad, None) == moe.MOE_ERR_INVALID


def test_null_and_misaligned_pointers_are_rejected(lib):
    cfg = _cfg()
    w = moe.MoeWeightsStruct()
    rc = lib.moe_route(ctypes.byref(cfg), None, ctypes.byref(w), None, 0, None, None, None, 0, None)
    assert rc == moe.MOE_ERR_INVALID and "NULL" in lib.moe_last_error().decode()
    rc = lib.moe_route(ctypes.byref(cfg), None, None, ctypes.c_void_p(0x1001), moe.MOE_LOGITS_GIVEN,
                       ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), None, 0, None)
    assert rc == moe.MOE_ERR_INVALID and "aligned" in lib.moe_last_error().decode()
    rc = lib.moe_combine(ctypes.byref(cfg), None, None, None, None)
    assert rc == moe.MOE_ERR_INVALID
    rc = lib.moe_forward(ctypes.byref(cfg), ctypes.c_void_p(0x1000), ctypes.byref(w), ctypes.c_void_p(0x1000),
                         ctypes.c_void_p(0x1000), 16, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    rc = lib.moe_quantize_weights_fp8(ctypes.c_void_p(0x1000), 1, 100, 128, ctypes.c_void_p(0x1000),
                                      ctypes.c_void_p(0x1000), None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    rc = lib.moe_quantize_weights_nvfp4(ctypes.c_void_p(0x1000), 1, 64, 128, ctypes.c_void_p(0x1000),
                                        ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), None)
    assert rc == moe.MOE_ERR_UNSUPPORTED


def test_eplb_plan_host_entry_point_matches_oracle(lib):
    """moe_eplb_plan runs on the host: checked here without a GPU against the oracle's planner."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(5)
    for E, cards, red in ((256, 8, 0), (256, 32, 32), (64, 8, 8), (16, 4, 4), (12, 3, 0)):
        load = rng.integers(0, 500, E)
        load[rng.integers(0, E)] = 3000  # one hot expert
        got = moe.eplb_plan(load, cards, red)
        reps, slot_expert, slot_replica, card = oracle.eplb_plan(load, cards, red)
        np.testing.assert_array_equal(got["replicas"], reps)
        np.testing.assert_array_equal(got["slot_expert"], slot_expert)
        np.testing.assert_array_equal(got["slot_replica"], slot_replica)
        np.testing.assert_array_equal(got["card_load"], card)
        for e in range(E):  # replica_slot is the inverse of (slot_expert, slot_replica)
            for i in range(reps[e]):
                s = got["replica_slot"][e, i]
                assert slot_expert[s] == e and slot_replica[s] == i
    rc = lib.moe_eplb_plan(None, 8, 3, 0, None, None, None, None, None)
    assert rc == moe.MOE_ERR_INVALID
