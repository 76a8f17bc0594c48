"""CPU oracle of the MoE layer hot path (route -> dispatch -> SwiGLU experts -> combine).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` leg may import this package. The product library never
does, and the oracle shares no code with it: the arithmetic lives in ``oracle.c`` (plain fp64
loops, compiled with gcc) and this wrapper only marshals numpy arrays.

Sources and readings are listed at the top of ``oracle.c``. Each wrapper names the step it
wraps. bf16 tensors are carried as ``uint16`` bit patterns, FP8 e4m3 tensors as ``uint8`` codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

SOFTMAX, SIGMOID = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no GPU toolchain involved)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", _SO, src,
                               "-lm"])
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            L.orc_router_logits.argtypes = [vp, vp, i64, i64, i64, vp]
            L.orc_route.argtypes = [vp, vp, i64, i32, i32, i32, i32, i32, i32, f32, vp, vp]
            L.orc_route.restype = i32
            L.orc_permute.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp]
            L.orc_permute.restype = i32
            L.orc_gather_rows.argtypes = [vp, i64, i32, vp, i64, vp]
            L.orc_permute_capacity.argtypes = [vp, i64, i32, i32, i32, vp, vp, vp, vp]
            L.orc_permute_capacity.restype = i32
            L.orc_expert_ffn_bf16.argtypes = [vp, i64, i64, i64, vp, vp, vp]
            L.orc_expert_ffn_fp8.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp, vp]
            L.orc_combine.argtypes = [vp, vp, vp, i64, i32, i64, vp]
            L.orc_quant_1x128.argtypes = [vp, i64, i64, vp, vp]
            L.orc_quant_weight_128x128.argtypes = [vp, i64, i64, vp, vp]
            L.orc_bf16_from_double_n.argtypes = [vp, i64, vp]
            L.orc_bf16_to_double_n.argtypes = [vp, i64, vp]
            L.orc_e4m3_encode_n.argtypes = [vp, i64, vp]
            L.orc_e4m3_decode_n.argtypes = [vp, i64, vp]
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_encode.argtypes = [f32]
            L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_quant_weight_nvfp4.argtypes = [vp, i64, i64, vp, vp, vp]
            L.orc_dequant_nvfp4.argtypes = [vp, vp, f32, i64, i64, vp]
            L.orc_expert_ffn_nvfp4.argtypes = [vp, i64, i64, i64, vp, vp, f32, vp, vp, f32, vp]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- number formats
def bf16_from_double(v) -> np.ndarray:
    v = _c(np.asarray(v, np.float64), np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_from_double_n(_p(v), v.size, _p(out))
    return out


def bf16_to_double(b) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().orc_bf16_to_double_n(_p(b), b.size, _p(out))
    return out


def e4m3_encode(f) -> np.ndarray:
    f = _c(np.asarray(f, np.float32), np.float32)
    out = np.empty(f.shape, np.uint8)
    lib().orc_e4m3_encode_n(_p(f), f.size, _p(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_n(_p(c), c.size, _p(out))
    return out


def quant_1x128(v) -> tuple[np.ndarray, np.ndarray]:
    """1x128 activation quantisation of a [m, n] array -> (codes [m, n], scales [m, n/128])"""
    v = _c(v, np.float64)
    m, n = v.shape
    assert n % 128 == 0
    q = np.empty((m, n), np.uint8)
    s = np.empty((m, n // 128), np.float32)
    lib().orc_quant_1x128(_p(v), m, n, _p(q), _p(s))
    return q, s


def quant_weight_128x128(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """128x128 static weight quantisation of a [rows, cols] bf16 matrix -> (codes, scales)"""
    w = _c(w_bf16, np.uint16)
    r, c = w.shape
    assert r % 128 == 0 and c % 128 == 0
    q = np.empty((r, c), np.uint8)
    s = np.empty((r // 128, c // 128), np.float32)
    lib().orc_quant_weight_128x128(_p(w), r, c, _p(q), _p(s))
    return q, s


def e2m1_decode(c) -> np.ndarray:
    """values of 4-bit e2m1 codes (low nibble)"""
    c = np.asarray(c, np.uint8)
    return np.array([lib().orc_e2m1_decode(int(v)) for v in c.ravel()], np.float64).reshape(c.shape)


def e2m1_encode(f) -> np.ndarray:
    """nearest e2m1 codes of fp32 values (ties to the even code, saturating at 6)"""
    f = np.asarray(f, np.float32)
    return np.array([lib().orc_e2m1_encode(float(v)) for v in f.ravel()], np.uint8).reshape(f.shape)


def quant_weight_nvfp4(w_bf16) -> tuple[np.ndarray, np.ndarray, float]:
    """NVFP4 quantisation of a [rows, cols] bf16 matrix -> (codes [rows, cols/2] two per byte, e4m3
    block scales [rows, cols/16], fp32 matrix scale)"""
    w = _c(w_bf16, np.uint16)
    r, c = w.shape
    assert c % 16 == 0
    q = np.empty((r, c // 2), np.uint8)
    sc = np.empty((r, c // 16), np.uint8)
    g = np.zeros(1, np.float32)
    lib().orc_quant_weight_nvfp4(_p(w), r, c, _p(q), _p(sc), _p(g))
    return q, sc, float(g[0])


def dequant_nvfp4(q, sc, g) -> np.ndarray:
    q, sc = _c(q, np.uint8), _c(sc, np.uint8)
    r, c2 = q.shape
    out = np.empty((r, 2 * c2), np.float64)
    lib().orc_dequant_nvfp4(_p(q), _p(sc), float(g), r, 2 * c2, _p(out))
    return out


# ---------------------------------------------------------------- step 1: route
def router_logits(x_bf16, w_r) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    w = _c(w_r, np.float32)
    T, h = x.shape
    E = w.shape[0]
    out = np.empty((T, E), np.float32)
    lib().orc_router_logits(_p(x), _p(w), T, h, E, _p(out))
    return out


def route(logits, bias, k, n_group=1, topk_group=1, score=SOFTMAX, renorm=False, routed_scale=1.0):
    """-> (topk_idx [T, k] int32, topk_w [T, k] fp32)"""
    l = _c(logits, np.float32)
    b = _c(bias, np.float32)
    T, E = l.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    rc = lib().orc_route(_p(l), _p(b), T, E, k, n_group, topk_group, score, int(bool(renorm)), routed_scale, _p(idx),
                         _p(w))
    if rc != 0:
        raise ValueError("invalid routing configuration")
    return idx, w


# ---------------------------------------------------------------- step 2: dispatch
def permute(topk_idx, E):
    """-> (counts [E], offsets [E+1], inv_pos [T, k], row_token [T*k])"""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    inv_pos = np.empty((T, k), np.int32)
    row_token = np.empty(T * k, np.int32)
    if lib().orc_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(inv_pos), _p(row_token)) != 0:
        raise ValueError("expert index out of range")
    return counts, offsets, inv_pos, row_token


def capacity(capacity_factor, T, k, E) -> int:
    """Assignments an expert may keep: ceil(capacity_factor * T * k / E); 0 = no limit."""
    if capacity_factor <= 0:
        return 0
    import math
    return int(math.ceil(capacity_factor * T * k / E))


def permute_capacity(topk_idx, E, cap):
    """permute() with at most `cap` rows per expert (earliest tokens); dropped entries get inv_pos -1.
    Returns (counts, offsets, inv_pos, row_token[:offsets[E]])."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    inv_pos = np.empty((T, k), np.int32)
    row_token = np.empty(T * k, np.int32)
    if lib().orc_permute_capacity(_p(idx), T, k, E, int(cap), _p(counts), _p(offsets), _p(inv_pos),
                                  _p(row_token)) != 0:
        raise ValueError("expert index out of range")
    return counts, offsets, inv_pos, row_token[:offsets[E]]


def gather_rows(x, row_token) -> np.ndarray:
    x = np.ascontiguousarray(x)
    rt = _c(row_token, np.int32)
    out = np.empty((rt.size,) + x.shape[1:], x.dtype)
    lib().orc_gather_rows(_p(x), x.shape[1], x.dtype.itemsize, _p(rt), rt.size, _p(out))
    return out


# ---------------------------------------------------------------- step 3: experts
def expert_ffn_bf16(x_bf16, w_gu, w_d) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    gu = _c(w_gu, np.uint16)
    d = _c(w_d, np.uint16)
    m, h = x.shape
    I = d.shape[1]
    assert gu.shape == (2 * I, h) and d.shape == (h, I)
    out = np.empty((m, h), np.float64)
    if m:
        lib().orc_expert_ffn_bf16(_p(x), m, h, I, _p(gu), _p(d), _p(out))
    return out


def expert_ffn_fp8(xq, xs, w_gu_q, w_gu_s, w_d_q, w_d_s) -> np.ndarray:
    xq, xs = _c(xq, np.uint8), _c(xs, np.float32)
    gq, gs = _c(w_gu_q, np.uint8), _c(w_gu_s, np.float32)
    dq, ds = _c(w_d_q, np.uint8), _c(w_d_s, np.float32)
    m, h = xq.shape
    I = dq.shape[1]
    out = np.empty((m, h), np.float64)
    if m:
        lib().orc_expert_ffn_fp8(_p(xq), _p(xs), m, h, I, _p(gq), _p(gs), _p(dq), _p(ds), _p(out))
    return out


def expert_ffn_nvfp4(x_bf16, w_gu, w_d) -> np.ndarray:
    """bf16 rows through one expert whose matrices are NVFP4 tuples (codes, scales, matrix scale)"""
    x = _c(x_bf16, np.uint16)
    (gq, gsc, gg), (dq, dsc, dg) = w_gu, w_d
    gq, gsc, dq, dsc = _c(gq, np.uint8), _c(gsc, np.uint8), _c(dq, np.uint8), _c(dsc, np.uint8)
    m, h = x.shape
    I = 2 * dq.shape[1]
    assert gq.shape == (2 * I, h // 2) and dq.shape == (h, I // 2)
    out = np.empty((m, h), np.float64)
    if m:
        lib().orc_expert_ffn_nvfp4(_p(x), m, h, I, _p(gq), _p(gsc), float(gg), _p(dq), _p(dsc), float(dg), _p(out))
    return out


# ---------------------------------------------------------------- step 4: combine
def combine(o, w, shared=None) -> np.ndarray:
    """o [n, k, h] fp64 expert outputs per (token, slot); w [n, k]; shared [n, h] or None -> y bf16 [n, h]"""
    o = _c(o, np.float64)
    w = _c(w, np.float32)
    s = _c(shared, np.float64)
    n, k, h = o.shape
    y = np.empty((n, h), np.uint16)
    lib().orc_combine(_p(o), _p(w), _p(s), n, k, h, _p(y))
    return y


# ---------------------------------------------------------------- expert placement
def eplb_plan(load, n_cards, n_redundant):
    """EPLB placement (inference guide 6.4, sections 5.2-5.3), the definition step by step:
    1. each of the n_redundant extra replicas goes to the expert with the largest load per replica;
    2. every replica carries load / replicas; replicas are taken heaviest first;
    3. each goes to the least-loaded card that still has a free slot ((E + R) / n_cards per card).
    Returns (replicas [E], slot_expert [E + R] card-major, slot_replica, card_load [n_cards])."""
    load = [int(v) for v in load]
    E = len(load)
    reps = [1] * E
    for _ in range(n_redundant):
        best = 0
        for e in range(1, E):
            if load[e] / reps[e] > load[best] / reps[best]:
                best = e
        reps[best] += 1
    copies = [(load[e] / reps[e], e) for e in range(E) for _ in range(reps[e])]
    order = sorted(range(len(copies)), key=lambda i: (-copies[i][0], i))  # heaviest first, stable
    per_card = (E + n_redundant) // n_cards
    used = [0] * n_cards
    card = [0.0] * n_cards
    slot_expert = [-1] * (E + n_redundant)
    slot_replica = [-1] * (E + n_redundant)
    placed = [0] * E
    for i in order:
        w, e = copies[i]
        g = min((c for c in range(n_cards) if used[c] < per_card), key=lambda c: (card[c], c))
        slot = g * per_card + used[g]
        slot_expert[slot], slot_replica[slot] = e, placed[e]
        placed[e] += 1
        used[g] += 1
        card[g] += w
    return (np.array(reps, np.int32), np.array(slot_expert, np.int32), np.array(slot_replica, np.int32),
            np.array(card, np.float64))


def permute_placed(topk_idx, E, slot_expert, slot_replica, replicas, cap=0):
    """The permutation over physical slots: the r-th kept token (token order) of expert e goes to its
    replica r % replicas[e], row r // replicas[e] of that slot; slots in slot order.
    Returns (counts [S], offsets [S + 1], inv_pos [T, k], row_token [offsets[S]])."""
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    S = len(slot_expert)
    slot_of = {(int(slot_expert[s]), int(slot_replica[s])): s for s in range(S)}
    members = [[] for _ in range(S)]  # (token, slot j) per physical slot, in order
    for e in range(E):
        r = 0
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    if cap <= 0 or r < cap:
                        members[slot_of[(e, r % int(replicas[e]))]].append((t, j))
                    r += 1
    counts = np.array([len(m) for m in members], np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    inv_pos = np.full((T, k), -1, np.int32)
    row_token = np.empty(int(offsets[-1]), np.int32)
    for s in range(S):
        for i, (t, j) in enumerate(members[s]):
            inv_pos[t, j] = offsets[s] + i
            row_token[offsets[s] + i] = t
    return counts, offsets, inv_pos, row_token


# ---------------------------------------------------------------- host-side statistics
def placement_imbalance(card_load) -> float:
    """Busiest card / mean card of a placement."""
    c = np.asarray(card_load, np.float64)
    return float(c.max() / c.mean())


def imbalance(counts, n_cards) -> float:
    """Load imbalance of a contiguous expert placement: busiest card / mean card (1 = balanced).
    (Inference guide 6.4, section 5.1: the layer waits for the busiest card.)"""
    c = np.asarray(counts, np.int64)
    per = c.size // n_cards
    load = c[: per * n_cards].reshape(n_cards, per).sum(axis=1)
    return float(load.max() / (load.sum() / n_cards))


# ---------------------------------------------------------------- whole layer (small shapes)
def forward(x_bf16, w_r, bias, experts, shared, *, k, n_group=1, topk_group=1, score=SOFTMAX, renorm=False,
            routed_scale=1.0, fp8=False, nvfp4=False, logits=None, capacity_factor=0.0):
    """The whole layer for shapes the oracle finishes in seconds.

    experts: list of (w_gu [2I, h], w_d [h, I]) bf16 per routed expert; shared: same tuple or None.
    FP8 layers quantise the expert weights 128x128 and the activations 1x128 first; NVFP4 layers
    quantise the expert weights to NVFP4 and keep the activations bf16.
    logits: router logits to route on (default: computed here from x and w_r).
    Returns a dict with every intermediate of the path.
    """
    x = _c(x_bf16, np.uint16)
    T, h = x.shape
    E = len(experts)
    if logits is None:
        logits = router_logits(x, w_r)
    idx, w = route(logits, bias, k, n_group, topk_group, score, renorm, routed_scale)
    cap = capacity(capacity_factor, T, k, E)
    if cap > 0:
        counts, offsets, inv_pos, row_token = permute_capacity(idx, E, cap)
    else:
        counts, offsets, inv_pos, row_token = permute(idx, E)
    R = int(offsets[E])
    out = dict(logits=logits, topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, inv_pos=inv_pos,
               row_token=row_token)
    if fp8:
        xq, xs = quant_1x128(bf16_to_double(x))
        xdq, xds = gather_rows(xq, row_token), gather_rows(xs, row_token)
        out.update(xq=xq, xs=xs, xd=xdq, xd_scales=xds)
        wq = [(quant_weight_128x128(gu), quant_weight_128x128(d)) for gu, d in experts]
        o_rows = np.empty((R, h), np.float64)
        for e in range(E):
            a, b = offsets[e], offsets[e + 1]
            (gq, gs), (dq, ds) = wq[e]
            o_rows[a:b] = expert_ffn_fp8(xdq[a:b], xds[a:b], gq, gs, dq, ds)
        sh = None
        if shared is not None:
            (gq, gs), (dq, ds) = quant_weight_128x128(shared[0]), quant_weight_128x128(shared[1])
            sh = expert_ffn_fp8(xq, xs, gq, gs, dq, ds)
    elif nvfp4:
        xd = gather_rows(x, row_token)
        out.update(xd=xd)
        q = lambda pair: (quant_weight_nvfp4(pair[0]), quant_weight_nvfp4(pair[1]))  # noqa: E731
        o_rows = np.empty((R, h), np.float64)
        for e in range(E):
            a, b = offsets[e], offsets[e + 1]
            if b > a:
                o_rows[a:b] = expert_ffn_nvfp4(xd[a:b], *q(experts[e]))
        sh = None if shared is None else expert_ffn_nvfp4(x, *q(shared))
    else:
        xd = gather_rows(x, row_token)
        out.update(xd=xd)
        o_rows = np.empty((R, h), np.float64)
        for e in range(E):
            a, b = offsets[e], offsets[e + 1]
            o_rows[a:b] = expert_ffn_bf16(xd[a:b], experts[e][0], experts[e][1])
        sh = None if shared is None else expert_ffn_bf16(x, shared[0], shared[1])
    # a dropped (token, slot) (inv_pos -1) contributes nothing: its expert output is zero
    flat = inv_pos.reshape(-1)
    o = np.where((flat >= 0)[:, None], o_rows[np.maximum(flat, 0)] if R > 0 else 0.0, 0.0).reshape(T, k, h)
    out.update(o_rows=o_rows, shared_out=sh, y=combine(o, w, sh))
    return out
