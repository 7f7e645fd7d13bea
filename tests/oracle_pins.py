"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when it disagrees
with a fixed fact: a hand-worked example from the format and routing rules (the
JSON fixtures under tests/golden, each carrying its source), a brute-force
enumeration on tiny inputs, a closed form, an exactness case, or an invariant.
They take the module as an argument so tests/test_oracle_mutations.py can run
every pin against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

from int4_grouped_expert_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------------------------------
# stored format
# ------------------------------------------------------------------------------------------

def pin_int4_worked_bytes(o):
    g = _load("int4_format.json")
    q = o.unpack_int4(np.array(g["packed"], np.uint8).reshape(1, -1), g["rows"], g["cols"])
    assert q.tolist() == [g["values"]], q


def pin_pack_roundtrip(o):
    rng_vals = synth.u64(synth.stream_seed(7, "rt"), 64 * 40)
    q = (rng_vals % np.uint64(16)).astype(np.int16).reshape(64, 40) - 8
    assert np.array_equal(o.unpack_int4(o.pack_int4(q), 64, 40), q)
    b = synth.random_bytes(synth.stream_seed(7, "rtb"), 33 * 20).reshape(33, 20)
    assert np.array_equal(o.pack_int4(o.unpack_int4(b, 33, 40)), b)
    # every byte value once: low nibble is the even column
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q = o.unpack_int4(allb, 1, 512).astype(np.int64)
    assert np.array_equal(q[0, 0::2], (np.arange(256) & 15) - 8)
    assert np.array_equal(q[0, 1::2], (np.arange(256) >> 4) - 8)


def pin_dequant_worked(o):
    g = _load("dequant_groups.json")
    packed = np.array(g["packed"], np.uint8)
    for case in g["cases"]:
        W = o.dequant(packed, np.array(case["scales"], np.float32), g["rows"], g["cols"], case["gs"])
        assert np.array_equal(W, np.array(case["W"], np.float64)), (case["gs"], W)


def pin_group_scale_equivalences(o):
    rows, cols = 12, 40
    packed = synth.random_bytes(synth.stream_seed(3, "p"), rows * cols // 2).reshape(rows, cols // 2)
    row_s = synth.uniform(synth.stream_seed(3, "s"), rows, 0.005, 0.02)
    W0 = o.dequant(packed, row_s, rows, cols, 0)
    # gs = I: a single group per row is per-row scaling, bit for bit
    assert np.array_equal(o.dequant(packed, row_s, rows, cols, cols), W0)
    # any even gs with every group scale equal to its row scale is per-row scaling
    for gs in (2, 4, 8, 6, 16, 38):
        G = -(-cols // gs)
        assert np.array_equal(o.dequant(packed, np.repeat(row_s, G), rows, cols, gs), W0), gs
    # distinct group scales act on their own column runs only (tail group included)
    gs = 16
    G = -(-cols // gs)
    gsc = synth.uniform(synth.stream_seed(3, "g"), rows * G, 0.005, 0.02).reshape(rows, G)
    Wg = o.dequant(packed, gsc.reshape(-1), rows, cols, gs)
    for r in range(rows):
        for gi in range(G):
            lo, hi = gi * gs, min(cols, (gi + 1) * gs)
            ref = o.dequant(packed[r:r + 1], gsc[r, gi:gi + 1], 1, cols, 0)[0, lo:hi]
            assert np.array_equal(Wg[r, lo:hi], ref), (r, gi)


# ------------------------------------------------------------------------------------------
# router
# ------------------------------------------------------------------------------------------

def _tied_scores(seed, E, levels):
    u = synth.u64(synth.stream_seed(seed, "tie"), E)
    return ((u % np.uint64(levels)).astype(np.float32) / np.float32(levels)).astype(np.float32)


def pin_topk_equals_stable_sort(o):
    for t in range(40):
        E = 8 + 9 * t
        c = _tied_scores(t, E, 5 + t % 7)
        K = 1 + t % min(E, 9)
        ref = np.argsort(-c.astype(np.float64), kind="stable")[:K]
        assert o.topk_by_choice(c, K).tolist() == ref.tolist(), t


def pin_topk_bruteforce(o):
    for t in range(12):
        E = 6
        c = _tied_scores(100 + t, E, 3)
        for K in range(1, E + 1):
            best = max(itertools.permutations(range(E), K),
                       key=lambda seq: [(float(c[e]), -e) for e in seq])
            assert o.topk_by_choice(c, K).tolist() == list(best), (t, K)


def pin_router_worked(o):
    g = _load("router_worked.json")
    tc = g["tie_case"]
    idx, w, n, _ = o.router_select(np.array([tc["x"]], np.float32), np.array(tc["Wr"], np.float32),
                                   np.array(tc["bias"], np.float32), tc["K"], tc["topp"],
                                   tc["norm_topk"], tc["routed_scale"])
    assert idx[0].tolist() == tc["idx"] and w[0].tolist() == tc["w"] and int(n[0]) == tc["n_sel"], (idx, w, n)
    for name in ("topp_case", "no_norm_case"):
        cse = g[name]
        i2, w2, m = o.route_weights(np.array(cse["s"], np.float32), np.array(cse["chosen"], np.int32),
                                    cse["topp"], cse["norm_topk"], cse["routed_scale"])
        assert i2.tolist() == cse["idx"] and w2.tolist() == cse["w"] and m == cse["n_sel"], (name, i2, w2, m)


def pin_sigmoid_closed_forms(o):
    D, E = 4, 5
    x = np.array([[1.0, 0.0, 0.0, 0.0]], np.float32)
    Wr = np.zeros((E, D), np.float32)
    Wr[:, 0] = [0.0, 30.0, -30.0, 2.0, -2.0]
    z, s, c = o.router_scores(x, Wr, None)
    assert z[0].tolist() == [0.0, 30.0, -30.0, 2.0, -2.0]
    assert s[0, 0] == np.float32(0.5)
    assert s[0, 1] == np.float32(1.0 / (1.0 + math.exp(-30.0)))
    assert abs(float(s[0, 2]) - math.exp(-30.0)) < 1e-19
    assert s[0, 3] == np.float32(1.0 / (1.0 + math.exp(-2.0)))
    assert abs(float(s[0, 3]) + float(s[0, 4]) - 1.0) < 1e-7
    assert np.array_equal(c, s)
    bias = np.array([0.25, 0, 0, 0, -0.5], np.float32)
    _, s2, c2 = o.router_scores(x, Wr, bias)
    assert c2[0, 0] == np.float32(0.75) and c2[0, 4] == np.float32(s2[0, 4] - np.float32(0.5))
    # logits are the plain matrix-vector product
    x3 = synth.normal(5, 3 * 16).reshape(3, 16)
    W3 = synth.normal(6, 7 * 16, 0.02).reshape(7, 16)
    z3, _, _ = o.router_scores(x3, W3, None)
    ref = np.array([[math.fsum(float(W3[e, j]) * float(x3[t, j]) for j in range(16)) for e in range(7)]
                    for t in range(3)], np.float32)
    assert np.array_equal(z3, ref)


def pin_route_invariants(o):
    for t in range(60):
        E, K = 32, 1 + t % 8
        s = synth.uniform(synth.stream_seed(t, "s"), E, 0.01, 0.99)
        chosen = o.topk_by_choice(s, K)
        rs = [1.0, 2.5, 0.5][t % 3]
        idx, w, m = o.route_weights(s, chosen, 0.0, True, rs)
        assert m == K and idx.tolist() == chosen.tolist()
        assert abs(float(np.sum(w.astype(np.float64))) - rs) <= 4e-7 * rs * K
        idx2, w2, m2 = o.route_weights(s, chosen, 0.0, False, rs)
        assert np.array_equal(w2, (s[chosen] * np.float32(rs)).astype(np.float32))
        # top-p keeps the shortest prefix reaching p (checked in float64, off-by-rounding excluded)
        p = [0.3, 0.5, 0.8, 0.95][t % 4]
        idx3, w3, m3 = o.route_weights(s, chosen, p, True, 1.0)
        raw = s[chosen].astype(np.float64)
        cum = np.cumsum(raw / raw.sum())
        assert 1 <= m3 <= K
        assert cum[m3 - 1] >= p - 1e-6
        if m3 > 1:
            assert cum[m3 - 2] < p + 1e-6
        assert idx3[:m3].tolist() == chosen[:m3].tolist() and (idx3[m3:] == -1).all() and (w3[m3:] == 0).all()
        assert abs(float(np.sum(w3[:m3].astype(np.float64))) - 1.0) < 1e-6 * K
        # top-p off for p <= 0 or p >= 1
        for off in (0.0, -1.0, 1.0, 2.0):
            assert o.route_weights(s, chosen, off, True, 1.0)[2] == K
    # K = E selects every expert exactly once
    s = synth.uniform(9, 16, 0.0, 1.0)
    assert sorted(o.topk_by_choice(s, 16).tolist()) == list(range(16))


# ------------------------------------------------------------------------------------------
# expert FFN and reduce
# ------------------------------------------------------------------------------------------

def _tensor_from_q(o, q, scales, gs=0):
    q = np.asarray(q, np.int16)
    return o.Tensor(o.pack_int4(q), np.asarray(scales, np.float32), q.shape[0], q.shape[1], gs)


def pin_ffn_worked(o):
    g = _load("ffn_worked.json")
    t = {k: _tensor_from_q(o, g[k]["q"], g[k]["scales"]) for k in ("gate", "up", "down")}
    ye = o.expert_ffn(np.array(g["x"]), t["gate"], t["up"], t["down"])
    assert np.allclose(ye, g["y_expert"], rtol=1e-14, atol=0), ye
    y = o.expert_group(np.array([g["x"]]), {0: (t["gate"], t["up"], t["down"])}, [[0]], [[g["w"]]],
                       None, np.array([g["resid"]]))
    assert np.allclose(y[0], g["y"], rtol=1e-14, atol=0), y


def _nib(packed_row, i):
    b = int(packed_row[i // 2])
    return ((b >> 4) if i % 2 else (b & 15)) - 8


def _scale(scales, r, i, cols, gs):
    if gs == 0:
        return float(scales[r])
    G = (cols + gs - 1) // gs
    return float(scales[r * G + i // gs])


def _matvec_brute(T, v):
    out = []
    for r in range(T.rows):
        acc = 0.0
        for i in range(T.cols):
            acc += _scale(T.scales, r, i, T.cols, T.gs) * _nib(T.packed[r], i) * float(v[i])
        out.append(acc)
    return out


def pin_ffn_bruteforce(o):
    D, I, E, K, S = 10, 6, 5, 2, 3
    for trial, gss in enumerate([(0, 0, 0), (2, 4, 0), (4, 0, 6), (6, 2, 2)]):
        experts = {}
        for e in range(E):
            ts = []
            for which, (rows, cols, gs) in zip(("g", "u", "d"), ((I, D, gss[0]), (I, D, gss[1]), (D, I, gss[2]))):
                p, s = synth.expert_tensor(synth.stream_seed(trial, e, which), rows, cols, gs)
                ts.append(o.Tensor(p, s, rows, cols, gs))
            experts[e] = tuple(ts)
        x = synth.normal(synth.stream_seed(trial, "x"), S * D).reshape(S, D)
        resid = synth.normal(synth.stream_seed(trial, "r"), S * D).reshape(S, D)
        idx = np.array([[3, 1], [0, 4], [2, 2]], np.int32)
        w = np.array([[0.7, 0.3], [1.5, -0.25], [0.5, 0.5]], np.float32)
        n_sel = np.array([2, 1, 2], np.int32)
        y = o.expert_group(x, experts, idx, w, n_sel, resid)
        for t in range(S):
            ref = [float(resid[t, d]) for d in range(D)]
            acc = [0.0] * D
            for k in range(int(n_sel[t])):
                G, U, Dn = experts[int(idx[t, k])]
                g = _matvec_brute(G, x[t])
                u = _matvec_brute(U, x[t])
                h = [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(I)]
                yd = _matvec_brute(Dn, h)
                acc = [acc[d] + float(w[t, k]) * yd[d] for d in range(D)]
            ref = [ref[d] + acc[d] for d in range(D)]
            assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-12), (trial, t)


def pin_ffn_closed_form(o):
    """All nibbles 9 (value +1): g_i = s_g Sum x, u_i = s_u Sum x, y_d = s_d * I * SiLU(g_0) u_0."""
    D, I = 16, 8
    sg, su, sd = 0.5, 0.25, 0.125
    ones = lambda r, c: o.Tensor(np.full((r, c // 2), 0x99, np.uint8), np.full(r, 1, np.float32), r, c, 0)
    gate, up, down = ones(I, D), ones(I, D), ones(D, I)
    gate.scales[:] = sg
    up.scales[:] = su
    down.scales[:] = sd
    x = synth.normal(11, D)
    sx = math.fsum(float(v) for v in x)
    g0, u0 = sg * sx, su * sx
    h0 = g0 / (1.0 + math.exp(-g0)) * u0
    y = o.expert_ffn(x, gate, up, down)
    assert np.allclose(y, sd * I * h0, rtol=1e-13, atol=0), (y, sd * I * h0)


def pin_ffn_exact_integers(o):
    """Integer activations and power-of-two scales: Wg x and Wu x are exact integers."""
    D, I = 24, 6
    for trial in range(4):
        q = ((synth.u64(synth.stream_seed(trial, "q"), I * D) % np.uint64(16)).astype(np.int16) - 8).reshape(I, D)
        xi = ((synth.u64(synth.stream_seed(trial, "x"), D) % np.uint64(9)).astype(np.int64) - 4)
        sc = np.array([2.0 ** (k - 3) for k in range(I)], np.float32)
        T = _tensor_from_q(o, q, sc)
        got = T.dense() @ xi.astype(np.float64)
        want = [sum(int(q[r, j]) * int(xi[j]) for j in range(D)) * 2.0 ** (r - 3) for r in range(I)]
        assert got.tolist() == want


def pin_f32_seq_worked(o):
    """The binary32 diagnosis mode, worked by hand.
    (1) Terms are added in column order. A row of value-1 weights times x = [2^24, 1, ..., 1] (sixteen
    columns) gives 2^24 in f32: every +1 is lost to round-to-even at 2^24 (spacing 2). The exact sum is
    2^24 + 15; a pairwise sum over eight partial sums gives 2^24 + 14.
    (2) The weight is the f32 product of scale and value, then the term the f32 product of weight and
    activation. With scale 1 + 2^-23 and value 7 the weight 7 + 7 2^-23 rounds to 7 + 2^-20 (the
    spacing in [4, 8) is 2^-21); times x = 3 that is 21 + 1.5 2^-19, a tie in [16, 32) (spacing 2^-19)
    that rounds to even: 21 + 2^-18. Rounding only once, (7 + 7 2^-23) 3 = 21 + 0.65625 2^-19 would
    round to 21 + 2^-19."""
    ones = _tensor_from_q(o, np.ones((1, 16), np.int16), [1.0])
    x = np.array([2.0 ** 24] + [1.0] * 15, np.float32)
    assert o.matvec_f32_seq(ones, x).tolist() == [2.0 ** 24]
    assert o.w4_linear(x, ones)[0].tolist() == [2.0 ** 24 + 15]
    s = np.float32(1.0 + 2.0 ** -23)
    seven = _tensor_from_q(o, np.array([[7, 0]], np.int16), [s])
    assert o.matvec_f32_seq(seven, np.array([1.0, 0.0], np.float32)).tolist() == [7.0 + 2.0 ** -20]
    assert o.matvec_f32_seq(seven, np.array([3.0, 0.0], np.float32)).tolist() == [21.0 + 2.0 ** -18]


def pin_f32_seq_exact_cases(o):
    """Integer activations, small integer weights and power-of-two scales keep every f32 product and
    partial sum exact: the binary32 mode then equals the float64 definition bit for bit, for the matvec,
    the expert FFN's gate/up/down chain up to h (where SiLU rounds) and the slot-ordered reduce of exact
    expert outputs."""
    D, I = 24, 6
    for trial in range(3):
        q = ((synth.u64(synth.stream_seed(trial, "q32"), I * D) % np.uint64(16)).astype(np.int16) - 8).reshape(I, D)
        xi = ((synth.u64(synth.stream_seed(trial, "x32"), D) % np.uint64(9)).astype(np.int64) - 4).astype(np.float32)
        sc = np.array([2.0 ** (k - 3) for k in range(I)], np.float32)
        T = _tensor_from_q(o, q, sc)
        assert o.matvec_f32_seq(T, xi).astype(np.float64).tolist() == (T.dense() @ xi.astype(np.float64)).tolist()
    # the FFN chain and the reduce: g = 32 * sum(x) = 128 makes SiLU(g) = g exactly in both precisions
    # (exp(-128) vanishes beside 1); expert 0 has u = 2 (h = 256), expert 1 u = 128 (h = 16384), and the
    # down rows are small integers times h / 16
    gate = _tensor_from_q(o, np.ones((2, 4), np.int16), [32.0, 32.0])
    up = _tensor_from_q(o, np.ones((2, 4), np.int16), [0.5, 0.5])
    down = _tensor_from_q(o, np.array([[1, -2], [3, 0], [-8, 7], [5, 5]], np.int16), [2.0 ** -4] * 4)
    ex = {0: (gate, up, down), 1: (gate, gate, down)}
    x = np.ones((1, 4), np.float32)
    r = np.array([[1.0, -2.0, 3.0, 0.5]], np.float32)
    y32 = o.expert_group_f32(x, ex, [[0, 1]], [[0.5, 2.0]], None, r)
    y64 = o.expert_group(x, ex, [[0, 1]], [[0.5, 2.0]], None, r)
    assert y32.astype(np.float64).tolist() == y64.tolist()
    # r + 0.5 * 16 * [-1, 3, -1, 10] + 2 * 1024 * [-1, 3, -1, 10]
    assert y64.tolist() == [[-2055.0, 6166.0, -2053.0, 20560.5]]


def pin_reduce_properties(o):
    D, I, E = 12, 4, 3
    experts = {}
    for e in range(E):
        trip = []
        for which, (r, c) in zip("gud", ((I, D), (I, D), (D, I))):
            p, s = synth.expert_tensor(synth.stream_seed(40, e, which), r, c, 0)
            trip.append(o.Tensor(p, s, r, c, 0))
        experts[e] = tuple(trip)
    x = synth.normal(41, D).reshape(1, D)
    resid = synth.normal(42, D).reshape(1, D)
    idx = np.array([[2, 0, 1]], np.int32)
    w = np.array([[0.5, 0.25, 1.0]], np.float32)
    y1 = o.expert_group(x, experts, idx, w, None, resid)
    y0 = o.expert_group(x, experts, idx, w, None, None)
    assert np.allclose(y1 - resid, y0, rtol=1e-13, atol=1e-13)  # residual joins additively
    y2 = o.expert_group(x, experts, idx, 2 * w, None, None)
    assert np.allclose(y2, 2 * y0, rtol=1e-13, atol=1e-13)       # linear in the weights
    single = [o.expert_group(x, experts, idx[:, k:k + 1], w[:, k:k + 1], None, None) for k in range(3)]
    assert np.allclose(y0, single[0] + single[1] + single[2], rtol=1e-12, atol=1e-12)
    yt = o.expert_group(x, experts, np.array([[2, 0, -1]], np.int32), w, np.array([2]), None)
    assert np.allclose(yt, single[0] + single[1], rtol=1e-12, atol=1e-12)  # truncated slot ignored
    yz = o.expert_group(x, experts, idx, w, np.array([0]), resid)
    assert np.array_equal(yz, resid.astype(np.float64))               # no slot: residual only


def pin_linear_bruteforce(o):
    """w4_linear against element-by-element sums over the packed nibbles, every scale layout."""
    O, I, S = 7, 12, 3
    for trial, gs in enumerate([0, 2, 4, 6, 12]):
        p, sc = synth.expert_tensor(synth.stream_seed(60 + trial, "W"), O, I, gs)
        T = o.Tensor(p, sc, O, I, gs)
        x = synth.normal(synth.stream_seed(60 + trial, "x"), S * I).reshape(S, I)
        resid = synth.normal(synth.stream_seed(60 + trial, "r"), S * O).reshape(S, O)
        y0 = o.w4_linear(x, T)
        y1 = o.w4_linear(x, T, resid)
        for t in range(S):
            ref = _matvec_brute(T, x[t])
            assert np.allclose(y0[t], ref, rtol=1e-12, atol=1e-12), (trial, t)
            assert np.allclose(y1[t], [float(resid[t, r]) + ref[r] for r in range(O)], rtol=1e-12, atol=1e-12), (trial, t)


def pin_linear_exact_and_transposed(o):
    """Integer x and power-of-two scales give exact integers; a one-hot x reads out a column."""
    O, I = 5, 8
    q = ((synth.u64(synth.stream_seed(70, "q"), O * I) % np.uint64(16)).astype(np.int16) - 8).reshape(O, I)
    sc = np.array([2.0 ** (r - 2) for r in range(O)], np.float32)
    T = _tensor_from_q(o, q, sc)
    xi = np.array([3, -1, 0, 2, -4, 1, 1, -2], np.int64)
    got = o.w4_linear(xi.astype(np.float64).reshape(1, I), T)[0]
    assert got.tolist() == [sum(int(q[r, j]) * int(xi[j]) for j in range(I)) * 2.0 ** (r - 2) for r in range(O)]
    for j in range(I):
        e = np.zeros((1, I))
        e[0, j] = 1.0
        col = o.w4_linear(e, T)[0]
        assert col.tolist() == [int(q[r, j]) * 2.0 ** (r - 2) for r in range(O)], j


def pin_shared_expert_bruteforce(o):
    """Routed slots plus an always-chosen shared expert of weight 1, by hand-written loops."""
    D, I, E, S = 8, 6, 4, 2
    def trip(tag):
        out = []
        for which, (r, c, gs) in zip("gud", ((I, D, 2), (I, D, 0), (D, I, 6))):
            p, sc = synth.expert_tensor(synth.stream_seed(80, tag, which), r, c, gs)
            out.append(o.Tensor(p, sc, r, c, gs))
        return tuple(out)
    experts = {e: trip(e) for e in range(E)}
    shared = trip("shared")
    x = synth.normal(synth.stream_seed(81, "x"), S * D).reshape(S, D)
    resid = synth.normal(synth.stream_seed(81, "r"), S * D).reshape(S, D)
    idx = np.array([[1, 3], [2, 0]], np.int32)
    w = np.array([[0.6, 0.4], [1.25, 0.5]], np.float32)
    n_sel = np.array([2, 1], np.int32)
    y = o.moe_block_with_shared(x, experts, idx, w, n_sel, shared, resid)
    y0 = o.moe_block_with_shared(x, experts, idx, w, np.array([0, 0], np.int32), shared, None)

    def ffn(trip_, v):
        G, U, Dn = trip_
        g, u = _matvec_brute(G, v), _matvec_brute(U, v)
        return _matvec_brute(Dn, [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(I)])
    for t in range(S):
        sh = ffn(shared, x[t])
        acc = [0.0] * D
        for k in range(int(n_sel[t])):
            yk = ffn(experts[int(idx[t, k])], x[t])
            acc = [acc[d] + float(w[t, k]) * yk[d] for d in range(D)]
        want = [float(resid[t, d]) + (acc[d] + sh[d]) for d in range(D)]
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-12), t
        assert np.allclose(y0[t], sh, rtol=1e-12, atol=1e-12), t  # no routed slot: the shared expert alone


def pin_append_shared_worked(o):
    """Hand-written rows: the shared slot lands right after the kept slots with weight 1."""
    idx = np.array([[4, 2, -1], [7, 1, 5]], np.int32)
    w = np.array([[0.75, 0.25, 0.0], [0.5, 0.3, 0.2]], np.float32)
    i2, w2, n2 = o.append_shared(idx, w, np.array([2, 3], np.int32), 9)
    assert i2.tolist() == [[4, 2, 9, -1], [7, 1, 5, 9]]
    assert w2.tolist() == [[0.75, 0.25, 1.0, 0.0], [0.5, 0.30000001192092896, 0.20000000298023224, 1.0]]
    assert n2.tolist() == [3, 4]


def pin_shard_routes_worked(o):
    """Hand-written rows over 2 and 3 ranks: owned kept slots first, in slot order; the rest -1/0."""
    idx = np.array([[4, 7, 2, 9], [3, 6, 1, -1]], np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.5, 0.25, 0.25, 0.0]], np.float32)
    n = np.array([3, 3], np.int32)
    i0, w0, n0 = o.shard_routes(idx, w, n, 0, 2)
    i1, w1, n1 = o.shard_routes(idx, w, n, 1, 2)
    assert i0.tolist() == [[4, 2, -1, -1], [6, -1, -1, -1]] and n0.tolist() == [2, 1]
    assert i1.tolist() == [[7, -1, -1, -1], [3, 1, -1, -1]] and n1.tolist() == [1, 2]
    assert w0[0].tolist()[:2] == [np.float32(0.4), np.float32(0.2)] and w1[1].tolist()[:2] == [0.5, 0.25]
    i2, _, n2 = o.shard_routes(idx, w, None, 2, 3)  # all four slots kept; 2 and 9 are not owned by rank 2
    assert i2.tolist() == [[2, -1, -1, -1], [-1, -1, -1, -1]] and n2.tolist() == [1, 0]


def pin_ep_layer_partition(o):
    """Every kept slot lands on exactly one rank; the rank-order sum equals the one-rank block up to
    rounding, and one rank is the one-rank block exactly."""
    D, I, E, K, S = 8, 6, 7, 3, 4
    experts = {}
    for e in range(E):
        trip = []
        for which, (r, c) in zip("gud", ((I, D), (I, D), (D, I))):
            p, sc = synth.expert_tensor(synth.stream_seed(90, e, which), r, c, 0)
            trip.append(o.Tensor(p, sc, r, c, 0))
        experts[e] = tuple(trip)
    x = synth.normal(synth.stream_seed(91, "x"), S * D).reshape(S, D)
    resid = synth.normal(synth.stream_seed(91, "r"), S * D).reshape(S, D)
    idx = np.array([[6, 1, 3], [0, 5, 2], [4, 4, 1], [2, 3, -1]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.6, 0.3, 0.1], [0.7, 0.2, 0.1], [0.75, 0.25, 0.0]], np.float32)
    n = np.array([3, 2, 3, 2], np.int32)
    ref = o.expert_group(x, experts, idx, w, n, resid)
    assert np.array_equal(o.ep_layer(x, experts, idx, w, n, 1, resid), ref)
    for world in (2, 3, 5):
        shards = [o.shard_routes(idx, w, n, r, world) for r in range(world)]
        for t in range(S):
            owned = sorted((int(i), float(v)) for (si, sw, sn) in shards for i, v in zip(si[t, :sn[t]], sw[t, :sn[t]]))
            assert owned == sorted((int(i), float(v)) for i, v in zip(idx[t, :n[t]], w[t, :n[t]])), (world, t)
        got = o.ep_layer(x, experts, idx, w, n, world, resid)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), world


def pin_ans_codec(o):
    """The block codec (oracle.ans): lossless round trips across block boundaries and odd lengths, a size
    within the entropy bound plus the per-block overhead, and a constant stream that needs no words."""
    import oracle.ans as A
    for n, sigma in ((1, 2.5), (31, 2.5), (4096, 2.0), (4097, 3.0), (9000, 1.5)):
        data = bytes(synth.gaussian_nibble_bytes(synth.stream_seed(95, n), n, sigma))
        enc = A.encode(data)
        assert A.decode(enc) == data, n
        nib = [b & 15 for b in data] + [b >> 4 for b in data]
        p = np.bincount(nib, minlength=16) / len(nib)
        h_bits = -sum(q * math.log2(q) for q in p if q > 0) * len(nib)
        blocks = (n + 4095) // 4096
        overhead = 56 + 4 * (blocks + 1) + blocks * (192 + 4 + 32 * 2)  # header, offsets, per-block states/counts/pad
        assert len(enc) <= h_bits / 8 * 1.01 + overhead + 16, (n, len(enc), h_bits / 8)
    rnd = bytes(synth.random_bytes(96, 5000))
    assert A.decode(A.encode(rnd)) == rnd
    const = bytes([0x88]) * 8192
    enc = A.encode(const)
    assert A.decode(enc) == const
    assert len(enc) == 56 + 4 * 3 + 2 * 192  # two blocks of states and counts, not one word


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
