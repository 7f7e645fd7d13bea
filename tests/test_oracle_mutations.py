"""Each plausible mistake, planted in a copy of the oracle on the CPU, must break at least one pin."""
import importlib.util
import os

import numpy as np
import pytest

from oracle_pins import ALL_PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_copy", os.path.join(ROOT, "oracle", "moe.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def swap_nibble_order(o):
    orig = o.unpack_int4

    def bad(packed, rows, cols):
        p = np.asarray(packed, np.uint8)
        return orig(((p >> 4) | (p << 4)).astype(np.uint8), rows, cols)
    o.unpack_int4 = bad


def offset_seven(o):
    orig = o.unpack_int4
    o.unpack_int4 = lambda p, r, c: (orig(p, r, c).astype(np.int16) + 1).astype(np.int8)


def tie_to_higher_index(o):
    def bad(c_row, K):
        c_row = np.asarray(c_row, np.float32)
        taken, out = np.zeros(len(c_row), bool), []
        for _ in range(K):
            best = -1
            for e in range(len(c_row)):
                if not taken[e] and (best < 0 or c_row[e] >= c_row[best]):
                    best = e
            taken[best] = True
            out.append(best)
        return np.array(out, np.int32)
    o.topk_by_choice = bad


def weights_from_choice(o):
    orig_sel = o.router_select

    def bad(x, Wr, bias, K, topp=0.0, norm_topk=True, routed_scale=1.0):
        x = np.atleast_2d(np.asarray(x))
        z, s, c = o.router_scores(x, Wr, bias)
        idx = np.zeros((x.shape[0], K), np.int32)
        w = np.zeros((x.shape[0], K), np.float32)
        n = np.zeros(x.shape[0], np.int32)
        for t in range(x.shape[0]):
            ch = o.topk_by_choice(c[t], K)
            idx[t], w[t], n[t] = o.route_weights(c[t], ch, topp, norm_topk, routed_scale)
        return idx, w, n, (z, s, c)
    o.router_select = bad


def scale_before_norm(o):
    orig = o.route_weights

    def bad(s_row, idx_row, topp, norm_topk, routed_scale):
        s2 = (np.asarray(s_row, np.float32) * np.float32(routed_scale)).astype(np.float32)
        return orig(s2, idx_row, topp, norm_topk, 1.0)
    o.route_weights = bad


def topp_drops_reaching_slot(o):
    orig = o.route_weights

    def bad(s_row, idx_row, topp, norm_topk, routed_scale):
        i, w, m = orig(s_row, idx_row, topp, False, 1.0)
        if 0 < topp < 1 and m > 1:
            m -= 1
        return orig(s_row, np.asarray(idx_row)[:len(idx_row)], 1.0, norm_topk, routed_scale) if m == len(idx_row) else \
            _truncate(orig, s_row, idx_row, m, norm_topk, routed_scale)
    o.route_weights = bad


def _truncate(orig, s_row, idx_row, m, norm_topk, routed_scale):
    i, w, _ = orig(s_row, np.asarray(idx_row)[:m], 1.0, norm_topk, routed_scale)
    K = len(idx_row)
    i2 = np.full(K, -1, np.int32)
    w2 = np.zeros(K, np.float32)
    i2[:m], w2[:m] = i, w
    return i2, w2, m


def norm_over_all_slots(o):
    orig = o.route_weights

    def bad(s_row, idx_row, topp, norm_topk, routed_scale):
        i, w, m = orig(s_row, idx_row, topp, False, 1.0)
        if norm_topk:
            tot = np.float32(np.sum(np.asarray(s_row, np.float32)[np.asarray(idx_row)], dtype=np.float32))
            w = (w / tot).astype(np.float32)
        return i, (w * np.float32(routed_scale)).astype(np.float32), m
    o.route_weights = bad


def sigmoid_sign(o):
    o.sigmoid64 = lambda z: 1.0 / (1.0 + np.exp(np.asarray(z, np.float64)))


def silu_on_up(o):
    def bad(x_row, gate, up, down):
        x64 = np.asarray(x_row, np.float64)
        g = gate.dense() @ x64
        u = up.dense() @ x64
        return down.dense() @ (o.silu64(u) * g)
    o.expert_ffn = bad


def drop_residual(o):
    orig = o.expert_group
    o.expert_group = lambda x, experts, idx, w, n_sel=None, resid=None: orig(x, experts, idx, w, n_sel, None)


def group_scales_column_major(o):
    def bad(scales, rows, cols, gs):
        scales = np.asarray(scales, np.float32).astype(np.float64)
        if gs == 0:
            return np.repeat(scales.reshape(rows, 1), cols, axis=1)
        G = (cols + gs - 1) // gs
        return scales.reshape(G, rows).T[:, np.arange(cols) // gs]
    o.scale_of = bad


def group_index_by_byte(o):
    def bad(scales, rows, cols, gs):
        scales = np.asarray(scales, np.float32).astype(np.float64)
        if gs == 0:
            return np.repeat(scales.reshape(rows, 1), cols, axis=1)
        G = (cols + gs - 1) // gs
        return scales.reshape(rows, G)[:, np.minimum(np.arange(cols) // (2 * gs) * 2, G - 1)]
    o.scale_of = bad


def down_transposed_roles(o):
    def bad(x_row, gate, up, down):
        x64 = np.asarray(x_row, np.float64)
        h = o.silu64(gate.dense() @ x64) * (up.dense() @ x64)
        Wd = down.dense()
        return (Wd.T @ h) if Wd.shape[0] == Wd.shape[1] else (Wd[:, ::-1] @ h)
    o.expert_ffn = bad


def gate_up_swapped(o):
    orig = o.expert_ffn
    o.expert_ffn = lambda x_row, gate, up, down: orig(x_row, up, gate, down)


def linear_drops_residual(o):
    orig = o.w4_linear
    o.w4_linear = lambda x, W, resid=None: orig(x, W, None)


def linear_reads_columns_reversed(o):
    orig = o.w4_linear
    o.w4_linear = lambda x, W, resid=None: orig(np.atleast_2d(np.asarray(x))[:, ::-1], W, resid)


def shared_weighted_like_slot0(o):
    orig = o.moe_block_with_shared

    def bad(x, experts, idx, w, n_sel, shared, resid=None):
        routed = orig(x, experts, idx, w, n_sel, shared, None) - orig(x, experts, idx, w, np.zeros(len(idx), np.int32),
                                                                        shared, None)
        sh = orig(x, experts, idx, w, np.zeros(len(idx), np.int32), shared, None)
        y = routed + np.asarray(w, np.float64)[:, :1] * sh
        return y if resid is None else np.asarray(resid, np.float64) + y
    o.moe_block_with_shared = bad


def shared_slot_at_row_end(o):
    orig = o.append_shared

    def bad(idx, w, n_sel, shared_id):
        i2, w2, n2 = orig(idx, w, n_sel, shared_id)
        for t in range(i2.shape[0]):
            m = int(n2[t]) - 1
            i2[t, m], w2[t, m] = -1, 0.0
            i2[t, -1], w2[t, -1] = shared_id, 1.0
        return i2, w2, n2
    o.append_shared = bad


def shard_by_block_not_modulo(o):
    o.expert_owner = lambda e, world: min(int(e) * int(world) // 8, int(world) - 1)


def ep_drops_last_rank(o):
    def bad(x, experts, idx, w, n_sel, world, resid=None):
        acc = 0.0
        for r in range(max(1, world - 1)):
            acc = acc + o.expert_group(x, experts, *o.shard_routes(idx, w, n_sel, r, world), None)
        return acc if resid is None else np.asarray(resid, np.float64) + acc
    o.ep_layer = bad


def f32_pairwise_sum(o):
    """The binary32 diagnosis mode summing each row pairwise (numpy's reduce) instead of in column order."""
    def bad(T, v):
        W32 = (o.scale_of(T.scales, T.rows, T.cols, T.gs).astype(np.float32) *
               o.unpack_int4(T.packed, T.rows, T.cols).astype(np.float32))
        return np.sum(W32 * np.asarray(v, np.float32)[None, :], axis=1, dtype=np.float32)
    o.matvec_f32_seq = bad


def f32_weights_unrounded(o):
    """The binary32 mode with each weight kept exact (float64 scale x value) before the f32 product."""
    def bad(T, v):
        W = T.dense()
        prod = (W * np.asarray(v, np.float32).astype(np.float64)[None, :]).astype(np.float32)
        return np.add.accumulate(prod, axis=1, dtype=np.float32)[:, -1]
    o.matvec_f32_seq = bad


MUTATIONS = [swap_nibble_order, offset_seven, tie_to_higher_index, weights_from_choice, scale_before_norm,
             topp_drops_reaching_slot, norm_over_all_slots, sigmoid_sign, silu_on_up, drop_residual,
             group_scales_column_major, group_index_by_byte, down_transposed_roles, gate_up_swapped,
             linear_drops_residual, linear_reads_columns_reversed, shared_weighted_like_slot0,
             shared_slot_at_row_end, shard_by_block_not_modulo, ep_drops_last_rank, f32_pairwise_sum,
             f32_weights_unrounded]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=[m.__name__ for m in MUTATIONS])
def test_mutation_is_caught(mutate):
    o = fresh_oracle()
    mutate(o)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutate.__name__}"


def test_unmutated_copy_passes_every_pin():
    o = fresh_oracle()
    for pin in ALL_PINS:
        pin(o)
