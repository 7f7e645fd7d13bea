"""CPU oracle for the decode-time int4 grouped-expert MoE block.

TEST INFRASTRUCTURE ONLY. This is a plain, slow, deliberately unoptimised restatement
of what the routed-expert block computes, used to check the CUDA library. Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path never does. It shares no code with the CUDA path:
inputs come from ``int4_grouped_expert_router_gb300.synth`` (random numbers only).

Sources (web pages about the "colibri" int4 MoE engine; cited by page and section):
  [g4]      c/backend_cuda.cu commit history, commit "grouped MoE kernels were per-row-only"
            (offset-8 nibbles, per-row fmt=2 / per-group fmt=4 scales, gs even, gs=0 per-row,
            tail group, mixed members in one launch)
  [router]  c/backend_cuda.cu commit history, commit "First increment of the #431 plan"
            (E x D f32 logits GEMV, sigmoid, bias-augmented top-K by choice, strict '>'
            tie-break, weights from the raw score, route-level TOPP, norm_topk, routed_scale)
  [tcgate]  c/backend_cuda.cu commit history, commit "The TC_W4A16 branch ..."
            (grouped 3-launch path: dual gate/up GEMV, SiLU, down GEMV)
  [resid]   PR #434 "COLI_CUDA_RESID=1", section "What"
            (per-expert weighting + fixed-order reduce, joined to the residual)
  [attn]    c/backend_cuda.cu commit history, commit "CUDA batch MLA attention, kv_b head-sharding,
            fused o_proj, expert-group dispatch, W4A16 kernels" (the shared expert on the device)
  [pipe]    c/backend_cuda.cu commit history, commit "GPU resident pipeline ..." (the shared-expert
            MLP beside the residual adds)
  [q651]    PR #651, comment "Follow-up decode experiments" (the generic quant_matmul's kernel share)

Precision: weights are dequantised exactly (float64) and every dot product, SiLU and
the weighted reduce run in float64. A binary32 sequential mode (matvec_f32_seq,
expert_ffn_f32, expert_group_f32) is kept beside it for diagnosis only: it measures how far
a plain f32 evaluation of the same sums falls from the float64 definition. The router's decisions (top-K, top-p) are taken in
float32, the precision of the pages' f32 logits, on float32 scores derived from the
float64 logits by one rounding each. Every reading of an ambiguous passage is marked
"Reading:" below.

Parity status: every function here is pinned by tests/test_oracle_pins.py (hand-worked
golden values, brute force, closed forms, invariants, textbook-routine equivalences).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


# ------------------------------------------------------------------------------------------
# Stored format [g4]
# ------------------------------------------------------------------------------------------

def unpack_int4(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Signed weights q = nibble - 8 as int8 [rows x cols] from packed bytes [rows x ceil(cols/2)].

    [g4]: stored nibbles are offset-8 ("offset->signed nibble conversion"), two per byte,
    fmt=4 packed identically to fmt=2. Reading: column 2m is the low nibble of byte m and
    column 2m+1 its high nibble (the pages fix only the offset, not the order).
    """
    packed = np.asarray(packed, dtype=np.uint8).reshape(rows, (cols + 1) // 2)
    lo = (packed & 0x0F).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    q = np.empty((rows, 2 * packed.shape[1]), dtype=np.int16)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    return (q[:, :cols] - 8).astype(np.int8)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Inverse of :func:`unpack_int4`: signed values in [-8, 7] -> packed offset-8 bytes."""
    q = np.asarray(q, dtype=np.int16)
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("int4 values must lie in [-8, 7]")
    rows, cols = q.shape
    n = (q + 8).astype(np.uint8)
    if cols % 2:
        n = np.concatenate([n, np.full((rows, 1), 8, np.uint8)], axis=1)
    return (n[:, 0::2] | (n[:, 1::2] << 4)).astype(np.uint8)


def scale_of(scales: np.ndarray, rows: int, cols: int, gs: int) -> np.ndarray:
    """The scale that multiplies W[o, i], expanded to [rows x cols] (float64).

    [g4]: gs = 0 means one scale per row (O floats); gs > 0 (even) means one scale per
    row and per run of gs input columns, O * ceil(I / gs) floats, row-major, the last
    run of a row being the (possibly shorter) tail group.
    """
    scales = np.asarray(scales, dtype=np.float32).astype(np.float64)
    if gs == 0:
        return np.repeat(scales.reshape(rows, 1), cols, axis=1)
    G = (cols + gs - 1) // gs
    per_group = scales.reshape(rows, G)
    group_of_col = np.arange(cols) // gs
    return per_group[:, group_of_col]


def dequant(packed: np.ndarray, scales: np.ndarray, rows: int, cols: int, gs: int) -> np.ndarray:
    """W[o, i] = scale(o, i) * (nibble(o, i) - 8), exact in float64 [g4]."""
    if gs < 0 or gs % 2:
        raise ValueError("gs must be 0 or a positive even number")
    return scale_of(scales, rows, cols, gs) * unpack_int4(packed, rows, cols).astype(np.float64)


# ------------------------------------------------------------------------------------------
# Router [router]
# ------------------------------------------------------------------------------------------

def sigmoid64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def router_scores(x: np.ndarray, Wr: np.ndarray, bias):
    """Per token: f32 logits z = Wr x, f32 scores s = sigmoid(z), f32 choice c = s + bias.

    [router]: "a tiny E x D logits GEMV + sigmoid" over f32 router weights, then the
    "bias-augmented" choice score. The GEMV is evaluated in float64 and rounded once to
    f32 (the logits are f32 on the pages); the sigmoid is evaluated in float64 on that
    f32 logit and rounded once; the bias add is one f32 addition.
    """
    x = np.asarray(x, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float32).astype(np.float64)
    z = (x @ Wr.T).astype(F32)                    # [S x E]
    s = sigmoid64(z.astype(np.float64)).astype(F32)
    if bias is None:
        c = s.copy()
    else:
        c = (s + np.asarray(bias, dtype=F32)).astype(F32)   # f32 + f32, rounded to f32
    if not (np.all(np.isfinite(s)) and np.all(np.isfinite(c))):
        raise FloatingPointError("non-finite router score")
    return z, s, c


def topk_by_choice(c_row: np.ndarray, K: int) -> np.ndarray:
    """K rounds of arg-max over the not-yet-chosen experts with a strict '>' comparison.

    [router]: "bias-augmented top-K by choice with strict-> tie-breaking". Scanning the
    experts in increasing index and replacing the best only on a strictly greater score
    makes the lower index win a tie. The output order is the order of selection.
    """
    c_row = np.asarray(c_row, dtype=F32)
    E = c_row.shape[0]
    if not 1 <= K <= E:
        raise ValueError("need 1 <= K <= E")
    taken = np.zeros(E, dtype=bool)
    out = []
    for _ in range(K):
        best = -1
        for e in range(E):
            if taken[e]:
                continue
            if best < 0 or c_row[e] > c_row[best]:
                best = e
        taken[best] = True
        out.append(best)
    return np.array(out, dtype=np.int32)


def route_weights(s_row: np.ndarray, idx_row: np.ndarray, topp: float, norm_topk: bool,
                  routed_scale: float):
    """Weights of the K selected experts, in slot order: (idx, w, n_sel), all f32 steps.

    [router]: "weights from the raw logit, route-level TOPP truncation, norm_topk,
    routed_scale".
    Reading (raw): the weight of a chosen expert is its sigmoid score s without the
      bias, i.e. the score before bias augmentation.
    Reading (TOPP): p_k = w_k / sum_{k<K} w_k; walking the slots in selection order,
      keep the shortest prefix m >= 1 whose running sum of p_k reaches topp. topp <= 0
      or >= 1 disables the truncation. Slots m..K-1 get idx = -1 and w = 0.
    Reading (norm_topk): w_k <- w_k / sum_{k<m} w_k over the kept slots.
    Reading (routed_scale): applied last, whether or not norm_topk is on.
    Every sum runs in slot order in float32.
    """
    idx_row = np.asarray(idx_row, dtype=np.int32)
    K = idx_row.shape[0]
    w = [F32(s_row[e]) for e in idx_row]
    m = K
    topp = F32(topp)
    if F32(0) < topp < F32(1):
        total = F32(0)
        for k in range(K):
            total = F32(total + w[k])
        cum = F32(0)
        for k in range(K):
            cum = F32(cum + F32(w[k] / total))
            if cum >= topp:
                m = k + 1
                break
    if norm_topk:
        denom = F32(0)
        for k in range(m):
            denom = F32(denom + w[k])
        w = [F32(w[k] / denom) if k < m else w[k] for k in range(K)]
    rs = F32(routed_scale)
    w_out = np.zeros(K, dtype=F32)
    idx_out = np.full(K, -1, dtype=np.int32)
    for k in range(m):
        w_out[k] = F32(w[k] * rs)
        idx_out[k] = idx_row[k]
    return idx_out, w_out, m


def router_select(x, Wr, bias, K: int, topp: float = 0.0, norm_topk: bool = True,
                  routed_scale: float = 1.0):
    """The whole device-router step for S tokens: idx [S x K], w [S x K], n_sel [S], plus scores."""
    x = np.atleast_2d(np.asarray(x))
    z, s, c = router_scores(x, Wr, bias)
    S = x.shape[0]
    idx = np.zeros((S, K), dtype=np.int32)
    w = np.zeros((S, K), dtype=F32)
    n_sel = np.zeros(S, dtype=np.int32)
    for t in range(S):
        chosen = topk_by_choice(c[t], K)
        idx[t], w[t], n_sel[t] = route_weights(s[t], chosen, topp, norm_topk, routed_scale)
    return idx, w, n_sel, (z, s, c)


# ------------------------------------------------------------------------------------------
# Expert FFN and reduce [tcgate], [g4], [resid]
# ------------------------------------------------------------------------------------------

class Tensor:
    """One uploaded int4 tensor in its stored form (packed bytes, scales, shape, gs)."""

    def __init__(self, packed, scales, rows: int, cols: int, gs: int):
        self.packed = np.asarray(packed, dtype=np.uint8).reshape(rows, (cols + 1) // 2)
        self.scales = np.asarray(scales, dtype=np.float32).reshape(-1)
        self.rows, self.cols, self.gs = rows, cols, gs
        need = rows if gs == 0 else rows * ((cols + gs - 1) // gs)
        if self.scales.shape[0] != need:
            raise ValueError("scale count does not match O, I and gs")
        self._w = None

    def dense(self) -> np.ndarray:
        if self._w is None:
            self._w = dequant(self.packed, self.scales, self.rows, self.cols, self.gs)
        return self._w

    def drop_cache(self):
        self._w = None


def silu64(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g) in float64."""
    return g * sigmoid64(g)


def expert_ffn(x_row: np.ndarray, gate: Tensor, up: Tensor, down: Tensor) -> np.ndarray:
    """y_e = Wd (SiLU(Wg x) * (Wu x)) for one token and one expert, float64 [tcgate]."""
    x64 = np.asarray(x_row, dtype=np.float64)
    g = gate.dense() @ x64
    u = up.dense() @ x64
    h = silu64(g) * u
    return down.dense() @ h


def expert_group(x, experts, idx, w, n_sel=None, resid=None) -> np.ndarray:
    """y[t] = resid[t] + sum_{k < n_sel[t]} w[t, k] * y_{idx[t, k]}(x[t]), slots in order.

    [resid]: per-expert weighting and a fixed-order reduce (no atomics), joined to the
    residual. Reading: the weighted slot sum is formed first, then added to the
    residual; with no residual the sum itself is the output. ``experts`` maps an expert
    id to a (gate, up, down) triple of :class:`Tensor`.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    idx = np.atleast_2d(np.asarray(idx))
    w = np.atleast_2d(np.asarray(w, dtype=np.float32))
    S, K = idx.shape
    D = x.shape[1]
    if n_sel is None:
        n_sel = np.full(S, K, dtype=np.int32)
    y = np.zeros((S, D), dtype=np.float64)
    for t in range(S):
        acc = np.zeros(D, dtype=np.float64)
        for k in range(int(n_sel[t])):
            gate, up, down = experts[int(idx[t, k])]
            acc = acc + float(w[t, k]) * expert_ffn(x[t], gate, up, down)
        y[t] = acc if resid is None else np.asarray(resid[t], dtype=np.float64) + acc
    return y


# ------------------------------------------------------------------------------------------
# Binary32 sequential evaluation (a diagnosis mode beside the float64 definition)
# ------------------------------------------------------------------------------------------

def matvec_f32_seq(T: Tensor, v) -> np.ndarray:
    """W v evaluated the plainest way in binary32: W[o, j] = f32(scale(o, j) * (nibble - 8)) ([g4]),
    each product W[o, j] * v[j] rounded to f32, and each row's products added to a running f32 sum in
    column order j = 0, 1, ..., L - 1. Not the definition (that is the exact float64 matvec): it sizes
    how far any binary32 evaluation of the same sums may fall from it."""
    W32 = (scale_of(T.scales, T.rows, T.cols, T.gs).astype(F32) *
           unpack_int4(T.packed, T.rows, T.cols).astype(F32))
    prod = W32 * np.asarray(v, dtype=F32)[None, :]
    return np.add.accumulate(prod, axis=1, dtype=F32)[:, -1]


def expert_ffn_f32(x_row, gate: Tensor, up: Tensor, down: Tensor) -> np.ndarray:
    """:func:`expert_ffn` in binary32: sequential f32 matvecs, h = g / (1 + exp(-g)) * u in f32."""
    x32 = np.asarray(x_row, dtype=F32)
    g = matvec_f32_seq(gate, x32)
    u = matvec_f32_seq(up, x32)
    with np.errstate(over="ignore"):
        h = (g / (F32(1) + np.exp(-g))).astype(F32) * u
    return matvec_f32_seq(down, h.astype(F32))


def expert_group_f32(x, experts, idx, w, n_sel=None, resid=None) -> np.ndarray:
    """:func:`expert_group` in binary32: acc = f32(acc + f32(w_k y_k)) in slot order, then resid + acc."""
    x = np.atleast_2d(np.asarray(x, dtype=F32))
    idx = np.atleast_2d(np.asarray(idx))
    w = np.atleast_2d(np.asarray(w, dtype=F32))
    S, K = idx.shape
    if n_sel is None:
        n_sel = np.full(S, K, dtype=np.int32)
    y = np.zeros((S, x.shape[1]), dtype=F32)
    for t in range(S):
        acc = np.zeros(x.shape[1], dtype=F32)
        for k in range(int(n_sel[t])):
            gate, up, down = experts[int(idx[t, k])]
            acc = (acc + (w[t, k] * expert_ffn_f32(x[t], gate, up, down)).astype(F32)).astype(F32)
        y[t] = acc if resid is None else (np.asarray(resid[t], dtype=F32) + acc).astype(F32)
    return y


# ------------------------------------------------------------------------------------------
# Dense int4 projection and the shared expert [tcgate], [q651], [attn], [pipe]
# ------------------------------------------------------------------------------------------

def w4_linear(x, W: Tensor, resid=None) -> np.ndarray:
    """y[t] = resid[t] + W x[t] for every token t, float64: the one-tensor int4 matmul that
    [tcgate] calls quant_matmul (the per-expert fallback) and [q651] measures as the largest
    kernel share of a decode step. W is dequantised exactly as in [g4]."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    y = x @ W.dense().T
    return y if resid is None else np.asarray(resid, dtype=np.float64) + y


def append_shared(idx, w, n_sel, shared_id: int):
    """Routes with the shared expert as one more kept slot of weight 1 right after each token's
    kept slots: idx, w [S x (K+1)] and n_sel + 1; the slots after it hold -1 and 0 ([attn], [pipe];
    the placement and the unscaled weight 1 are our reading, see moe_block_with_shared)."""
    idx = np.atleast_2d(np.asarray(idx, np.int32))
    w = np.atleast_2d(np.asarray(w, np.float32))
    S, K = idx.shape
    n_sel = np.full(S, K, np.int32) if n_sel is None else np.asarray(n_sel, np.int32)
    idx2 = np.full((S, K + 1), -1, np.int32)
    w2 = np.zeros((S, K + 1), np.float32)
    for t in range(S):
        m = int(n_sel[t])
        idx2[t, :m] = idx[t, :m]
        w2[t, :m] = w[t, :m]
        idx2[t, m] = shared_id
        w2[t, m] = 1.0
    return idx2, w2, n_sel + 1


def moe_block_with_shared(x, experts, idx, w, n_sel, shared, resid=None) -> np.ndarray:
    """y[t] = resid[t] + (routed[t] + E_shared(x[t])), float64.

    routed[t] is the slot-ordered weighted sum of :func:`expert_group` (no residual); the
    shared expert is a (gate, up, down) triple applied to every token with weight 1 ([attn]
    runs it on the device, [pipe] beside the residual adds). Reading: the pages give no
    formula; we take the usual one, an always-chosen expert whose output is added unscaled
    (no routing weight, no routed scale), and sum routed then shared before the residual.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    routed = expert_group(x, experts, idx, w, n_sel, None)
    gate, up, down = shared
    sh = np.stack([expert_ffn(x[t], gate, up, down) for t in range(x.shape[0])])
    y = routed + sh
    return y if resid is None else np.asarray(resid, dtype=np.float64) + y


# ------------------------------------------------------------------------------------------
# Expert parallelism over ranks [resid], [pipe]
# ------------------------------------------------------------------------------------------

def expert_owner(e: int, world: int) -> int:
    """Rank that holds expert e. Reading: the pages spread expert groups over the cards without a
    rule; we take e mod world (experts of neighbouring ids land on different ranks)."""
    return int(e) % int(world)


def shard_routes(idx, w, n_sel, rank: int, world: int):
    """Rank ``rank``'s share of the routes: each token's kept slots whose expert it owns, moved to
    the front in slot order; idx, w [S x K] (the rest -1 and 0) and the count n [S]."""
    idx = np.atleast_2d(np.asarray(idx, np.int32))
    w = np.atleast_2d(np.asarray(w, np.float32))
    S, K = idx.shape
    n_sel = np.full(S, K, np.int32) if n_sel is None else np.asarray(n_sel, np.int32)
    idx2 = np.full((S, K), -1, np.int32)
    w2 = np.zeros((S, K), np.float32)
    n2 = np.zeros(S, np.int32)
    for t in range(S):
        j = 0
        for k in range(int(n_sel[t])):
            if idx[t, k] >= 0 and expert_owner(idx[t, k], world) == rank:
                idx2[t, j], w2[t, j] = idx[t, k], w[t, k]
                j += 1
        n2[t] = j
    return idx2, w2, n2


def ep_layer(x, experts, idx, w, n_sel, world: int, resid=None) -> np.ndarray:
    """The expert-parallel block: every rank's partial sum over its own routes (expert_group with
    no residual), added in rank order, then the residual ([resid]: a fixed-order reduce of the
    device groups' partial sums). Equal to expert_group up to the grouping of the terms."""
    parts = [expert_group(x, experts, *shard_routes(idx, w, n_sel, r, world), None) for r in range(world)]
    acc = parts[0]
    for p in parts[1:]:
        acc = acc + p
    return acc if resid is None else np.asarray(resid, dtype=np.float64) + acc
