"""fp64 CPU oracle of the routed-expert SwiGLU MoE layer.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The library's CUDA path
never calls it and shares no code with it.

What it computes, step by step, for token rows x_t (all in float64, nothing
rounded; stored inputs are decoded exactly: fp32 as is, bf16 bits -> float):

1. router logits  l[t, e] = sum_i x[t, i] * Wr[e, i]  (+ b[e] when a bias is
   given).  "Optimizing on-device inference for Apple Silicon", section "Qwen
   creates three different workload shapes": a router scores the 256 experts
   of every token.
2. selection: the k experts with the largest logits (ties go to the lower
   expert id).  Same section: eight of the 256 are chosen.
3. weights: p = softmax over all E logits; the k selected probabilities are
   renormalised to sum to one (the pages do not spell the weighting out; the
   plain reading used here is softmax-then-renormalise).
4. canonical order: each token's k (expert, weight) pairs sorted by expert id.
5. grouping (same page, section "Keeping expert routing on the GPU"): per-expert
   counts, their exclusive prefix sum as start offsets, and the permutation
   that lists, for expert 0, 1, ... in turn, the tokens that chose it in
   ascending token order; ``slot[t, j]`` is the position of (t, idx[t, j]).
6. expert FFN, SwiGLU: g = W_gate x, u = W_up x, h = silu(g) * u,
   o = W_down h, with gate_up rows [0, I) the gate and [I, 2I) the up
   projection ("two input projections of the experts with their gated
   activation", same page, section "Reducing intermediate and state traffic").
7. shared expert: the same FFN with the shared weights, applied to every token
   with weight one (section "Qwen creates three different workload shapes").
8. output y_t = sum_j w[t, j] * o_{idx[t, j]}(x_t) + o_shared(x_t), summed over
   j in ascending expert order.

Variants the pages do not describe (plain readings, each pinned on its own):
- bias for selection only: the router bias decides which experts are picked,
  and the picks' weights are the softmax of the unbiased logits over them.
- sigmoid-gated shared expert: o_shared(x_t) is scaled by sigmoid(x_t . g) for
  a gate vector g of d fp32 values (no bias).
- 4-bit group-affine expert weights ("Optimizing on-device inference for Apple
  Silicon", section "Dequantizing weights during matrix multiplication": the
  checkpoint stores the experts in 4 bits and the kernels expand them inside
  the multiplication).  Reading: along each weight row, groups of 64
  consecutive input columns share one scale and one bias (bf16); a weight is
  scale * q + bias for its 4-bit code q in 0..15; eight codes are packed per
  32-bit word, the lowest nibble first.  The layer is then the same layer over
  the expanded weights (``dequant_affine4`` and ``moe_layer(weights_f64=True)``).

Library primitives used as steps: numpy matmul (a dot product per output
element), ``numpy.exp``, ``numpy.argsort`` (stable) and ``numpy.bincount``.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, brute force on tiny inputs, hand-worked golden values and invariants.
"""
from __future__ import annotations

import numpy as np


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.ascontiguousarray(bits).view(np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray, bf16: bool) -> np.ndarray:
    """Stored tensor -> float64: bf16 bit patterns when ``bf16``, else fp32/fp64 values."""
    return decode_bf16(a) if bf16 else np.asarray(a, dtype=np.float64)


def router_logits(x: np.ndarray, router_w: np.ndarray, router_b=None) -> np.ndarray:
    """Step 1: l[t, e] = sum_i x[t, i] Wr[e, i] (+ b[e]); x [T, d], Wr [E, d], fp64."""
    logits = x @ router_w.T
    if router_b is not None:
        logits = logits + np.asarray(router_b, dtype=np.float64)[None, :]
    return logits


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row softmax over the last axis, shifted by the row maximum."""
    m = logits.max(axis=-1, keepdims=True)
    p = np.exp(logits - m)
    return p / p.sum(axis=-1, keepdims=True)


def select_top_k(logits: np.ndarray, k: int):
    """Steps 2 and 4: the k largest logits per row, returned in ascending expert id.

    Returns (idx [T, k] int32, margin [T]) where margin is the gap between the
    k-th and the (k+1)-th largest logit (+inf when k == E)."""
    T, E = logits.shape
    order = np.argsort(-logits, axis=1, kind="stable")  # equal logits: lower id first
    rows = np.arange(T)
    if k < E:
        margin = logits[rows, order[:, k - 1]] - logits[rows, order[:, k]]
    else:
        margin = np.full(T, np.inf)
    idx = np.sort(order[:, :k], axis=1).astype(np.int32)
    return idx, margin


def route(logits: np.ndarray, k: int, weight_logits: np.ndarray | None = None):
    """Steps 2-4: (idx [T, k] int32 ascending, w [T, k] fp64, margin [T]).

    The k experts are picked on ``logits``; their weights come from
    ``weight_logits`` (default: the same logits).  The variant with a router
    bias that only balances load picks on l + b and weights on l."""
    idx, margin = select_top_k(logits, k)
    p = softmax(logits if weight_logits is None else weight_logits)
    p_sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    w = p_sel / p_sel.sum(axis=1, keepdims=True)
    return idx, w, margin


def group(idx: np.ndarray, n_experts: int):
    """Step 5: (counts [E], offsets [E+1], perm [T*k], slot [T, k]), all int32.

    perm lists token ids grouped by expert (ascending), tokens ascending within
    a group; slot[t, j] is where (t, idx[t, j]) landed in perm."""
    T, k = idx.shape
    e_flat = idx.astype(np.int64).ravel()
    t_flat = np.repeat(np.arange(T, dtype=np.int64), k)
    counts = np.bincount(e_flat, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(e_flat * max(T, 1) + t_flat, kind="stable")
    perm = t_flat[order]
    slot = np.empty(T * k, dtype=np.int64)
    slot[order] = np.arange(T * k)
    return (counts.astype(np.int32), offsets.astype(np.int32), perm.astype(np.int32),
            slot.reshape(T, k).astype(np.int32))


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_ffn(x_rows: np.ndarray, gate_up: np.ndarray, down: np.ndarray) -> np.ndarray:
    """Step 6: o = W_down (silu(W_gate x) * (W_up x)) for each row of x_rows.

    x_rows [n, d]; gate_up [2I, d] (gate rows first); down [d, I]; fp64."""
    inter = down.shape[1]
    g = x_rows @ gate_up[:inter].T
    u = x_rows @ gate_up[inter:].T
    h = silu(g) * u
    return h @ down.T


def unpack_u4(words: np.ndarray) -> np.ndarray:
    """uint32 words [..., n] -> 4-bit codes [..., 8 n] (uint8), lowest nibble first."""
    w = np.ascontiguousarray(words, dtype=np.uint32)
    shifts = np.arange(8, dtype=np.uint32) * 4
    codes = (w[..., None] >> shifts) & np.uint32(15)
    return codes.reshape(*w.shape[:-1], w.shape[-1] * 8).astype(np.uint8)


def dequant_affine4(words: np.ndarray, scales: np.ndarray, biases: np.ndarray, group: int = 64) -> np.ndarray:
    """Expanded weights, fp64 [..., K]: scale[g] * q + bias[g] for the group g = k // group of
    each column k.  words uint32 [..., K / 8]; scales, biases bf16 bits [..., K / group]."""
    q = unpack_u4(words).astype(np.float64)
    s = np.repeat(decode_bf16(scales), group, axis=-1)
    b = np.repeat(decode_bf16(biases), group, axis=-1)
    assert q.shape == s.shape == b.shape, (q.shape, s.shape, b.shape)
    return s * q + b


def sigmoid(z: np.ndarray) -> np.ndarray:
    """sigmoid(z) = 1 / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def moe_layer(x, router_w, router_b, gate_up, down, shared, k, *, x_bf16: bool,
              shared_inter: int | None = None, tokens=None, expert_ids=None, bias_select_only: bool = False,
              shared_gate_w=None, weights_f64: bool = False):
    """Steps 1-8 for the token rows ``tokens`` (default: all).

    x        [T, d]  fp32 values, or bf16 bits when ``x_bf16``
    router_w [E, d]  fp32;  router_b [E] fp32 or None
    gate_up  [n, 2I, d] bf16 bits;  down [n, d, I] bf16 bits
    shared   flat bf16 bits: gate_up [2I_s, d] then down [d, I_s]; or None
    expert_ids  which expert each of the n stacked matrices is (default
             0..n-1); lets a caller pass only the experts the sampled tokens use.
    bias_select_only  the router bias picks the experts but their weights are
             the softmax of the unbiased logits over the picks.
    shared_gate_w  [d] fp32 gate vector, or None: the shared expert's output
             is scaled by sigmoid(x_t . shared_gate_w).
    weights_f64  the expert weights are given as float64 values (for example
             expanded 4-bit weights) instead of bf16 bits: gate_up [n, 2I, d],
             down [n, d, I], and shared, if any, as the pair (gate_up [2I_s, d],
             down [d, I_s]).

    Returns dict(y [n_tok, d] fp64, idx, w, margin, logits) for those tokens."""
    xs = as_f64(x, x_bf16)
    tokens = np.arange(xs.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xs = xs[tokens]
    wr = np.asarray(router_w, dtype=np.float64)
    logits = router_logits(xs, wr, router_b)
    unbiased = router_logits(xs, wr, None) if (bias_select_only and router_b is not None) else None
    idx, w, margin = route(logits, k, weight_logits=unbiased)
    n_tok, d = xs.shape
    y = np.zeros((n_tok, d), dtype=np.float64)

    where = {int(e): j for j, e in enumerate(range(gate_up.shape[0]) if expert_ids is None else expert_ids)}
    counts, offsets, perm, slot = group(idx, wr.shape[0])
    for e in range(wr.shape[0]):               # ascending e: each token sums its j in order
        rows = perm[offsets[e]:offsets[e + 1]]
        if rows.size == 0:
            continue
        j = where[e]
        if weights_f64:
            o = swiglu_ffn(xs[rows], np.asarray(gate_up[j], dtype=np.float64), np.asarray(down[j], dtype=np.float64))
        else:
            o = swiglu_ffn(xs[rows], decode_bf16(gate_up[j]), decode_bf16(down[j]))
        w_e = w[rows, np.argmax(idx[rows] == e, axis=1)]
        y[rows] += w_e[:, None] * o
    if shared is not None:
        if weights_f64:
            o_s = swiglu_ffn(xs, np.asarray(shared[0], dtype=np.float64), np.asarray(shared[1], dtype=np.float64))
        else:
            i_s = shared_inter if shared_inter is not None else len(shared) // (3 * d)
            sh = decode_bf16(shared)
            o_s = swiglu_ffn(xs, sh[: 2 * i_s * d].reshape(2 * i_s, d), sh[2 * i_s * d:].reshape(d, i_s))
        if shared_gate_w is not None:
            o_s = sigmoid(xs @ np.asarray(shared_gate_w, dtype=np.float64))[:, None] * o_s
        y += o_s
    return dict(y=y, idx=idx, w=w, margin=margin, logits=logits)
