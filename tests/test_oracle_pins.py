"""Pins of the fp64 oracle to facts outside itself (no GPU needed).

Each test checks one oracle function against a closed form, a brute-force
evaluation on tiny inputs written independently here, a value the pages print,
or an invariant the pages state.  Together they are chosen so that a dropped
term, a wrong sign, a swapped gate/up half, a transposed weight or a wrong
index anywhere in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import moe_workloads as mw
import oracle
from oracle.inputs import MARGIN, enforce_margin, layer_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(a):
    return mw.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


# ----------------------------------------------------------------- decoding

def test_decode_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x0001, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127]
    got = oracle.decode_bf16(bits)
    assert got.dtype == np.float64
    assert list(got) == want


# ------------------------------------------------------------------- router

def test_router_logits_brute_force():
    rng = np.random.default_rng(0)
    T, E, d = 3, 5, 7
    x, wr, b = rng.normal(size=(T, d)), rng.normal(size=(E, d)), rng.normal(size=E)
    got = oracle.router_logits(x, wr, b)
    for t in range(T):
        for e in range(E):
            s = b[e]
            for i in range(d):
                s += x[t, i] * wr[e, i]
            assert abs(got[t, e] - s) < 1e-12


def test_router_weight_orientation():
    # Wr is [E, d]: a single nonzero Wr[e0, i0] only lifts expert e0, and only
    # through feature i0.  A transposed read would lift a different expert.
    E, d = 6, 9
    wr = np.zeros((E, d))
    wr[4, 2] = 1.0
    x = np.zeros((1, d))
    x[0, 2] = 5.0
    logits = oracle.router_logits(x, wr)
    assert np.argmax(logits[0]) == 4 and logits[0, 4] == 5.0
    idx, _, _ = oracle.route(logits, 1)
    assert idx[0, 0] == 4


def brute_top_k(row, k):
    """All k-subsets; the best has the largest sum of logits, ties to lower ids."""
    best = None
    for sub in itertools.combinations(range(len(row)), k):
        key = (sum(row[e] for e in sub), [-e for e in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    return list(best[1])


def test_select_top_k_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(50):
        E, k = int(rng.integers(2, 8)), None
        k = int(rng.integers(1, E + 1))
        row = rng.normal(size=E)
        idx, margin = oracle.select_top_k(row[None, :], k)
        assert list(idx[0]) == brute_top_k(row, k)
        srt = sorted(row, reverse=True)
        assert margin[0] == (srt[k - 1] - srt[k] if k < E else np.inf)


def test_select_ties_go_to_lower_expert():
    idx, margin = oracle.select_top_k(np.array([[1.0, 3.0, 1.0, 1.0]]), 2)
    assert list(idx[0]) == [0, 1] and margin[0] == 0.0


def test_route_hand_worked():
    # logits ln(1..4); top-2 = experts 2, 3; renormalised: 3/7, 4/7.
    logits = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    idx, w, margin = oracle.route(logits, 2)
    assert list(idx[0]) == [2, 3]
    assert abs(w[0, 0] - 3 / 7) < 1e-15 and abs(w[0, 1] - 4 / 7) < 1e-15
    assert abs(margin[0] - math.log(3 / 2)) < 1e-15


def test_route_weights_closed_forms():
    rng = np.random.default_rng(2)
    logits = rng.normal(size=(64, 16)) * 3
    # renormalised top-k weights = softmax over the selected logits alone
    for k in (1, 3, 8):
        idx, w, _ = oracle.route(logits, k)
        assert np.allclose(w.sum(1), 1.0, atol=1e-15, rtol=0)
        sel = np.take_along_axis(logits, idx.astype(np.int64), 1)
        assert np.allclose(w, scipy.special.softmax(sel, axis=1), atol=1e-15, rtol=0)
        # weights follow the logit order
        for t in range(8):
            order = np.argsort(sel[t])
            assert np.all(np.diff(w[t][order]) >= 0)
    # k = E: the full softmax (library routine), k = 1: weight one
    idx, w, _ = oracle.route(logits, 16)
    assert np.array_equal(idx, np.tile(np.arange(16), (64, 1)))
    assert np.allclose(w, scipy.special.softmax(logits, axis=1), atol=1e-15, rtol=0)
    _, w1, _ = oracle.route(logits, 1)
    assert np.all(w1 == 1.0)


def test_router_bias_only_routing():
    # Wr = 0 with a strictly decreasing bias: every token picks experts 0..k-1.
    E, k, T, d = 16, 4, 10, 8
    bias = np.array([1.2 * math.log(1.0 / (e + 1)) for e in range(E)])
    logits = oracle.router_logits(np.ones((T, d)), np.zeros((E, d)), bias)
    idx, w, _ = oracle.route(logits, k)
    assert np.all(idx == np.arange(k))
    counts, _, _, _ = oracle.group(idx, E)
    assert list(counts[:k]) == [T] * k and counts[k:].sum() == 0
    # weights: renormalised (e+1)^-1.2
    p = np.array([(e + 1) ** -1.2 for e in range(k)])
    assert np.allclose(w[0], p / p.sum(), atol=1e-15)


def test_bias_for_selection_only_hand_worked():
    # logits ln(1..4), bias +10 on expert 0, k = 2: the bias makes expert 0 a
    # pick (with expert 3); its weight comes from the unbiased logits:
    # exp(0) / (exp(0) + 4) = 1/5, expert 3: 4/5.  With the bias in the weights
    # expert 0 would carry e^10 / (e^10 + 4).
    l = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    b = np.array([10.0, 0.0, 0.0, 0.0])
    idx, w, _ = oracle.route(l + b, 2, weight_logits=l)
    assert list(idx[0]) == [0, 3]
    assert abs(w[0, 0] - 0.2) < 1e-15 and abs(w[0, 1] - 0.8) < 1e-15
    _, w_biased, _ = oracle.route(l + b, 2)
    assert abs(w_biased[0, 0] - math.exp(10) / (math.exp(10) + 4)) < 1e-15


def test_bias_for_selection_only_properties():
    rng = np.random.default_rng(11)
    l = rng.normal(size=(40, 16))
    # no bias: the variant is the plain routing
    a = oracle.route(l, 4)
    b = oracle.route(l, 4, weight_logits=l)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # a bias that keeps the picks changes no weight, whatever its size
    idx0, w0, _ = oracle.route(l, 4)
    bias = np.zeros(16)
    for scale in (1e-3, 1e-1):
        bias_t = scale * rng.normal(size=16)
        idx1, w1, _ = oracle.route(l + bias_t, 4, weight_logits=l)
        same = np.all(idx1 == idx0, axis=1)
        assert np.allclose(w1[same], w0[same], atol=1e-15, rtol=0)
    # the layer: identical to routing on l + b with weights from the softmax of
    # the unbiased logits over the picks, written out token by token
    E, k = 6, 3
    x, wr, gu, dn, sh = tiny_layer(rng, E=E, k=k)
    bias = rng.normal(size=E) * 2
    r = oracle.moe_layer(x, wr, bias, gu, dn, sh, k, x_bf16=False, bias_select_only=True)
    lu = x.astype(np.float64) @ wr.astype(np.float64).T
    for t in range(x.shape[0]):
        chosen = sorted(range(E), key=lambda e: (-(lu[t, e] + bias[e]), e))[:k]
        z = sum(math.exp(lu[t, e]) for e in chosen)
        assert list(r["idx"][t]) == sorted(chosen)
        assert np.allclose(r["w"][t], [math.exp(lu[t, e]) / z for e in sorted(chosen)], atol=1e-14)


# ----------------------------------------------------------------- grouping

def brute_group(idx, E):
    T, k = idx.shape
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    perm, slot = [], {}
    for e in range(E):
        for t in range(T):
            if e in list(idx[t]):
                slot[(t, e)] = len(perm)
                perm.append(t)
    return counts, offsets, perm, slot


def test_group_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(20):
        T, E = int(rng.integers(1, 12)), int(rng.integers(1, 10))
        k = int(rng.integers(1, E + 1))
        idx = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), 1)
        counts, offsets, perm, slot = oracle.group(idx.astype(np.int32), E)
        bc, bo, bp, bs = brute_group(idx, E)
        assert list(counts) == bc and list(offsets) == bo and list(perm) == bp
        for t in range(T):
            for j in range(k):
                assert slot[t, j] == bs[(t, idx[t, j])]


def test_group_invariants_and_pages_worked_example():
    g = {}
    for line in open(os.path.join(GOLDEN, "routing_worked_example.txt")):
        if line.strip() and not line.startswith("#"):
            key, val = line.split()
            g[key] = int(val)
    T, E, k = g["tokens"], g["experts"], g["top_k"]
    rng = np.random.default_rng(4)
    logits = rng.normal(size=(T, E))
    idx, _, _ = oracle.route(logits, k)
    counts, offsets, perm, slot = oracle.group(idx, E)
    assert counts.sum() == g["assignments"] == offsets[-1] == len(perm)
    assert counts.sum() / E == g["mean_rows_per_expert"]
    assert np.array_equal(np.bincount(perm, minlength=T), np.full(T, k))  # each token k times
    expert_of = np.repeat(np.arange(E), counts)
    key = expert_of.astype(np.int64) * T + perm
    assert np.all(np.diff(key) > 0)                                          # sorted by (expert, token)
    assert np.array_equal(perm[slot], np.tile(np.arange(T)[:, None], (1, k)))  # slot inverts perm
    assert np.array_equal(expert_of[slot], idx)


# -------------------------------------------------------------- expert FFN

def test_silu_closed_forms():
    l3 = math.log(3.0)
    g = np.array([0.0, l3, -l3, 40.0, -40.0, 1000.0, -1000.0])
    s = oracle.silu(g)
    assert s[0] == 0.0
    assert abs(s[1] - 0.75 * l3) < 1e-15 and abs(s[2] + 0.25 * l3) < 1e-15
    assert abs(s[3] - 40.0) < 1e-12 and abs(s[4]) < 1e-15
    assert s[5] == 1000.0 and s[6] == 0.0
    z = np.linspace(-6, 6, 101)
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, atol=1e-14)  # x*s(x) + x*s(-x) = x


def test_swiglu_hand_worked():
    # d = 2, I = 2.  g = [ln3, 0], u = [3, 0.5], h = [2.25 ln3, 0],
    # o = down h = [1*2.25 ln3, 3*2.25 ln3].  Swapping gate and up, or reading
    # down transposed, gives a different o.
    l3 = math.log(3.0)
    x = np.array([[1.0, 2.0]])
    gate_up = np.array([[l3, 0.0], [0.0, 0.0], [1.0, 1.0], [0.5, 0.0]])
    down = np.array([[1.0, 2.0], [3.0, 4.0]])
    o = oracle.swiglu_ffn(x, gate_up, down)
    assert np.allclose(o, [[2.25 * l3, 6.75 * l3]], atol=1e-15, rtol=0)


def test_swiglu_linear_in_up_and_down_not_gate():
    rng = np.random.default_rng(5)
    d, inter = 12, 5
    x, gu, dn = rng.normal(size=(4, d)), rng.normal(size=(2 * inter, d)), rng.normal(size=(d, inter))
    o = oracle.swiglu_ffn(x, gu, dn)
    gu_up = gu.copy()
    gu_up[inter:] *= 3.0
    assert np.allclose(oracle.swiglu_ffn(x, gu_up, dn), 3.0 * o, atol=1e-12)
    assert np.allclose(oracle.swiglu_ffn(x, gu, 3.0 * dn), 3.0 * o, atol=1e-12)
    gu_gate = gu.copy()
    gu_gate[:inter] *= 3.0
    assert not np.allclose(oracle.swiglu_ffn(x, gu_gate, dn), 3.0 * o, atol=1e-3)


def test_swiglu_neuron_bundles_and_order():
    # "LLM in a flash", section 3.2 "Bundling columns and rows": neuron i owns
    # up-projection row i and down-projection column i; section 3.3: the order
    # of intermediate neurons does not change the FFN output.
    rng = np.random.default_rng(6)
    d, inter = 10, 7
    x, gu, dn = rng.normal(size=(3, d)), rng.normal(size=(2 * inter, d)), rng.normal(size=(d, inter))
    o = oracle.swiglu_ffn(x, gu, dn)
    acc = np.zeros_like(o)
    for i in range(inter):                      # one bundle at a time
        g = x @ gu[i]
        u = x @ gu[inter + i]
        acc += ((g / (1 + np.exp(-g))) * u)[:, None] * dn[:, i][None, :]
    assert np.allclose(o, acc, atol=1e-12)
    p = rng.permutation(inter)
    gu_p = np.concatenate([gu[:inter][p], gu[inter:][p]])
    assert np.allclose(oracle.swiglu_ffn(x, gu_p, dn[:, p]), o, atol=1e-12)


# ------------------------------------------------------------------- layer

def tiny_layer(rng, T=5, E=6, d=4, inter=3, k=2, shared=True):
    x = rng.normal(size=(T, d)).astype(np.float32)
    wr = (rng.normal(size=(E, d)) * 0.5).astype(np.float32)
    gu = bf16_bits(rng.normal(size=(E, 2 * inter, d)) * 0.5)
    dn = bf16_bits(rng.normal(size=(E, d, inter)) * 0.5)
    sh = bf16_bits(rng.normal(size=3 * inter * d) * 0.5) if shared else None
    return x, wr, gu, dn, sh


def test_layer_brute_force_dense_masked():
    # Every expert on every token, masked by weights that are zero off the
    # top-k; selection by explicit sorting, weights by exp / sum written out.
    rng = np.random.default_rng(7)
    for trial in range(10):
        E, k = 6, int(rng.integers(1, 5))
        x, wr, gu, dn, sh = tiny_layer(rng, E=E, k=k)
        r = oracle.moe_layer(x, wr, None, gu, dn, sh, k, x_bf16=False)
        xf = x.astype(np.float64)
        for t in range(x.shape[0]):
            l = [sum(float(xf[t, i]) * float(wr[e, i]) for i in range(x.shape[1])) for e in range(E)]
            chosen = sorted(range(E), key=lambda e: (-l[e], e))[:k]
            z = sum(math.exp(l[e]) for e in chosen)
            y = np.zeros(x.shape[1])
            for e in range(E):
                m = math.exp(l[e]) / z if e in chosen else 0.0
                gu_e, dn_e = oracle.decode_bf16(gu[e]), oracle.decode_bf16(dn[e])
                inter = dn_e.shape[1]
                h = [0.0] * inter
                for i in range(inter):
                    g = sum(gu_e[i, c] * xf[t, c] for c in range(x.shape[1]))
                    u = sum(gu_e[inter + i, c] * xf[t, c] for c in range(x.shape[1]))
                    h[i] = g / (1 + math.exp(-g)) * u
                y += m * np.array([sum(dn_e[r_, i] * h[i] for i in range(inter)) for r_ in range(x.shape[1])])
            s = oracle.decode_bf16(sh)
            inter = dn.shape[2]
            d = x.shape[1]
            y += oracle.swiglu_ffn(xf[t:t + 1], s[:2 * inter * d].reshape(2 * inter, d),
                                   s[2 * inter * d:].reshape(d, inter))[0]
            assert np.allclose(r["y"][t], y, atol=1e-12), (trial, t)
            assert list(r["idx"][t]) == sorted(chosen)


def test_layer_single_expert_is_dense_swiglu():
    rng = np.random.default_rng(8)
    x, wr, gu, dn, _ = tiny_layer(rng, T=7, E=1, d=16, inter=8, k=1, shared=False)
    r = oracle.moe_layer(x, wr, None, gu, dn, None, 1, x_bf16=False)
    assert np.all(r["w"] == 1.0) and np.all(r["idx"] == 0)
    dense = oracle.swiglu_ffn(x.astype(np.float64), oracle.decode_bf16(gu[0]), oracle.decode_bf16(dn[0]))
    assert np.array_equal(r["y"], dense)


def test_layer_identical_experts_ignore_routing():
    # sum of weights is one, so with identical experts y = FFN(x) + shared(x)
    rng = np.random.default_rng(9)
    x, wr, gu, dn, sh = tiny_layer(rng, T=9, E=5, d=8, inter=4, k=3)
    gu[:] = gu[0]
    dn[:] = dn[0]
    r = oracle.moe_layer(x, wr, None, gu, dn, sh, 3, x_bf16=False)
    xf = x.astype(np.float64)
    s = oracle.decode_bf16(sh)
    want = oracle.swiglu_ffn(xf, oracle.decode_bf16(gu[0]), oracle.decode_bf16(dn[0])) + \
        oracle.swiglu_ffn(xf, s[:64].reshape(8, 8), s[64:].reshape(8, 4))
    assert np.allclose(r["y"], want, atol=1e-12)


def test_layer_shared_and_routed_parts_separate():
    rng = np.random.default_rng(10)
    x, wr, gu, dn, sh = tiny_layer(rng, T=6, E=4, d=8, inter=4, k=2)
    full = oracle.moe_layer(x, wr, None, gu, dn, sh, 2, x_bf16=False)["y"]
    routed = oracle.moe_layer(x, wr, None, gu, dn, None, 2, x_bf16=False)["y"]
    zero = np.zeros_like(gu)
    shared_only = oracle.moe_layer(x, wr, None, zero, np.zeros_like(dn), sh, 2, x_bf16=False)["y"]
    assert np.allclose(full, routed + shared_only, atol=1e-12)
    assert np.all(oracle.moe_layer(x, wr, None, gu, dn, np.zeros_like(sh), 2, x_bf16=False)["y"] == routed)


def test_sigmoid_closed_forms():
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0, -40.0, -800.0])
    got = oracle.sigmoid(z)
    assert got[0] == 0.5
    assert abs(got[1] - 0.75) < 1e-15 and abs(got[2] - 0.25) < 1e-15
    assert got[3] == 1.0 and 0.0 < got[4] < 1e-17 and got[5] == 0.0
    r = np.random.default_rng(3).normal(size=50) * 5
    assert np.allclose(oracle.sigmoid(r) + oracle.sigmoid(-r), 1.0, atol=1e-15, rtol=0)
    assert np.allclose(oracle.sigmoid(r), scipy.special.expit(r), atol=1e-16, rtol=1e-15)


def test_shared_gate_scales_only_the_shared_expert():
    # g = the first unit vector, so token t's gate logit is x[t, 0]: gates of
    # exactly 1/2, 3/4, 1/4, ~1 and ~0 (sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4).
    rng = np.random.default_rng(12)
    x, wr, gu, dn, sh = tiny_layer(rng, T=5, E=4, d=8, inter=4, k=2)
    x = x.astype(np.float64)
    x[:, 0] = [0.0, math.log(3.0), -math.log(3.0), 40.0, -40.0]
    g = np.zeros(8)
    g[0] = 1.0
    want_gate = np.array([0.5, 0.75, 0.25, 1.0, 0.0])
    gated = oracle.moe_layer(x, wr, None, gu, dn, sh, 2, x_bf16=False, shared_gate_w=g)
    plain = oracle.moe_layer(x, wr, None, gu, dn, sh, 2, x_bf16=False)
    routed = oracle.moe_layer(x, wr, None, gu, dn, None, 2, x_bf16=False)["y"]
    # the gate changes neither the picks nor their weights
    assert np.array_equal(gated["idx"], plain["idx"]) and np.array_equal(gated["w"], plain["w"])
    shared_part = plain["y"] - routed
    assert np.all(np.abs(shared_part).max(axis=1) > 1e-3)
    assert np.allclose(gated["y"], routed + want_gate[:, None] * shared_part, atol=1e-12, rtol=0)
    # without a shared expert the gate vector is ignored
    r = oracle.moe_layer(x, wr, None, gu, dn, None, 2, x_bf16=False, shared_gate_w=g)["y"]
    assert np.array_equal(r, routed)
    # a general gate vector: the logit is the dot product with the token row
    g2 = rng.normal(size=8)
    gated2 = oracle.moe_layer(x[:3], wr, None, gu, dn, sh, 2, x_bf16=False, shared_gate_w=g2)["y"]
    for t in range(3):
        z = sum(float(x[t, i]) * float(g2[i]) for i in range(8))
        s_t = 1.0 / (1.0 + math.exp(-z))
        assert np.allclose(gated2[t], routed[t] + s_t * shared_part[t], atol=1e-12, rtol=0)


# ------------------------------------------------------- 4-bit group-affine weights

def _bf16_value(bits: int) -> float:
    # an independent bf16 decoder: the bits are the high half of an fp32
    import struct
    return struct.unpack(">f", ((bits & 0xFFFF) << 16).to_bytes(4, "big"))[0]


def test_unpack_u4_hand_worked():
    words = np.array([0x76543210, 0xFEDCBA98], dtype=np.uint32)
    assert list(oracle.unpack_u4(words)) == list(range(16))
    assert list(oracle.unpack_u4(np.array([0xF0F0F0F0], dtype=np.uint32))) == [0, 15] * 4


def test_dequant_affine4_hand_worked():
    # one row of 128 columns, two groups: scale 0.5 / bias -1 with every code
    # 3 (-> 0.5), then scale 2 / bias 0.25 with codes 0, 15, 0, 15, ...
    # (-> 0.25, 30.25, ...)
    words = np.array([[0x33333333] * 8 + [0xF0F0F0F0] * 8], dtype=np.uint32)
    scales = np.array([[0x3F00, 0x4000]], dtype=np.uint16)
    biases = np.array([[0xBF80, 0x3E80]], dtype=np.uint16)
    w = oracle.dequant_affine4(words, scales, biases)
    assert w.shape == (1, 128)
    assert np.all(w[0, :64] == 0.5)
    assert list(w[0, 64:68]) == [0.25, 30.25, 0.25, 30.25]
    # all-zero codes give the bias, all-15 codes 15 scale + bias
    z = oracle.dequant_affine4(np.zeros((1, 16), np.uint32), scales, biases)
    assert np.all(z[0, :64] == -1.0) and np.all(z[0, 64:] == 0.25)
    f = oracle.dequant_affine4(np.full((1, 16), 0xFFFFFFFF, np.uint32), scales, biases)
    assert np.all(f[0, :64] == 6.5) and np.all(f[0, 64:] == 30.25)


def test_dequant_affine4_brute_force():
    rng = np.random.default_rng(21)
    rows, K, g = 3, 256, 64
    words = rng.integers(0, 2 ** 32, size=(rows, K // 8), dtype=np.uint64).astype(np.uint32)
    scales = bf16_bits(rng.normal(size=(rows, K // g)) * 0.01)
    biases = bf16_bits(rng.normal(size=(rows, K // g)) * 0.05)
    got = oracle.dequant_affine4(words, scales, biases, group=g)
    for r in range(rows):
        for k in range(K):
            q = (int(words[r, k // 8]) >> (4 * (k % 8))) & 15
            want = _bf16_value(int(scales[r, k // g])) * q + _bf16_value(int(biases[r, k // g]))
            assert got[r, k] == want, (r, k)


def test_layer_on_expanded_4bit_weights():
    # 4-bit weights whose expansion (q - 8) / 32 is exact in bf16: the layer
    # on the expanded fp64 weights equals the layer on those bf16 weights
    rng = np.random.default_rng(22)
    E, d, inter, k, T = 4, 64, 64, 2, 5
    x = rng.normal(size=(T, d)).astype(np.float32)
    wr = (rng.normal(size=(E, d)) * 0.5).astype(np.float32)

    def q4(rows, cols):
        words = rng.integers(0, 2 ** 32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
        sc = np.full((rows, cols // 64), 0x3D00, np.uint16)  # 2^-5
        bi = np.full((rows, cols // 64), 0xBE80, np.uint16)  # -2^-2
        return oracle.dequant_affine4(words, sc, bi)

    gu = np.stack([q4(2 * inter, d) for _ in range(E)])
    dn = np.stack([q4(d, inter) for _ in range(E)])
    sh = (q4(2 * inter, d), q4(d, inter))
    assert np.all(gu * 32 == np.round(gu * 32)) and np.abs(gu).max() <= 0.25
    r64 = oracle.moe_layer(x, wr, None, gu, dn, sh, k, x_bf16=False, weights_f64=True)
    flat_sh = np.concatenate([bf16_bits(sh[0]).ravel(), bf16_bits(sh[1]).ravel()])
    rb = oracle.moe_layer(x, wr, None, bf16_bits(gu), bf16_bits(dn), flat_sh, k, x_bf16=False)
    assert np.array_equal(r64["idx"], rb["idx"])
    assert np.array_equal(r64["y"], rb["y"])


def test_layer_token_permutation_equivariance_and_subsets():
    rng = np.random.default_rng(11)
    x, wr, gu, dn, sh = tiny_layer(rng, T=11, E=7, d=8, inter=4, k=3)
    full = oracle.moe_layer(x, wr, None, gu, dn, sh, 3, x_bf16=False)
    p = rng.permutation(11)
    perm_r = oracle.moe_layer(x[p], wr, None, gu, dn, sh, 3, x_bf16=False)
    assert np.allclose(perm_r["y"], full["y"][p], atol=1e-13)
    assert np.array_equal(perm_r["idx"], full["idx"][p])
    sub = [9, 2, 5]
    r = oracle.moe_layer(x, wr, None, gu, dn, sh, 3, x_bf16=False, tokens=sub)
    assert np.allclose(r["y"], full["y"][sub], atol=1e-13)
    used = sorted(set(r["idx"].ravel().tolist()))
    r2 = oracle.moe_layer(x, wr, None, gu[used], dn[used], sh, 3, x_bf16=False, tokens=sub,
                          expert_ids=used)
    assert np.array_equal(r2["y"], r["y"])


def test_layer_x_bf16_decoding():
    rng = np.random.default_rng(12)
    x, wr, gu, dn, sh = tiny_layer(rng, T=4, E=4, d=8, inter=4, k=2)
    xb = bf16_bits(x)
    a = oracle.moe_layer(xb, wr, None, gu, dn, sh, 2, x_bf16=True)["y"]
    b = oracle.moe_layer(oracle.decode_bf16(xb), wr, None, gu, dn, sh, 2, x_bf16=False)["y"]
    assert np.array_equal(a, b)


# ------------------------------------------------------------------- inputs

def test_margin_enforcement_tiny_workload():
    w = mw.WORKLOADS["tiny"]
    inp = layer_inputs(w)
    logits = oracle.router_logits(oracle.as_f64(inp["x"], False), inp["router_w"].astype(np.float64))
    _, gap = oracle.select_top_k(logits, w.k)
    assert gap.min() >= MARGIN
    # deterministic: same draw twice
    again = enforce_margin(w, 0, mw.draw_x(w), inp["router_w"], None)
    assert np.array_equal(again, inp["x"])


def test_skewed_bias_matches_recipe():
    w = mw.WORKLOADS["prefill_skewed"]
    _, b = mw.draw_router(w)
    assert b[0] == 0.0 and abs(b[1] - 1.2 * math.log(0.5)) < 1e-6 and np.all(np.diff(b) < 0)


def test_4bit_inputs_recipe():
    # the seeded 4-bit experts expand to weights of mean ~0 and spread ~0.02,
    # like the bf16 experts; codes are uniform over 0..15
    w = mw.WORKLOADS["decode"]
    (gu, dn) = mw.draw_expert_q4(w, 0, 5)
    assert gu[0].shape == (2 * w.I, w.d // 8) and gu[1].shape == (2 * w.I, w.d // 64)
    assert dn[0].shape == (w.d, w.I // 8) and dn[2].shape == (w.d, w.I // 64)
    W = oracle.dequant_affine4(*gu)
    assert abs(W.mean()) < 1e-3 and 0.019 < W.std() < 0.021
    counts = np.bincount(oracle.unpack_u4(gu[0]).ravel(), minlength=16)
    assert counts.min() > 0.95 * counts.mean() and counts.max() < 1.05 * counts.mean()
    sh = mw.draw_expert_q4(w, 0, -1)
    assert not np.array_equal(sh[0][0], mw.draw_expert_q4(w, 0, 0)[0][0])
