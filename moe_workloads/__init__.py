"""Seeded synthetic inputs for the routed-expert SwiGLU MoE layer.

This module only *draws* tensors.  It holds none of the layer's arithmetic:
no router logits, no softmax, no selection, no FFN.  Both the CUDA path (via
the tests and the benchmark) and the fp64 oracle consume what it returns.

Workload shapes follow the MoE layer of "Optimizing on-device inference for
Apple Silicon" (section "Qwen creates three different workload shapes"): a
router over 256 experts that picks eight of them plus one shared expert that
every token goes through.  Model width ``d`` and the expert inner size ``I``
are not printed on that page; the workloads below fix them (d=2048, I=512,
and a tiny d=512, I=128 case).

Value recipe (all draws are float32 standard normals from numpy's PCG64,
each tensor from its own ``SeedSequence``):

* ``x``            ~ N(0, 1), stored fp32 (tiny workload) or rounded to bf16;
* ``router_w``     ~ N(0, 0.02^2), fp32, shape [E, d];
* ``router_b``     b_e = 1.2 * ln(1 / (e + 1)) (skewed workloads only), fp32;
* expert weights   ~ N(0, 0.02^2) rounded to bf16 (round-to-nearest-even):
  ``gate_up`` [E, 2I, d] (rows 0..I-1 gate, I..2I-1 up), ``down`` [E, d, I];
* shared expert    same distribution, one flat bf16 buffer holding its
  gate_up [2I_s, d] followed by its down [d, I_s].
* shared gate      (the sigmoid-gated shared-expert variant) g ~ N(0, 0.9^2 / d),
  fp32 [d]: with x ~ N(0, 1) the gate logit x . g has a spread of about 0.9,
  so the gates cover most of (0, 1).
* 4-bit experts    (the 4-bit group-affine variant) per weight matrix: uniformly
  random 32-bit words (eight uniform 4-bit codes each), and per 64-column group
  a bf16 scale s = 0.02 / sqrt(21.25) * (1 + 0.1 N(0, 1)) and bias -7.5 s (21.25
  is the variance of a uniform code in 0..15), so that the expanded weights have
  mean ~0 and spread ~0.02 like the bf16 experts.

Each expert is drawn from its own stream, so a caller that needs only a few
experts (the oracle on a sample of tokens) can draw just those.

A token row of ``x`` can be redrawn (``redraw_x_rows``) from a stream keyed by
(token, attempt); the tests use that to enforce a gap between the 8th and 9th
router logit without this module computing any logit itself.

bf16 tensors are returned as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

SEED_BASE = 20261202

# tensor-kind tags for SeedSequence keys
_X, _X_REDRAW, _ROUTER_W, _GATE_UP, _DOWN, _SHARED, _SHARED_GATE, _Q4 = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE-layer workload: shapes, dtype of x, routing skew, layer count."""

    name: str
    T: int                 # tokens
    d: int = 2048          # model width
    E: int = 256           # routed experts
    I: int = 512           # routed expert inner size
    I_s: int = 512         # shared expert inner size (0 = no shared expert)
    k: int = 8             # experts selected per token
    x_dtype: str = "bf16"  # "bf16" or "f32"
    skewed: bool = False   # add the Zipf-like router bias
    layers: int = 1        # distinct weight sets run back to back
    cid: int = 0           # workload id, part of every seed

    @property
    def seed(self) -> int:
        return SEED_BASE + self.cid


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", T=32, d=512, I=128, I_s=128, x_dtype="f32", cid=1),
        Workload("decode", T=1, layers=10, cid=2),
        Workload("prefill_balanced", T=4096, cid=3),
        Workload("prefill_skewed", T=4096, skewed=True, cid=4),
        Workload("sweep_T2", T=2, cid=5),
        Workload("sweep_T8", T=8, cid=5),
        Workload("sweep_T32", T=32, cid=5),
        Workload("sweep_T128", T=128, cid=5),
        Workload("sweep_T32768", T=32768, cid=5),
    ]
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(v) for v in key])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the 16-bit patterns."""
    import torch  # torch's CPU cast is round-to-nearest-even and multithreaded

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal(scale: float, n: int, *key: int) -> np.ndarray:
    a = _rng(*key).standard_normal(n, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def draw_x(w: Workload, layer: int = 0, T: Optional[int] = None) -> np.ndarray:
    """Token activations x [T, d]: float32, or bf16 bits when ``x_dtype == 'bf16'``."""
    T = w.T if T is None else T
    a = _normal(1.0, T * w.d, w.seed, layer, _X, T).reshape(T, w.d)
    return a if w.x_dtype == "f32" else f32_to_bf16_bits(a)


def redraw_x_rows(w: Workload, layer: int, rows, attempt: int) -> np.ndarray:
    """Fresh draws for the given token rows; row t's value depends only on (t, attempt)."""
    out = np.stack([_normal(1.0, w.d, w.seed, layer, _X_REDRAW, int(t), attempt) for t in rows])
    return out if w.x_dtype == "f32" else f32_to_bf16_bits(out)


def draw_router(w: Workload, layer: int = 0):
    """Router weights [E, d] fp32 and the optional bias [E] fp32 (None when unskewed)."""
    wr = _normal(0.02, w.E * w.d, w.seed, layer, _ROUTER_W).reshape(w.E, w.d)
    b = None
    if w.skewed:
        b = np.array([1.2 * math.log(1.0 / (e + 1)) for e in range(w.E)], dtype=np.float32)
    return wr, b


def draw_expert(w: Workload, layer: int, e: int):
    """One routed expert: gate_up [2I, d] and down [d, I], bf16 bits."""
    gu = _normal(0.02, 2 * w.I * w.d, w.seed, layer, _GATE_UP, e)
    dn = _normal(0.02, w.d * w.I, w.seed, layer, _DOWN, e)
    return (f32_to_bf16_bits(gu).reshape(2 * w.I, w.d), f32_to_bf16_bits(dn).reshape(w.d, w.I))


def _q4_matrix(rows: int, cols: int, *key: int):
    rng = _rng(*key)
    words = rng.integers(0, 2 ** 32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
    s = np.float32(0.02 / math.sqrt(21.25)) * (1 + np.float32(0.1) * rng.standard_normal((rows, cols // 64),
                                                                                          dtype=np.float32))
    return words, f32_to_bf16_bits(s), f32_to_bf16_bits(np.float32(-7.5) * s)


def draw_expert_q4(w: Workload, layer: int, e: int):
    """One routed expert in 4 bits (``e = -1``: the shared expert): for gate_up [2I, d]
    and down [d, I], (words uint32 [rows, cols / 8], scales, biases bf16 [rows, cols / 64])."""
    inter = w.I if e >= 0 else w.I_s
    return (_q4_matrix(2 * inter, w.d, w.seed, layer, _Q4, e + 1, 0),
            _q4_matrix(w.d, inter, w.seed, layer, _Q4, e + 1, 1))


def draw_experts_q4(w: Workload, layer: int = 0, experts=None, threads: int = 16):
    """Stacked 4-bit routed experts (``draw_expert_q4``) for ``experts`` (default all):
    dict of gu_words [n, 2I, d/8] u32, gu_scales / gu_biases [n, 2I, d/64] bf16 bits,
    dn_words [n, d, I/8], dn_scales / dn_biases [n, d, I/64]."""
    ids = list(range(w.E)) if experts is None else [int(e) for e in experts]
    n = len(ids)
    out = dict(gu_words=np.empty((n, 2 * w.I, w.d // 8), np.uint32),
               gu_scales=np.empty((n, 2 * w.I, w.d // 64), np.uint16),
               gu_biases=np.empty((n, 2 * w.I, w.d // 64), np.uint16),
               dn_words=np.empty((n, w.d, w.I // 8), np.uint32),
               dn_scales=np.empty((n, w.d, w.I // 64), np.uint16),
               dn_biases=np.empty((n, w.d, w.I // 64), np.uint16))

    def one(j):
        (gw, gs, gb), (dw, ds, db) = draw_expert_q4(w, layer, ids[j])
        out["gu_words"][j], out["gu_scales"][j], out["gu_biases"][j] = gw, gs, gb
        out["dn_words"][j], out["dn_scales"][j], out["dn_biases"][j] = dw, ds, db

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(one, range(n)))
    return out


def pack_q4(words: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """The library's byte layout of 4-bit matrices (MOE_W_Q4G64): every row as
    its code words, then its scales, then its biases (9 K / 16 bytes for K
    columns), rows back to back.  Pure data movement (no arithmetic): words
    [..., R, K/8] u32, scales and biases [..., R, K/64] bf16 bits -> uint8 [bytes]."""
    rows = np.concatenate([np.ascontiguousarray(words).view(np.uint8),
                           np.ascontiguousarray(scales).view(np.uint8),
                           np.ascontiguousarray(biases).view(np.uint8)], axis=-1)
    return np.ascontiguousarray(rows).ravel()


def draw_experts(w: Workload, layer: int = 0, experts=None, threads: int = 16):
    """Stacked routed experts: gate_up [n, 2I, d] and down [n, d, I] bf16 bits.

    ``experts`` selects which ones (default: all E, in order)."""
    ids = list(range(w.E)) if experts is None else [int(e) for e in experts]
    gu = np.empty((len(ids), 2 * w.I, w.d), dtype=np.uint16)
    dn = np.empty((len(ids), w.d, w.I), dtype=np.uint16)

    def one(j):
        gu[j], dn[j] = draw_expert(w, layer, ids[j])

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(one, range(len(ids))))
    return gu, dn


def draw_shared(w: Workload, layer: int = 0) -> Optional[np.ndarray]:
    """Shared expert as one flat bf16 buffer: gate_up [2I_s, d] then down [d, I_s]."""
    if w.I_s == 0:
        return None
    a = _normal(0.02, 3 * w.I_s * w.d, w.seed, layer, _SHARED)
    return f32_to_bf16_bits(a)


def draw_shared_gate(w: Workload, layer: int = 0) -> np.ndarray:
    """Gate vector of the sigmoid-gated shared-expert variant, fp32 [d]."""
    return _normal(0.9 / math.sqrt(w.d), w.d, w.seed, layer, _SHARED_GATE)


def split_shared(w: Workload, shared: np.ndarray):
    """View the flat shared buffer as (gate_up [2I_s, d], down [d, I_s])."""
    n = 2 * w.I_s * w.d
    return shared[:n].reshape(2 * w.I_s, w.d), shared[n:].reshape(w.d, w.I_s)
