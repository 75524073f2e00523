"""Layer inputs with a guaranteed routing margin (TEST INFRASTRUCTURE).

The routed-expert layer must pick the same k experts on the GPU (fp32 logits)
as in this fp64 oracle.  Selection is an integer decision taken from floating
point, so the inputs are drawn such that, for every token, the k-th and the
(k+1)-th largest router logit differ by at least ``MARGIN`` (1e-3): far above
the ~1e-6 error of an fp32 dot product of length 2048.  A token row that
misses the margin is replaced by the next draw of its own per-token stream
(``moe_workloads.redraw_x_rows``) until it passes.  Logits are evaluated here,
in fp64, on the *stored* values (after the bf16 rounding of x).
"""
from __future__ import annotations

import numpy as np

import moe_workloads as mw

from .moe_oracle import as_f64, router_logits, select_top_k

MARGIN = 1e-3


def enforce_margin(w: mw.Workload, layer: int, x: np.ndarray, router_w, router_b,
                   margin: float = MARGIN, max_attempts: int = 200) -> np.ndarray:
    """Return x with every row's k-th/(k+1)-th logit gap >= ``margin``."""
    x = x.copy()
    wr = np.asarray(router_w, dtype=np.float64)
    bf16 = w.x_dtype == "bf16"
    _, gap = select_top_k(router_logits(as_f64(x, bf16), wr, router_b), w.k)
    bad = np.nonzero(gap < margin)[0]
    attempt = 0
    while bad.size:
        if attempt >= max_attempts:
            raise RuntimeError(f"could not reach routing margin {margin} for rows {bad[:8]}")
        fresh = mw.redraw_x_rows(w, layer, bad, attempt)
        _, g = select_top_k(router_logits(as_f64(fresh, bf16), wr, router_b), w.k)
        ok = g >= margin
        x[bad[ok]] = fresh[ok]
        bad = bad[~ok]
        attempt += 1
    return x


def layer_inputs(w: mw.Workload, layer: int = 0, *, margin: float | None = MARGIN,
                 with_experts: bool = True):
    """All inputs of one layer as numpy arrays (bf16 as uint16 bits).

    Keys: x, router_w, router_b, gate_up, down, shared."""
    router_w, router_b = mw.draw_router(w, layer)
    x = mw.draw_x(w, layer)
    if margin is not None:
        x = enforce_margin(w, layer, x, router_w, router_b, margin)
    out = dict(x=x, router_w=router_w, router_b=router_b, shared=mw.draw_shared(w, layer))
    if with_experts:
        out["gate_up"], out["down"] = mw.draw_experts(w, layer)
    return out
