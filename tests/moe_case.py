"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
layer through the C ABI, and compare with the fp64 oracle.

Parity bar (fixed here, used by every test):
  * routing indices, per-expert counts, offsets and the permutation: bit-exact;
  * routing weights: |w_gpu - w_oracle| <= 1e-5 * w_oracle + 1e-7;
  * y: relative L2 error <= 1e-2 and max-abs error <= 2e-2 against the fp64
    oracle evaluated on the same stored inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_workloads as mw
import oracle
from oracle.inputs import layer_inputs
import expert_routed_ffn_moe_gb300 as moe

REL_L2 = 1e-2
MAX_ABS = 2e-2
W_REL = 1e-5


def bf16_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def device_inputs(w: mw.Workload, inp: dict, dev="cuda"):
    x = torch.from_numpy(inp["x"]).to(dev) if w.x_dtype == "f32" else bf16_dev(inp["x"], dev)
    return dict(
        x=x,
        router_w=torch.from_numpy(inp["router_w"]).to(dev),
        router_b=None if inp["router_b"] is None else torch.from_numpy(inp["router_b"]).to(dev),
        gate_up=bf16_dev(inp["gate_up"], dev),
        down=bf16_dev(inp["down"], dev),
        shared=None if inp["shared"] is None else bf16_dev(inp["shared"], dev),
    )


def make_layer(w: mw.Workload, max_tokens=None, path=moe.MOE_PATH_AUTO, router=moe.MOE_ROUTER_AUTO,
               bias_select_only=False, shared_gate=False):
    layer = moe.MoeLayer(w.d, w.E, w.I, w.k, max_tokens or w.T,
                         x_dtype=moe.MOE_F32 if w.x_dtype == "f32" else moe.MOE_BF16,
                         has_router_bias=w.skewed, has_shared=w.I_s > 0, bias_select_only=bias_select_only,
                         shared_gate=shared_gate)
    moe.moe_set_path(layer.ctx, path)
    moe.moe_set_router(layer.ctx, router)
    return layer


def gpu_run(w, inp, layer, dev_in=None, top_k=None, with_forward_tables=False):
    """moe_route's tables and y from moe_forward; with ``with_forward_tables``
    also the tables moe_forward itself computed (read back with moe_last_routing)."""
    d = dev_in or device_inputs(w, inp)
    k = top_k or w.k
    r = layer.route(d["x"], d["router_w"], d["router_b"], top_k=k)
    r = {key: v.cpu().numpy() for key, v in r.items()}
    y = layer.forward(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"], top_k=k)
    fwd = {key: v.cpu().numpy() for key, v in layer.last_routing().items()}
    torch.cuda.synchronize()
    status = layer.status()
    assert status == moe.MOE_OK, moe.moe_strerror(status)
    return (r, y, fwd) if with_forward_tables else (r, y)


def oracle_routing(w, inp, k=None, bias_select_only=False):
    k = k or w.k
    x = oracle.as_f64(inp["x"], w.x_dtype == "bf16")
    logits = oracle.router_logits(x, inp["router_w"].astype(np.float64), inp["router_b"])
    unbiased = (oracle.router_logits(x, inp["router_w"].astype(np.float64), None)
                if bias_select_only and inp["router_b"] is not None else None)
    idx, wts, margin = oracle.route(logits, k, weight_logits=unbiased)
    counts, offsets, perm, slot = oracle.group(idx, w.E)
    return dict(idx=idx, w=wts, margin=margin, counts=counts, offsets=offsets, perm=perm, slot=slot)


def check_routing(got, ref, what="moe_route"):
    """Bit-exact idx, counts, offsets, perm (and slot when ``got`` has it);
    weights within W_REL relative."""
    assert np.array_equal(got["idx"], ref["idx"]), f"{what}: routing indices differ"
    assert np.array_equal(got["counts"], ref["counts"]), f"{what}: per-expert counts differ"
    assert np.array_equal(got["offsets"], ref["offsets"]), f"{what}: expert offsets differ"
    assert np.array_equal(got["perm"], ref["perm"]), f"{what}: permutation differs"
    if "slot" in got:
        assert np.array_equal(got["slot"], ref["slot"]), f"{what}: slots differ"
    err = np.abs(got["w"] - ref["w"])
    assert np.all(err <= W_REL * ref["w"] + 1e-7), f"{what}: routing weights differ (max {err.max():.3e})"


def oracle_y(w, inp, tokens, k=None, bias_select_only=False, shared_gate_w=None):
    """fp64 oracle output rows for `tokens`, drawing only the experts they use."""
    k = k or w.k
    r = oracle.moe_layer(inp["x"], inp["router_w"], inp["router_b"], inp["gate_up"], inp["down"], inp["shared"],
                         k, x_bf16=w.x_dtype == "bf16", tokens=tokens, bias_select_only=bias_select_only,
                         shared_gate_w=shared_gate_w)
    return r["y"]


def check_y(got: np.ndarray, ref: np.ndarray, what=""):
    got = got.astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{what}: rel L2 {rel:.3e} max abs {mx:.3e}"
    return rel, mx


def tile_position_tokens(ref, T: int, n: int, bm: int = 128, seed: int = 0) -> np.ndarray:
    """At least ``n`` tokens (all if T <= n) that cover every grouped-GEMM m-tile
    position: for each expert group (``ref`` = oracle routing) the first, second
    and last rows of its first, second and last tiles of ``bm`` rows, the same
    for the shared expert's group (all T tokens in order), the first and last
    token, then random tokens up to ``n``."""
    if T <= n:
        return np.arange(T)
    pick = {0, T - 1}
    offsets, perm = ref["offsets"], ref["perm"]
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        c = hi - lo
        if c == 0:
            continue
        n_tiles = (c + bm - 1) // bm
        for tile in {0, 1, n_tiles - 1}:
            if tile >= n_tiles:
                continue
            r0, r1 = tile * bm, min(c, (tile + 1) * bm)
            for r in {r0, r0 + 1, r1 - 1}:
                if r0 <= r < r1:
                    pick.add(int(perm[lo + r]))
    for t0 in (0, bm, T - T % bm if T % bm else T - bm):
        for t in (t0, t0 + 1, min(T, t0 + bm) - 1):
            if 0 <= t < T:
                pick.add(t)
    rng = np.random.default_rng(seed)
    while len(pick) < n:
        pick.update(rng.choice(T, n - len(pick), replace=False).tolist())
    return np.array(sorted(pick))


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """All tokens if T <= n, else n tokens spread over the range incl. both ends."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(pick))


def y_host(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy()


__all__ = ["bf16_dev", "device_inputs", "make_layer", "gpu_run", "oracle_routing", "check_routing", "oracle_y",
           "check_y", "sample_tokens", "tile_position_tokens", "layer_inputs", "y_host"]
