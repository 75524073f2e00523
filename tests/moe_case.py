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


def gpu_run(w, inp, layer, dev_in=None, top_k=None):
    d = dev_in or device_inputs(w, inp)
    k = top_k or w.k
    r = layer.route(d["x"], d["router_w"], d["router_b"], top_k=k)
    y = layer.forward(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"], top_k=k)
    torch.cuda.synchronize()
    status = layer.status()
    assert status == moe.MOE_OK, moe.moe_strerror(status)
    return {key: v.cpu().numpy() for key, v in r.items()}, y


def oracle_routing(w, inp, k=None, bias_select_only=False):
    k = k or w.k
    x = oracle.as_f64(inp["x"], w.x_dtype == "bf16")
    logits = oracle.router_logits(x, inp["router_w"].astype(np.float64), inp["router_b"])
    unbiased = (oracle.router_logits(x, inp["router_w"].astype(np.float64), None)
                if bias_select_only and inp["router_b"] is not None else None)
    idx, wts, margin = oracle.route(logits, k, weight_logits=unbiased)
    counts, offsets, perm, slot = oracle.group(idx, w.E)
    return dict(idx=idx, w=wts, margin=margin, counts=counts, offsets=offsets, perm=perm, slot=slot)


def check_routing(got, ref):
    assert np.array_equal(got["idx"], ref["idx"]), "routing indices differ"
    assert np.array_equal(got["counts"], ref["counts"]), "per-expert counts differ"
    assert np.array_equal(got["offsets"], ref["offsets"]), "expert offsets differ"
    assert np.array_equal(got["perm"], ref["perm"]), "permutation differs"
    err = np.abs(got["w"] - ref["w"])
    assert np.all(err <= W_REL * ref["w"] + 1e-7), f"routing weights differ (max {err.max():.3e})"


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
           "check_y", "sample_tokens", "layer_inputs", "y_host"]
