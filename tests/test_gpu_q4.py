"""4-bit group-affine experts (MOE_W_Q4G64) on the GPU against the fp64 oracle.

The oracle expands the codes exactly (``oracle.dequant_affine4``: w = s q + b
per 64-column group) and runs the same layer on the expanded weights
(``moe_layer(weights_f64=True)``); the library reads the packed planes and
expands the codes inside its kernels.  Routing is unchanged by the weight
format (the router is fp32), so indices and tables must match bit for bit and
y must be within the usual tolerance.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle
import expert_routed_ffn_moe_gb300 as moe
from moe_case import check_routing, check_y, layer_inputs, oracle_routing, y_host

pytestmark = pytest.mark.gpu


def q4_inputs(w, layer=0):
    """Router and x from the usual seeded inputs (margin enforced); 4-bit experts."""
    inp = layer_inputs(w, layer, with_experts=False)
    q = mw.draw_experts_q4(w, layer)
    sh = mw.draw_expert_q4(w, layer, -1) if w.I_s else None
    return inp, q, sh


def packed_device(q, sh, dev="cuda"):
    def dev_u8(a):
        return torch.from_numpy(a).to(dev)

    gu = dev_u8(mw.pack_q4(q["gu_words"], q["gu_scales"], q["gu_biases"]))
    dn = dev_u8(mw.pack_q4(q["dn_words"], q["dn_scales"], q["dn_biases"]))
    shared = None
    if sh is not None:
        (gw, gs, gb), (dw, ds, db) = sh
        shared = dev_u8(np.concatenate([mw.pack_q4(gw, gs, gb), mw.pack_q4(dw, ds, db)]))
    return gu, dn, shared


class _Expand:
    """Stacked 4-bit matrices expanded one expert at a time on access (the
    oracle indexes its expert weights by position), so that a full layer does
    not hold every expert in float64 at once."""

    def __init__(self, words, scales, biases, ids):
        self.words, self.scales, self.biases, self.ids = words, scales, biases, ids

    def __getitem__(self, j):
        e = self.ids[j]
        return oracle.dequant_affine4(self.words[e], self.scales[e], self.biases[e])


def oracle_q4_y(w, inp, q, sh, tokens, k=None):
    """fp64 layer on the exactly expanded 4-bit weights, for `tokens` (only the experts they use)."""
    k = k or w.k
    ref = oracle_routing(w, dict(inp, x=inp["x"][tokens]), k)
    used = np.unique(ref["idx"])
    gu = _Expand(q["gu_words"], q["gu_scales"], q["gu_biases"], used)
    dn = _Expand(q["dn_words"], q["dn_scales"], q["dn_biases"], used)
    shared = None
    if sh is not None:
        (gw, gs, gb), (dw, ds, db) = sh
        shared = (oracle.dequant_affine4(gw, gs, gb), oracle.dequant_affine4(dw, ds, db))
    r = oracle.moe_layer(inp["x"], inp["router_w"], inp["router_b"], gu, dn, shared, k, x_bf16=w.x_dtype == "bf16",
                         tokens=tokens, expert_ids=used, weights_f64=True)
    return r["y"]


def run_q4(w, inp, q, sh, path=moe.MOE_PATH_AUTO):
    dev = "cuda"
    x = (torch.from_numpy(inp["x"]).to(dev) if w.x_dtype == "f32"
         else torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev))
    wr = torch.from_numpy(inp["router_w"]).to(dev)
    rb = None if inp["router_b"] is None else torch.from_numpy(inp["router_b"]).to(dev)
    gu, dn, shared = packed_device(q, sh)
    layer = moe.MoeLayer(w.d, w.E, w.I, w.k, w.T, x_dtype=moe.MOE_F32 if w.x_dtype == "f32" else moe.MOE_BF16,
                         has_router_bias=w.skewed, has_shared=w.I_s > 0, weight_format=moe.MOE_W_Q4G64)
    moe.moe_set_path(layer.ctx, path)
    y = layer.forward(x, wr, rb, gu, dn, shared)
    fwd = {key: v.cpu().numpy() for key, v in layer.last_routing().items()}
    torch.cuda.synchronize()
    status = layer.status()
    layer.close()
    assert status == moe.MOE_OK, moe.moe_strerror(status)
    return y, fwd


@pytest.mark.parametrize("T", [1, 3, 4])
def test_q4_fused_decode_kernel_decode_shapes(T):
    # d = 2048, 256 experts of inner size 512, top-8 + shared, bf16 x
    w = mw.Workload(f"q4_dec{T}", T=T, cid=40)
    inp, q, sh = q4_inputs(w)
    y, fwd = run_q4(w, inp, q, sh)
    check_routing(fwd, oracle_routing(w, inp), "moe_forward")
    toks = np.arange(w.T)
    check_y(y_host(y), oracle_q4_y(w, inp, q, sh, toks), f"4-bit decode T={T}")


@pytest.mark.parametrize("T,x_dtype,skewed", [(2, "bf16", False), (7, "f32", False), (16, "bf16", True)])
def test_q4_fused_decode_kernel_small_shapes(T, x_dtype, skewed):
    # d = 512, 64 experts of inner size 256, top-4 + shared; every token bound up to 16
    w = mw.Workload(f"q4_small{T}", T=T, d=512, E=64, I=256, I_s=256, k=4, x_dtype=x_dtype, skewed=skewed, cid=41)
    inp, q, sh = q4_inputs(w)
    y, fwd = run_q4(w, inp, q, sh, path=moe.MOE_PATH_GEMV)
    check_routing(fwd, oracle_routing(w, inp), "moe_forward")
    check_y(y_host(y), oracle_q4_y(w, inp, q, sh, np.arange(w.T)), f"4-bit decode small T={T}")


def test_q4_no_shared_expert():
    w = mw.Workload("q4_noshared", T=2, d=512, E=64, I=256, I_s=0, k=4, cid=42)
    inp, q, sh = q4_inputs(w)
    y, _ = run_q4(w, inp, q, sh)
    check_y(y_host(y), oracle_q4_y(w, inp, q, sh, np.arange(w.T)), "4-bit, no shared expert")


def test_q4_rejects_inner_size_not_multiple_of_256():
    with pytest.raises(moe.MoeError) as e:
        moe.MoeLayer(512, 64, 128, 4, 8, weight_format=moe.MOE_W_Q4G64)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


# ------------------------------------------------------------ grouped GEMMs (codes expanded inside the GEMM)

@pytest.mark.parametrize("T,d,E,I,k", [(64, 512, 64, 256, 4), (300, 1024, 64, 512, 8), (8, 2048, 256, 512, 8)])
def test_q4_grouped_gemm(T, d, E, I, k):
    # inner size 256 loads each row's 4 scales and 4 biases in one box; 512 and
    # d = 1024 / 2048 in boxes of 8 groups; T = 8 at the decode shapes forced
    # onto the GEMMs
    w = mw.Workload(f"q4_gemm{T}_{d}", T=T, d=d, E=E, I=I, I_s=I, k=k, cid=43)
    inp, q, sh = q4_inputs(w)
    y, fwd = run_q4(w, inp, q, sh, path=moe.MOE_PATH_GEMM)
    ref = oracle_routing(w, inp)
    check_routing(fwd, ref, "moe_forward")
    check_y(y_host(y), oracle_q4_y(w, inp, q, sh, np.arange(w.T)), f"4-bit grouped GEMM T={T}")


@pytest.mark.parametrize("name", ["prefill_balanced", "prefill_skewed"])
def test_q4_prefill_every_token(name):
    # T = 4096, d = 2048, 256 experts of 512, top-8 + shared; every token's y
    import dataclasses

    w = dataclasses.replace(mw.WORKLOADS[name], name=name + "_q4", cid=mw.WORKLOADS[name].cid + 40)
    inp, q, sh = q4_inputs(w)
    y, fwd = run_q4(w, inp, q, sh)
    ref = oracle_routing(w, inp)
    check_routing(fwd, ref, "moe_forward")
    check_y(y_host(y), oracle_q4_y(w, inp, q, sh, np.arange(w.T)), f"4-bit {name}")
