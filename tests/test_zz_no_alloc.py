"""The allocation-free decode entry point (moe_decode_noalloc) against the
regular context-based one (moe_forward, small-T path), through the C ABI.

Callers that cannot allocate device memory -- a plugin whose host application
owns every device buffer, or a serving loop that must not risk the device
synchronisation an allocation may cause -- use moe_decode_noalloc, whose
scratch is a fixed device array inside the library.
Two calls in a row must both match moe_forward (the second one runs on the
scratch contents the first one left behind).  This file is collected last so
that a stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import expert_routed_ffn_moe_gb300 as moe
from moe_case import check_y, device_inputs, layer_inputs, make_layer, oracle_y, y_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 4])
def test_noalloc_matches_context_path_twice(T):
    w = mw.Workload("noalloc", T=T, cid=77)
    inp = layer_inputs(w)
    d = device_inputs(w, inp)
    layer = make_layer(w)
    ref = layer.forward(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    layer.close()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        y = torch.full_like(d["x"], float("nan"))
        moe.moe_decode_noalloc(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"], w.k, y,
                               status=status)
        torch.cuda.synchronize()
        outs.append(y)
    assert int(status[0]) == 0
    for y in outs:
        check_y(y_host(y), y_host(ref).astype(np.float64), "noalloc vs moe_forward")
    check_y(y_host(outs[1]), oracle_y(w, inp, list(range(T))), "noalloc vs oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = mw.Workload("noalloc_big", T=17, d=512, E=64, I=256, I_s=256, k=4, cid=78)
    d = device_inputs(w, layer_inputs(w, margin=None))
    y = torch.empty_like(d["x"])
    with pytest.raises(moe.MoeError) as e:
        moe.moe_decode_noalloc(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"], w.k, y)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
