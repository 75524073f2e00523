"""Expert-parallel dispatch/combine bookkeeping on two gloo ranks (CPU).

Each rank owns half of the experts and its own share of the tokens.  The test
routes each rank's tokens with the oracle, dispatches the picks with
``expert_parallel``, runs each rank's local experts on the rows it received
(the oracle's SwiGLU FFN, fp64), returns the outputs with the reverse exchange
and forms the weighted sum; the result must equal the single-process oracle
layer over all tokens.  It also checks that the rows an expert receives,
concatenated over source ranks, are exactly that expert's group of the global
stable permutation (expert ascending, token ascending), and the count
bookkeeping of both exchanges.  Unmeasured on GPUs: nothing here runs NCCL.
"""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, wl, split, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from oracle.inputs import layer_inputs
    from expert_routed_ffn_moe_gb300 import expert_parallel as ep

    inp = layer_inputs(wl)
    lo, hi = split[rank], split[rank + 1]
    x_all = oracle.as_f64(inp["x"], wl.x_dtype == "bf16")
    x = x_all[lo:hi]
    T, k, E = hi - lo, wl.k, wl.E
    # 1. route this rank's tokens (router replicated)
    idx, w, _ = oracle.route(oracle.router_logits(x, inp["router_w"].astype(np.float64), inp["router_b"]), k)
    idx_t = torch.from_numpy(idx.astype(np.int64))
    # 2. dispatch the rows, and (for the bookkeeping check) their global token ids
    plan, rows, experts = ep.dispatch(torch.from_numpy(x), idx_t, E)
    _, tok_ids, _ = ep.dispatch(torch.arange(lo, hi, dtype=torch.int64)[:, None], idx_t, E)
    # 3. local experts on the received rows
    n_local = ep.experts_per_rank(E, world)
    first = rank * n_local
    counts, offsets, perm = ep.local_groups(experts, first, n_local)
    out_rows = torch.zeros_like(rows)
    local_perm = {}
    for i in range(n_local):
        sel = perm[offsets[i]:offsets[i + 1]]
        local_perm[first + i] = tok_ids[sel, 0].numpy()
        if sel.numel() == 0:
            continue
        gu, dn = oracle.decode_bf16(inp["gate_up"][first + i]), oracle.decode_bf16(inp["down"][first + i])
        out_rows[sel] = torch.from_numpy(oracle.swiglu_ffn(rows[sel].numpy(), gu, dn))
    # 4. combine: outputs back in pick order, weighted sum in ascending expert order, shared expert locally
    per_pick = ep.combine_rows(out_rows, plan, T, k).numpy()
    y = np.zeros((T, wl.d))
    for j in range(k):
        y += w[:, j:j + 1] * per_pick[:, j]
    if inp["shared"] is not None:
        sh = oracle.decode_bf16(inp["shared"])
        i_s = wl.I_s
        y += oracle.swiglu_ffn(x, sh[:2 * i_s * wl.d].reshape(2 * i_s, wl.d), sh[2 * i_s * wl.d:].reshape(wl.d, i_s))
    sends = [torch.empty(world, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sends, torch.tensor(plan.send_counts, dtype=torch.int64))
    out[rank] = dict(y=y, lo=lo, hi=hi, send=plan.send_counts, recv=plan.recv_counts,
                     sends=[s.tolist() for s in sends], counts=counts.numpy(), local_perm=local_perm,
                     n_rows=int(rows.shape[0]))
    dist.barrier()
    dist.destroy_process_group()


def _run(wl, split):
    world = len(split) - 1
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, wl, split, out), nprocs=world, join=True)
        return dict(out)


@pytest.mark.parametrize("skewed,split", [(False, (0, 16, 32)), (True, (0, 21, 32))])
def test_expert_parallel_two_ranks_matches_single_layer(skewed, split):
    import sys

    sys.path.insert(0, ROOT)
    import moe_workloads as mw
    import oracle
    from oracle.inputs import layer_inputs

    wl = dataclasses.replace(mw.WORKLOADS["tiny"], name=f"ep_tiny_{int(skewed)}", skewed=skewed, cid=60 + skewed)
    res = _run(wl, split)
    world = len(split) - 1
    inp = layer_inputs(wl)
    ref = oracle.moe_layer(inp["x"], inp["router_w"], inp["router_b"], inp["gate_up"], inp["down"], inp["shared"],
                           wl.k, x_bf16=wl.x_dtype == "bf16")
    counts, offsets, perm, _ = oracle.group(ref["idx"], wl.E)
    for r in range(world):
        got = res[r]
        # the layer over this rank's tokens equals the single-process layer
        np.testing.assert_allclose(got["y"], ref["y"][got["lo"]:got["hi"]], rtol=1e-10, atol=1e-12)
        # every pick leaves once; what r receives from s is what s sends to r
        assert sum(got["send"]) == (got["hi"] - got["lo"]) * wl.k
        assert got["recv"] == [res[s]["send"][r] for s in range(world)]
        assert got["sends"] == [res[s]["send"] for s in range(world)]
        assert got["n_rows"] == sum(got["recv"])
        # each owned expert receives exactly its global group, in stable (token) order
        n_local = wl.E // world
        for e in range(r * n_local, (r + 1) * n_local):
            np.testing.assert_array_equal(got["local_perm"][e], perm[offsets[e]:offsets[e + 1]])
        np.testing.assert_array_equal(got["counts"], counts[r * n_local:(r + 1) * n_local])
    if skewed:
        # the Zipf-like bias sends most picks to the owner of the low expert ids
        assert sum(res[0]["recv"]) > 2 * sum(res[1]["recv"])


def test_partition_rejects_uneven_split():
    import sys

    sys.path.insert(0, ROOT)
    from expert_routed_ffn_moe_gb300 import expert_parallel as ep

    with pytest.raises(ValueError):
        ep.experts_per_rank(256, 3)
    assert ep.expert_owner(torch.tensor([0, 127, 128, 255]), 256, 2).tolist() == [0, 0, 1, 1]
    plan = ep.plan_dispatch(torch.tensor([[1, 200], [3, 130]]), 256, 2)
    # sending order: owner 0 (experts 1, 3), then owner 1 (experts 130, 200)
    assert plan.send_counts == [2, 2]
    assert plan.order.tolist() == [0, 2, 3, 1]
