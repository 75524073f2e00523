"""GPU path vs the fp64 oracle, through the C ABI, on the seeded workloads.

Routing (indices, counts, offsets, permutation, slots) must match bit for bit
and y must be within relative L2 1e-2 / max-abs 2e-2 (tests/moe_case.py).  The
routing is checked twice: the tables moe_route returns, and the tables
moe_forward itself computed and used (read back with moe_last_routing).  y is
compared on every token up to T = 4096; at T = 32768 on 4096 tokens that cover
the first, second and last rows of the first, second and last m-tile of every
expert group and of the shared expert's group.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_workloads as mw
import expert_routed_ffn_moe_gb300 as moe
from moe_case import (check_routing, check_y, device_inputs, gpu_run, layer_inputs, make_layer, oracle_routing,
                      oracle_y, tile_position_tokens, y_host)

pytestmark = pytest.mark.gpu

W = mw.WORKLOADS


def custom(name, **kw):
    base = dict(T=64, d=512, E=64, I=256, I_s=256, k=4, cid=90)
    base.update(kw)
    return mw.Workload(name, **base)


def full_case(w, layer_id=0, path=moe.MOE_PATH_AUTO, router=moe.MOE_ROUTER_AUTO, n_sample=4096, inp=None):
    inp = inp or layer_inputs(w, layer_id)
    layer = make_layer(w, path=path, router=router)
    got, y, fwd = gpu_run(w, inp, layer, with_forward_tables=True)
    layer.close()
    ref = oracle_routing(w, inp)
    check_routing(got, ref)
    check_routing(fwd, ref, "moe_forward")
    toks = tile_position_tokens(ref, w.T, n_sample)
    return check_y(y_host(y)[toks], oracle_y(w, inp, toks), f"{w.name} layer {layer_id}")


# ------------------------------------------------------------ the workloads

def test_tiny_fp32_x():
    full_case(W["tiny"])


@pytest.mark.parametrize("layer_id", [0, 7])
def test_decode_layer(layer_id):
    full_case(W["decode"], layer_id)


def test_decode_on_grouped_gemm_path():
    full_case(W["decode"], 3, path=moe.MOE_PATH_GEMM)


@pytest.mark.parametrize("name", ["sweep_T2", "sweep_T8", "sweep_T32", "sweep_T128"])
def test_sweep_small(name):
    full_case(W[name])


def test_prefill_balanced():
    full_case(W["prefill_balanced"])


def test_prefill_skewed():
    full_case(W["prefill_skewed"])


def test_long_prefill_32768():
    full_case(W["sweep_T32768"])


def test_prefill_simt_router_matches():
    full_case(W["prefill_balanced"], router=moe.MOE_ROUTER_SIMT)


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("T", [1, 31, 33, 129, 300, 1000])
def test_ragged_token_counts(T):
    full_case(custom(f"ragged{T}", T=T))


def test_gemv_and_gemm_paths_agree_fp32_x():
    w = custom("gemv_f32", T=8, x_dtype="f32")
    inp = layer_inputs(w)
    a = full_case(w, path=moe.MOE_PATH_GEMV, inp=inp)
    b = full_case(w, path=moe.MOE_PATH_GEMM, inp=inp)
    assert a[0] < 1e-2 and b[0] < 1e-2


@pytest.mark.parametrize("w", [
    # groups of ~512 rows: two full pairs, some a single tile more; the shared group 8 tiles
    custom("pairs_e8", T=1024, E=8, k=4),
    # groups of ~525 rows: two full pairs and a single tile; the shared group's last pair is part-filled
    custom("pairs_e4", T=700, E=4, k=3),
    # ragged groups of ~525 rows, no shared expert
    custom("pairs_e16_noshared", T=2100, E=16, k=4, I_s=0),
], ids=lambda w: w.name)
def test_paired_gate_up_groups(w):
    # T k >= 512 E: the gate/up GEMM multiplies two m-tiles of a group per weight tile
    assert w.T * w.k >= 4 * 128 * w.E
    full_case(w)


@pytest.mark.parametrize("path", [moe.MOE_PATH_GEMV, moe.MOE_PATH_GEMM])
def test_no_shared_expert(path):
    full_case(custom("noshared", T=8, I_s=0), path=path)


def test_router_bias_small():
    full_case(custom("bias", T=200, skewed=True))


def test_single_expert_is_dense_ffn():
    full_case(custom("dense", T=100, E=1, k=1, I_s=0))


def test_top_k_below_configured():
    w = custom("k2", T=150, k=8)
    inp = layer_inputs(dataclasses.replace(w, k=2))
    w2 = dataclasses.replace(w, k=2)
    layer = make_layer(w)  # configured for top-8, called with top-2
    got, y, fwd = gpu_run(w2, inp, layer, top_k=2, with_forward_tables=True)
    layer.close()
    ref = oracle_routing(w2, inp)
    check_routing(got, ref)
    check_routing(fwd, ref, "moe_forward")
    check_y(y_host(y), oracle_y(w2, inp, np.arange(w.T)), "top-2")


def test_many_experts_per_token():
    full_case(custom("k32", T=40, E=64, k=32))


def test_zero_tokens_is_a_noop():
    w = custom("zero", T=4)
    layer = make_layer(w)
    d = device_inputs(w, layer_inputs(w))
    y = torch.full_like(d["x"], 7.0)
    moe.moe_forward(layer.ctx, d["x"][:0], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"],
                    w.k, y[:0])
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK and bool((y == 7.0).all())
    layer.close()


# ------------------------------------------------------------ properties

def test_deterministic_and_token_permutation_equivariant():
    w = custom("equiv", T=300, d=1024, E=128, I=256, k=8)
    inp = layer_inputs(w)
    layer = make_layer(w)
    d = device_inputs(w, inp)
    args = (d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    y1 = layer.forward(d["x"], *args).clone()
    y2 = layer.forward(d["x"], *args).clone()
    p = torch.from_numpy(np.random.default_rng(5).permutation(w.T)).cuda()
    yp = layer.forward(d["x"][p].contiguous(), *args).clone()
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    layer.close()
    assert torch.equal(y1, y2), "two runs differ"
    assert torch.equal(yp, y1[p]), "not equivariant under token permutation"


# ------------------------------------------------------------ errors

def test_argument_errors():
    w = custom("errs", T=16)
    layer = make_layer(w)
    d = device_inputs(w, layer_inputs(w))
    y = torch.empty_like(d["x"])
    base = [d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"]]
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(layer.ctx, d["x"], *base, 0, y)
    assert e.value.code == moe.MOE_ERR_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(layer.ctx, d["x"], *base, w.k + 1, y)
    assert e.value.code == moe.MOE_ERR_ARG
    big = torch.cat([d["x"], d["x"]])
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(layer.ctx, big, *base, w.k, torch.empty_like(big))
    assert e.value.code == moe.MOE_ERR_ARG
    flat = torch.empty(d["x"].numel() + 8, dtype=d["x"].dtype, device="cuda")
    xm = flat[1:1 + d["x"].numel()].view_as(d["x"])  # 2-byte offset: not 16-byte aligned
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(layer.ctx, xm, *base, w.k, y)
    assert e.value.code == moe.MOE_ERR_ALIGN
    assert moe.lib().moe_forward(layer.ctx, None, 4, None, None, None, None, None, w.k, None, None) == moe.MOE_ERR_ARG
    layer.close()


def test_bounded_wait_reports_timeout_and_context_recovers():
    # The injected stall makes the grouped GEMM's MMA thread wait on a barrier
    # nothing signals; with a 1 ms limit the wait runs out, the kernel must
    # return with MOE_ERR_TIMEOUT latched (no trap, no hang), and the same
    # context must then run correctly again.
    w = custom("timeout", T=256)
    inp = layer_inputs(w)
    layer = make_layer(w, path=moe.MOE_PATH_GEMM)
    d = device_inputs(w, inp)
    args = (d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    moe.moe_set_spin_limit(layer.ctx, 1_000_000)
    moe.moe_inject_stall(layer.ctx, True)
    layer.forward(d["x"], *args)
    assert layer.status() == moe.MOE_ERR_TIMEOUT
    moe.moe_inject_stall(layer.ctx, False)
    moe.moe_set_spin_limit(layer.ctx, 0)
    y = layer.forward(d["x"], *args)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    layer.close()
    toks = np.arange(w.T)
    check_y(y_host(y)[toks], oracle_y(w, inp, toks), "after timeout")


def test_modular_gemv_path_beyond_fused_limit():
    # T = 24 with d = 512, I = 256: above the fused decode kernel's 16-token
    # limit, still inside the GEMV kernels' shared-memory limit
    full_case(custom("gemv24", T=24), path=moe.MOE_PATH_GEMV)


def test_fused_decode_barrier_timeout_and_recovery():
    # The injected stall makes every block wait for router logits tagged with
    # an epoch that no block writes; with a 1 ms limit the wait runs out, the
    # status word reports it, and the next call on the same context (a new
    # epoch) is correct and does not take the failed call's values as ready.
    w = W["decode"]
    inp = layer_inputs(w, 2)
    layer = make_layer(w)
    d = device_inputs(w, inp)
    args = (d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    moe.moe_set_spin_limit(layer.ctx, 1_000_000)
    moe.moe_inject_stall(layer.ctx, True)
    layer.forward(d["x"], *args)
    assert layer.status() == moe.MOE_ERR_TIMEOUT
    moe.moe_inject_stall(layer.ctx, False)
    moe.moe_set_spin_limit(layer.ctx, 0)
    y = layer.forward(d["x"], *args)
    y2 = layer.forward(d["x"], *args)
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    layer.close()
    assert torch.equal(y, y2)
    check_y(y_host(y), oracle_y(w, inp, [0]), "after barrier timeout")


def test_overlapped_decode_launches_match_plain():
    # Programmatic launch overlap lets a layer's blocks start while the
    # previous layer's kernel finishes; they must read x (the previous
    # layer's output) only after waiting for it.  Chain three layers through
    # x -> y -> x on one stream, with and without overlap, eagerly and from a
    # CUDA graph: all four results must be bitwise equal.
    w = W["decode"]
    inps = [layer_inputs(w, i) for i in range(3)]
    devs = [device_inputs(w, inp) for inp in inps]
    layer = make_layer(w)
    st = torch.cuda.Stream()

    def chain():
        x = devs[0]["x"]
        for d in devs:
            y = torch.empty_like(x)
            moe.moe_forward(layer.ctx, x, d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"],
                            w.k, y, st)
            x = y
        return x

    outs = []
    for on in (False, True):
        moe.moe_set_overlap(layer.ctx, on)
        with torch.cuda.stream(st):
            outs.append(chain().clone())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                yg = chain()
            g.replay()
        st.synchronize()
        outs.append(yg.clone())
    assert layer.status() == moe.MOE_OK
    layer.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_prefetch_hint_does_not_change_results():
    # moe_set_prefetch only moves the next layer's weights into L2: the layer
    # computed with the hint must equal the one computed without it, bitwise.
    w = W["decode"]
    d0, d1 = device_inputs(w, layer_inputs(w, 0)), device_inputs(w, layer_inputs(w, 1))
    layer = make_layer(w)
    args = (d0["router_w"], d0["router_b"], d0["gate_up"], d0["down"], d0["shared"])
    y_plain = layer.forward(d0["x"], *args).clone()
    moe.moe_set_prefetch(layer.ctx, d1["router_w"], d1["shared"])
    y_hint = layer.forward(d0["x"], *args).clone()
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    layer.close()
    assert torch.equal(y_plain, y_hint)


def test_chunked_prefill_matches_oracle_and_unchunked():
    # moe_set_chunk_tokens: a context sized for 256 tokens runs T = 700 in
    # slices of 256, 256 and 188; every token must match the oracle, and the
    # same tokens through a context sized for all 700 must agree (each slice
    # takes the grouped-GEMM path, whose per-row arithmetic does not depend on
    # which other rows share a tile).
    w = custom("chunked", T=700)
    inp = layer_inputs(w)
    d = device_inputs(w, inp)
    args = (d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    small = make_layer(w, max_tokens=256)
    moe.moe_set_chunk_tokens(small.ctx, 256)
    y_chunked = small.forward(d["x"], *args).clone()
    last = {key: v.cpu().numpy() for key, v in small.last_routing().items()}
    torch.cuda.synchronize()
    assert small.status() == moe.MOE_OK
    # the tables of the last slice (tokens 512..699) are those of that slice alone
    tail = dict(inp, x=inp["x"][512:])
    check_routing(last, oracle_routing(dataclasses.replace(w, T=188), tail), "last slice")
    with pytest.raises(moe.MoeError):
        moe.moe_set_chunk_tokens(small.ctx, 257)  # above max_tokens
    small.close()
    full = make_layer(w)
    y_full = full.forward(d["x"], *args).clone()
    torch.cuda.synchronize()
    assert full.status() == moe.MOE_OK
    full.close()
    assert torch.equal(y_chunked, y_full)
    toks = np.arange(w.T)
    check_y(y_host(y_chunked)[toks], oracle_y(w, inp, toks), "chunked prefill")


@pytest.mark.parametrize("T,path", [(1, moe.MOE_PATH_AUTO), (4, moe.MOE_PATH_GEMV), (200, moe.MOE_PATH_AUTO),
                                    (8, moe.MOE_PATH_GEMM)])
def test_router_bias_for_selection_only(T, path):
    # bias_select_only: the Zipf-like bias picks the experts, the weights are
    # the softmax of the unbiased logits over the picks (fused decode kernel at
    # T = 1 and 4, grouped GEMMs at T = 200 and T = 8 forced)
    w = custom(f"biassel{T}", T=T, skewed=True)
    inp = layer_inputs(w)
    layer = make_layer(w, path=path, bias_select_only=True)
    got, y, fwd = gpu_run(w, inp, layer, with_forward_tables=True)
    layer.close()
    ref = oracle_routing(w, inp, bias_select_only=True)
    check_routing(got, ref)
    check_routing(fwd, ref, "moe_forward")
    toks = np.arange(w.T)
    check_y(y_host(y)[toks], oracle_y(w, inp, toks, bias_select_only=True), f"bias for selection only, T={T}")
    # the plain reading differs on these inputs: the bias also scales the weights there
    ref_plain = oracle_routing(w, inp)
    assert not np.allclose(got["w"], ref_plain["w"], rtol=1e-3)


@pytest.mark.parametrize("T,path,x_dtype", [(1, moe.MOE_PATH_AUTO, "bf16"), (4, moe.MOE_PATH_GEMV, "bf16"),
                                            (24, moe.MOE_PATH_GEMV, "bf16"), (200, moe.MOE_PATH_AUTO, "bf16"),
                                            (8, moe.MOE_PATH_GEMM, "bf16"), (3, moe.MOE_PATH_AUTO, "f32"),
                                            (40, moe.MOE_PATH_GEMM, "f32")])
def test_sigmoid_gated_shared_expert(T, path, x_dtype):
    # shared_gate: router row E is a gate vector g and the shared expert's
    # output is scaled by sigmoid(x_t . g); the fused decode kernel at T = 1,
    # 3 and 4, the GEMV kernels at T = 24, the grouped GEMMs at T = 200, 8, 40
    w = custom(f"sgate{T}{x_dtype}", T=T, x_dtype=x_dtype)
    inp = layer_inputs(w)
    g = mw.draw_shared_gate(w)
    d = device_inputs(w, inp)
    d["router_w"] = torch.cat([d["router_w"], torch.from_numpy(g)[None].to(d["router_w"].device)]).contiguous()
    layer = make_layer(w, path=path, shared_gate=True)
    got, y, fwd = gpu_run(w, inp, layer, dev_in=d, with_forward_tables=True)
    layer.close()
    ref = oracle_routing(w, inp)
    check_routing(got, ref)
    check_routing(fwd, ref, "moe_forward")
    toks = np.arange(w.T)
    got_y = y_host(y)[toks]
    check_y(got_y, oracle_y(w, inp, toks, shared_gate_w=g), f"sigmoid-gated shared expert, T={T}")
    # the gate matters on these inputs: the ungated layer is outside the tolerance
    plain = oracle_y(w, inp, toks)
    assert np.linalg.norm(got_y - plain) / np.linalg.norm(plain) > 10 * 1e-2


def test_shared_gate_needs_a_shared_expert():
    with pytest.raises(moe.MoeError):
        moe.MoeLayer(512, 64, 256, 4, 16, has_shared=False, shared_gate=True)


@pytest.mark.parametrize("T", [2, 3, 4, 5, 7, 8, 9, 10, 11])
def test_fused_kernel_each_token_bound(T):
    # the fused kernel is instantiated for token bounds 1, 2, 4, 8 and 16; run
    # each bound at the decode shapes (d = 2048, 256 experts, inter 512,
    # top-8 + shared), at and between the bounds; the largest T here go to the
    # modular GEMV kernels (the fused kernel needs a weight ring of at least 6
    # slots beside its activations in shared memory; T = 11 is the GEMV
    # kernels' limit at these shapes)
    full_case(mw.Workload(f"fused_T{T}", T=T, cid=91), path=moe.MOE_PATH_GEMV)


def test_fused_kernel_sixteen_tokens():
    full_case(custom("fused_T16", T=16), path=moe.MOE_PATH_GEMV)


def test_fused_kernel_rejects_tokens_beyond_shared_memory():
    # T = 12 at the decode shapes: neither the fused kernel nor the GEMV
    # kernels (up to T = 11) hold its activations in shared memory; the forced
    # small-T path says so
    w = mw.Workload("fused_T12", T=12, cid=91)
    layer = make_layer(w, path=moe.MOE_PATH_GEMV)
    d = device_inputs(w, layer_inputs(w))
    with pytest.raises(moe.MoeError) as e:
        layer.forward(d["x"], d["router_w"], d["router_b"], d["gate_up"], d["down"], d["shared"])
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
    layer.close()


@pytest.mark.parametrize("T,path,router", [(1, moe.MOE_PATH_GEMV, moe.MOE_ROUTER_AUTO),
                                           (3, moe.MOE_PATH_GEMV, moe.MOE_ROUTER_AUTO),
                                           (64, moe.MOE_PATH_GEMM, moe.MOE_ROUTER_AUTO),
                                           (200, moe.MOE_PATH_GEMM, moe.MOE_ROUTER_TENSOR),
                                           (200, moe.MOE_PATH_GEMM, moe.MOE_ROUTER_SIMT)])
def test_exact_ties_go_to_the_lower_expert(T, path, router):
    # Router rows repeat with period 4 (expert e gets row e mod 4), so a
    # token's 256 logits take 4 values, each shared by 64 experts: the top-8
    # boundary always falls inside an exact tie, which the selection must break
    # toward the lower expert ids as the oracle does.  (The one-reduction-per-
    # pick rounds cannot decide such a boundary; the exact rounds must run.)
    w = custom(f"ties_T{T}", T=T, d=512, E=256, I=256, I_s=256, k=8, cid=97)
    inp = layer_inputs(w, 0)
    inp = dict(inp, router_w=np.ascontiguousarray(inp["router_w"][np.arange(w.E) % 4]))
    full_case(w, path=path, router=router, inp=inp)
