"""Host-side logic of bench.py that needs no GPU: the traffic record lookup
(an ncu figure is reported only for the kernel source it was taken of) and
the multi-rank aggregation."""
import os
import shutil

import pytest

import bench


def test_traffic_record_matches_only_current_source(tmp_path, monkeypatch):
    # a private copy of the sources and profiles: changing a byte of the
    # kernel source must void the recorded traffic
    root = tmp_path / "repo"
    shutil.copytree(bench.CSRC, root / "expert_routed_ffn_moe_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "HERE", str(root))
    monkeypatch.setattr(bench, "CSRC", str(root / "expert_routed_ffn_moe_gb300" / "csrc"))
    h = bench.kernel_source_hash("decode_fused_kernel")
    (root / "profiles" / "k.md").write_text(
        f"text\ntraffic-record: kernel=decode_fused_kernel workload=decode source_sha256={h} bytes_per_launch=12345\n")
    assert bench.profiled_traffic("decode_fused_kernel", "decode") == 12345
    # another workload (another token count, a variant) moves other bytes
    assert bench.profiled_traffic("decode_fused_kernel", "sweep_T2") is None
    assert bench.profiled_traffic("grouped_gemm_kernel<gate_up>", "decode") is None
    src = root / "expert_routed_ffn_moe_gb300" / "csrc" / "moe_decode_kernel.cuh"
    src.write_text(src.read_text() + "\n// a comment changes no kernel\n")
    assert bench.profiled_traffic("decode_fused_kernel", "decode") == 12345
    src.write_text(src.read_text() + "\nstatic int changed_code = 1;\n")
    assert bench.profiled_traffic("decode_fused_kernel", "decode") is None


def test_aggregate_single_rank():
    value, ms_step, e2e = bench.aggregate(ms=100.0, ms_e2e=200.0, steps=10, tokens_per_step=5, world=1, dev=None)
    assert ms_step == pytest.approx(10.0)
    assert value == pytest.approx(5 / 0.010)
    assert e2e == pytest.approx(5 / 0.020)


def test_algorithmic_bytes_and_flops_per_unit():
    import numpy as np

    import moe_workloads as mw

    expert = 3 * 2048 * 512 * 2  # gate_up [1024, 2048] + down [2048, 512], bf16
    assert expert == 6_291_456
    # decode: one token, 8 distinct routed experts + the shared one, the fp32
    # router, x and y in bf16
    c = bench.layer_costs(mw.WORKLOADS["decode"], np.arange(8)[None, :] * 3)
    assert c["distinct"] == 9
    assert c["layer_bytes"] == 9 * expert + 256 * 2048 * 4 + 2 * 2048 * 2 == 58_728_448
    assert c["layer_flops"] == 2 * 9 * 3 * 2048 * 512
    # balanced prefill: all 256 experts + shared; gate/up reads two thirds of
    # each expert plus the token rows once
    w = mw.WORKLOADS["prefill_balanced"]
    idx = (np.arange(w.T * 8).reshape(w.T, 8)) % 256
    c = bench.layer_costs(w, idx)
    assert c["gate_up_bytes"] == 257 * 2 * 512 * 2048 * 2 + 4096 * 2048 * 2 == 1_094_713_344
    assert c["gate_up_flops"] == 2 * 4096 * 9 * 2048 * 1024
    # the shared-gate variant adds its fp32 gate row to the router bytes
    c2 = bench.layer_costs(w, idx, shared_gate=True)
    assert c2["layer_bytes"] - c["layer_bytes"] == 2048 * 4


def test_q4_bytes_and_plane_roundtrip():
    import numpy as np

    import moe_workloads as mw

    # one 4-bit expert at d = 2048, I = 512: half a byte per weight + a bf16 scale and bias per 64
    q4_expert = 3 * 2048 * 512 // 2 + 3 * 2048 * 512 // 64 * 4
    assert bench.expert_matrix_bytes(1024, 2048, True) + bench.expert_matrix_bytes(2048, 512, True) == q4_expert
    c = bench.layer_costs(mw.WORKLOADS["decode"], np.arange(8)[None, :] * 3, q4=True)
    assert c["layer_bytes"] == 9 * q4_expert + 256 * 2048 * 4 + 2 * 2048 * 2
    # the bench's plane reader inverts moe_workloads.pack_q4
    w = mw.Workload("q4rt", T=1, d=512, E=3, I=256, I_s=256, k=2, cid=9)
    q = mw.draw_experts_q4(w)
    buf = mw.pack_q4(q["dn_words"], q["dn_scales"], q["dn_biases"])
    words, scales, biases = bench.unpack_q4_planes(buf, w.E, w.d, w.I)
    assert np.array_equal(words, q["dn_words"]) and np.array_equal(scales, q["dn_scales"])
    assert np.array_equal(biases, q["dn_biases"])


def test_committed_traffic_records_are_well_formed():
    # every ncu summary's record names a kernel whose sources bench.py hashes
    # and a workload it runs (variant suffixes included), and gives a byte
    # count; a record of stale sources is allowed (it just stops matching)
    import glob
    import re

    import moe_workloads as mw

    pat = re.compile(r"traffic-record: kernel=(\S+) workload=(\S+) source_sha256=([0-9a-f]{16}) bytes_per_launch=(\d+)$")
    n = 0
    for path in sorted(glob.glob(os.path.join(bench.HERE, "profiles", "*.md"))):
        for line in open(path):
            if not line.startswith("traffic-record:"):
                continue
            m = pat.match(line.strip())
            assert m, (path, line)
            kernel, workload, _, nbytes = m.groups()
            assert kernel in bench.KERNEL_SOURCES, (path, kernel)
            base = workload.split("+")[0]
            assert base in mw.WORKLOADS, (path, workload)
            assert all(v in ("q4", "shared_gate") or v.startswith("chunk") for v in workload.split("+")[1:]), workload
            assert int(nbytes) > 0
            n += 1
    assert n > 0
