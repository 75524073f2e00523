"""Benchmark of the GB300 routed-expert MoE layer (one JSON line on stdout).

Metric: MoE-layer tokens per second -- tokens pushed through one MoE layer per
second, summed over the layers of a step and over all ranks.

Workloads (``--workload``, default ``decode``):
  decode            T = 1 token through 10 stacked, distinct MoE layers per step
                    (d = 2048, 256 experts of inner size 512, top-8 + shared),
                    each layer with its own token; 10 x ~59 MB of weights per
                    step, far larger than L2, so no flush is needed.
  prefill_balanced  T = 4096 tokens through one layer (1.6 GB of weights > L2).
  prefill_skewed    same with the Zipf-like router bias.
  sweep_T<n>        one layer at T = n.

The default run (decode) prints the decode figures as the line's ``value`` and
adds the metric's other half as two nested objects, ``prefill_balanced`` and
``prefill_skewed``, each measured the same way (its own value, roofline with
both the HBM and the tensor fraction, e2e, cpu_baseline and clocks);
``--no-prefill`` leaves them out.  Every roofline gives its fraction of the
measured peak (``frac``) and of the nominal one (``frac_of_nominal``).

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA graphs
and bracketed by a barrier and a device synchronisation on both sides, CUDA
events on the launching stream, max over ranks.  The dominant kernel of the
path is bracketed by its own CUDA events inside the replayed graph (through the
library's profiling hook), which gives its average launch duration for the
roofline.  ``e2e`` repeats the measurement with each step's x (every layer's
tokens, one pinned block) copied in from host memory and y copied back out, one
copy each way per step, inside the timed region.  As a serving loop would, it
overlaps the copies with the layers of the neighbouring steps: device x and y
are double-buffered, step s + 1's upload and step s - 1's download run on two
copy streams while step s computes, ordered by events on the buffer each step
reuses.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (data
parallel replicas, no collective on the data path); ``value`` counts the
tokens of all ranks over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the only reference there is) on
a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_workloads as mw  # noqa: E402

METRIC = "MoE-layer tokens/s (decode T=1, prefill T=4096) on 1 GB300; % HBM / bf16 roofline"
UNIT = "tokens/s"
L2_BYTES = 126 * 1024 * 1024  # GB300 L2 (cudaDeviceProp.l2CacheSize)
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "expert_routed_ffn_moe_gb300", "csrc")
# sources that decide each dominant kernel's code (its traffic record is void once they change)
KERNEL_SOURCES = {
    "decode_fused_kernel": ["moe_decode_kernel.cuh", "moe_decode.cu", "moe_decode_k1.cu", "moe_decode_q4_k1.cu",
                            "moe_common.cuh", "moe_internal.h"],
    "grouped_gemm_kernel<gate_up>": ["moe_gemm.cu", "moe_common.cuh", "moe_internal.h"],
    # the other kernels of a layer (their records in profiles/ are evidence only; no line reads them)
    "grouped_gemm_kernel<down>": ["moe_gemm.cu", "moe_common.cuh", "moe_internal.h"],
    "grouped_gemm_kernel<router>": ["moe_gemm.cu", "moe_common.cuh", "moe_internal.h"],
    "router_split_kernel": ["moe_route.cu", "moe_common.cuh", "moe_internal.h"],
    "select_kernel": ["moe_route.cu", "moe_common.cuh", "moe_internal.h"],
    "group_scan_kernel": ["moe_route.cu", "moe_common.cuh", "moe_internal.h"],
    "group_scatter_rows_kernel": ["moe_route.cu", "moe_common.cuh", "moe_internal.h"],
    "combine_kernel": ["moe_combine.cu", "moe_common.cuh", "moe_internal.h"],
}


def _code_only(text: str) -> str:
    """C/C++ source with comments and blank space removed: comment edits do not
    change the kernel, so they must not void a traffic record."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from the ncu
    summaries under profiles/, if one was taken of the current source on that
    workload; else None."""
    want = kernel_source_hash(kernel)
    for path in sorted(glob.glob(os.path.join(HERE, "profiles", "*.md"))):
        with open(path) as fh:
            for line in fh:
                m = re.match(r"traffic-record: kernel=(\S+) workload=(\S+) source_sha256=(\w+) bytes_per_launch=(\d+)",
                             line.strip())
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == want:
                    return int(m.group(4))
    return None
GRAPH_STEPS = 50  # steps per captured graph; longer runs replay it
EVENT_EVERY = 5   # steps between two event-timed launches of the dominant kernel


# Nominal GB300 figures, reported beside the measured ones: HBM3e ~8 TB/s and
# 2.25 PFLOP/s dense bf16 on the tensor cores.
NOMINAL = dict(hbm_gbs=8000.0, bf16_tflops=2250.0)


def with_nominal(roof):
    """Add the fractions of the nominal peaks to a roofline object (its own
    ``frac`` stays against the measured peak)."""
    if roof.get("unit") == "GB/s":
        roof["frac_of_nominal"] = round(roof["achieved"] / NOMINAL["hbm_gbs"], 4)
        roof["nominal_peak"] = NOMINAL["hbm_gbs"]
    else:
        roof["frac_of_nominal"] = round(roof["achieved"] / NOMINAL["bf16_tflops"], 4)
        roof["nominal_peak"] = NOMINAL["bf16_tflops"]
    if "hbm_frac" in roof:
        roof["hbm_frac_of_nominal"] = round(roof["hbm_frac"] * roof.get("_hbm_peak", 0) / NOMINAL["hbm_gbs"], 4)
        roof["tensor_frac_of_nominal"] = round(roof["tensor_frac"] * roof.get("_tc_peak", 0) / NOMINAL["bf16_tflops"],
                                               4)
        roof.pop("_hbm_peak", None)
        roof.pop("_tc_peak", None)
    return roof


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm_gbs=j["hbm_gbs"], bf16_tflops=j["bf16_tflops"],
                    bf16_tflops_sustained=j.get("bf16_tflops_sustained", j["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), util=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
        busy = [r for r in rows if r["util"] > 0] or rows
        reasons = sorted({name for r in busy for name, key in
                          (("hw_slowdown", "hw"), ("hw_thermal_slowdown", "hwt"), ("sw_thermal_slowdown", "swt"),
                           ("sw_power_cap", "pcap")) if r[key].lower() == "active"})
        return dict(sm_mhz=statistics.median(r["sm"] for r in busy), sm_max_mhz=max(r["smax"] for r in rows),
                    reasons=reasons, samples=len(busy))


# ------------------------------------------------------------------ inputs
def device_weights(w: mw.Workload, layer: int, dev, shared_gate=False, q4=False):
    """Seeded device-side weights of one layer (torch CUDA generator).  With
    ``shared_gate`` the router gets a row E: the gate vector of a sigmoid-gated
    shared expert, ~ N(0, 0.9^2 / d) like ``moe_workloads.draw_shared_gate``.
    With ``q4`` the experts are 4-bit planes (MOE_W_Q4G64) drawn like
    ``moe_workloads.draw_expert_q4``: uniform codes, per-group scale
    0.02 / sqrt(21.25) (1 + 0.1 N(0, 1)) and bias -7.5 scale."""
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 1000 + layer)

    def q4_planes(n_mats, rows, cols):
        # every row: codes (cols / 8 u32), then scales and biases (cols / 64 bf16 each)
        codes = torch.randint(-2 ** 31, 2 ** 31 - 1, (n_mats * rows, cols // 8), generator=g, device=dev,
                              dtype=torch.int64).to(torch.int32)
        s = (0.02 / 21.25 ** 0.5) * (1 + 0.1 * torch.randn(n_mats * rows, cols // 64, generator=g, device=dev))
        params = torch.cat([s, -7.5 * s], dim=1).to(torch.bfloat16)
        return torch.cat([codes.view(torch.uint8), params.view(torch.uint8)], dim=1).reshape(-1)

    def normal(*shape):
        out = torch.empty(*shape, dtype=torch.bfloat16, device=dev)
        flat = out.view(-1)
        step = 1 << 26
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            flat[i:i + n] = (torch.randn(n, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        return out

    router_w = torch.randn(w.E, w.d, generator=g, device=dev) * 0.02
    if shared_gate:
        gate = torch.randn(1, w.d, generator=g, device=dev) * (0.9 / w.d ** 0.5)
        router_w = torch.cat([router_w, gate])
    router_b = None
    if w.skewed:
        router_b = torch.tensor(mw.draw_router(w, layer)[1], device=dev)
    if q4:
        shared = (torch.cat([q4_planes(1, 2 * w.I_s, w.d), q4_planes(1, w.d, w.I_s)]) if w.I_s else None)
        return dict(router_w=router_w.contiguous(), router_b=router_b, gate_up=q4_planes(w.E, 2 * w.I, w.d),
                    down=q4_planes(w.E, w.d, w.I), shared=shared)
    return dict(router_w=router_w.contiguous(), router_b=router_b, gate_up=normal(w.E, 2 * w.I, w.d),
                down=normal(w.E, w.d, w.I), shared=normal(3 * w.I_s * w.d) if w.I_s else None)


def host_x(w: mw.Workload, layer: int):
    import torch

    x = mw.draw_x(w, layer)
    if w.x_dtype == "f32":
        return torch.from_numpy(x)
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------------ algorithmic bytes / flops
def expert_matrix_bytes(rows: int, cols: int, q4: bool) -> int:
    """Stored bytes of one expert weight matrix: bf16, or 4-bit codes (half a
    byte per weight) plus a bf16 scale and bias per 64 weights."""
    return rows * cols // 2 + rows * (cols // 64) * 4 if q4 else rows * cols * 2


def layer_costs(w: mw.Workload, idx: np.ndarray, shared_gate=False, q4=False):
    """Bytes and flops a layer must move/compute, from its actual routing
    (with ``shared_gate``, the router's extra gate row as well; with ``q4``,
    4-bit expert weights)."""
    distinct = len(np.unique(idx)) + (1 if w.I_s else 0)
    gate_up_w = expert_matrix_bytes(2 * w.I, w.d, q4)
    expert_bytes = gate_up_w + expert_matrix_bytes(w.d, w.I, q4)
    xb = 2 if w.x_dtype == "bf16" else 4
    rows = w.T * (w.k + (1 if w.I_s else 0))
    return dict(
        distinct=distinct,
        gate_up_bytes=distinct * gate_up_w + w.T * w.d * xb,
        layer_bytes=distinct * expert_bytes + (w.E + int(shared_gate)) * w.d * 4 + 2 * w.T * w.d * xb,
        gate_up_flops=2.0 * rows * w.d * 2 * w.I,
        layer_flops=2.0 * rows * 3 * w.d * w.I,
    )


def dominant_kernel(path: int):
    """The kernel whose roofline the bench line reports: for the small-T path
    the fused decode kernel is the whole layer; for the grouped-GEMM path the
    gate/up GEMM moves two thirds of the expert bytes."""
    import expert_routed_ffn_moe_gb300 as moe

    return moe.MOE_K_DECODE_FUSED if path == moe.MOE_PATH_GEMV else moe.MOE_K_GEMM_GATE_UP


# ------------------------------------------------------------------ oracle leg
def oracle_sample(w: mw.Workload, budget_s: float, host_inputs):
    """Time the fp64 oracle on a bounded sample of tokens; returns (tokens/s, tokens, seconds, threads).

    Each host input holds the tokens to evaluate and exactly the experts the
    oracle's own routing of those tokens selects (see ``host_layer_for_oracle``)."""
    import oracle

    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    done, t0 = 0, time.perf_counter()
    while True:
        for inp in host_inputs:
            gu, dn, sh, f64 = inp["gate_up"], inp["down"], inp["shared"], False
            if inp.get("q4_gate_up") is not None:  # 4-bit experts: the oracle expands them (step of its definition)
                gu, dn, f64 = oracle.dequant_affine4(*inp["q4_gate_up"]), oracle.dequant_affine4(*inp["q4_down"]), True
                if inp["q4_shared"] is not None:
                    sh = tuple(oracle.dequant_affine4(*m)[0] for m in inp["q4_shared"])
            oracle.moe_layer(inp["x"], inp["router_w"], inp["router_b"], gu, dn, sh,
                             w.k, x_bf16=w.x_dtype == "bf16", tokens=inp["tokens"], expert_ids=inp["expert_ids"],
                             shared_gate_w=inp.get("shared_gate_w"), weights_f64=f64)
            done += len(inp["tokens"])
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done / el, done, el, threads


def unpack_q4_planes(buf: np.ndarray, n: int, rows: int, cols: int):
    """The MOE_W_Q4G64 rows of n stacked [rows, cols] matrices in a byte buffer
    -> (words [n, rows, cols / 8] u32, scales, biases [n, rows, cols / 64] bf16 bits)."""
    r = buf[:n * rows * cols // 16 * 9].reshape(n, rows, cols // 16 * 9)
    words = np.ascontiguousarray(r[..., :cols // 2]).view(np.uint32)
    params = np.ascontiguousarray(r[..., cols // 2:]).view(np.uint16)
    return words, params[..., :cols // 64], params[..., cols // 64:]


def host_layer_for_oracle(w, layer, dev_w, x_host, n_tokens=8, seed=0, q4=False):
    """Host copies of what the oracle needs for a sample of one layer's tokens:
    x, the router, the experts the oracle routes those tokens to, the shared expert
    (with ``q4``: their 4-bit planes, which the timed oracle expands itself)."""
    import torch

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    x = x_host.numpy() if w.x_dtype == "f32" else bits(x_host)
    wr_all = dev_w["router_w"].cpu().numpy()
    wr, gate = wr_all[:w.E], (wr_all[w.E] if wr_all.shape[0] > w.E else None)
    rb = None if dev_w["router_b"] is None else dev_w["router_b"].cpu().numpy()
    rng = np.random.default_rng(seed + layer)
    toks = np.sort(rng.choice(w.T, min(w.T, n_tokens), replace=False))
    logits = oracle.router_logits(oracle.as_f64(x, w.x_dtype == "bf16")[toks], wr.astype(np.float64), rb)
    used = np.unique(oracle.route(logits, w.k)[0])
    if q4:
        gu = unpack_q4_planes(dev_w["gate_up"].cpu().numpy(), w.E, 2 * w.I, w.d)
        dn = unpack_q4_planes(dev_w["down"].cpu().numpy(), w.E, w.d, w.I)
        sh = None
        if dev_w["shared"] is not None:
            b = dev_w["shared"].cpu().numpy()
            n_gu = 2 * w.I_s * (w.d // 16 * 9)
            sh = (unpack_q4_planes(b[:n_gu], 1, 2 * w.I_s, w.d), unpack_q4_planes(b[n_gu:], 1, w.d, w.I_s))
        return dict(x=x, router_w=wr, router_b=rb, q4_gate_up=tuple(a[used] for a in gu),
                    q4_down=tuple(a[used] for a in dn), q4_shared=sh, gate_up=None, down=None, shared=None,
                    expert_ids=used, tokens=toks, shared_gate_w=gate)
    return dict(x=x, router_w=wr, router_b=rb, gate_up=bits(dev_w["gate_up"][torch.from_numpy(used).to(
        dev_w["gate_up"].device)]), down=bits(dev_w["down"][torch.from_numpy(used).to(dev_w["down"].device)]),
        shared=None if dev_w["shared"] is None else bits(dev_w["shared"]), expert_ids=used, tokens=toks,
        shared_gate_w=gate)


# ------------------------------------------------------------------ multi-rank bookkeeping
def aggregate(ms, ms_e2e, steps, tokens_per_step, world, dev):
    """Whole-job throughput: every rank ran `steps` steps of `tokens_per_step`
    tokens; the job took as long as its slowest rank (all-reduce MAX).

    Returns (tokens/s over all ranks, ms per step of the slowest rank, e2e tokens/s)."""
    if world > 1:
        import torch

        t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, ms_e2e = t.tolist()
    ms_step = ms / steps
    value = tokens_per_step * world / (ms_step / 1e3)
    e2e_value = tokens_per_step * world / (ms_e2e / steps / 1e3)
    return value, ms_step, e2e_value


def replica_layer(layer: int, rank: int) -> int:
    """Seed index of a rank's inputs: every replica draws its own tokens."""
    return layer + 1000 * rank


# ------------------------------------------------------------------ main arm
def run_ours(args, rank, world, dev, workload=None, cpu_seconds=None, chunk=None):
    """One workload (default: ``args.workload``) timed through the library;
    returns its JSON object on rank 0 (None elsewhere)."""
    import torch

    import expert_routed_ffn_moe_gb300 as moe

    moe.build()
    main_run = workload is None
    w = mw.WORKLOADS[workload or args.workload]
    layers = (args.layers if main_run else 0) or w.layers
    chunk = args.chunk if chunk is None else chunk
    cpu_seconds = args.cpu_seconds if cpu_seconds is None else cpu_seconds
    peaks = load_peaks()
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)

    q4 = args.weights == "q4"
    weights = [device_weights(w, L, dev, args.shared_gate, q4) for L in range(layers)]
    # one pinned host block and one device block for all layers' tokens, so an
    # end-to-end step moves its inputs and results in one copy each way
    xh_all = torch.stack([host_x(w, replica_layer(L, rank)) for L in range(layers)]).pin_memory()
    xd_all = xh_all.to(dev)
    yd_all = torch.empty_like(xd_all)
    yh_all = torch.empty_like(xh_all).pin_memory()
    xh, xd, yd, yh = list(xh_all), list(xd_all), list(yd_all), list(yh_all)
    # end-to-end steps: two device buffers for x and for y, and the copy streams
    xd2, yd2 = [xd_all, torch.empty_like(xd_all)], [yd_all, torch.empty_like(yd_all)]
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in, ev_done, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    max_tokens = chunk if chunk else w.T
    ctx = moe.MoeLayer(w.d, w.E, w.I, w.k, max_tokens, x_dtype=moe.MOE_F32 if w.x_dtype == "f32" else moe.MOE_BF16,
                       has_router_bias=w.skewed, has_shared=w.I_s > 0, shared_gate=args.shared_gate,
                       weight_format=moe.MOE_W_Q4G64 if q4 else moe.MOE_W_BF16)
    if chunk:  # chunked prefill: workspace for `chunk` tokens, the layer over all T in slices
        moe.moe_set_chunk_tokens(ctx.ctx, chunk)
    path = moe.MOE_PATH_AUTO if args.path == "auto" else (moe.MOE_PATH_GEMV if args.path == "gemv"
                                                          else moe.MOE_PATH_GEMM)
    moe.moe_set_path(ctx.ctx, path)
    eff_path = path if path != moe.MOE_PATH_AUTO else (moe.MOE_PATH_GEMV if w.T <= 7 else moe.MOE_PATH_GEMM)  # the library's rule
    dom = dominant_kernel(eff_path)

    whole_layer = eff_path == moe.MOE_PATH_GEMV  # the dominant kernel is the whole layer
    # the configuration a traffic record must have been taken on (per-launch traffic
    # does not depend on the number of stacked layers)
    traffic_key = (w.name + ("+shared_gate" if args.shared_gate else "") + (f"+chunk{chunk}" if chunk else "")
                   + ("+q4" if q4 else ""))
    if layers > 1:
        # stacked layers with fixed weights: a layer's blocks may start on its
        # weights while the previous layer's kernel finishes (moe_set_overlap)
        moe.moe_set_overlap(ctx.ctx, True)

    def step(ev_pair=None, e2e=False, s=0):
        if ev_pair is not None and whole_layer:
            # every launch of the step is the dominant kernel: bracket the
            # step's back-to-back launches with one event pair
            moe.moe_record_event(ev_pair[0], stream)
        xs, ys = xd, yd
        if e2e:
            # upload into buffer b once step s - 2's layers are done reading it
            # (step 0 joins the copy stream behind the stream's earlier work)
            b = s & 1
            if s == 0:
                cs_in.wait_stream(stream)
            elif s >= 2:
                cs_in.wait_event(ev_done[b])
            with torch.cuda.stream(cs_in):
                xd2[b].copy_(xh_all, non_blocking=True)
            ev_in[b].record(cs_in)
            stream.wait_event(ev_in[b])
            if s >= 2:
                stream.wait_event(ev_out[b])  # step s - 2's download of y buffer b is done
            xs, ys = list(xd2[b]), list(yd2[b])
        for L in range(layers):
            if ev_pair is not None and L == 0 and not whole_layer:
                moe.moe_time_kernel(ctx.ctx, dom, *ev_pair)
            p = weights[L]
            if layers > 1:  # stacked layers: name the next layer's first reads as a prefetch hint
                q = weights[(L + 1) % layers]
                moe.moe_set_prefetch(ctx.ctx, q["router_w"], q["shared"])
            moe.moe_forward(ctx.ctx, xs[L], p["router_w"], p["router_b"], p["gate_up"], p["down"], p["shared"], w.k,
                            ys[L], stream, packed_weights=q4)
        if e2e:
            ev_done[b].record(stream)
            cs_out.wait_event(ev_done[b])
            with torch.cuda.stream(cs_out):
                yh_all.copy_(yd2[b], non_blocking=True)
            ev_out[b].record(cs_out)
        if ev_pair is not None and whole_layer:
            moe.moe_record_event(ev_pair[1], stream)

    # routing of every layer (for the algorithmic byte counts) and warm-up
    costs = []
    with torch.cuda.stream(stream):
        for L in range(layers):
            p = weights[L]
            step_t = chunk or w.T  # moe_route keeps the T <= max_tokens limit: route slice by slice
            idx = [ctx.route(xd[L][t0:t0 + step_t], p["router_w"], p["router_b"], stream=stream)["idx"].cpu().numpy()
                   for t0 in range(0, w.T, step_t)]
            costs.append(layer_costs(w, np.concatenate(idx), args.shared_gate, q4))
        for _ in range(max(args.warmup, 0)):
            step()
    stream.synchronize()
    st = ctx.status()
    if st != moe.MOE_OK:
        raise RuntimeError("device status after warm-up: " + moe.moe_strerror(st))

    def make_events(n):
        evs = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            b.record(stream)
            evs.append((a, b))
        return evs

    def capture(n_steps, e2e, with_events):
        # The dominant kernel is bracketed by events on layer 0 of every
        # EVENT_EVERY-th step only: an event-record node costs a few
        # microseconds of serialisation, which must not inflate the step time.
        g = torch.cuda.CUDAGraph()
        sampled = [s for s in range(n_steps) if s % EVENT_EVERY == 0] if with_events else []
        evs = make_events(len(sampled))
        stream.synchronize()
        before = moe.moe_launch_count(ctx.ctx)
        with torch.cuda.graph(g, stream=stream):
            for s in range(n_steps):
                step(evs[sampled.index(s)] if s in sampled else None, e2e, s)
            if e2e:  # join the copy streams: the graph ends when the last download has landed
                stream.wait_stream(cs_in)
                stream.wait_stream(cs_out)
        launches = moe.moe_launch_count(ctx.ctx) - before
        return g, evs, launches

    def timed(n_steps, e2e):
        gsteps = min(n_steps, GRAPH_STEPS)
        g, evs, launches_per_graph = capture(gsteps, e2e, with_events=not e2e)
        reps, rem = divmod(n_steps, gsteps)
        g_rem = capture(rem, e2e, with_events=False)[0] if rem else None
        with torch.cuda.stream(stream):
            g.replay()  # untimed: uploads the graph
            if g_rem:
                g_rem.replay()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(reps):
                g.replay()
            if g_rem:
                g_rem.replay()
            stop.record(stream)
        stop.synchronize()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        ms = start.elapsed_time(stop)
        kern = [a.elapsed_time(b) / (layers if whole_layer else 1) for a, b in evs] if evs else []
        total_launches = launches_per_graph * reps + (launches_per_graph // gsteps) * rem
        return ms, kern, total_launches

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    ms, kern_ms, launches = timed(args.steps, e2e=False)
    clk = clocks.stop()
    ms_e2e, _, _ = timed(args.steps, e2e=True)
    # the downloaded y of the last end-to-end step must be the device run's y, bit for bit
    torch.cuda.synchronize(dev)
    if not all(torch.equal(yh_all, yd2[b].cpu()) for b in range(min(2, args.steps))):
        raise RuntimeError("end-to-end steps returned a y that differs from the device-resident run")
    st = ctx.status()
    if st != moe.MOE_OK:
        raise RuntimeError("device status after timing: " + moe.moe_strerror(st))

    tokens_step = w.T * layers
    value, ms_step, e2e_value = aggregate(ms, ms_e2e, args.steps, tokens_step, world, dev)

    # roofline of the dominant kernel: algorithmic bytes (or flops) per launch / mean launch time
    kern_avg_ms = statistics.mean(kern_ms) if kern_ms else None
    if eff_path == moe.MOE_PATH_GEMV:
        per_launch = statistics.mean(c["layer_bytes"] for c in costs)
        achieved = per_launch / (kern_avg_ms / 1e3) / 1e9
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(achieved / peaks["hbm_gbs"], 4), traffic=profiled_traffic("decode_fused_kernel", traffic_key),
                    kernel="decode_fused_kernel (whole layer)", algorithmic_bytes_per_launch=int(per_launch),
                    avg_launch_us=round(kern_avg_ms * 1e3, 2), peak_source=peaks["source"])
    else:
        per_launch_b = statistics.mean(c["gate_up_bytes"] for c in costs)
        per_launch_f = statistics.mean(c["gate_up_flops"] for c in costs)
        gbs = per_launch_b / (kern_avg_ms / 1e3) / 1e9
        tfs = per_launch_f / (kern_avg_ms / 1e3) / 1e12
        hbm_frac, tc_frac = gbs / peaks["hbm_gbs"], tfs / peaks["bf16_tflops"]
        if hbm_frac >= tc_frac:
            roof = dict(bound="hbm", achieved=round(gbs, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                        frac=round(hbm_frac, 4), traffic=None)
        else:
            roof = dict(bound="tensor", achieved=round(tfs, 1), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                        frac=round(tc_frac, 4), traffic=None)
        roof["traffic"] = profiled_traffic("grouped_gemm_kernel<gate_up>", traffic_key)
        roof.update(kernel="grouped_gemm_kernel<gate_up>", algorithmic_bytes_per_launch=int(per_launch_b),
                    algorithmic_flops_per_launch=int(per_launch_f), avg_launch_us=round(kern_avg_ms * 1e3, 2),
                    tensor_frac=round(tc_frac, 4), hbm_frac=round(hbm_frac, 4), peak_source=peaks["source"],
                    _hbm_peak=peaks["hbm_gbs"], _tc_peak=peaks["bf16_tflops"])
    layer_bytes = statistics.mean(c["layer_bytes"] for c in costs)
    layer_flops = statistics.mean(c["layer_flops"] for c in costs)
    ms_layer = ms_step / layers
    if chunk and chunk < w.T:
        # chunked: the event hook times one slice's launch, not the layer's; report the
        # whole layer against the layer's minimum bytes (weights read once), which the
        # chunked run exceeds by design (the selected experts are read once per slice)
        gbs = layer_bytes / (ms_layer / 1e3) / 1e9
        roof = dict(bound="hbm", achieved=round(gbs, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(gbs / peaks["hbm_gbs"], 4), traffic=None, kernel="whole layer, chunked",
                    algorithmic_bytes_per_launch=int(layer_bytes), peak_source=peaks["source"])
    roof = with_nominal(roof)
    whole = dict(ms_per_layer=round(ms_layer, 5),
                 hbm_frac_of_layer=round(layer_bytes / (ms_layer / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                 tensor_frac_of_layer=round(layer_flops / (ms_layer / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                 hbm_frac_of_layer_nominal=round(layer_bytes / (ms_layer / 1e3) / 1e9 / NOMINAL["hbm_gbs"], 4),
                 tensor_frac_of_layer_nominal=round(layer_flops / (ms_layer / 1e3) / 1e12 / NOMINAL["bf16_tflops"],
                                                    4),
                 algorithmic_bytes_per_layer=int(layer_bytes), algorithmic_flops_per_layer=int(layer_flops),
                 distinct_experts_per_layer=round(statistics.mean(c["distinct"] for c in costs), 1))

    out = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            hosts = [host_layer_for_oracle(w, L, weights[L], xh[L], q4=q4) for L in range(layers)]
            v, n, el, thr = oracle_sample(w, cpu_seconds, hosts)
            cpu = dict(value=round(v, 3), unit=UNIT, cores=thr, kind="oracle",
                       sample=f"{n} token-layers (8 random tokens per layer, all {layers} layers, repeated) "
                              f"in {el:.1f} s; fp64 numpy, BLAS threads = {thr}")
        out = dict(metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=world, steps=args.steps,
                   warmup=args.warmup, ms_per_step=round(ms_step, 5), higher_is_better=True, scaling="weak",
                   vs_baseline=None, dtype="q4" if q4 else "bf16", data="synthetic",
                   config=dict(workload=w.name, tokens_per_layer=w.T, layers_per_step=layers, d=w.d, experts=w.E,
                               weights="q4g64 (4-bit codes, bf16 scale + bias per 64)" if q4 else "bf16",
                               inter=w.I, shared_inter=w.I_s, top_k=w.k,
                               path="gemv" if eff_path == moe.MOE_PATH_GEMV else "grouped_gemm",
                               l2=(f"inputs larger than L2 (distinct weights per layer, "
                                   f"{layer_bytes * layers / 1e6:.0f} MB touched per step)"
                                   if layer_bytes * layers > L2_BYTES else
                                   f"inputs fit in L2 ({layer_bytes * layers / 1e6:.0f} MB per step): "
                                   f"a profiling run, not a bench number"),
                               parallelism=f"replicas x{world}", **({"chunk_tokens": chunk} if chunk else {}),
                               **({"shared_gate": "sigmoid"} if args.shared_gate else {})),
                   e2e=dict(value=round(e2e_value, 1), unit=UNIT,
                            h2d_bytes_per_step=int(sum(t.numel() * t.element_size() for t in xh)),
                            d2h_bytes_per_step=int(sum(t.numel() * t.element_size() for t in yh)),
                            copies="overlapped with the neighbouring steps' layers: two copy streams, "
                                   "double-buffered device x and y"),
                   gpu_launches=int(launches), roofline=roof, layer=whole, clocks=clk, cpu_baseline=cpu)
    ctx.close()
    return out


NESTED_PREFILL = ("prefill_balanced", "prefill_skewed")


def nested(sub):
    """The per-workload part of a JSON line, for nesting inside the main line."""
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "config", "e2e", "gpu_launches", "roofline", "layer",
            "clocks", "cpu_baseline")
    return {k: sub[k] for k in keep if k in sub}


def run_reference(args):
    """The fp64 oracle on the host cores, on a bounded sample of the same workload."""
    w = mw.WORKLOADS[args.workload]
    import oracle as orc

    hosts = []
    for L in range(w.layers):
        wr, b = mw.draw_router(w, L)
        x = mw.draw_x(w, L)
        toks = np.sort(np.random.default_rng(L).choice(w.T, min(w.T, 8), replace=False))
        logits = orc.router_logits(orc.as_f64(x, w.x_dtype == "bf16")[toks], wr.astype(np.float64), b)
        used = np.unique(orc.route(logits, w.k)[0])
        gu, dn = mw.draw_experts(w, L, used)
        hosts.append(dict(x=x, router_w=wr, router_b=b, gate_up=gu, down=dn, shared=mw.draw_shared(w, L),
                          expert_ids=used, tokens=toks))
    for _ in range(max(args.warmup, 0)):
        oracle_sample(w, 0.0, hosts)
    per = []
    for _ in range(args.steps):
        v, n, el, thr = oracle_sample(w, args.ref_step_seconds, hosts)
        per.append((n, el))
    n = sum(a for a, _ in per)
    el = sum(b for _, b in per)
    value = n / el
    return dict(metric=METRIC, value=round(value, 3), unit=UNIT, n_gpus=1, steps=args.steps, warmup=args.warmup,
                ms_per_step=round(el / args.steps * 1e3, 3), higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=w.name, tokens_per_layer=w.T, layers_per_step=w.layers, d=w.d, experts=w.E,
                            inter=w.I, top_k=w.k),
                cpu_baseline=dict(value=round(value, 3), unit=UNIT, cores=thr, kind="oracle",
                                  sample=f"{n} token-layers in {el:.1f} s"),
                e2e=dict(value=round(value, 3), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(mw.WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "gemm"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk", type=int, default=0,
                    help="chunked prefill: size the workspace for this many tokens and run T in slices")
    ap.add_argument("--layers", type=int, default=0,
                    help="stacked layers per step (default: the workload's own; fewer only for small profiling runs)")
    ap.add_argument("--shared-gate", action="store_true",
                    help="the sigmoid-gated shared-expert variant (a gate row appended to the router)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "q4"],
                    help="expert weight format: bf16, or 4-bit group-affine (MOE_W_Q4G64)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode only: skip the nested prefill_balanced / prefill_skewed measurements")
    ap.add_argument("--prefill-cpu-seconds", type=float, default=6.0,
                    help="oracle time budget of each nested prefill measurement's cpu_baseline")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch

    dev = torch.device("cuda", local)
    if world > 1:
        torch.cuda.set_device(dev)
        torch.distributed.init_process_group("nccl", device_id=dev)
    out = run_ours(args, rank, world, dev)
    if args.workload == "decode" and not args.no_prefill:
        # the metric's second half: the T = 4096 prefill layer, balanced and
        # skewed routing, each measured the same way and nested in the line
        torch.cuda.empty_cache()
        for name in NESTED_PREFILL:
            sub = run_ours(args, rank, world, dev, workload=name, cpu_seconds=args.prefill_cpu_seconds, chunk=0)
            torch.cuda.empty_cache()
            if rank == 0:
                out[name] = nested(sub)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
