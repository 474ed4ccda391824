"""Benchmark: Q4_0 MUL_MAT over a 7B-like 32-layer weight sweep on GB300.

One step = one pass of the whole hot path over the sweep:
  decode   224 MUL_MATs at N = 1 through gq_mul_mat_q4_0 (decode kernel),
           replayed as one CUDA graph;
  prefill  224 MUL_MATs at N = 512: per layer one gq_f32_to_bf16 over its four
           activations (one buffer),
           then gq_mul_mat_q4_0_bf16x (tensor-core kernel), CUDA events
           around the tensor-core launches.
Per layer: q, k, v, o 4096 x 4096, gate and up 11008 x 4096, down 4096 x 11008
("Binding GGUF weights to the compute graph", section 2.4), 3.64 GB of Q4_0
weights in total, all resident in HBM and larger than L2, so every pass
streams them from DRAM.  Weights and activations are seeded synthetic data
(synth.py).

Prints ONE JSON line.  `value` is decode weight throughput (weight bytes of the
sweep / decode time); prefill TFLOP/s, the roofline of the dominant kernel
(tensor-core prefill), the decode roofline, the end-to-end number through
host buffers, clocks and the CPU-oracle baseline are extra keys.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gq|reference]
Under torchrun (N > 1) every rank runs its own replica of the sweep (weak
scaling); rank 0 prints.  `--impl reference` times the CPU oracle on the host
cores for the same metric (bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4_0 mul_mat weight GB/s (decode N=1) and TFLOP/s (prefill N=512) vs roofline"
DECODE_N, PREFILL_N = 1, 512
WORKLOAD = ("7B-like 32-layer Q4_0 weight sweep: per layer q/k/v/o 4096x4096, gate/up 11008x4096, "
            "down 4096x11008 (3.64 GB of weights); decode N=1 then prefill N=512")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def layer_inputs():
    """Per layer: which activation feeds which matrix (q/k/v share one input, gate/up another)."""
    # input ids: 0 attn input (K=4096), 1 attn-output input (4096), 2 ffn input (4096), 3 down input (11008)
    return [0, 0, 0, 1, 2, 2, 3], [4096, 4096, 4096, 11008]


def make_weights(n_layers, rank):
    host = []
    for layer in range(n_layers):
        for j, (_, M, K) in enumerate(synth.LAYER_MATRICES):
            seed = synth.seed_for(5, j, layer) + 7919 * rank
            host.append((M, K, synth.q4_0_weights(M, K, seed)))
    return host


def make_acts(n_layers, N, rank, tag):
    _, ks = layer_inputs()
    return [[synth.activations(N, K, synth.seed_for(5, 8 + i, layer) + 104729 * rank + tag)
             for i, K in enumerate(ks)] for layer in range(n_layers)]


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of a list of floats over all ranks (the slowest rank
    sets the time); the identity when there is no process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.rows, self.proc, self.dev = [], None, device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "", 1).isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------------------ CPU oracle leg
def oracle_decode_rate(weights, acts, budget_s, nthreads, max_passes=64, gpu_out=None, check=None):
    """Oracle MUL_MAT at N=1 over the sweep's matrices, pass after pass, until
    budget_s elapses (at least one matrix, at most max_passes passes).
    Returns (weight GB/s, matrices done, weight bytes done, seconds).  With
    gpu_out (matrix index -> the GPU's y of that matrix) the first pass also
    compares each result it computes with the GPU's, element by element, and
    records the worst tolerance ratio in check (outside the timing)."""
    import oracle
    orc = oracle.get()
    order, _ = layer_inputs()
    done_bytes, done, t0 = 0, 0, time.perf_counter()
    paused = 0.0
    for p in range(max_passes):
        for idx, (M, K, W) in enumerate(weights):
            layer, j = divmod(idx, len(order))
            y_ref, s_ref = orc.mul_mat(W, M, K, acts[layer][order[j]], nthreads=nthreads)
            if p == 0 and gpu_out is not None and idx in gpu_out:
                tc = time.perf_counter()
                _, worst = oracle.within_tolerance(gpu_out[idx], y_ref, s_ref)
                check["decode_worst_ratio"] = max(check.get("decode_worst_ratio", 0.0), float(worst))
                check["decode_matrices"] = check.get("decode_matrices", 0) + 1
                check["decode_outputs"] = check.get("decode_outputs", 0) + int(y_ref.size)
                paused += time.perf_counter() - tc
            done_bytes += W.nbytes
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        else:
            continue
        break
    dt = time.perf_counter() - t0 - paused
    return done_bytes / dt / 1e9, done, done_bytes, dt


def prefill_parity(weights, acts, order, pre_rows, nthreads, check):
    """The oracle on the sampled rows of the prefill outputs (all 512 tokens),
    compared element by element with the GPU's; returns the parity summary."""
    import oracle
    orc = oracle.get()
    worst, n_out = 0.0, 0
    for i, (rows, y_gpu) in pre_rows.items():
        M, K, W = weights[i]
        layer, j = divmod(i, len(order))
        y_ref, s_ref = orc.mul_mat(np.ascontiguousarray(W[rows]), len(rows), K, acts[layer][order[j]],
                                   nthreads=nthreads)
        _, w = oracle.within_tolerance(y_gpu, y_ref, s_ref)
        worst = max(worst, float(w))
        n_out += int(y_ref.size)
    check["prefill_worst_ratio"] = worst
    check["prefill_outputs"] = n_out
    d = check.get("decode_worst_ratio")
    return {"parity_worst_ratio": round(max(worst, d if d is not None else 0.0), 4),
            "tolerance": "|y - y_ref| <= 1e-3 * sum|w x| + 1e-5 (ratio < 1 passes)",
            "decode": {"worst_ratio": round(d, 4) if d is not None else None,
                       "matrices": check.get("decode_matrices", 0), "outputs": check.get("decode_outputs", 0),
                       "what": "the last step's Y of every matrix the CPU leg's first pass computed"},
            "prefill": {"worst_ratio": round(worst, 4), "outputs": n_out,
                        "what": "32 sampled rows x 512 tokens of each matrix of the first and last layer"}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    nthreads = os.cpu_count() or 1
    oracle.get()
    layers = 2
    weights = make_weights(layers, 0)
    acts = make_acts(layers, DECODE_N, 0, 0)
    for _ in range(args.warmup):
        oracle_decode_rate(weights[:1], acts, 1e9, nthreads, max_passes=1)
    total_bytes, total_t, mats = 0, 0.0, 0
    for _ in range(args.steps):
        _, n, b, dt = oracle_decode_rate(weights, acts, args.ref_budget, nthreads, max_passes=1)
        total_bytes += b
        total_t += dt
        mats += n
    value = total_bytes / total_t / 1e9
    sample = (f"oracle MUL_MAT at N=1 over the first {layers} layers of the sweep "
              f"({sum(w.nbytes for _, _, w in weights) / 1e6:.0f} MB of Q4_0 weights), "
              f"{mats} matrix calls over {args.steps} steps, fp64 sums, {nthreads} OpenMP threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sampled": True},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU leg
def run_gpu(args, rank, world, dist):
    import torch
    import quantized_block_q4_gb300 as gq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # weights are uploaded once and never written by the kernels that run
    # before each MUL_MAT, so the decode kernel may stream W early
    gq.gq_set_option(gq.GQ_OPT_WEIGHTS_STATIC, 1)
    # each MUL_MAT's activations are prepared before the sweep, never written by
    # the MUL_MAT launched before it, so decode launches may read X early
    gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    order, ks = layer_inputs()
    L = args.layers

    t_gen = time.perf_counter()
    host_w = make_weights(L, rank)
    W = [torch.from_numpy(w).to(dev) for _, _, w in host_w]
    shapes = [(M, K) for M, K, _ in host_w]
    acts1 = make_acts(L, DECODE_N, rank, 0)
    actsP = make_acts(L, PREFILL_N, rank, 1)
    X1 = [[torch.from_numpy(a).to(dev) for a in la] for la in acts1]
    # each layer's four prefill activations in one buffer (fp32 and bf16), so
    # that one conversion call covers them; XP / XPb are views of it
    XPflat = [torch.from_numpy(np.concatenate([a.ravel() for a in la])).to(dev) for la in actsP]
    XPbflat = [torch.empty(x.numel(), dtype=torch.int16, device=dev) for x in XPflat]
    XP, XPb = [], []
    for layer, la in enumerate(actsP):
        off, xs, xbs = 0, [], []
        for a in la:
            xs.append(XPflat[layer][off:off + a.size].view(a.shape))
            xbs.append(XPbflat[layer][off:off + a.size].view(a.shape))
            off += a.size
        XP.append(xs)
        XPb.append(xbs)
    Y1 = [torch.empty(DECODE_N, M, device=dev) for M, _ in shapes]
    YP = [torch.empty(PREFILL_N, M, device=dev) for M, _ in shapes]
    gen_s = time.perf_counter() - t_gen
    wbytes = sum(w.numel() for w in W)
    flops_p = sum(2.0 * M * K * PREFILL_N for M, K in shapes)
    dec_alg_bytes = sum(M * K * 18 // 32 + 4 * DECODE_N * K + 4 * DECODE_N * M for M, K in shapes)

    s = torch.cuda.Stream(device=dev)

    def decode_pass():
        for i, (M, K) in enumerate(shapes):
            layer, j = divmod(i, len(order))
            gq.gq_mul_mat_q4_0(W[i], M, K, X1[layer][order[j]], DECODE_N, Y1[i], stream=s)

    # one event pair per layer around its run of tensor-core launches
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]

    def prefill_pass(record, promise=True):
        # activation conversion for each layer's inputs, then the tensor-core
        # MUL_MATs: the first without the x-static promise (its X was converted
        # right before), which orders the conversions before everything after
        # it; the other six with it (their X was written before that call)
        for layer in range(L):
            gq.gq_f32_to_bf16(XPflat[layer], XPbflat[layer], XPflat[layer].numel(), stream=s)
            if record:
                ev_pairs[layer][0].record(s)
            for j in range(len(order)):
                i = layer * len(order) + j
                M, K = shapes[i]
                gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1 if promise and j > 0 else 0)
                gq.gq_mul_mat_q4_0_bf16x(W[i], M, K, XPb[layer][order[j]], PREFILL_N, YP[i], stream=s)
            gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1)
            if record:
                ev_pairs[layer][1].record(s)

    # decode sweep as one CUDA graph (224 short launches)
    with torch.cuda.stream(s):
        decode_pass()
        prefill_pass(False)
    torch.cuda.synchronize(dev)
    gq.gq_sync_status(s)
    g_dec = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_dec, stream=s):
            decode_pass()
    torch.cuda.synchronize(dev)
    # the same sweep without the x-static promise: every launch reads its X
    # only after the kernel before it has finished (a dependent chain)
    gq.gq_set_option(gq.GQ_OPT_X_STATIC, 0)
    g_dep = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        decode_pass()
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g_dep, stream=s):
            decode_pass()
    torch.cuda.synchronize(dev)
    gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1)

    def step(record):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(s):
            e0.record(s)
            g_dec.replay()
            e1.record(s)
            prefill_pass(record)
            e2.record(s)
        return e0, e1, e2

    for _ in range(max(args.warmup, 3)):
        step(False)
    torch.cuda.synchronize(dev)
    gq.gq_sync_status(s)

    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    marks = [step(False) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall0
    if dist is not None:
        dist.barrier()
    # The same K steps again with an event pair around each layer's 7
    # back-to-back tensor-core launches, for the kernel's own time (roofline):
    # the mean launch duration is that time over the launches, with consecutive
    # launches overlapping as they do in the steps above.  The events keep the
    # conversions outside, so these steps are not the ones the throughput
    # above is taken from.
    k3_ms = 0.0
    for _ in range(args.steps):
        step(True)
        torch.cuda.synchronize(dev)  # per step, so that its K3 events can be read
        k3_ms += sum(a.elapsed_time(b) for a, b in ev_pairs)
    if dist is not None:
        dist.barrier()
    # the prefill pass with no x-static promise at all, K passes, timed alone
    with torch.cuda.stream(s):
        prefill_pass(False, promise=False)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(s)
        for _ in range(args.steps):
            prefill_pass(False, promise=False)
        p1.record(s)
    p1.synchronize()
    pre_dep_ms = p0.elapsed_time(p1)
    # the dependent decode sweep, K steps, timed alone
    with torch.cuda.stream(s):
        for _ in range(3):
            g_dep.replay()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(s)
        for _ in range(args.steps):
            g_dep.replay()
        d1.record(s)
    d1.synchronize()
    dep_ms = d0.elapsed_time(d1)
    clocks = clk.stop()
    gq.gq_sync_status(s)
    # outputs of the last step, for the parity check of the CPU leg: every
    # decode Y, and 32 sampled rows of each prefill Y of the first and last layer
    with torch.cuda.stream(s):
        g_dec.replay()
        prefill_pass(False)
    torch.cuda.synchronize(dev)
    gq.gq_sync_status(s)
    dec_out = {i: Y1[i].cpu().numpy() for i in range(len(shapes))}
    rng = np.random.default_rng(0x51A7)
    pre_rows = {}
    for i in list(range(len(order))) + list(range(len(shapes) - len(order), len(shapes))):
        M = shapes[i][0]
        rows = np.sort(rng.choice(M, size=32, replace=False))
        pre_rows[i] = (rows, YP[i][:, torch.from_numpy(rows).to(dev)].cpu().numpy())

    dec_ms = sum(a.elapsed_time(b) for a, b, _ in marks)
    pre_ms = sum(b.elapsed_time(c) for _, b, c in marks)
    step_ms = sum(a.elapsed_time(c) for a, _, c in marks)
    dec_ms, pre_ms, step_ms, k3_ms, dep_ms, pre_dep_ms = max_over_ranks(
        [dec_ms, pre_ms, step_ms, k3_ms, dep_ms, pre_dep_ms], dist, dev)

    K_ = args.steps
    value = world * wbytes * K_ / (dec_ms * 1e-3) / 1e9
    prefill_tflops = world * flops_p * K_ / (pre_ms * 1e-3) / 1e12
    k3_avg_us = k3_ms / (K_ * len(shapes)) * 1e3
    k3_tflops = flops_p * K_ / (k3_ms * 1e-3) / 1e12
    dec_avg_us = dec_ms / (K_ * len(shapes)) * 1e3
    dec_gbs_alg = dec_alg_bytes * K_ / (dec_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers (decode, N = 1)
    e2e = run_e2e(gq, torch, dev, s, W, shapes, acts1, order, L, args)
    aux = run_aux(gq, torch, dev, s, peaks["hbm_gbs"]) if rank == 0 else {}
    if rank == 0:
        aux["mul_mat_id"] = run_moe_aux(gq, torch, dev, s, peaks)
        aux["block_formats"] = run_formats_aux(gq, torch, dev, s, peaks)
        aux["prepared_layout"] = run_prepared_aux(gq, torch, dev, s, peaks)
        aux["library_reference"] = run_library_reference(gq, torch, dev, s, peaks)
    if rank == 0:
        aux["per_config"] = run_per_config(gq, torch, dev, s, peaks)
    e2e["ms"] = max_over_ranks([e2e["ms"]], dist, dev)[0]
    e2e_value = world * wbytes / (e2e["ms"] * 1e-3) / 1e9

    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        check = {}
        gbs, n, b, dt = oracle_decode_rate(host_w, acts1, args.cpu_budget, nthreads, gpu_out=dec_out, check=check)
        parity = prefill_parity(host_w, actsP, order, pre_rows, nthreads, check)
        gbs1, n1, b1, dt1 = oracle_decode_rate(host_w, acts1, args.cpu_budget / 5, 1, max_passes=1)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
               "sample": f"oracle MUL_MAT at N=1, {n} matrices taken in order from the same "
                         f"{len(host_w)}-matrix sweep, repeated ({b / 1e6:.0f} MB of weights, {dt:.1f} s), "
                         f"fp64 sums",
               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                 "sample": f"the first {n1} matrices of the sweep ({b1 / 1e6:.0f} MB, {dt1:.1f} s)"}}

    if rank != 0:
        return 0
    sust = peaks["bf16_tflops_sustained"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K_,
        "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms / K_, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 x f16 -> f32 (decode), bf16 x bf16 -> f32 (prefill)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": L, "matrices": len(shapes), "decode_n": DECODE_N,
                   "prefill_n": PREFILL_N, "weight_bytes": wbytes,
                   "l2": "inputs larger than L2 (3.64 GB of weights streamed per pass)",
                   "weights_static": True, "x_static": True,
                   "parallelism": f"replicas x{world}"},
        "decode": {"value": round(value, 2), "unit": "GB/s", "ms": round(dec_ms / K_, 4),
                   "avg_launch_us": round(dec_avg_us, 3), "frac": round(value / peaks["hbm_gbs"], 4),
                   "promises": "weights static and x static (each launch may read X and compute before the "
                               "kernel before it ends; Y is written after it)"},
        "decode_no_x_static": {"value": round(world * wbytes * K_ / (dep_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                               "ms": round(dep_ms / K_, 4),
                               "frac": round(world * wbytes * K_ / (dep_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                               "promises": "weights static only: every launch reads X after the kernel before "
                                           "it has finished, as in a chain where each input is the last output"},
        "prefill": {"value": round(prefill_tflops, 2), "unit": "TFLOP/s", "ms": round(pre_ms / K_, 4),
                    "includes": "fp32->bf16 activation conversion + tensor-core MUL_MAT",
                    "launch": "eager, programmatic dependent launch between consecutive kernels; per layer "
                              "the first MUL_MAT without the x-static promise, the other six with it"},
        "prefill_no_x_static": {"value": round(world * flops_p * K_ / (pre_dep_ms * 1e-3) / 1e12, 2),
                                "unit": "TFLOP/s", "ms": round(pre_dep_ms / K_, 4),
                                "promises": "weights static only: every MUL_MAT reads X after the kernel "
                                            "before it has finished"},
        "roofline": {"kernel": "k_prefill_q4_0 (tcgen05 prefill)", "bound": "tensor",
                     "achieved": round(k3_tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(k3_tflops / peaks["bf16_tflops"], 4), "traffic": sweep_traffic("prefill", shapes),
                     "traffic_unit": "bytes per launch (ncu, mean over the sweep's shapes)",
                     "peak_kind": f"bf16 burst ({peaks['source']}): the timed region is under a second at "
                                  f"full clock", "frac_of_sustained": round(k3_tflops / sust, 4),
                     "avg_launch_us": round(k3_avg_us, 3),
                     "per_launch": "2*M*K*512 flops of the launch's matrix",
                     "timing": "event pair around each layer's 7 back-to-back launches (conversions outside), "
                               "over K further steps of the same sweep; avg = their time / 224"},
        "roofline_decode": {"kernel": "k_decode_q4_0 (decode)", "bound": "hbm", "achieved": round(dec_gbs_alg, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(dec_gbs_alg / peaks["hbm_gbs"], 4),
                            "traffic": sweep_traffic("decode", shapes),
                            "traffic_unit": "bytes per launch (ncu, mean over the sweep's shapes)",
                            "peak_kind": f"HBM copy ({peaks['source']})",
                            "per_launch": "M*K*18/32 + 4*N*K + 4*N*M bytes; graph-replay time incl. launch gaps"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"],
                "path": "per step: the step's activations pinned host -> device in one copy, the 224 "
                        "gq_mul_mat_q4_0 calls, every Y -> pinned host in one copy (decode sweep)"},
        "dequant": aux.get("dequant"),
        "quantize": aux.get("quantize"),
        "validate": aux.get("validate"),
        "mul_mat_id": aux.get("mul_mat_id"),
        "block_formats": aux.get("block_formats"),
        "prepared_layout": aux.get("prepared_layout"),
        "library_reference": aux.get("library_reference"),
        "gpu_launches": K_ * (len(shapes) + len(shapes) + L),  # decode + tensor-core MUL_MATs + one conversion per layer
        "clocks": clocks,
        "cpu_baseline": cpu,
        "parity": parity,
        "parity_worst_ratio": parity["parity_worst_ratio"] if parity else None,
        "per_config": aux.get("per_config"),
        "wall_s": round(wall, 3), "setup_s": round(gen_s, 1),
    }
    print(json.dumps(line), flush=True)
    return 0


AUX_M, AUX_K, AUX_REPS = 14336, 4096, 10

# (name, M, K, N list): the workloads besides the sweep, each timed on its own
PER_CONFIG = [("small mat-vec", 256, 1024, [1]),
              ("7B FFN gate/up mat-vec", 11008, 4096, [1]),
              ("7B FFN down mat-vec", 4096, 11008, [1]),
              ("7B attention projection, small batches", 4096, 4096, [1, 2, 4, 8, 16]),
              ("32000-row output projection, small batches", 32000, 4096, [1, 2, 4, 8, 16]),
              ("14336-row prefill, 512 tokens", 14336, 4096, [512])]


def graph_time(torch, s, fn, reps, replays=10):
    """Median of `replays` replays of a CUDA graph of `reps` calls fn(0..reps-1), per call, seconds."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for i in range(reps):
            fn(i)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for i in range(reps):
                fn(i)
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / reps * 1e-3)
    return statistics.median(times)


def eager_time(torch, s, fn, reps, replays=10):
    """Median of `replays` runs of `reps` back-to-back eager calls fn(0..reps-1), per call, seconds."""
    times = []
    with torch.cuda.stream(s):
        for i in range(reps):
            fn(i)
    torch.cuda.synchronize()
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for i in range(reps):
                fn(i)
            e1.record(s)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / reps * 1e-3)
    return statistics.median(times)


def graph_or_eager_time(gq, torch, s, fn, reps):
    """graph_time, or eager_time where the calls cannot be captured (the
    tensor-core path takes stream-ordered scratch); returns (seconds, how)."""
    try:
        return graph_time(torch, s, fn, reps), "graph"
    except Exception as e:  # a refused capture is an API error, not a device fault
        torch.cuda.synchronize()
        gq.gq_last_error()
        return eager_time(torch, s, fn, reps), f"eager ({type(e).__name__} on capture)"


def run_per_config(gq, torch, dev, s, peaks):
    """Every workload besides the sweep, device-timed: a CUDA graph of 50 to
    200 back-to-back calls, each on its own weight copy (together more than
    4x L2, so every call streams its weights from DRAM), median of 10
    replays.  Decode shapes
    (N < 16) are timed with the x-static promise (as in the sweep) and
    without it (each call reads X only after the kernel before it ends);
    N >= 16 runs the bf16 conversion and the tensor-core kernel (the promise
    does not apply: X is converted right before); the 512-token prefill also
    the tensor-core kernel alone on bf16 activations, with the promise (the
    next call's MMAs start while the previous call finishes) and without."""
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    out = []
    old_x = gq.gq_get_option(gq.GQ_OPT_X_STATIC)
    try:
        for name, M, K, ns in PER_CONFIG:
            nb = gq.gq_q4_0_nbytes(M, K)
            # at least 50 calls per graph, on enough copies for 4x L2 (capped
            # at 200: the 256 x 1024 matrix stays L2-resident, a latency figure)
            copies = min(200, max(50, int(4 * 130e6 // nb) + 1))
            W0 = torch.from_numpy(synth.q4_0_weights(M, K, seed=0x5C00 + M + K)).to(dev)
            Ws = [W0] + [W0.clone() for _ in range(copies - 1)]
            for n in ns:
                X = torch.randn(n, K, device=dev, generator=torch.Generator(device=dev).manual_seed(n))
                Y = torch.empty(n, M, device=dev)
                alg = nb + 4 * n * K + 4 * n * M
                e = {"workload": name, "shape": f"{M}x{K}", "n": n, "calls_per_graph": copies}

                def call(i):
                    gq.gq_mul_mat_q4_0(Ws[i % copies], M, K, X, n, Y, stream=s)
                if n < gq.gq_get_option(gq.GQ_OPT_PREFILL_MIN_N):
                    for xs, key in ((1, "x_static"), (0, "dependent")):
                        gq.gq_set_option(gq.GQ_OPT_X_STATIC, xs)
                        t = graph_time(torch, s, call, copies)
                        gbs = alg / t / 1e9
                        e[key] = {"us": round(t * 1e6, 2), "achieved": round(gbs, 1), "unit": "GB/s",
                                  "frac": round(gbs / hbm, 4)}
                    e.update({"bound": "hbm", "peak": hbm, "bytes": alg,
                              "kernel": "k_decode_q4_0 (mma.sync decode)"})
                else:
                    t, how = graph_or_eager_time(gq, torch, s, call, copies)
                    tf = 2 * M * K * n / t / 1e12
                    e.update({"us": round(t * 1e6, 2), "achieved": round(tf, 2), "unit": "TFLOP/s", "timing": how,
                              "frac": round(tf / tc, 4), "bound": "tensor", "peak": tc,
                              "weight_gbs": round(nb / t / 1e9, 1),
                              "kernel": "k_f32_to_bf16 + k_prefill_q4_0 (tcgen05)"})
                    # the tensor-core kernel alone (bf16 X given), with and
                    # without the x-static promise
                    Xb = X.to(torch.bfloat16).view(torch.int16)
                    e["tensor_core_kernel_only"] = {}
                    for xs, key in ((1, "x_static"), (0, "dependent")):
                        gq.gq_set_option(gq.GQ_OPT_X_STATIC, xs)
                        t3, how3 = graph_or_eager_time(gq, torch, s, lambda i: gq.gq_mul_mat_q4_0_bf16x(
                            Ws[i % copies], M, K, Xb, n, Y, stream=s), copies)
                        tf3 = 2 * M * K * n / t3 / 1e12
                        e["tensor_core_kernel_only"][key] = {"us": round(t3 * 1e6, 2), "achieved": round(tf3, 2),
                                                             "unit": "TFLOP/s", "frac": round(tf3 / tc, 4),
                                                             "weight_gbs": round(nb / t3 / 1e9, 1),
                                                             "weight_frac_of_hbm": round(nb / t3 / 1e9 / hbm, 4),
                                                             "timing": how3}
                out.append(e)
            del Ws, W0
    finally:
        gq.gq_set_option(gq.GQ_OPT_X_STATIC, old_x)
    gq.gq_sync_status(s)
    return {"peak_kind": f"HBM copy / bf16 burst ({peaks['source']})",
            "timing": "CUDA graph of 50-200 back-to-back calls, one weight copy each (> 4x L2 together, "
                      "except the 256 x 1024 matrix: 200 copies, L2-resident), median of 10 replays, "
                      "with GQ_OPT_WEIGHTS_STATIC", "entries": out}


def run_aux(gq, torch, dev, s, hbm_gbs):
    """The dequant and quantise kernels on the 14336 x 4096 matrix (fp32 side
    235 MB, larger than L2), timed with CUDA events on the bench stream, each
    against the HBM roofline with its algorithmic bytes."""
    M, K = AUX_M, AUX_K
    g = torch.Generator(device=dev).manual_seed(0x51A0)
    Wf = torch.randn(M, K, device=dev, generator=g) * 0.05
    Q = torch.empty(M, K // 32 * 18, dtype=torch.uint8, device=dev)
    D = torch.empty(M, K, dtype=torch.float32, device=dev)
    qbytes, fbytes = M * K // 32 * 18, 4 * M * K

    def timed(fn):
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(AUX_REPS):
                fn()
            e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / AUX_REPS * 1e-3

    tq = timed(lambda: gq.gq_quantize_q4_0(Wf, M, K, Q, stream=s))
    td = timed(lambda: gq.gq_dequant_q4_0(Q, M, K, D, stream=s))
    R = torch.empty(2, dtype=torch.int64, device=dev)
    Qs = [Q] + [Q.clone() for _ in range(5)]  # 6 x 33 MB: each call reads W from DRAM
    calls = [0]

    def validate():
        gq.gq_validate_q4_0(Qs[calls[0] % len(Qs)], M, K, R, stream=s)
        calls[0] += 1
    tv = timed(validate)
    gq.gq_sync_status(s)
    out = {}
    vgbs = qbytes / tv / 1e9
    out["validate"] = {"kernel": "k_validate", "shape": f"{M}x{K}", "us": round(tv * 1e6, 2),
                       "achieved": round(vgbs, 1), "unit": "GB/s", "peak": hbm_gbs, "frac": round(vgbs / hbm_gbs, 4),
                       "bound": "hbm", "bytes": qbytes, "bytes_note": "M*K/32*18 Q4_0 read (every sector holds a scale)",
                       "includes": "the one-thread reset of the result (overlapped under programmatic dependent launch)"}
    for name, t, kern in (("quantize", tq, "k_quantize_q4_0"), ("dequant", td, "k_dequant_vec")):
        gbs = (qbytes + fbytes) / t / 1e9
        out[name] = {"kernel": kern, "shape": f"{M}x{K}", "us": round(t * 1e6, 2), "achieved": round(gbs, 1),
                     "unit": "GB/s", "peak": hbm_gbs, "frac": round(gbs / hbm_gbs, 4), "bound": "hbm",
                     "bytes": qbytes + fbytes, "bytes_note": "4*M*K fp32 + M*K/32*18 Q4_0, one read, one written"}
    return out


def run_library_reference(gq, torch, dev, s, peaks):
    """Library reference point, timed only (not part of any value): what a
    caller without these kernels would do on the 14336 x 4096 matrix, namely
    dequantise W to dense bf16 and multiply with torch.matmul (cuBLAS), either
    once per call or once up front with the dense copy kept (4x the weight
    bytes).  Against it: the Q4_0 MUL_MAT of this library on the same shapes."""
    M, K = AUX_M, AUX_K
    Wq = [torch.from_numpy(synth.q4_0_weights(M, K, seed=0x51B0 + i)).to(dev) for i in range(3)]
    Wd = []
    for w in Wq:
        f = torch.empty(M, K, dtype=torch.float32, device=dev)
        gq.gq_dequant_q4_0(w, M, K, f, stream=s)
        Wd.append(f.to(torch.bfloat16))  # 117 MB each: three copies rotate past L2 at N = 1
        del f
    Ws = torch.empty(M, K, dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev).manual_seed(0x51B8)
    X = {n: torch.randn(n, K, device=dev, generator=g) for n in (1, 512)}
    Xb = {n: x.to(torch.bfloat16) for n, x in X.items()}
    Y = {n: torch.empty(n, M, device=dev) for n in (1, 512)}
    reps = 12

    def timed(fn):
        with torch.cuda.stream(s):
            for i in range(3):
                fn(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for i in range(reps):
                fn(i)
            e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps * 1e-3

    def per_call(i, n):  # dequantise, convert, multiply: nothing cached
        gq.gq_dequant_q4_0(Wq[i % 3], M, K, Ws, stream=s)
        torch.matmul(Xb[n], Ws.to(torch.bfloat16).t())

    out = {"note": "timed only; torch.matmul is cuBLAS bf16, fp32 accumulate; W dequantised by gq_dequant_q4_0"}
    for n in (1, 512):
        flops = 2.0 * M * K * n
        t_dense = timed(lambda i: torch.matmul(Xb[n], Wd[i % 3].t()))
        t_call = timed(lambda i: per_call(i, n))
        t_ours = timed(lambda i: gq.gq_mul_mat_q4_0(Wq[i % 3], M, K, X[n], n, Y[n], stream=s))
        out[f"n{n}"] = {
            "dense_bf16_matmul_us": round(t_dense * 1e6, 2),
            "dequant_then_matmul_us": round(t_call * 1e6, 2),
            "gq_mul_mat_q4_0_us": round(t_ours * 1e6, 2),
            "dense_bf16_matmul_tflops": round(flops / t_dense / 1e12, 1),
            "gq_mul_mat_q4_0_tflops": round(flops / t_ours / 1e12, 1),
            "weight_bytes": {"dense_bf16": 2 * M * K, "q4_0": M * K // 32 * 18},
        }
    gq.gq_sync_status(s)
    return out


# MUL_MAT_ID workloads: experts the shape of the prefill matrix (14336 x 4096),
# 8 experts, 2 used per token; 512 tokens (the probe batch) and 1 or 8 tokens.
MOE_E, MOE_M, MOE_K, MOE_S = 8, 14336, 4096, 2
MOE_SETS, MOE_REPS = 4, 8


def moe_weights_dev(torch, dev, rows, K, seed):
    """Seeded Q4_0 blocks generated on the device: qs uniform random bytes, d =
    fp16 of U[0.005, 0.02] (the distribution synth.py uses)."""
    g = torch.Generator(device=dev).manual_seed(seed)
    nb = K // 32
    blk = torch.randint(0, 256, (rows, nb, 18), dtype=torch.uint8, device=dev, generator=g)
    d = (torch.rand((rows, nb), device=dev, generator=g, dtype=torch.float64) * 0.015 + 0.005).to(torch.float16)
    blk[:, :, 0:2] = d.view(torch.uint8).view(rows, nb, 2)
    return blk.view(rows, nb * 18)


def run_moe_aux(gq, torch, dev, s, peaks):
    """gq_mul_mat_id_q4_0 on MOE_SETS distinct expert sets (264 MB each), used in
    turn so that every call streams its experts from DRAM; CUDA events on the
    bench stream around MOE_REPS calls.  Each call = routing + (gather +
    tensor-core | decode) kernels; a single token runs the decode kernel
    alone, reading the ids itself."""
    E, M, K, S = MOE_E, MOE_M, MOE_K, MOE_S
    Ws = [moe_weights_dev(torch, dev, E * M, K, 0x3E00 + i) for i in range(MOE_SETS)]
    out = {}
    for name, T in (("prefill", 512), ("decode", 1), ("decode_t8", 8)):
        X = torch.randn(T, S, K, device=dev, generator=torch.Generator(device=dev).manual_seed(T))
        ids = torch.from_numpy(synth.expert_ids(T, S, E, seed=0x1D00 + T)).to(dev)
        Y = torch.empty(T, S, M, device=dev)
        used = int(torch.unique(ids).numel())

        def call(i):
            gq.gq_mul_mat_id_q4_0(Ws[i % MOE_SETS], E, M, K, X, S, ids, T, Y, stream=s)

        with torch.cuda.stream(s):
            for i in range(MOE_SETS):
                call(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for i in range(MOE_REPS):
                call(i)
            e1.record(s)
        e1.synchronize()
        gq.gq_sync_status(s)
        t = e0.elapsed_time(e1) / MOE_REPS * 1e-3
        P = T * S
        wbytes = used * M * K // 32 * 18
        entry = {"shape": f"{E} experts x {M}x{K}, T={T} tokens x {S} slots", "used_experts": used,
                 "us": round(t * 1e6, 2)}
        if name == "prefill":
            tf = 2 * P * M * K / t / 1e12
            entry.update({"path": "routing + bf16 gather + tcgen05 kernel", "achieved": round(tf, 2),
                          "unit": "TFLOP/s", "peak": peaks["bf16_tflops"], "bound": "tensor",
                          "frac": round(tf / peaks["bf16_tflops"], 4), "flops": 2 * P * M * K,
                          "peak_kind": f"bf16 burst ({peaks['source']})"})
        else:
            b = wbytes + 4 * P * K + 4 * P * M
            gbs = b / t / 1e9
            path = "decode kernel reading the ids itself (no routing)" if T == 1 else "routing + decode kernel"
            entry.update({"path": path, "achieved": round(gbs, 1), "unit": "GB/s",
                          "peak": peaks["hbm_gbs"], "bound": "hbm", "frac": round(gbs / peaks["hbm_gbs"], 4),
                          "bytes": b, "bytes_note": "used experts' Q4_0 weights + fp32 x and y"})
        out[name] = entry
    return out


def run_formats_aux(gq, torch, dev, s, peaks):
    """Q4_1, Q8_0, Q4_K, Q5_0 and Q5_1 on the 14336 x 4096 matrix: dequant (GB/s), MUL_MAT
    at N = 1 (weight GB/s) and N = 512 (TFLOP/s), CUDA events over repeated
    calls on 8 rotating weight copies (264 MB and more together, so each call
    streams its copy from DRAM)."""
    M, K = MOE_M, MOE_K
    out = {}
    for name, qt in (("q4_1", gq.GQ_TYPE_Q4_1), ("q8_0", gq.GQ_TYPE_Q8_0), ("q4_k", gq.GQ_TYPE_Q4_K),
                     ("q5_0", gq.GQ_TYPE_Q5_0), ("q5_1", gq.GQ_TYPE_Q5_1)):
        nbytes = gq.gq_type_nbytes(qt, M, K)
        W0 = torch.from_numpy(synth.typed_weights(qt, M, K, seed=0x7E00 + qt)).to(dev)
        Ws = [W0.clone() for _ in range(8)]
        D = torch.empty(M, K, device=dev)
        X1 = torch.randn(1, K, device=dev)
        XP = torch.randn(512, K, device=dev)
        Y1 = torch.empty(1, M, device=dev)
        YP = torch.empty(512, M, device=dev)

        def timed(fn, reps=6):
            with torch.cuda.stream(s):
                for i in range(3):
                    fn(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                for i in range(reps):
                    fn(i)
                e1.record(s)
            e1.synchronize()
            return e0.elapsed_time(e1) / reps * 1e-3

        td = timed(lambda i: gq.gq_dequant(qt, Ws[i % 8], M, K, D, stream=s))
        t1 = timed(lambda i: gq.gq_mul_mat(qt, Ws[i % 8], M, K, X1, 1, Y1, stream=s), reps=16)
        tp = timed(lambda i: gq.gq_mul_mat(qt, Ws[i % 8], M, K, XP, 512, YP, stream=s))
        gq.gq_sync_status(s)
        dq = (nbytes + 4 * M * K) / td / 1e9
        g1 = (nbytes + 4 * K + 4 * M) / t1 / 1e9
        tf = 2 * M * K * 512 / tp / 1e12
        out[name] = {
            "shape": f"{M}x{K}", "block_bytes": gq.TYPE_BLOCK_BYTES[qt],
            "block_weights": gq.TYPE_BLOCK_WEIGHTS[qt],
            "dequant": {"us": round(td * 1e6, 2), "achieved": round(dq, 1), "unit": "GB/s", "bound": "hbm",
                        "frac": round(dq / peaks["hbm_gbs"], 4)},
            "mul_mat_n1": {"us": round(t1 * 1e6, 2), "achieved": round(g1, 1), "unit": "GB/s", "bound": "hbm",
                           "frac": round(g1 / peaks["hbm_gbs"], 4),
                           "kernel": "k_decode_q4_0<..., type> (mma.sync decode on this block format)",
                           "timing": "eager back-to-back calls (launch gaps included)"},
            "mul_mat_n512": {"us": round(tp * 1e6, 2), "achieved": round(tf, 2), "unit": "TFLOP/s",
                             "bound": "tensor", "frac": round(tf / peaks["bf16_tflops"], 4),
                             "kernel": "k_f32_to_bf16 + k_prefill_q4_0<256, 0, 0, type>"},
        }
    return out


def run_prepared_aux(gq, torch, dev, s, peaks):
    """The repacked layout on an 11008 x 2880 matrix (2880 = 11.25 x 256, a K
    the packed fast paths do not take): gq_prepare_q4_0 (GB/s), then MUL_MAT on
    the prepared weights at N = 1 (weight GB/s, rotating copies) and N = 512."""
    M, K = 11008, 2880
    W = torch.from_numpy(synth.q4_0_weights(M, K, seed=0x9E00)).to(dev)
    pb = gq.gq_prepared_q4_0_nbytes(M, K)
    Wps = [torch.empty(pb, dtype=torch.uint8, device=dev) for _ in range(8)]
    X1 = torch.randn(1, K, device=dev)
    XP = torch.randn(512, K, device=dev)
    Y1 = torch.empty(1, M, device=dev)
    YP = torch.empty(512, M, device=dev)

    def timed(fn, reps=8):
        with torch.cuda.stream(s):
            for i in range(8):
                fn(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for i in range(reps):
                fn(i)
            e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps * 1e-3

    tpre = timed(lambda i: gq.gq_prepare_q4_0(W, M, K, 0, Wps[i % 8], stream=s))
    t1 = timed(lambda i: gq.gq_mul_mat_q4_0_prepared(Wps[i % 8], M, K, X1, 1, Y1, stream=s))
    tp = timed(lambda i: gq.gq_mul_mat_q4_0_prepared(Wps[i % 8], M, K, XP, 512, YP, stream=s))
    gq.gq_sync_status(s)
    wbytes = gq.gq_q4_0_nbytes(M, K)
    return {
        "shape": f"{M}x{K}",
        "prepare": {"us": round(tpre * 1e6, 2), "achieved": round((wbytes + pb) / tpre / 1e9, 1), "unit": "GB/s",
                    "bound": "hbm", "frac": round((wbytes + pb) / tpre / 1e9 / peaks["hbm_gbs"], 4)},
        "mul_mat_n1": {"us": round(t1 * 1e6, 2), "achieved": round(wbytes / t1 / 1e9, 1), "unit": "GB/s",
                       "bound": "hbm", "frac": round(wbytes / t1 / 1e9 / peaks["hbm_gbs"], 4)},
        "mul_mat_n512": {"us": round(tp * 1e6, 2), "achieved": round(2 * M * K * 512 / tp / 1e12, 2),
                         "unit": "TFLOP/s", "bound": "tensor",
                         "frac": round(2 * M * K * 512 / tp / 1e12 / peaks["bf16_tflops"], 4)},
    }


def run_e2e(gq, torch, dev, s, W, shapes, acts1, order, L, args):
    """Decode sweep through gq_mul_mat_q4_0 with host buffers.  Every step
    copies the step's inputs (all layers' activations, one pinned buffer) to
    the device in one copy, runs the 224 calls, and copies the step's results
    (every Y, one device buffer) back to pinned host memory in one copy, as a
    decode step moves its inputs and outputs once."""
    xs = [a for la in acts1 for a in la]
    x_off = np.cumsum([0] + [a.size for a in xs])
    hx = torch.from_numpy(np.concatenate([a.reshape(-1) for a in xs])).pin_memory()
    dx = torch.empty(hx.numel(), dtype=torch.float32, device=dev)
    y_sizes = [DECODE_N * M for M, _ in shapes]
    y_off = np.cumsum([0] + y_sizes)
    dy = torch.empty(int(y_off[-1]), device=dev)
    hy = torch.empty(int(y_off[-1])).pin_memory()
    nper = len(acts1[0])
    xview = [[dx[int(x_off[l * nper + i]):int(x_off[l * nper + i + 1])].view(acts1[l][i].shape)
              for i in range(nper)] for l in range(L)]
    yview = [dy[int(y_off[i]):int(y_off[i + 1])] for i in range(len(shapes))]

    def one():
        dx.copy_(hx, non_blocking=True)
        for layer in range(L):
            for j in range(len(order)):
                i = layer * len(order) + j
                M, K = shapes[i]
                gq.gq_mul_mat_q4_0(W[i], M, K, xview[layer][order[j]], DECODE_N, yview[i], stream=s)
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(s):
        one()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            one()
    torch.cuda.synchronize(dev)
    for _ in range(3):
        with torch.cuda.stream(s):
            g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            g.replay()
        e1.record(s)
    e1.synchronize()
    return {"ms": e0.elapsed_time(e1) / args.steps, "h2d": hx.numel() * 4, "d2h": hy.numel() * 4}


# DRAM bytes (read + write) per launch, from one ncu capture per shape of the
# sweep (profiles/dram_traffic_sweep_shapes.md); refresh when a kernel changes.
MEASURED_TRAFFIC = {
    "decode": {(4096, 4096): 9512704, (11008, 4096): 25442048, (4096, 11008): 25465344},
    "prefill": {(4096, 4096): 13682944, (11008, 4096): 29627136, (4096, 11008): 36686336},
}

def sweep_traffic(kind, shapes):
    """Mean measured DRAM bytes per launch over the sweep's launches, or None."""
    table = MEASURED_TRAFFIC[kind]
    if not all(sh in table for sh in shapes):
        return None
    return round(sum(table[sh] for sh in shapes) / len(shapes))


PROFILE_CASES = {
    # name: (M, K, N, entry point)
    "decode": (11008, 4096, 1, "f32"),
    "decode_down": (4096, 11008, 1, "f32"),
    "decode_small": (4096, 4096, 1, "f32"),
    "decode_big": (32000, 4096, 1, "f32"),
    "decode_big_n8": (32000, 4096, 8, "f32"),
    "prefill": (14336, 4096, 512, "bf16"),
    "prefill_small": (4096, 4096, 512, "bf16"),
    "prefill_gate": (11008, 4096, 512, "bf16"),
    "prefill_down": (4096, 11008, 512, "bf16"),
    "moe_prefill": (MOE_M, MOE_K, 512, "moe"),
    "moe_decode": (MOE_M, MOE_K, 1, "moe"),
    "q4_1_decode": (14336, 4096, 1, "q4_1"),
    "q8_0_decode": (14336, 4096, 1, "q8_0"),
    "q4_k_decode": (14336, 4096, 1, "q4_k"),
    "q4_k_prefill": (14336, 4096, 512, "q4_k"),
    "q4_k_dequant": (14336, 4096, 0, "q4_k"),
    "quantize": (14336, 4096, 0, "quantize"),
}


def run_profile_case(name, pair=False):
    """One small invocation for an ncu capture: two launches of one MUL_MAT."""
    import torch
    import quantized_block_q4_gb300 as gq
    M, K, N, mode = PROFILE_CASES[name]
    gq.gq_set_option(gq.GQ_OPT_WEIGHTS_STATIC, 1)
    gq.gq_set_option(gq.GQ_OPT_X_STATIC, 1)
    gq.gq_set_option(gq.GQ_OPT_PREFILL_PAIR, 1 if pair else 0)
    if mode == "moe":  # MUL_MAT_ID: N tokens x MOE_S slots over MOE_E experts
        W = moe_weights_dev(torch, "cuda", MOE_E * M, K, 1)
        X = torch.randn(N, MOE_S, K, device="cuda")
        ids = torch.from_numpy(synth.expert_ids(N, MOE_S, MOE_E, seed=3)).cuda()
        Y = torch.empty(N, MOE_S, M, device="cuda")
        for _ in range(2):
            gq.gq_mul_mat_id_q4_0(W, MOE_E, M, K, X, MOE_S, ids, N, Y)
        torch.cuda.synchronize()
        gq.gq_sync_status()
        print(f"profile case {name}: {MOE_E} experts {M}x{K}, {N} tokens x {MOE_S} ok")
        return 0
    if mode in ("q4_1", "q8_0", "q4_k"):  # the other block formats (N = 0: dequantisation)
        qt = {"q4_1": gq.GQ_TYPE_Q4_1, "q8_0": gq.GQ_TYPE_Q8_0, "q4_k": gq.GQ_TYPE_Q4_K}[mode]
        W = torch.from_numpy(synth.typed_weights(qt, M, K, seed=1)).cuda()
        X = torch.from_numpy(synth.activations(max(N, 1), K, seed=2)).cuda()
        Y = torch.empty(max(N, 1), M, device="cuda")
        D = torch.empty(M, K, device="cuda") if N == 0 else None
        for _ in range(2):
            if N == 0:
                gq.gq_dequant(qt, W, M, K, D)
            else:
                gq.gq_mul_mat(qt, W, M, K, X, N, Y)
        torch.cuda.synchronize()
        gq.gq_sync_status()
        print(f"profile case {name}: M={M} K={K} N={N} ok")
        return 0
    if mode == "quantize":  # fp32 -> Q4_0
        Wf = torch.from_numpy(synth.activations(M, K, seed=3)).cuda() * 0.05
        Q = torch.empty(M, K // 32 * 18, dtype=torch.uint8, device="cuda")
        for _ in range(2):
            gq.gq_quantize_q4_0(Wf, M, K, Q)
        torch.cuda.synchronize()
        gq.gq_sync_status()
        print(f"profile case {name}: M={M} K={K} ok")
        return 0
    W = torch.from_numpy(synth.q4_0_weights(M, K, seed=1)).cuda()
    X = torch.from_numpy(synth.activations(N, K, seed=2)).cuda()
    Y = torch.empty(N, M, device="cuda")
    for _ in range(2):
        if mode == "bf16":
            gq.gq_mul_mat_q4_0_bf16x(W, M, K, X.to(torch.bfloat16).view(torch.int16), N, Y)
        else:
            gq.gq_mul_mat_q4_0(W, M, K, X, N, Y)
    torch.cuda.synchronize()
    gq.gq_sync_status()
    print(f"profile case {name}: M={M} K={K} N={N} ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run one MUL_MAT twice (for an ncu capture) and exit")
    ap.add_argument("--pair", action="store_true", help="with --profile-case: use the 2-SM prefill kernel")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gq", "reference"], default="gq")
    ap.add_argument("--layers", type=int, default=synth.N_LAYERS)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=5.0, help="seconds of oracle work per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args.profile_case, args.pair)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend=backend)
        dist = tdist
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_gpu(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
