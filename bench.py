"""Benchmark: one LLaDA-8B-shaped diffusion denoising step at canvas L = 148 on GB300.

A step = embedding of the canvas, 32 layers (RMSNorm + Q8_K, Q|K Q4_K, V Q6_K, NORM RoPE,
non-causal attention, O Q4_K + residual, RMSNorm + Q8_K, gate|up Q4_K, SwiGLU + Q8_K, down
Q6_K + residual), then the masked-rows-only LM head (Q6_K 126464 x 4096) with softmax
confidence and the top-4 commit of the current block; 32 steps fill 4 blocks of 32 positions.
Weights are seeded random (synthetic) with the LLaDA-8B shapes; total weight bytes per step
(4.9 GB) exceed L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. `--impl reference` times the CPU oracle (f64, OpenMP) on a bounded
sample of the same step (two of the 32 layers plus the LM head), scaled to one step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms/denoising step at L=148 (LLaDA-8B shapes); Q4_K GEMM TOPS vs roofline"
WORKLOAD = "llada8b_denoise_step_L148"
# the pages' benchmark protocol: 20 prompt + 128 generated tokens, blocks of 32, 32 steps (the
# library's schedule then commits 4 tokens per step)
L_CANVAS, PROMPT, GEN, BLOCK, STEPS = 148, 20, 128, 32, 32
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _env_dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _schedule():
    """(schedule, kinds, kind index per step): the library's transfer schedule of the protocol,
    its distinct (block_begin, block_end, k) step kinds, and each step's kind."""
    import quantized_gemm_q8_gb300 as dl

    sched = dl.schedule(PROMPT, GEN, BLOCK, STEPS)
    kinds = sorted(set(sched))
    return sched, kinds, [kinds.index(t) for t in sched]


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs."""

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"]}
        hi = [v for v in sm if v > 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(hi), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def gemm_source_sha1() -> str:
    """sha1 of the GEMM kernel's code (the kernel and the PTX wrappers it is built from), with
    comments, indentation and blank lines left out, so that a comment edit keeps the record."""
    h = hashlib.sha1()
    for name in ("qgemm.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "quantized_gemm_q8_gb300", "csrc", name), encoding="utf-8") as f:
            src = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).strip() for ln in src.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()


def _traffic_for(kernel_file: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", kernel_file)
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("gemm_src_sha1") == gemm_source_sha1():
            return rec.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def oracle_step_sample(dims, seed, n_layers_sample=2):
    """Time the CPU oracle on two of the 32 layers (with attention) plus the masked LM head and
    scale to one step. Returns (ms per step, threads, description)."""
    import numpy as np

    import oracle as orc
    from quantized_gemm_q8_gb300 import synth

    canvas = synth.canvas(seed)
    table = synth.embed_weights(seed, dims)
    head = synth.head_weights(seed, dims)
    lws = [synth.layer_weights(seed, i, dims) for i in range(n_layers_sample)]
    t0 = time.perf_counter()
    x = orc.embed(table, canvas)
    t1 = time.perf_counter()
    for lw in lws:
        x, _ = orc.layer(lw, x, dims, attention_on=True)
    t2 = time.perf_counter()
    cv = canvas.copy()
    b0, b1, k = _schedule()[0][0]
    orc.lmhead_commit(x, cv, dims["mask_id"], b0, b1, k, head["out_norm"], head["w_out"], dims["eps"])
    t3 = time.perf_counter()
    per_layer = (t2 - t1) / n_layers_sample
    ms = 1e3 * ((t1 - t0) + dims["n_layers"] * per_layer + (t3 - t2))
    desc = (f"estimate: embedding + {n_layers_sample} of {dims['n_layers']} layers (L=148, with attention) + masked "
            f"LM head (32 rows x 126464 x 4096) of one step, measured; the layer time scaled "
            f"x{dims['n_layers']}/{n_layers_sample} to the full depth")
    return ms, orc.num_threads(), desc


def run_reference(args, rank):
    from quantized_gemm_q8_gb300 import synth

    if rank != 0:
        return
    dims = dict(synth.LLADA)
    seed = synth.config_seed(4)
    for _ in range(args.warmup):
        oracle_step_sample(dims, seed)
    vals = []
    desc, cores = "", 0
    for _ in range(args.steps):
        ms, cores, desc = oracle_step_sample(dims, seed)
        vals.append(ms)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "ms/step", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random LLaDA-8B-shaped weights)",
        "config": {"workload": WORKLOAD, "L": L_CANVAS, "layers": dims["n_layers"], "block": BLOCK,
                   "k_commit": _schedule()[0][0][2], "l2": "weights (4.9 GB) > L2",
                   "value_kind": "estimate: 2 of the 32 layers timed, scaled to 32 (a full oracle step takes "
                                 "about half a minute per layer pair on these cores)"},
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": "ms/step", "cores": cores, "sample": desc},
        "e2e": {"value": value, "unit": "ms/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def job_timing(ms_local, steps, world, dist=None, device="cpu"):
    """Whole-job timing of N replicas: the slowest rank's timed region (max over ranks), its
    per-step time, and the job-wide ms per step (N replicas complete N * steps steps in that
    time). `dist` is torch.distributed with an initialized process group when world > 1."""
    import torch

    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, ms_max / steps, ms_max / (steps * world)


def run_ours(args, rank, local_rank, world):
    import numpy as np
    import torch

    import quantized_gemm_q8_gb300 as dl
    from quantized_gemm_q8_gb300 import synth

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dims = dict(synth.LLADA)
    seed = synth.config_seed(4)
    model = dl.model_from_seed(dims, seed)
    canvas0 = torch.from_numpy(synth.canvas(seed)).cuda()
    canvas = canvas0.clone()
    sched, kinds, kind_of = _schedule()
    graphs = dl.StepGraphs(model, canvas, kinds)

    def block_of(s):  # the graph of step s of the protocol's schedule (repeated past its end)
        return kind_of[s % len(sched)]

    stream = graphs.stream
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):  # graph replays launch on the current stream
        for s in range(args.warmup):
            graphs.replay(block_of(s))
    torch.cuda.synchronize()
    dl.check(stream)
    canvas.copy_(canvas0)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        ev0.record(stream)
        for s in range(args.steps):
            graphs.replay(block_of(s))
        ev1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    dl.check(stream)
    ms_max, ms_per_step, value = job_timing(ev0.elapsed_time(ev1), args.steps, world, dist, "cuda")

    # ---- end-to-end through the public call with host buffers (H2D canvas, D2H commits) ----
    # one dllm_step_graph_host call per step: the pinned host canvas in, the step's graph, the
    # commits out and applied to the host canvas (torch builds without a raw graph handle fall
    # back to the same copies issued from Python)
    canvas_h = torch.from_numpy(synth.canvas(seed)).pin_memory()
    kmax = max(k for _, _, k in kinds)
    out_h = torch.empty(2 * kmax, dtype=torch.int32).pin_memory()
    e2e_steps = min(args.steps, 32)
    via_c = hasattr(torch.cuda.CUDAGraph, "raw_cuda_graph_exec")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        if via_c:
            graphs.step_host(block_of(s), canvas_h, out_h)
            continue
        with torch.cuda.stream(stream):
            canvas.copy_(canvas_h, non_blocking=True)
            graphs.replay(block_of(s))
            out_h.copy_(graphs.pos_id, non_blocking=True)
        stream.synchronize()
        k = sched[s % len(sched)][2]
        pos, ids = out_h[:k].numpy(), out_h[kmax:kmax + k].numpy()
        for p, i in zip(pos, ids):
            if p >= 0:
                canvas_h[p] = int(i)
    e2e_ms = 1e3 * (time.perf_counter() - t0) / e2e_steps
    dl.check(stream)
    committed = int((canvas_h.numpy()[PROMPT:] != dims["mask_id"]).sum())

    # ---- dominant kernel: the gate|up Q4_K GEMM alone, CUDA events on its stream ----
    peaks, peak_src = _peaks()
    L, d, f = L_CANVAS, dims["d_model"], dims["d_ff"]
    x = torch.randn(L, d, device="cuda")
    act = dl.quantize_act(x, plain=False)["act"]
    lays = model.struct.layers
    gemms = {
        "gate_up_q4k": (dl.Q4_K, 2 * f, d, lambda i: lays[i].wgu),
        "qk_q4k": (dl.Q4_K, 2 * d, d, lambda i: lays[i].wqk),
        "v_q6k": (dl.Q6_K, d, d, lambda i: lays[i].wv),
        "o_q4k": (dl.Q4_K, d, d, lambda i: lays[i].wo),
    }
    actf = dl.quantize_act(torch.randn(L, f, device="cuda"), plain=False)["act"]
    kern = {}
    with torch.cuda.stream(stream):
        for name, (ty, n, k, wp) in list(gemms.items()) + [("down_q6k", (dl.Q6_K, d, f, lambda i: lays[i].wdown))]:
            a = actf if name == "down_q6k" else act
            nb = int(dl.lib().dllm_qgemm_partials_bytes(ty, L, n, k))
            part = torch.empty(nb // 4, dtype=torch.float32, device="cuda")

            class _W:  # wrap a raw device pointer for the binding
                def __init__(self, ptr):
                    self.p = ptr

                def data_ptr(self):
                    return self.p

            for i in range(3):
                dl.qgemm_partials(ty, a, L, k, _W(wp(i)), n, partials=part, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(dims["n_layers"]):
                dl.qgemm_partials(ty, a, L, k, _W(wp(i)), n, partials=part, stream=stream)
            e1.record(stream)
            stream.synchronize()
            kern[name] = e0.elapsed_time(e1) / dims["n_layers"]
    dl.check(stream)
    gu_ms = kern["gate_up_q4k"]
    gu_flops = 2.0 * L * (2 * f) * d
    achieved = gu_flops / (gu_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    q4k_bytes = (2 * f) * d // 256 * 144
    layer_gemm_ms = sum(kern.values())
    ops_step = 2.0 * L * dims["n_layers"] * (4 * d * d + 3 * d * f) + 2.0 * 32 * dims["vocab"] * d
    bytes_step = dims["n_layers"] * ((4 * d * d + 2 * d * f) // 256 * 144 + (d * d + d * f) // 256 * 210) + \
        dims["vocab"] * d // 256 * 210
    t_roof_ms = max(ops_step / (peak * 1e12), bytes_step / (peaks["hbm_gbs"] * 1e9)) * 1e3
    # the second roofline: the legacy int8 tensor path's dense rate (mma.sync m16n8k32), measured
    i8_tops = dl.peak_mma_i8_tops(stream=stream)
    t_roof_i8_ms = max(ops_step / (i8_tops * 1e12), bytes_step / (peaks["hbm_gbs"] * 1e9)) * 1e3

    line = {
        "metric": METRIC, "value": value, "unit": "ms/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded random LLaDA-8B-shaped Q4_K/Q6_K weights, 20 random prompt ids + 128 masks)",
        "config": {"workload": WORKLOAD, "L": L, "layers": dims["n_layers"], "d_model": d, "d_ff": f,
                   "vocab": dims["vocab"], "block": BLOCK, "k_commit": sched[0][2],
                   "schedule": f"dllm_schedule({PROMPT}, {GEN}, {BLOCK}, {STEPS})", "graph": "one CUDA graph per block",
                   "l2": "no flush: weights read per step (4.9 GB) exceed L2",
                   "parallelism": f"replicas x{world}",
                   "arith": "Q8_K x Q4_K/Q6_K integer sums exact in f16 tcgen05 MMA, f32 accumulate/epilogue"},
        "tok_per_s": (sum(k for _, _, k in sched) / len(sched)) * world / (value * 1e-3),
        "step_roofline_ms": t_roof_ms, "step_roofline_frac": t_roof_ms / ms_per_step,
        "roofline_int8_mma_sync": {"peak_tops": i8_tops, "source": "measured in this run (dllm_peak_mma_i8)",
                                   "step_roofline_ms": t_roof_i8_ms, "step_frac": t_roof_i8_ms / ms_per_step,
                                   "gate_up_frac": achieved / i8_tops},
        "algorithmic_tops": ops_step / (ms_per_step * 1e-3) / 1e12,
        "gpu_launches": int(graphs.launches_per_step[0]) * args.steps,
        "roofline": {"kernel": "qgemm_kernel<Q4_K, NT=160> (gate|up 148x24576x4096)", "bound": "tensor",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"bf16 burst, {peak_src} (MEASURED_PEAKS.json); f16 runs at the bf16 rate",
                     "traffic": _traffic_for("qgemm_q4k_gateup_L148.json"),
                     "algorithmic_bytes": q4k_bytes, "ms_per_launch": gu_ms},
        "kernel_ms_per_layer": {k: round(v, 4) for k, v in kern.items()},
        "layer_gemm_ms": layer_gemm_ms,
        "clocks": clk.summary(),
        "e2e": {"value": e2e_ms, "unit": "ms/step", "h2d_bytes_per_step": int(canvas_h.numel() * 4),
                "d2h_bytes_per_step": int(2 * max(k for _, _, k in sched) * 4), "steps": e2e_steps,
                "committed_after": committed, "path": "dllm_step_graph_host" if via_c else "python copies"},
        "context": {"pages_rtx3050_ms_per_step": 221, "pages_i5_13420h_ms_per_step": 3005},
    }
    if rank == 0 and not args.no_cpu_baseline:
        ms_cpu, cores, desc = oracle_step_sample(dims, seed)
        line["cpu_baseline"] = {"value": ms_cpu, "unit": "ms/step", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


ONLY_KERNELS = {  # name: (type, n, k) of one layer's GEMM at L = 148
    "gate_up_q4k": ("q4k", 2 * 12288, 4096), "qk_q4k": ("q4k", 2 * 4096, 4096), "v_q6k": ("q6k", 4096, 4096),
    "o_q4k": ("q4k", 4096, 4096), "down_q6k": ("q6k", 4096, 12288),
}


def run_only_layer(args):
    """One LLaDA-8B-shaped layer's full forward (embedding, attention, FFN) at L = 148 on a
    one-layer model: the profiling target of the glue kernels (--steps launches after --warmup)."""
    import torch

    import quantized_gemm_q8_gb300 as dl
    from quantized_gemm_q8_gb300 import synth

    torch.cuda.set_device(0)
    dims = dict(synth.LLADA, n_layers=1)
    model = dl.model_from_seed(dims, synth.config_seed(4))
    canvas = torch.from_numpy(synth.canvas(synth.config_seed(4))).cuda()
    x = torch.empty((L_CANVAS, dims["d_model"]), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup):
        dl.step_linear_stream(model, x, dl.STREAM_FULL, canvas=canvas)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        dl.step_linear_stream(model, x, dl.STREAM_FULL, canvas=canvas)
    e1.record()
    torch.cuda.synchronize()
    dl.check()
    print(json.dumps({"kernel": "layer_full", "L": L_CANVAS, "ms_per_layer": e0.elapsed_time(e1) / max(args.steps, 1),
                      "note": "one-layer model, embedding + layer; a profiling target"}))


def run_only_lmhead(args):
    """Config 3's masked-rows LM head alone (126464 x 4096 Q6_K on the 32 rows of block 0, softmax
    confidence, top-4 commit): the profiling target of the narrow-tile GEMM (--steps calls)."""
    import torch

    import quantized_gemm_q8_gb300 as dl
    from quantized_gemm_q8_gb300 import synth

    torch.cuda.set_device(0)
    dims = dict(synth.LLADA)
    seed = synth.config_seed(3)
    d, vocab = dims["d_model"], dims["vocab"]
    head = synth.head_weights(seed, dims)
    w_out = dl.pack_weights(dl.Q6_K, torch.from_numpy(head["w_out"].reshape(-1)).cuda(), vocab, d)
    out_norm = torch.from_numpy(head["out_norm"]).cuda()
    canvas0 = torch.from_numpy(synth.canvas(seed)).cuda()
    canvas = canvas0.clone()
    hidden = torch.from_numpy(synth.activations(seed, L_CANVAS, d)).cuda()
    b0, b1, k_commit = _schedule()[0][0]
    ws = torch.empty(max(dl.lmhead_workspace_bytes(b1 - b0, vocab, d), 1), dtype=torch.uint8, device="cuda")

    def run():
        canvas.copy_(canvas0)
        dl.lmhead_masked_select(hidden, canvas, dims["mask_id"], b0, b1, k_commit, out_norm, w_out, vocab,
                                dims["eps"], ws=ws)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    dl.check()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    wbytes = vocab * d // 256 * 210
    print(json.dumps({"kernel": "lm_head", "rows": b1 - b0, "vocab": vocab, "d": d, "ms_per_call": ms,
                      "weight_gbs": wbytes / (ms * 1e-3) / 1e9,
                      "note": "weights (425 MB) exceed L2: read from HBM every call; a profiling target"}))


def run_only_kernel(args):
    """Time one GEMM of the step alone (the profiling target): --steps launches after --warmup."""
    import torch

    import quantized_gemm_q8_gb300 as dl
    from quantized_gemm_q8_gb300 import synth

    if args.only_kernel == "layer_full":
        return run_only_layer(args)
    if args.only_kernel == "lm_head":
        return run_only_lmhead(args)

    ty_name, n, k = ONLY_KERNELS[args.only_kernel]
    ty = dl.Q4_K if ty_name == "q4k" else dl.Q6_K
    torch.cuda.set_device(0)
    blocks = torch.from_numpy(synth.blocks(ty, synth.config_seed(4), n, k).reshape(-1)).cuda()
    pk = dl.pack_weights(ty, blocks, n, k)
    del blocks
    act = dl.quantize_act(torch.from_numpy(synth.activations(synth.config_seed(4), L_CANVAS, k)).cuda(),
                          plain=False)["act"]
    part, splits = dl.qgemm_partials(ty, act, L_CANVAS, k, pk, n)
    for _ in range(args.warmup):
        dl.qgemm_partials(ty, act, L_CANVAS, k, pk, n, partials=part)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        dl.qgemm_partials(ty, act, L_CANVAS, k, pk, n, partials=part)
    e1.record()
    torch.cuda.synchronize()
    dl.check()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    flops = 2.0 * L_CANVAS * n * k
    print(json.dumps({"kernel": args.only_kernel, "m": L_CANVAS, "n": n, "k": k, "splits": splits,
                      "ms_per_launch": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                      "note": "weights L2-resident after the first launch (single copy): a profiling target"}))


def run_configs(args):
    """One JSON line per configuration other than the step (config 4, the default run): the
    single Q4_K GEMM (config 1), the layer stream at L = 148 (2), the masked-rows LM head + commit
    (3) and the canvas-length sweep of the layer stream (5), each against its roofline, and the
    CPU oracle timed on configs 1-3."""
    import numpy as np
    import torch

    import quantized_gemm_q8_gb300 as dl
    from quantized_gemm_q8_gb300 import synth

    torch.cuda.set_device(0)
    peaks, peak_src = _peaks()
    hbm, tens = peaks["hbm_gbs"], peaks["bf16_tflops"]
    stream = torch.cuda.Stream()
    lines = []

    def timed(fn, reps):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        dl.check(stream)
        return e0.elapsed_time(e1) / reps

    # ---- config 1: quantize 16 x 4096 + Q4_K GEMM 4096 x 4096, 16 weight copies (151 MB) rotated
    m1, n1, k1 = 16, 4096, 4096
    seed1 = synth.config_seed(1)
    wblk = synth.blocks(dl.Q4_K, seed1, n1, k1)
    copies = [dl.pack_weights(dl.Q4_K, torch.from_numpy(wblk.reshape(-1)).cuda(), n1, k1) for _ in range(16)]
    x1 = torch.from_numpy(synth.activations(seed1, m1, k1)).cuda()
    act1 = torch.empty(dl.act_bytes(m1, k1), dtype=torch.uint8, device="cuda")
    y1 = torch.empty((m1, n1), dtype=torch.float32, device="cuda")
    ws1 = torch.empty(max(dl.qgemm_workspace_bytes(dl.Q4_K, m1, n1, k1), 1), dtype=torch.uint8, device="cuda")
    per_graph = 64
    with torch.cuda.stream(stream):
        for i in range(3):  # warm-up, also loads the kernels
            dl.quantize_act(x1, plain=False, act=act1, stream=stream)
            dl.qgemm(dl.Q4_K, act1, m1, k1, copies[i % 16], n1, y=y1, ws=ws1, stream=stream)
    torch.cuda.synchronize()
    dl.check(stream)
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        for i in range(per_graph):
            dl.quantize_act(x1, plain=False, act=act1, stream=stream)
            dl.qgemm(dl.Q4_K, act1, m1, k1, copies[i % 16], n1, y=y1, ws=ws1, stream=stream)
    g1.replay()
    ms1 = timed(g1.replay, 8) / per_graph
    bytes1 = n1 * k1 // 256 * 144 + m1 * (k1 + k1 // 256 * 4 + k1 // 16 * 2) + m1 * n1 * 4
    ln1 = {"config": 1, "workload": "quantize 16x4096 + Q4_K GEMM 4096x4096 -> 16x4096 f32", "value": ms1 * 1e3,
           "unit": "us/GEMM", "launch": f"CUDA graph of {per_graph} back-to-back calls, 16 weight copies rotated",
           "roofline": {"bound": "hbm", "achieved": bytes1 / (ms1 * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": bytes1 / (ms1 * 1e-3) / 1e9 / hbm, "algorithmic_bytes": bytes1},
           "tops": 2.0 * m1 * n1 * k1 / (ms1 * 1e-3) / 1e12}
    lines.append(ln1)
    del copies, g1

    # ---- configs 2 and 5: the layer stream (no attention) over a 4-layer model (560 MB of weights)
    dims = dict(synth.LLADA, n_layers=4)
    seed2 = synth.config_seed(2)
    model = dl.model_from_seed(dims, seed2)
    d, f = dims["d_model"], dims["d_ff"]
    wbytes_layer = (4 * d * d + 2 * d * f) // 256 * 144 + (d * d + d * f) // 256 * 210
    for L in (148, 32, 512, 2048):
        x0 = torch.from_numpy(synth.activations(seed2 if L == 148 else synth.config_seed(5) + L, L, d)).cuda()
        x = x0.clone()
        ws = torch.empty(dl.step_workspace_bytes(model, L, dl.STREAM_LINEAR) + 1024, dtype=torch.uint8, device="cuda")

        def run_stream():
            x.copy_(x0, non_blocking=True)
            dl.step_linear_stream(model, x, dl.STREAM_LINEAR, ws=ws, stream=stream)

        run_stream()
        reps = 20 if L <= 512 else 6
        ms = timed(run_stream, reps) / dims["n_layers"]
        ops = 2.0 * L * (4 * d * d + 3 * d * f)
        t_roof = max(ops / (tens * 1e12), wbytes_layer / (hbm * 1e9)) * 1e3
        bound = "tensor" if ops / (tens * 1e12) >= wbytes_layer / (hbm * 1e9) else "hbm"
        lines.append({"config": 2 if L == 148 else 5, "workload": f"LLaDA-8B layer stream (no attention), L={L}",
                      "value": ms, "unit": "ms/layer", "tops": ops / (ms * 1e-3) / 1e12,
                      "roofline": {"bound": bound, "t_roof_ms": t_roof, "frac": t_roof / ms,
                                   "peak": {"tensor_tflops": tens, "hbm_gbs": hbm}},
                      "note": "per layer of a 4-layer pass; the input copy (L x 4096 f32) is inside the timed region"})
    del model

    # ---- config 3: masked-rows LM head 126464 x 4096 Q6_K + softmax confidence + top-4 commit
    dims3 = dict(synth.LLADA)
    seed3 = synth.config_seed(3)
    head = synth.head_weights(seed3, dims3)
    vocab = dims3["vocab"]
    w_out = dl.pack_weights(dl.Q6_K, torch.from_numpy(head["w_out"].reshape(-1)).cuda(), vocab, d)
    out_norm = torch.from_numpy(head["out_norm"]).cuda()
    canvas0 = torch.from_numpy(synth.canvas(seed3)).cuda()
    canvas = canvas0.clone()
    hidden = torch.from_numpy(synth.activations(seed3, L_CANVAS, d)).cuda()
    b0, b1, K_COMMIT = _schedule()[0][0]  # the protocol's first step: block 0, 4 commits
    ws3 = torch.empty(max(dl.lmhead_workspace_bytes(b1 - b0, vocab, d), 1), dtype=torch.uint8, device="cuda")

    def run_head():
        canvas.copy_(canvas0, non_blocking=True)
        dl.lmhead_masked_select(hidden, canvas, dims3["mask_id"], b0, b1, K_COMMIT, out_norm, w_out, vocab,
                                dims3["eps"], ws=ws3, stream=stream)

    run_head()
    ms3 = timed(run_head, 20)
    bytes3 = vocab * d // 256 * 210
    ln3 = {"config": 3, "workload": "masked-rows LM head 126464x4096 Q6_K (32 block rows) + confidence + top-4",
           "value": ms3 * 1e3, "unit": "us/call",
           "roofline": {"bound": "hbm", "achieved": bytes3 / (ms3 * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": bytes3 / (ms3 * 1e-3) / 1e9 / hbm, "algorithmic_bytes": bytes3}}
    lines.append(ln3)

    # ---- config 3 with temperature sampling (T = 0.8): Gumbel-max draws in the same epilogue
    def run_head_sample():
        canvas.copy_(canvas0, non_blocking=True)
        dl.lmhead_select(hidden, canvas, dims3["mask_id"], b0, b1, K_COMMIT, out_norm, w_out, vocab, dl.CONF_PMAX,
                         dims3["eps"], ws=ws3, stream=stream, temperature=0.8, seed=42, step=0)

    run_head_sample()
    ms3s = timed(run_head_sample, 20)
    lines.append({"config": "3-sample", "workload": "config 3 with temperature 0.8: Gumbel-max draws from counter-based "
                  "SplitMix64 noise in the head's epilogue + probability of the draw + top-4",
                  "value": ms3s * 1e3, "unit": "us/call",
                  "roofline": {"bound": "hbm", "achieved": bytes3 / (ms3s * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                               "frac": bytes3 / (ms3s * 1e-3) / 1e9 / hbm, "algorithmic_bytes": bytes3}})

    # ---- the same head over every masked position of the canvas (block = the whole canvas,
    # 148 rows of which 128 masked): the tensor work per weight byte grows 4.6x
    ws3b = torch.empty(max(dl.lmhead_workspace_bytes(L_CANVAS, vocab, d), 1), dtype=torch.uint8, device="cuda")

    def run_head_all():
        canvas.copy_(canvas0, non_blocking=True)
        dl.lmhead_masked_select(hidden, canvas, dims3["mask_id"], 0, L_CANVAS, K_COMMIT, out_norm, w_out, vocab,
                                dims3["eps"], ws=ws3b, stream=stream)

    run_head_all()
    ms3b = timed(run_head_all, 20)
    flops3b = 2.0 * L_CANVAS * vocab * d
    t_roof3b = max(bytes3 / (hbm * 1e9), flops3b / (tens * 1e12)) * 1e3
    lines.append({"config": "3-all", "workload": "LM head over every masked position: 126464x4096 Q6_K, block = whole "
                  "canvas (148 rows, 128 masked) + confidence + top-4",
                  "value": ms3b * 1e3, "unit": "us/call", "tops": flops3b / (ms3b * 1e-3) / 1e12,
                  "roofline": {"bound": "tensor" if flops3b / (tens * 1e12) > bytes3 / (hbm * 1e9) else "hbm",
                               "t_roof_ms": t_roof3b, "frac": t_roof3b / ms3b,
                               "peak": {"tensor_tflops": tens, "hbm_gbs": hbm}}})

    # ---- the same, ranked by entropy (Dream's ranking): one more partial per (tile, row)
    def run_head_ent():
        canvas.copy_(canvas0, non_blocking=True)
        dl.lmhead_select(hidden, canvas, dims3["mask_id"], 0, L_CANVAS, K_COMMIT, out_norm, w_out, vocab,
                         dl.CONF_NEG_ENTROPY, dims3["eps"], ws=ws3b, stream=stream)

    run_head_ent()
    ms3e = timed(run_head_ent, 20)
    lines.append({"config": "3-all-entropy", "workload": "LM head over every masked position ranked by entropy: "
                  "126464x4096 Q6_K, block = whole canvas (148 rows, 128 masked) + -entropy + top-4",
                  "value": ms3e * 1e3, "unit": "us/call", "tops": flops3b / (ms3e * 1e-3) / 1e12,
                  "roofline": {"bound": "tensor" if flops3b / (tens * 1e12) > bytes3 / (hbm * 1e9) else "hbm",
                               "t_roof_ms": t_roof3b, "frac": t_roof3b / ms3e,
                               "peak": {"tensor_tflops": tens, "hbm_gbs": hbm}}})

    if not args.no_cpu_baseline:
        import oracle as orc

        t0 = time.perf_counter()
        q, dq, _ = orc.quantize_q8k(synth.activations(seed1, m1, k1))
        orc.qgemm(dl.Q4_K, wblk, q, dq)
        ln1["cpu_baseline"] = {"value": 1e3 * (time.perf_counter() - t0), "unit": "ms/GEMM",
                               "cores": orc.num_threads(), "kind": "oracle", "sample": "the whole config"}
        lw = synth.layer_weights(seed2, 0, dims)
        xa = np.asarray(synth.activations(seed2, L_CANVAS, d), np.float64)
        t0 = time.perf_counter()
        orc.layer(lw, xa, dims, attention_on=False)
        lines[1]["cpu_baseline"] = {"value": 1e3 * (time.perf_counter() - t0), "unit": "ms/layer",
                                    "cores": orc.num_threads(), "kind": "oracle", "sample": "one layer at L=148"}
        cv = synth.canvas(seed3)
        t0 = time.perf_counter()
        orc.lmhead_commit(np.asarray(hidden.cpu().numpy(), np.float64), cv, dims3["mask_id"], b0, b1, K_COMMIT,
                          head["out_norm"], head["w_out"], dims3["eps"])
        ln3["cpu_baseline"] = {"value": 1e3 * (time.perf_counter() - t0), "unit": "ms/call",
                                     "cores": orc.num_threads(), "kind": "oracle", "sample": "the whole config"}
    # ---- the step with the inter-step K/V cache: per block one refreshing step and seven
    # block-only steps, against the uncached step on the same model and canvas (32 steps each)
    del w_out
    dims4 = dict(synth.LLADA)
    seed4 = synth.config_seed(4)
    model4 = dl.model_from_seed(dims4, seed4)
    canvas_a = torch.from_numpy(synth.canvas(seed4)).cuda()
    canvas_b = canvas_a.clone()
    start = canvas_a.clone()
    sched, kinds, kind_of = _schedule()
    plain = dl.StepGraphs(model4, canvas_a, kinds)
    cached = dl.CachedStepGraphs(model4, canvas_b, kinds)

    def run_plain():
        for st in range(len(sched)):
            plain.replay(kind_of[st])

    def run_cached():  # a block's first step refreshes the cache
        for st in range(len(sched)):
            cached.replay(kind_of[st], st == 0 or sched[st][0] != sched[st - 1][0])

    def timed_on(st, fn):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        torch.cuda.synchronize()
        dl.check(st)
        return e0.elapsed_time(e1) / 32

    for cv, fn in ((canvas_a, run_plain), (canvas_b, run_cached)):  # warm-up pass each
        cv.copy_(start)
        fn()
    canvas_a.copy_(start)
    ms_plain = timed_on(plain.stream, run_plain)
    canvas_b.copy_(start)
    ms_cached = timed_on(cached.stream, run_cached)
    ga, gb = canvas_a.cpu().numpy(), canvas_b.cpu().numpy()
    gen = slice(PROMPT, PROMPT + GEN)
    lines.append({"config": "4-dual-cache", "workload": "denoising step at L=148 (LLaDA-8B shapes, 32 layers) with the "
                  "inter-step K/V cache: per 32-token block 1 refreshing step + 7 block-only steps (32 rows), 32 steps",
                  "value": ms_cached, "unit": "ms/step", "uncached_ms_per_step": ms_plain,
                  "speedup": ms_plain / ms_cached, "kv_cache_bytes": dl.kv_cache_bytes(model4, L_CANVAS),
                  "divergence": {"tokens_differing_after_32_steps": int((ga[gen] != gb[gen]).sum()),
                                 "generated_tokens": GEN,
                                 "note": "final canvases of the cached and uncached runs from the same start"}})
    del plain, cached, model4

    for ln in lines:
        ln["peak_source"] = peak_src
        print(json.dumps(ln), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-kernel", choices=sorted(ONLY_KERNELS) + ["layer_full", "lm_head"], default=None,
                    help="time one GEMM of the step alone (profiling target) instead of the step")
    ap.add_argument("--configs", action="store_true",
                    help="one JSON line per other configuration (1, 2, 3, 5) instead of the step")
    args = ap.parse_args()
    rank, local_rank, world = _env_dist()
    if args.gpus != world and args.impl == "ours" and not (args.only_kernel or args.configs):
        # N replicas come from the launcher (one process per GPU); a plain run would measure one GPU
        sys.stderr.write(f"bench.py --gpus {args.gpus}: WORLD_SIZE is {world}; launch N > 1 replicas with "
                         f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus "
                         f"{args.gpus} ...\n")
        sys.exit(2)
    if args.only_kernel:
        run_only_kernel(args)
    elif args.configs:
        run_configs(args)
    elif args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
