"""Benchmark of the sparse-depth layer stack on GB300.

Default (the headline): one step = one pass of the whole X-MoD A3K16 stack, the largest
single-GPU configuration (Eq. 3 with N0=2, N1=2, 48 Sparse(K=16) layers per block with
Eq. 7 gating: 2 Dense + (48 Sparse + 1 Dense) x 2 = 100 layers; d=2048, 16 q / 4 kv
heads, head_dim 128, SwiGLU d_ff=5632, B=4 sequences of T=16384 tokens) through the
library's stack entry point. Metric: selected tokens processed by sparse layers per
second (B * T/K * 96 per step), whole job over all ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl xmod|reference]

Other workloads: --workload a4k8_bf16 | mod_bf16 | tiny_fp32 (the same stack step),
--workload routing_bf16 (the routing-only microbench: router + top-(T/K) + gather +
Eq. 7 scatter of a given block output), --pass bwd (the backward of every layer).

Under torchrun every rank runs its own B sequences (sequences are independent;
no data-path collective), the timing is the max over ranks.
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

from sparse_depth_token_gb300 import inputs as I  # noqa: E402

METRIC = "selected tokens/s per X-MoD sparse-layer fwd (bf16, 1xGB300); % HBM / tensor roofline"
UNIT = "selected tokens/s"
WORKLOAD = "a3k16_bf16"
ABI_NAMES = {"w_r": "w_router", "g1": "rms1", "wq": "wq", "wk": "wk", "wv": "wv", "wo": "wo",
             "g2": "rms2", "wg": "w_gate", "wu": "w_up", "wd": "w_down"}


DENSE, SPARSE, ATTN, RFFN, FULLKV = 0, 1, 2, 3, 4   # the library's layer kinds
VARIANT = "xmod"   # set from --variant before any schedule is built
ONLY = None        # --only: a stack of one layer kind (profiling), set before any schedule
ONLY_LAYERS = {"sparse": 16, "dense": 2}


def schedule(w: I.Workload, variant=None):
    """Layer kinds in execution order. xmod: the Eq. 3 stack; routed_ffn: the Routed-FFN
    control (([FullAttn] + [Routed-FFN] x K) x A between the anchors); fullkv: the
    Selected-Q / full-KV control (the Eq. 3 stack with full-sequence keys and values)."""
    variant = variant or VARIANT
    if ONLY is not None:   # one kind only, at the workload's shapes
        return [SPARSE if ONLY == "sparse" else DENSE] * ONLY_LAYERS[ONLY]
    ak = int(round(w.A * w.K))
    if variant == "routed_ffn":
        A = ak // w.K
        return [DENSE] * w.N0 + (([ATTN] + [RFFN] * w.K) * A + [DENSE]) * w.N1
    sp = FULLKV if variant == "fullkv" else SPARSE
    return [DENSE] * w.N0 + ([sp] * ak + [DENSE]) * w.N1


def routed(k) -> bool:
    return k in (SPARSE, RFFN, FULLKV)


def workload_config(w: I.Workload) -> dict:
    kinds = schedule(w)
    n_routed = sum(1 for k in kinds if routed(k))
    if ONLY is not None:
        what = f"{len(kinds)} {ONLY} layers only (profiling stack)"
    elif VARIANT == "routed_ffn":
        what = (f"Routed-FFN control {n_routed} Routed-FFN(K={w.K}) + {kinds.count(ATTN)} "
                f"FullAttn + {kinds.count(DENSE)} Dense")
    elif VARIANT == "fullkv":
        what = f"Selected-Q/full-KV control {n_routed} Sparse(K={w.K}) + {kinds.count(DENSE)} Dense"
    else:
        what = f"X-MoD stack {n_routed} Sparse(K={w.K}) + {kinds.count(DENSE)} Dense"
    return {
        "workload": f"{w.name}: {what} "
                    + ("" if ONLY is not None else f"(Eq. 3, N0={w.N0}, N1={w.N1}, A={w.A}), ")
                    + f"Eq. "
                    f"{'7' if w.gate == 0 else '6'} gating, d={w.d}, {w.hq}/{w.hkv} heads, "
                    f"head_dim {w.hd}, SwiGLU d_ff={w.F}",
        "B_per_gpu": w.B, "T": w.T, "K": w.K,
        "selected_tokens_per_step_per_gpu": n_routed * w.B * (w.T // w.K),
        "l2": l2_note(w),
        "inputs": "seeded synthetic: x~N(0,1), matrices~N(0,0.02^2), w_r~N(0,1/d), "
                  + (f"bias~N(0,{w.bias_std}^2), " if w.bias_std else "no router bias, ")
                  + ("varsigma~U(0.5,1.5), " if w.gate == 0 else "")
                  + "RMSNorm gains 1",
    }


def l2_note(w: I.Workload) -> str:
    """Why the timed steps need no L2 flush: the distinct bytes one step streams."""
    es = 2 if w.dtype == "bf16" else 4
    per_layer = es * (w.d * (w.hq + 2 * w.hkv) * w.hd + w.hq * w.hd * w.d + 3 * w.d * w.F + w.d)
    weights = per_layer * len(schedule(w))
    stream = es * w.B * w.T * w.d
    if weights + stream > 2 * 129e6:
        return (f"no flush: one step streams {weights / 1e9:.1f} GB of distinct layer weights "
                f"and a {stream / 1e6:.0f} MB stream, both larger than the 129 MB L2"
                if stream > 129e6 else
                f"no flush: one step streams {weights / 1e9:.1f} GB of distinct layer weights "
                f"(the 129 MB L2 holds under a tenth of a step's bytes)")
    return "no flush: a latency-bound tiny step (its bytes fit in L2)"


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def algorithmic_work(w: I.Workload, sel_counts=None) -> dict:
    """Algorithmic FLOPs (tensor kinds) or bytes (memory kinds) per step, per kernel kind.
    Sparse layers count only the selected tokens; attention is causal (half the square).
    sel_counts [n_sparse, B]: tokens each sparse layer routed per sequence (threshold
    routing); None: T / K each."""
    es = 2 if w.dtype == "bf16" else 4
    out = {}

    def add(kind, v):
        out[kind] = out.get(kind, 0.0) + float(v)

    kinds = schedule(w)
    run_left = 0   # layers left in the current run of sparse layers (logits kept current)
    ls = 0
    for l, kind in enumerate(kinds):
        sparse = routed(kind)
        n = w.T // w.K if sparse else w.T
        M = w.B * n
        ns = [n] * w.B
        if sparse and sel_counts is not None:
            ns = [int(v) for v in sel_counts[ls]]
            M = sum(ns)
        if sparse:
            ls += 1
        if sparse:
            if run_left == 0:   # one pass over the stream: logits of up to 32 layers
                run = 1
                while run < ROUTER_RUN and l + run < len(kinds) and kinds[l + run] == kind:
                    run += 1
                run_left = run
                add("router", w.B * w.T * w.d * es + 4 * run * w.B * w.T)
            run_left -= 1
            if run_left > 0:    # logits of the updated rows for the rest of the run
                add("router_refresh", M * w.d * es + 4 * run_left * M)
            add("topk", 4 * w.B * w.T + 8 * M)
        if kind == RFFN:   # FFN half only: RMSNorm2 fused into the gather
            add("gather_rmsnorm", 2 * M * w.d * es)
            add("gemm_gate_up_swiglu", 4 * M * w.d * w.F)
            add("gemm_down_scatter", 2 * M * w.F * w.d)
            continue
        if kind == FULLKV:   # every token's RMSNorm1 and k, v; q for the selected
            BT = w.B * w.T
            add("gather_rmsnorm", 2 * (BT + M) * w.d * es)
            add("gemm_qkv", 2 * BT * w.d * 2 * w.hkv * w.hd + 2 * M * w.d * w.hq * w.hd)
            # a query at position p sees p + 1 keys: T / 2 on average
            add("attention", 4 * M * (w.T / 2) * w.hd * w.hq)
        else:
            add("gather_rmsnorm", 2 * M * w.d * es)
            add("gemm_qkv", 2 * M * w.d * (w.hq + 2 * w.hkv) * w.hd)
            add("attention", 2 * sum(v * v for v in ns) * w.hd * w.hq)
        add("gemm_o_residual", 2 * M * w.hq * w.hd * w.d)
        if kind == ATTN:
            continue
        add("rmsnorm2", M * w.d * (4 + es))
        add("gemm_gate_up_swiglu", 4 * M * w.d * w.F)
        add("gemm_down_scatter", 2 * M * w.F * w.d)
    return out


# Sparse layers whose router logits one pass over the stream computes (the library's
# run length; later layers of a run only refresh the logits of the rows that changed).
ROUTER_RUN = 32

TENSOR_KINDS = {"gemm_qkv", "attention", "gemm_o_residual", "gemm_gate_up_swiglu",
                "gemm_down_scatter"}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a bench
# line's dominant kernel, from one ncu capture of that kernel in that configuration, with
# the summary that records it; used only while the kernel is unchanged and the run is
# the captured configuration. Key: (workload, B, variant / routing tag, kernel kind).
RECORDED_TRAFFIC = {
    # the gate/up launches of one step, mean: A3K16 (96 sparse layers + 4 dense), A4K8
    # (32 sparse layers + the dense one)
    ("a3k16_bf16", 4, "xmod", "gemm_gate_up_swiglu"):
        (137.35e6, "profiles/gemm_gate_up_dram.md"),
    ("a4k8_bf16", 8, "xmod", "gemm_gate_up_swiglu"):
        (52.54e6, "profiles/gemm_gate_up_dram.md"),
    # the router's x read + logits write at B = 8, scaled by 8 to B = 64 (x is read once)
    ("routing_bf16", 64, "routing", "router"):
        (8 * 540.3e6, "profiles/routing_kernels_c2_microbench.md"),
}


def recorded_traffic(w: I.Workload, tag: str, kernel: str):
    return RECORDED_TRAFFIC.get((w.name, w.B, tag, kernel), (None, None))


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------- CPU oracle baseline

def oracle_sample(w: I.Workload, budget_s: float = 15.0, max_reps: int = 50,
                  row_frac: float = 1.0):
    """The CPU oracle on a bounded sample of the workload: one sparse layer of the stack
    (layer 0 weights) on sequence 0 of the batch, repeated until `budget_s` elapses.
    row_frac < 1: only the selected tokens in the first row_frac of the positions are
    computed (the router and top-k still cover the whole sequence; keys and values up
    to the last wanted row); the tokens counted are those rows.
    Returns (selected tokens/s, threads, description)."""
    import oracle as O
    lw = I.layer_weights(w, 0)
    L = O.Layer({k: I.to_f64(v, w.dtype) for k, v in lw.items() if k in ABI_NAMES},
                lw["varsigma"])
    w1 = w.replace(B=1)
    x = I.to_f64(I.residual_stream(w1), w.dtype)
    bias = I.router_bias(w1)
    dm = O.dims(1, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    n = w.T // w.K
    kind = {"routed_ffn": O.RFFN, "fullkv": O.FULLKV}.get(VARIANT, O.SPARSE)
    mask, counted, what = None, n, f"n={n} selected"
    if row_frac < 1.0 and kind != O.FULLKV:
        cut = int(w.T * row_frac)
        mask = (np.arange(w.T) < cut).astype(np.int32)[None, :]
        idx = O.topk(O.router(x, L.arrays["w_r"], bias)[0], n)   # the layer's own selection
        counted = int((idx[0] < cut).sum())
        what = f"the {counted} of its n={n} selected tokens before position {cut}"
    reps, t0 = 0, time.perf_counter()
    while True:
        O.layer_fwd(dm, kind, w.K, w.gate, L, x, bias=bias, row_mask=mask)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    return reps * counted / el, O.num_threads(), (
        f"one Sparse(K={w.K}) layer on 1 of the {w.B} sequences (T={w.T}, {what}), "
        f"{reps} repetition(s) in {el:.1f} s")


def single_thread_variant(sample_fn, budget_s: float) -> dict:
    """The same oracle sample on one host thread (OpenMP limited to 1), then the thread
    count restored: the single-thread variant of the oracle timing."""
    import oracle as O
    cores = O.num_threads()
    O.set_num_threads(1)
    try:
        v, _, sample = sample_fn(budget_s)
    finally:
        O.set_num_threads(cores)
    return {"value": v, "cores": 1, "sample": sample}


def run_reference(args):
    """--impl reference: the oracle as it stands, timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = I.WORKLOADS[args.workload]
    import oracle as O
    lw = I.layer_weights(w, 0)
    L = O.Layer({k: I.to_f64(v, w.dtype) for k, v in lw.items() if k in ABI_NAMES},
                lw["varsigma"])
    w1 = w.replace(B=1)
    x = I.to_f64(I.residual_stream(w1), w.dtype)
    bias = I.router_bias(w1)
    dm = O.dims(1, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    n = w.T // w.K

    def step():
        O.layer_fwd(dm, {"routed_ffn": O.RFFN, "fullkv": O.FULLKV}.get(VARIANT, O.SPARSE), w.K,
                    w.gate, L, x, bias=bias)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * n / el
    sample = (f"each step: one Sparse(K={w.K}) layer of the workload on 1 of its {w.B} "
              f"sequences (n={n} selected tokens)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.num_threads(),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- GPU arm

def run_xmod(args):
    import torch
    from sparse_depth_token_gb300 import xmod as X

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    X.load()

    w = I.WORKLOADS[args.workload]
    kinds = schedule(w)
    n_sparse = sum(1 for k in kinds if routed(k))
    sel_per_step = n_sparse * w.B * (w.T // w.K)
    # per-rank data: the same weights, different sequences
    wr = w.replace(seed=w.seed + 1000 * rank) if rank else w
    layers = I.all_layer_weights(w, len(kinds))
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def to_dev(a):
        if w.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    dev_layers = [{ABI_NAMES[k]: to_dev(v) for k, v in l.items() if k in ABI_NAMES} for l in layers]
    if args.qwen3:   # QK-norm (unit gains) and RoPE at the tokens' original positions
        ones = to_dev(np.ones(w.hd, np.float32) if w.dtype != "bf16" else
                      I.f32_to_bf16_bits(np.ones(w.hd, np.float32)))
        for dl in dev_layers:
            dl["q_norm"] = dl["k_norm"] = ones
    theta = 1e6 if args.qwen3 else 0.0
    abi = [X.layer_weights(d, l["varsigma"], theta) for d, l in zip(dev_layers, layers)]
    x_host = I.residual_stream(wr)
    bias_host = I.router_bias(wr)
    x0 = to_dev(x_host)
    x = torch.empty_like(x0)
    bias = torch.from_numpy(bias_host).to(dev) if bias_host is not None else None
    dm = X.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, X.BF16 if w.dtype == "bf16" else X.FP32,
                w.eps)
    ws = torch.zeros(X.workspace_bytes(dm, w.K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    plain = args.routing == "topk" and args.bias_step == 0.0

    def run_stack(stats=None, xb=None, bb=None):
        xb = x if xb is None else xb
        bb = bias if bb is None else bb
        if VARIANT != "xmod" or ONLY is not None:
            X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xb, bb, ws,
                              bias_step=args.bias_step, layer_stats=stats,
                              routing=X.ROUTE_THRESHOLD if args.routing == "threshold"
                              else X.ROUTE_TOPK, stream=stream)
        elif plain and stats is None:
            X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xb, bb, ws, stream)
        else:
            X.stack_fwd_ex(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xb, bb, ws,
                           bias_step=args.bias_step, layer_stats=stats,
                           routing=X.ROUTE_THRESHOLD if args.routing == "threshold" else X.ROUTE_TOPK,
                           stream=stream)

    def step():
        x.copy_(x0, non_blocking=True)
        run_stack()

    sel_counts = None
    if not plain:
        # tokens each sparse layer routes (the same every step: the input is restored)
        stats = torch.zeros((n_sparse, w.B, 4), dtype=torch.int32, device=dev)
        x.copy_(x0)
        run_stack(stats)
        sel_counts = stats[:, :, 0].cpu().numpy()
        sel_per_step = int(sel_counts.sum())

    def barrier():
        if dist is not None:
            dist.barrier()

    X.reset_status(ws)
    for _ in range(max(args.warmup, 3)):
        step()
    st = X.sync_status(ws)
    if st != X.OK:
        raise RuntimeError(f"device status after warm-up: {X.status_string(st)}")

    # ---- timed region
    clocks = ClockSampler(local if world > 1 else 0)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = X.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = (X.launch_count() - launches0) // args.steps
    clock_info = clocks.stop()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = ms
    if dist is not None:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    value = world * sel_per_step / (ms_max / 1e3)

    # ---- profiled pass: per-kernel CUDA-event times on the launching stream
    X.profile_read()
    X.profile_enable(True)
    prof_steps = max(1, min(args.steps, 3))
    e0.record(stream)
    for _ in range(prof_steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    prof_ms = e0.elapsed_time(e1)
    X.profile_enable(False)
    prof = X.profile_read()
    work = algorithmic_work(w, sel_counts)
    peaks = measured_peaks()
    total_ms = sum(v[1] for v in prof.values())
    kernels = {}
    for kind, (cnt, kms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        per_step_ms = kms / prof_steps
        wk = work.get(kind)
        entry = {"launches_per_step": cnt // prof_steps, "ms_per_step": per_step_ms,
                 "share": kms / total_ms if total_ms else None}
        if wk is not None and kms > 0:
            if kind in TENSOR_KINDS:
                entry["tflops"] = wk / (per_step_ms / 1e3) / 1e12
            else:
                entry["gbs"] = wk / (per_step_ms / 1e3) / 1e9
        kernels[kind] = entry
    top = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roofline = None
    if top is not None and top in work:
        cnt, kms = prof[top]
        if top in TENSOR_KINDS:
            ach = work[top] / (kms / prof_steps / 1e3) / 1e12
            peak = peaks["bf16_tflops"]
            tag = "xmod" if (VARIANT == "xmod" and plain and not args.qwen3) else "other"
            traffic, tsrc = recorded_traffic(w, tag, top)
            roofline = {"kernel": top, "bound": "tensor", "achieved": ach, "peak": peak,
                        "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic,
                        "peak_source": f"{peaks['source']} bf16 burst (the kernel is timed "
                                       f"in a profiled pass of {prof_steps} step(s), "
                                       f"{prof_ms:.0f} ms: not a seconds-long run)",
                        "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                        "algorithmic_per_launch": work[top] / (cnt / prof_steps)}
            if tsrc:
                roofline["traffic_source"] = tsrc
        else:
            ach = work[top] / (kms / prof_steps / 1e3) / 1e9
            peak = peaks["hbm_gbs"]
            roofline = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peak,
                        "unit": "GB/s", "frac": ach / peak, "traffic": None,
                        "peak_source": f"{peaks['source']} HBM copy",
                        "algorithmic_per_launch": work[top] / (cnt / prof_steps)}
    step_flops = sum(v for k, v in work.items() if k in TENSOR_KINDS)

    # ---- end to end through the C ABI call with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(np.ascontiguousarray(x_host).view(np.int16)).view(torch.bfloat16) \
            if w.dtype == "bf16" else torch.from_numpy(x_host)
        xh = xh.pin_memory()
        out_h = torch.empty_like(xh).pin_memory()
        bh = torch.from_numpy(bias_host).pin_memory() if bias_host is not None else None

        def e2e_step():
            x.copy_(xh, non_blocking=True)
            if bh is not None:
                bias.copy_(bh, non_blocking=True)
            run_stack()
            out_h.copy_(x, non_blocking=True)

        for _ in range(2):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1) / args.steps
        if dist is not None:
            t = torch.tensor([ems], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())
        e2e_serial = {"value": world * sel_per_step / (ems / 1e3), "unit": UNIT,
                      "ms_per_step": ems,
                      "transfers": "serial: copy in, stack, copy out on one stream"}

        # Double-buffered, as a serving loop would run it: step i computes on buffer
        # i % 2 while one copy stream brings in step i+1's input (pinned host -> device)
        # and another takes out step i's result once it is done (device -> pinned host).
        # Every step still copies its whole input in and its whole result out.
        x2 = [x, torch.empty_like(x)]
        b2 = [bias, torch.empty_like(bias) if bias is not None else None]
        outs = [out_h, torch.empty_like(xh).pin_memory()]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def h2d(k):
            s_in.wait_event(ev_out[k])   # buffer k's previous result has left
            with torch.cuda.stream(s_in):
                x2[k].copy_(xh, non_blocking=True)
                if bh is not None:
                    b2[k].copy_(bh, non_blocking=True)
            ev_in[k].record(s_in)

        def pipelined(nsteps, t0=None, t1=None):
            if t0 is not None:
                t0.record(stream)
                s_in.wait_event(t0)
            h2d(0)
            for i in range(nsteps):
                k = i & 1
                stream.wait_event(ev_in[k])
                run_stack(xb=x2[k], bb=b2[k])
                ev_done[k].record(stream)
                if i + 1 < nsteps:
                    h2d(1 - k)
                s_out.wait_event(ev_done[k])
                with torch.cuda.stream(s_out):
                    outs[k].copy_(x2[k], non_blocking=True)
                ev_out[k].record(s_out)
            stream.wait_event(ev_out[(nsteps - 1) & 1])
            if t1 is not None:
                t1.record(stream)

        pipelined(3)
        barrier()
        torch.cuda.synchronize()
        pipelined(args.steps, e0, e1)
        torch.cuda.synchronize()
        pms = e0.elapsed_time(e1) / args.steps
        if dist is not None:
            t = torch.tensor([pms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            pms = float(t.item())
        e2e = {"value": world * sel_per_step / (pms / 1e3), "unit": UNIT,
               "ms_per_step": pms,
               "h2d_bytes_per_step": int(xh.numel() * xh.element_size() +
                                         (bh.numel() * 4 if bh is not None else 0)),
               "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()),
               "transfers": "double-buffered: step i+1's input copy and step i's result copy "
                            "run on their own streams while step i computes",
               "serial": e2e_serial}
    st = X.sync_status(ws)
    if st != X.OK:
        raise RuntimeError(f"device status after the run: {X.status_string(st)}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_sample(w, budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "cpu_model": cpu_model(),
               "kind": "oracle", "sample": sample,
               "single_thread": single_thread_variant(
                   lambda bs: oracle_sample(w, budget_s=bs, max_reps=1,
                                            row_frac=min(1.0, 256 / (w.T // w.K))),
                   args.cpu_budget / 3)}

    if rank == 0:
        cfg = workload_config(w)
        cfg["parallelism"] = f"replicas x{world} (sequences sharded, no collective)"
        if VARIANT != "xmod":
            cfg["variant"] = VARIANT
        if args.qwen3:
            cfg["attention"] = "QK-norm + RoPE (theta 1e6) at original positions"
        if not plain:
            cfg["routing"] = args.routing
            cfg["bias_step"] = args.bias_step
            cfg["selected_tokens_per_step_per_gpu"] = sel_per_step
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "fp32",
                "data": "synthetic (seeded; random-init weights)", "config": cfg,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches) * args.steps,
                "gpu_launches_per_step": int(launches),
                "clocks": clock_info,
                "step_tflops": step_flops / (ms_max / 1e3) / 1e12,
                "kernels": kernels}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------- backward pass

BWD_METRIC = "selected tokens/s per X-MoD sparse-layer bwd (bf16, 1xGB300); % tensor roofline"


def backward_work(w: I.Workload) -> dict:
    """Algorithmic FLOPs per backward step (every layer of the stack once, in reverse):
    the forward each layer recomputes, the activation- and weight-gradient GEMMs (each
    as many FLOPs as the forward projection) and the attention backward (S recomputed,
    dP, dV, dQ, dK: five causal n x n x head_dim products per head)."""
    out = {}

    def add(kind, v):
        out[kind] = out.get(kind, 0.0) + float(v)

    qw, kw = w.hq * w.hd, w.hkv * w.hd
    BT = w.B * w.T
    es = 2 if w.dtype == "bf16" else 4

    def r8(v):
        return (v + 7) // 8 * 8

    def tr(R, Rpad, C, e=es):   # one transpose: R x C read, C x Rpad written (zero padding)
        return e * (R * C + C * Rpad)

    for kind in schedule(w):
        n = w.T // w.K if routed(kind) else w.T
        M = w.B * n
        Mp = r8(M)
        proj = 0
        # the transposes that feed the gradient GEMMs token-contiguous operands (bytes)
        tb = 0
        if kind != ATTN:   # df, H, W_down, [dG | dU], v2, W_gate, W_up
            tb += tr(M, Mp, w.d) + tr(M, Mp, w.F) + tr(w.d, w.d, w.F) + tr(M, Mp, 2 * w.F)
            tb += tr(M, Mp, w.d) + 2 * tr(w.F, w.F, w.d)
        if kind != RFFN:   # da, o, W_o; the attention backward's per-sequence transposes
            tb += tr(M, Mp, w.d) + tr(M, Mp, qw) + tr(w.d, w.d, qw)
            nk = w.T if kind == FULLKV else n
            tb += w.B * (tr(nk, nk, kw) + 2 * tr(n, n, qw) + tr(n, n, w.hq, 4))
            if kind == FULLKV:   # dq, u_sel, W_q; [dk | dv], u of every token, W_k, W_v
                tb += tr(M, Mp, qw) + tr(M, Mp, w.d) + tr(qw, qw, w.d)
                tb += tr(BT, r8(BT), 2 * kw) + tr(BT, r8(BT), w.d) + 2 * tr(kw, kw, w.d)
            else:                # [dq | dk | dv], u, W_q, W_k, W_v
                tb += tr(M, Mp, qw + 2 * kw) + tr(M, Mp, w.d) + tr(qw, qw, w.d)
                tb += 2 * tr(kw, kw, w.d)
        add("bwd_transpose", tb)
        if kind != RFFN:   # the attention half
            if kind == FULLKV:   # k, v of every token; a query at position p sees p + 1 keys
                qkv = 2 * BT * w.d * 2 * kw + 2 * M * w.d * qw
                att = 2 * M * (w.T / 2) * w.hd * w.hq    # one product, T / 2 keys on average
            else:
                qkv = 2 * M * w.d * (qw + 2 * kw)
                att = w.B * n * n * w.hd * w.hq          # one causal n x n x hd product
            add("gemm_qkv", qkv)
            add("attention", 2 * att)
            add("gemm_o_residual", 2 * M * qw * w.d)
            add("bwd_attention", 5 * att)
            proj += qkv + 2 * M * qw * w.d
        if kind != ATTN:   # the FFN half
            add("gemm_gate_up", 4 * M * w.d * w.F)
            add("gemm_down", 2 * M * w.F * w.d)
            proj += 6 * M * w.d * w.F
        add("bwd_gemm_dw", proj)
        add("bwd_gemm_dx", proj)
    return out


BWD_TENSOR_KINDS = {"gemm_qkv", "attention", "gemm_o_residual", "gemm_gate_up", "gemm_down",
                    "bwd_gemm_dw", "bwd_gemm_dx", "bwd_attention"}


def run_backward(args):
    """--pass bwd: the backward of the whole stack, layer by layer in reverse
    (xmod_layer_bwd, Eq. 9 coefficient 1e-4 as the pages chose), from the layer inputs a
    forward pass stored, with a synthetic upstream gradient dy ~ N(0, 1) at the top. One
    step = every layer's backward once; the weight gradients of a layer are written to
    one shared set of fp32 buffers (a trainer would keep one set per layer)."""
    import torch
    from sparse_depth_token_gb300 import xmod as X

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    X.load()
    w = I.WORKLOADS[args.workload]
    kinds = schedule(w)
    n_routed = sum(1 for k in kinds if routed(k))
    sel_per_step = n_routed * w.B * (w.T // w.K)
    layers = I.all_layer_weights(w, len(kinds))

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    dev_layers = [{ABI_NAMES[k]: to_dev(v) for k, v in l.items() if k in ABI_NAMES} for l in layers]
    abi = [X.layer_weights(d, l["varsigma"]) for d, l in zip(dev_layers, layers)]
    bias_host = I.router_bias(w)
    bias = torch.from_numpy(bias_host).to(dev) if bias_host is not None else None
    dm = X.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, X.BF16, w.eps)
    # the layer inputs of one forward pass
    ws_f = torch.zeros(X.workspace_bytes(dm, w.K), dtype=torch.uint8, device=dev)
    xs = [to_dev(I.residual_stream(w))]
    for l, kind in enumerate(kinds):
        x = xs[-1].clone()
        X.layer_fwd(dm, kind, w.K, w.gate, abi[l], x, bias if routed(kind) else None, None,
                    None, ws_f)
        xs.append(x)
    del ws_f
    ws = torch.zeros(X.bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    dy_top = torch.randn(xs[0].shape, generator=g, device=dev).to(torch.bfloat16)
    dbuf = [torch.empty_like(dy_top), torch.empty_like(dy_top)]
    qw, kw = w.hq * w.hd, w.hkv * w.hd
    shapes = {"w_router": (w.d,), "rms1": (w.d,), "wq": (qw, w.d), "wk": (kw, w.d),
              "wv": (kw, w.d), "wo": (w.d, qw), "rms2": (w.d,), "w_gate": (w.F, w.d),
              "w_up": (w.F, w.d), "w_down": (w.d, w.F), "varsigma": (4,), "route_loss": (4,)}
    gd = {k: torch.empty(v, dtype=torch.float32, device=dev) for k, v in shapes.items()}
    grads = X.layer_grads(gd)
    stream = torch.cuda.current_stream()
    coef = 1e-4

    def step():
        dy = dy_top
        for l in range(len(kinds) - 1, -1, -1):
            dx = dbuf[l & 1]
            X.layer_bwd(dm, kinds[l], w.K, w.gate, abi[l], xs[l],
                        bias if routed(kinds[l]) else None, dy, coef, dx, grads, ws, stream)
            dy = dx

    X.reset_status(ws)
    for _ in range(max(args.warmup, 3)):
        step()
    st = X.sync_status(ws)
    if st != X.OK:
        raise RuntimeError(f"device status after warm-up: {X.status_string(st)}")
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = X.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = (X.launch_count() - launches0) // args.steps
    clock_info = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    X.profile_read()
    X.profile_enable(True)
    prof_steps = max(1, min(args.steps, 2))
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize()
    X.profile_enable(False)
    prof = X.profile_read()
    st = X.sync_status(ws)
    if st != X.OK:
        raise RuntimeError(f"device status after the run: {X.status_string(st)}")
    work = backward_work(w)
    peaks = measured_peaks()
    total_ms = sum(v[1] for v in prof.values())
    kernels = {}
    for kind, (cnt, kms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        pms = kms / prof_steps
        e = {"launches_per_step": cnt // prof_steps, "ms_per_step": pms,
             "share": kms / total_ms if total_ms else None}
        if kind in work and pms > 0:
            if kind in BWD_TENSOR_KINDS:
                e["tflops"] = work[kind] / (pms / 1e3) / 1e12
            else:
                e["gbs"] = work[kind] / (pms / 1e3) / 1e9
        kernels[kind] = e
    top = max(prof.items(), key=lambda kv: kv[1][1])[0]
    roofline = None
    if top in work:
        cnt, kms = prof[top]
        if top in BWD_TENSOR_KINDS:
            ach = work[top] / (kms / prof_steps / 1e3) / 1e12
            peak = peaks["bf16_tflops"]
            roofline = {"kernel": top, "bound": "tensor", "achieved": ach, "peak": peak,
                        "unit": "TFLOP/s", "frac": ach / peak, "traffic": None,
                        "peak_source": f"{peaks['source']} bf16 burst (profiled pass of "
                                       f"{prof_steps} step(s))",
                        "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                        "algorithmic_per_launch": work[top] / (cnt / prof_steps)}
        else:   # data movement (the transposes): compulsory bytes over the HBM copy rate
            ach = work[top] / (kms / prof_steps / 1e3) / 1e9
            peak = peaks["hbm_gbs"]
            roofline = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peak,
                        "unit": "GB/s", "frac": ach / peak, "traffic": None,
                        "peak_source": f"{peaks['source']} HBM copy",
                        "algorithmic_per_launch": work[top] / (cnt / prof_steps)}
    cfg = workload_config(w)
    cfg["pass"] = "backward of every layer (xmod_layer_bwd, forward recomputed inside), " \
                  "Eq. 9 coefficient 1e-4, synthetic upstream gradient dy~N(0,1)"
    print(json.dumps({
        "metric": BWD_METRIC, "value": sel_per_step / (ms / 1e3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights)", "config": cfg,
        "roofline": roofline, "gpu_launches": int(launches) * args.steps,
        "gpu_launches_per_step": int(launches), "clocks": clock_info,
        "step_tflops": sum(v for k, v in work.items() if k in BWD_TENSOR_KINDS) / (ms / 1e3) / 1e12,
        "kernels": kernels}), flush=True)


# ---------------------------------------------------------------------- routing microbench

ROUTING_KS = (2, 8, 16)
ROUTING_HEADLINE_K = 8


def routing_work(w: I.Workload, K: int) -> dict:
    """Compulsory HBM bytes per step of the routing-only pipeline, per kernel kind: the
    router reads x once and writes the logits; top-k reads the logits and writes idx and
    the gates; the gather reads and writes M rows; the scatter reads a+f and the x rows
    and writes the x rows."""
    es = 2 if w.dtype == "bf16" else 4
    BT, M = w.B * w.T, w.B * (w.T // K)
    return {"router": BT * w.d * es + 4 * BT,
            "topk": 4 * BT + 8 * M,
            "gather": 2 * M * w.d * es + 4 * M,
            "gated_scatter": 3 * M * w.d * es + 8 * M}


def routing_config(w: I.Workload, K: int) -> dict:
    return {
        "workload": f"{w.name}: routing-only microbench (router GEMV + top-(T/K) + gather + "
                    f"Eq. 7 gated scatter of a given block output a+f~N(0,1)), "
                    f"B={w.B}, T={w.T}, d={w.d}, K={K}",
        "B_per_gpu": w.B, "T": w.T, "d": w.d, "K": K,
        "selected_tokens_per_step_per_gpu": w.B * (w.T // K),
        "l2": f"no flush: x is {w.B * w.T * w.d * 2 / 1e9:.2f} GB, far above the 129 MB L2",
        "inputs": "seeded synthetic: x~N(0,1), w_r~N(0,1/d), bias 0, a+f~N(0,1), varsigma 1",
    }


def oracle_routing_sample(w: I.Workload, K: int, budget_s: float = 15.0, max_reps: int = 5000):
    """The oracle's router, top-k, gather and Eq. 7 scatter on one sequence of the
    workload, repeated until `budget_s` elapses. Returns (selected tokens/s, threads,
    description)."""
    import oracle as O
    w1 = w.replace(B=1)
    n = w.T // K
    x = I.to_f64(I.residual_stream(w1), w.dtype).reshape(w.T, w.d)
    w_r = I.to_f64(I.layer_weights(w1, 0)["w_r"], w.dtype)
    af = I.to_f64(I.given_block_output(w1, n), w.dtype)
    reps, t0 = 0, time.perf_counter()
    while True:
        s, r = O.router(x[None], w_r)
        idx = O.topk(s, n)[0]
        xs = x[idx]                                   # the position-ordered gather
        O.gated_scatter(x, idx, af, None, r[0, idx], 1.0, O.GATE_XMOD)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    del xs
    return reps * n / el, O.num_threads(), (
        f"router + top-{n} + gather + Eq. 7 scatter on 1 of the {w.B} sequences "
        f"(T={w.T}, d={w.d}, K={K}), {reps} repetition(s) in {el:.1f} s")


def run_routing_reference(args):
    """--impl reference on the routing microbench: the oracle, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = I.WORKLOADS[args.workload]
    K = args.K or ROUTING_HEADLINE_K
    import oracle as O
    n = w.T // K
    w1 = w.replace(B=1)
    x = I.to_f64(I.residual_stream(w1), w.dtype).reshape(w.T, w.d)
    w_r = I.to_f64(I.layer_weights(w1, 0)["w_r"], w.dtype)
    af = I.to_f64(I.given_block_output(w1, n), w.dtype)

    def step():
        s, r = O.router(x[None], w_r)
        idx = O.topk(s, n)[0]
        _ = x[idx]
        O.gated_scatter(x, idx, af, None, r[0, idx], 1.0, O.GATE_XMOD)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * n / el
    sample = (f"each step: router + top-{n} + gather + Eq. 7 scatter on 1 of the workload's "
              f"{w.B} sequences (T={w.T}, d={w.d})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": routing_config(w, K),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.num_threads(),
                         "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_routing(args):
    """The routing-only microbench: per step, xmod_router_topk (router GEMV + top-(T/K)),
    xmod_gather and xmod_gated_scatter (Eq. 7, varsigma 1) of a given block output a+f,
    on the B x T x d stream, which the scatter updates in place. K = 8 is the headline;
    K = 2 and 16 are timed too and reported under "sweep"."""
    import torch
    from sparse_depth_token_gb300 import xmod as X

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    X.load()
    w = I.WORKLOADS[args.workload]
    wr = w.replace(seed=w.seed + 1000 * rank) if rank else w
    Ks = [args.K] if args.K else list(ROUTING_KS)
    head_K = args.K or ROUTING_HEADLINE_K

    def bf16_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    x_host = I.residual_stream(wr)
    x = bf16_dev(x_host)
    w_r = bf16_dev(I.layer_weights(w, 0)["w_r"])
    M_max = w.B * (w.T // min(Ks))
    af_host = I.given_block_output(wr, M_max)
    af_all = bf16_dev(af_host)
    # the block's widths do not enter the routing kernels: one head of 8, d_ff 8
    dm = X.dims(w.B, w.T, w.d, 1, 1, 8, 8, X.BF16, w.eps)
    ws = torch.zeros(X.workspace_bytes(dm, min(Ks)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(ms):
        if dist is None:
            return ms
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    results = {}
    for K in Ks:
        n = w.T // K
        M = w.B * n
        idx = torch.empty((w.B, n), dtype=torch.int32, device=dev)
        r_sel = torch.empty((w.B, n), dtype=torch.float32, device=dev)
        logits = torch.empty((w.B, w.T), dtype=torch.float32, device=dev)
        xs = torch.empty((M, w.d), dtype=torch.bfloat16, device=dev)
        af = af_all[:M]

        def step():
            X.router_topk(dm, K, x, w_r, None, logits, None, idx, r_sel, ws, stream)
            X.gather(dm, K, x, idx, xs, stream)
            X.gated_scatter(dm, K, x, idx, r_sel, af, None, 1.0, X.GATE_XMOD, stream)

        X.reset_status(ws)
        for _ in range(max(args.warmup, 3)):
            step()
        st = X.sync_status(ws)
        if st != X.OK:
            raise RuntimeError(f"device status after warm-up: {X.status_string(st)}")
        clocks = ClockSampler(local if world > 1 else 0)
        barrier()
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)
        launches0 = X.launch_count()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        launches = (X.launch_count() - launches0) // args.steps
        clock_info = clocks.stop()
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)

        # per-kernel CUDA-event times on the launching stream
        X.profile_read()
        X.profile_enable(True)
        prof_steps = max(1, min(args.steps, 5))
        for _ in range(prof_steps):
            step()
        torch.cuda.synchronize()
        X.profile_enable(False)
        prof = X.profile_read()
        work = routing_work(w, K)
        kernels = {}
        for kind, (cnt, kms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
            pms = kms / prof_steps
            e = {"launches_per_step": cnt // prof_steps, "ms_per_step": pms}
            if kind in work and pms > 0:
                e["gbs"] = work[kind] / (pms / 1e3) / 1e9
                e["frac_hbm"] = e["gbs"] / peaks["hbm_gbs"]
            kernels[kind] = e
        top = max(prof.items(), key=lambda kv: kv[1][1])[0]
        cnt, kms = prof[top]
        ach = work[top] / (kms / prof_steps / 1e3) / 1e9
        traffic, tsrc = recorded_traffic(w, "routing", top)
        roofline = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                    "peak_source": f"{peaks['source']} HBM copy",
                    "algorithmic_per_launch": work[top] / (cnt / prof_steps)}
        if tsrc:
            roofline["traffic_source"] = tsrc
        total = sum(work.values())
        results[K] = {"value": world * M / (ms / 1e3), "ms_per_step": ms,
                      "pipeline_gbs": total / (ms / 1e3) / 1e9,
                      "pipeline_frac_hbm": total / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                      "roofline": roofline, "kernels": kernels, "clocks": clock_info,
                      "gpu_launches_per_step": int(launches)}
        st = X.sync_status(ws)
        if st != X.OK:
            raise RuntimeError(f"device status after K={K}: {X.status_string(st)}")
        del idx, r_sel, logits, xs

    # ---- end to end through the C ABI with host buffers: x and a+f in, x out, each step
    e2e = None
    K = head_K
    if not args.no_e2e:
        n = w.T // K
        M = w.B * n
        xh = torch.from_numpy(np.ascontiguousarray(x_host).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        afh = torch.from_numpy(np.ascontiguousarray(af_host[:M]).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        out_h = torch.empty_like(xh).pin_memory()
        idx = torch.empty((w.B, n), dtype=torch.int32, device=dev)
        r_sel = torch.empty((w.B, n), dtype=torch.float32, device=dev)
        logits = torch.empty((w.B, w.T), dtype=torch.float32, device=dev)
        xs = torch.empty((M, w.d), dtype=torch.bfloat16, device=dev)
        af = af_all[:M]

        def e2e_step():
            x.copy_(xh, non_blocking=True)
            af.copy_(afh, non_blocking=True)
            X.router_topk(dm, K, x, w_r, None, logits, None, idx, r_sel, ws, stream)
            X.gather(dm, K, x, idx, xs, stream)
            X.gated_scatter(dm, K, x, idx, r_sel, af, None, 1.0, X.GATE_XMOD, stream)
            out_h.copy_(x, non_blocking=True)

        e2e_step()
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e_steps = max(1, min(args.steps, 5))
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1) / e_steps)
        e2e_serial = {"value": world * M / (ems / 1e3), "unit": UNIT, "ms_per_step": ems,
                      "transfers": "serial: copies in, routing, copy out on one stream"}

        # double-buffered: step i's routing runs on one pair of device buffers while one
        # copy stream brings in step i+1's x and a+f and another takes out step i's x
        x2, af2 = [x, torch.empty_like(x)], [af, torch.empty_like(af)]
        outs = [out_h, torch.empty_like(xh).pin_memory()]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def h2d(k):
            s_in.wait_event(ev_out[k])
            with torch.cuda.stream(s_in):
                x2[k].copy_(xh, non_blocking=True)
                af2[k].copy_(afh, non_blocking=True)
            ev_in[k].record(s_in)

        def pipelined(nsteps, t0=None, t1=None):
            if t0 is not None:
                t0.record(stream)
                s_in.wait_event(t0)
            h2d(0)
            for i in range(nsteps):
                k = i & 1
                stream.wait_event(ev_in[k])
                X.router_topk(dm, K, x2[k], w_r, None, logits, None, idx, r_sel, ws, stream)
                X.gather(dm, K, x2[k], idx, xs, stream)
                X.gated_scatter(dm, K, x2[k], idx, r_sel, af2[k], None, 1.0, X.GATE_XMOD, stream)
                ev_done[k].record(stream)
                if i + 1 < nsteps:
                    h2d(1 - k)
                s_out.wait_event(ev_done[k])
                with torch.cuda.stream(s_out):
                    outs[k].copy_(x2[k], non_blocking=True)
                ev_out[k].record(s_out)
            stream.wait_event(ev_out[(nsteps - 1) & 1])
            if t1 is not None:
                t1.record(stream)

        pipelined(2)
        barrier()
        torch.cuda.synchronize()
        pipelined(e_steps, e0, e1)
        torch.cuda.synchronize()
        pms = max_over_ranks(e0.elapsed_time(e1) / e_steps)
        e2e = {"value": world * M / (pms / 1e3), "unit": UNIT, "ms_per_step": pms,
               "steps": e_steps,
               "h2d_bytes_per_step": int(xh.numel() * 2 + afh.numel() * 2),
               "d2h_bytes_per_step": int(out_h.numel() * 2),
               "transfers": "double-buffered: step i+1's copies in and step i's copy out run "
                            "on their own streams while step i's routing runs",
               "serial": e2e_serial}
        del x2, af2
        st = X.sync_status(ws)
        if st != X.OK:
            raise RuntimeError(f"device status after the e2e run: {X.status_string(st)}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_routing_sample(w, K, budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "cpu_model": cpu_model(),
               "kind": "oracle", "sample": sample,
               "single_thread": single_thread_variant(
                   lambda bs: oracle_routing_sample(w, K, budget_s=bs), args.cpu_budget / 3)}

    if rank == 0:
        h = results[K]
        cfg = routing_config(w, K)
        cfg["parallelism"] = f"replicas x{world} (sequences sharded, no collective)"
        line = {"metric": METRIC, "value": h["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded)", "config": cfg,
                "roofline": h["roofline"], "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": h["gpu_launches_per_step"] * args.steps,
                "gpu_launches_per_step": h["gpu_launches_per_step"],
                "clocks": h["clocks"],
                "pipeline_gbs": h["pipeline_gbs"], "pipeline_frac_hbm": h["pipeline_frac_hbm"],
                "kernels": h["kernels"],
                "sweep": {str(k): {kk: v[kk] for kk in ("value", "ms_per_step", "pipeline_gbs",
                                                        "pipeline_frac_hbm", "kernels")}
                          for k, v in results.items() if k != K}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["xmod", "reference"], default="xmod")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--B", type=int, default=None,
                    help="override sequences per GPU (small profiling cases only)")
    ap.add_argument("--A", type=float, default=None,
                    help="override the anchor stride A (small profiling cases only)")
    ap.add_argument("--routing", choices=["topk", "threshold"], default="topk",
                    help="token selection of the sparse layers (threshold: r >= 1/2)")
    ap.add_argument("--bias-step", type=float, default=0.0,
                    help="token-choice bias growth per selection inside a block (0: constant)")
    ap.add_argument("--variant", choices=["xmod", "routed_ffn", "fullkv"], default="xmod",
                    help="X-MoD stack, or one of the mechanism controls")
    ap.add_argument("--qwen3", action="store_true",
                    help="QK-norm and RoPE (base 1e6) in every attending layer")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="bwd: time the backward of every layer of the stack (xmod_layer_bwd)")
    ap.add_argument("--only", choices=["sparse", "dense"], default=None,
                    help="profiling: a stack of 16 sparse or 2 dense layers of the workload "
                         "instead of its Eq. 3 schedule (not a headline configuration)")
    ap.add_argument("--K", type=int, default=None,
                    help="routing_bf16 only: one sparsity K (default: 8 as the headline, with "
                         "2 and 16 under \"sweep\")")
    args = ap.parse_args()
    global VARIANT, ONLY
    VARIANT = args.variant
    ONLY = args.only
    if args.B is not None or args.A is not None:
        w = I.WORKLOADS[args.workload]
        A = w.A if args.A is None else args.A
        n_layers = w.N0 + w.N1 * (int(round(A * w.K)) + 1)
        I.WORKLOADS[args.workload] = w.replace(B=args.B or w.B, A=A, n_layers=n_layers)
    if args.pass_ == "bwd":
        run_backward(args)
    elif args.workload == "routing_bf16":   # the routing-only microbench: no block
        if args.impl == "reference":
            run_routing_reference(args)
        else:
            run_routing(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_xmod(args)


if __name__ == "__main__":
    main()
