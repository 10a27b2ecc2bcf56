#!/usr/bin/env python3
"""Benchmark of the headwise-chunked (UPipe) causal GQA attention layer, fwd+bwd.

One step = one forward and one backward pass of the whole layer (every stage:
projection, exchange, attention, exchange back, output projection, and the
matching backward work) over one synthetic batch.  Default workload: the
Llama3-8B-shaped layer, S=32768, d_model=4096, H=32, G=8, d_head=128, U=8,
C=8 virtual ranks, bf16 in / fp32 accumulate.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead (the only other code path allowed to run it), on a bounded sample.
Under torchrun with N > 1 every rank runs an independent replica on its own
GPU (the layer does not shard across GPUs here); value = tokens over all
ranks / max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn-layer fwd+bwd tokens/s & TFLOP/s (% BF16 peak) at 1 GB300; peak bytes vs U"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "llama3_8b_32k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.th:
            self.th.join(timeout=2)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1])]
        mx = [num(r[2]) for r in self.rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


KERNEL_SOURCES = {"attn_bwd": "attn_bwd.cu", "attn_fwd": "attn_fwd.cu", "gemm": "gemm.cu",
                  "seq2head": "permute.cu", "head2seq": "permute.cu", "bwd_prep": "attn_bwd.cu"}


def source_sha(kernel):
    import hashlib
    path = os.path.join(ROOT, "headwise_chunked_ulysses_gb300", "csrc", KERNEL_SOURCES[kernel])
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def measured_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu figure
    profiles/traffic_<kernel>_<workload>.json, if that capture was taken from
    the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        if rec.get("source_sha256_16") != source_sha(kernel):
            return None
        return float(rec["dram_bytes_per_launch"])
    except (ValueError, KeyError, TypeError):
        return None


def max_over_ranks(value, device=None):
    """The largest of a per-rank float over the default process group (the
    value itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(world, tokens_per_rank_step, steps, max_elapsed_ms):
    """Whole-job throughput: every rank processes its own replica of the
    workload; the job takes as long as the slowest rank."""
    return world * tokens_per_rank_step * steps / (max_elapsed_ms / 1e3)


def model_flops_step(sh):
    """Model FLOPs of one fwd+bwd step: 3x the forward, which is the QKV
    projection, the output projection and causal attention (QK^T and PV over
    the S(S+1)/2 visible pairs).  Recomputation is not counted."""
    S, dm, H, G, d = sh.S, sh.d_model, sh.H, sh.G, sh.d_head
    fwd = 2 * S * dm * (H + 2 * G) * d + 2 * S * H * d * dm + 2 * 2 * d * H * S * (S + 1) / 2
    return 3 * fwd


def oracle_sample(sh, S_sample, seed=0):
    """Time the fp64 oracle (fwd+bwd) on the workload's widths at S_sample tokens.
    Returns (seconds, tokens/s extrapolated to the workload by model-FLOP ratio)."""
    import numpy as np
    from oracle import upipe_oracle as orc
    from synthetic import layer_inputs, bf16_bits_to_f64
    small = sh.replace(S=S_sample, U=sh.U, C=sh.C)
    bits = layer_inputs(small, seed)
    X, Wqkv, Wo, dY = (bf16_bits_to_f64(bits[k]) for k in ("X", "W_qkv", "W_o", "dY"))
    t0 = time.perf_counter()
    orc.layer_forward(X, Wqkv, Wo, small.H, small.G, small.d_head)
    orc.layer_backward(X, Wqkv, Wo, small.H, small.G, small.d_head, dY)
    dt = time.perf_counter() - t0
    ratio = model_flops_step(sh) / model_flops_step(small)
    return dt, sh.S / (dt * ratio)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, sh):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    S_sample = args.ref_sample_tokens
    for _ in range(args.warmup):
        oracle_sample(sh, S_sample)
    times, vals = [], []
    for _ in range(args.steps):
        dt, v = oracle_sample(sh, S_sample)
        times.append(dt)
        vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.median(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, sh),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"fp64 numpy oracle fwd+bwd at the workload's widths with S={S_sample} "
                                   f"per step, tokens/s extrapolated to S={sh.S} by the model-FLOP ratio"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(args, sh):
    return {"workload": args.workload, "S": sh.S, "d_model": sh.d_model, "H": sh.H, "G": sh.G,
            "d_head": sh.d_head, "U": sh.U, "C": sh.C, "schedule": "gqa_out_of_order" if args.sched else "in_order",
            "causal": True, "l2": "inputs larger than L2 (X and dY are 2*S*d_model bf16 each; every step streams "
                                  "GBs through HBM)"}


def run_kernel_profile(args, sh):
    """One stage's attention kernels in isolation (U query slots, in-order KV
    copies), for ncu captures on small cases and quick kernel timing."""
    import torch
    import headwise_chunked_ulysses_gb300 as upipe
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    n_q = n_kv = sh.U
    shape = (n_q, sh.S, sh.d_head)
    Q, K, V, dO = (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
    kv = list(range(n_q))
    O, lse = upipe.attention_fwd(Q, K, V, kv)
    pairs = sh.S * (sh.S + 1) / 2
    res = {}
    for name, fn, flops in (("attn_fwd", lambda: upipe.attention_fwd(Q, K, V, kv, O=O, lse=lse),
                             4 * sh.d_head * pairs * n_q),
                            ("attn_bwd", lambda: upipe.attention_bwd(Q, K, V, O, dO, lse, kv),
                             10 * sh.d_head * pairs * n_q)):
        if args.profile_kernel not in (name, "all"):
            continue
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.reps
        res[name] = {"ms": ms, "tflops": flops / (ms / 1e3) / 1e12}
    upipe.sync_status()
    print(json.dumps({"profile_kernel": args.profile_kernel, "S": sh.S, "U": sh.U, "d_head": sh.d_head,
                      "note": "bwd time includes its preprocessing kernel", "kernels": res}), flush=True)
    return 0


DEFAULT_SWEEP = ("llama3_8b_256k_usweep", "qwen3_32b_128k", "llama3_8b_512k_gqa", "llama3_8b_256k_fp8")


def sweep_cases(names=None, extra=False):
    """(workload, shape, schedule, sequence chunks (0: none; -1: FP8 heads),
    offload store) of the other workloads: the U sweep at 256K, the Qwen3-32B
    layer at 128K, the 512K layer under both schedules (the GQA schedule's
    exchange bytes against the in-order ones), the 256K layer with FP8 heads;
    with extra, also the sequence-chunked rows and FP8 heads at 32K."""
    from synthetic import SHAPES
    cases = []
    us = SHAPES["llama3_8b_256k_usweep"]
    for U in (8, 16, 32):
        cases.append(("llama3_8b_256k_usweep", us.replace(U=U), 0, 0, None))
    cases.append(("qwen3_32b_128k", SHAPES["qwen3_32b_128k"], 0, 0, None))
    gq = SHAPES["llama3_8b_512k_gqa"]
    cases += [("llama3_8b_512k_gqa", gq, 1, 0, None), ("llama3_8b_512k_gqa", gq, 0, 0, None)]
    if extra:
        # head stages on sequence chunks, K/V offloaded to page-locked host memory
        cases += [("llama3_8b_256k_chunked", us, 0, 8, "host"), ("llama3_8b_256k_chunked", us, 0, 16, "host"),
                  ("llama3_8b_512k_chunked", gq, 0, 16, "host")]
        # every head's scores in FP8, forward and backward
        cases += [("llama3_8b_32k_fp8", SHAPES["llama3_8b_32k"], 0, -1, None)]
    # every head's scores in FP8 at 256K: the backward arena against the bf16 row's
    cases.append(("llama3_8b_256k_fp8", us, 0, -1, None))
    if names:
        cases = [c for c in cases if c[0] in names]
    return cases


def sweep_entries(cases, steps, warmup):
    """Time each case (warmup untimed steps, then `steps` fwd+bwd steps on the
    device) and yield one dict per case: tokens/s, TFLOP/s and their fractions
    of the burst and sustained bf16 peaks, the attention backward kernel's own
    rate, the stage arenas against the pages' forms, and the exchange bytes."""
    import numpy as np
    import torch
    import headwise_chunked_ulysses_gb300 as upipe
    dev = torch.device("cuda", 0)
    pk = peaks()
    for name, sh, sched, n_chunks, where in cases:
        s = upipe.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, sched)
        g = torch.Generator(device=dev).manual_seed(0)
        w_std = 1.0 / np.sqrt(sh.d_model)

        def randn(*shape, std=1.0):
            return (torch.randn(*shape, generator=g, device=dev) * std).to(torch.bfloat16)
        X, dY = randn(sh.S, sh.d_model), randn(sh.S, sh.d_model)
        Wqkv, Wo = randn(sh.d_model, sh.qkv_cols, std=w_std), randn(sh.H * sh.d_head, sh.d_model, std=w_std)
        store = None
        if n_chunks < 0:
            all_heads = set(range(sh.H))
            wsf = torch.empty(upipe.fwd_workspace_bytes(s), dtype=torch.uint8, device=dev)
            wsb = torch.empty(upipe.bwd_workspace_bytes_fp8(s, all_heads), dtype=torch.uint8, device=dev)

            def fwd(**kw):
                return upipe.attn_fwd_fp8(X, Wqkv, Wo, s, all_heads, ws=wsf, **kw)

            def bwd(O, lse, **kw):
                return upipe.attn_bwd_fp8(X, Wqkv, Wo, O, lse, dY, s, all_heads, ws=wsb, **kw)
        elif n_chunks:
            wsf = torch.empty(upipe.chunked_workspace_bytes(s, n_chunks, False), dtype=torch.uint8, device=dev)
            wsb = torch.empty(upipe.chunked_workspace_bytes(s, n_chunks, True), dtype=torch.uint8, device=dev)
            store = torch.empty(upipe.chunked_store_bytes(s, n_chunks, True), dtype=torch.uint8)
            store = store.pin_memory() if where == "host" else store.to(dev)

            def fwd(**kw):
                return upipe.attn_fwd_chunked(X, Wqkv, Wo, s, n_chunks, store, ws=wsf, **kw)

            def bwd(O, lse, **kw):
                return upipe.attn_bwd_chunked(X, Wqkv, Wo, O, lse, dY, s, n_chunks, store, ws=wsb, **kw)
        else:
            wsf = torch.empty(upipe.fwd_workspace_bytes(s), dtype=torch.uint8, device=dev)
            wsb = torch.empty(upipe.bwd_workspace_bytes(s), dtype=torch.uint8, device=dev)

            def fwd(**kw):
                return upipe.attn_fwd(X, Wqkv, Wo, s, ws=wsf, **kw)

            def bwd(O, lse, **kw):
                return upipe.attn_bwd(X, Wqkv, Wo, O, lse, dY, s, ws=wsb, **kw)
        Y, O, lse, _ = fwd()
        dX, dWqkv, dWo, _ = bwd(O, lse)
        for _ in range(max(0, warmup - 1)):
            fwd(Y=Y, O_saved=O, lse=lse)
            bwd(O, lse, dX=dX, dW_qkv=dWqkv, dW_o=dWo)
        torch.cuda.synchronize()
        upipe.sync_status()
        clocks = ClockSampler(0)
        clocks.start()
        upipe.profile_enable(True)
        upipe.profile_read()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e0.record()
        for i in range(steps):
            _, _, _, stf = fwd(Y=Y, O_saved=O, lse=lse)
            _, _, _, stb = bwd(O, lse, dX=dX, dW_qkv=dWqkv, dW_o=dWo)
            marks[i].record()
        e1.record()
        torch.cuda.synchronize()
        per_step = [e0.elapsed_time(marks[0])] + [marks[i - 1].elapsed_time(marks[i]) for i in range(1, steps)]
        clk = clocks.stop()
        prof = upipe.profile_read()
        upipe.profile_enable(False)
        upipe.sync_status()
        ms = e0.elapsed_time(e1) / steps
        tf = model_flops_step(sh) / (ms / 1e3) / 1e12
        k_ms = {k: v[0] / steps for k, v in prof.items()}
        bwd_fl = stb["flops_by_kind"]["attn_bwd"]
        bwd_tf = bwd_fl / (k_ms["attn_bwd"] / 1e3) / 1e12 if k_ms.get("attn_bwd") else None
        closed, ulysses = stf["stage_closed_form_bytes"], 12 * sh.S * sh.H * sh.d_head
        yield {
            "sweep": name, "S": sh.S, "U": sh.U, "C": sh.C, "H": sh.H, "G": sh.G, "d_model": sh.d_model,
            "schedule": "gqa_out_of_order" if sched else "in_order", "steps": steps, "warmup": warmup,
            "ms_per_step": ms, "ms_per_step_min_max": [min(per_step), max(per_step)],
            "tokens_per_s": sh.S / (ms / 1e3), "tflops": tf,
            "frac_of_bf16_peak": tf / pk["bf16_tflops"],
            "frac_of_bf16_peak_sustained": tf / pk["bf16_tflops_sustained"],
            "attn_bwd_tflops": bwd_tf,
            "attn_bwd_frac": bwd_tf / pk["bf16_tflops"] if bwd_tf else None,
            "attn_bwd_frac_sustained": bwd_tf / pk["bf16_tflops_sustained"] if bwd_tf else None,
            "stage_arena_fwd_bytes": stf["arena_peak_bytes"], "stage_arena_bwd_bytes": stb["arena_peak_bytes"],
            "closed_form_12SUd": closed, "ulysses_form_12SHd": ulysses,
            "arena_fwd_over_12SUd": stf["arena_peak_bytes"] / closed,
            "arena_fwd_over_12SHd": stf["arena_peak_bytes"] / ulysses,
            "arena_bwd_over_12SHd": stb["arena_peak_bytes"] / ulysses,
            "permute_bytes_fwd": stf["permute_bytes"], "permute_bytes_bwd": stb["permute_bytes"],
            "persistent_bytes": stf["persistent_bytes"], "clocks": clk,
            "workspace_fwd_bytes": wsf.numel(), "workspace_bwd_bytes": wsb.numel(),
            "sequence_chunks": max(n_chunks, 0), "fp8_heads": "all" if n_chunks < 0 else "none",
            "offload_store": where, "offload_bytes": stb["offload_bytes"],
            "offload_copy_bytes": stf["offload_copy_bytes"] + stb["offload_copy_bytes"],
            "kernel_ms_per_step": k_ms}
        del X, dY, Wqkv, Wo, wsf, wsb, Y, O, lse, dX, dWqkv, dWo, store, fwd, bwd
        torch.cuda.empty_cache()


def with_schedule_ratio(entries):
    """Adds, to each out-of-order entry with an in-order twin, the ratio of
    its exchange bytes to the in-order schedule's."""
    for e in entries:
        if e["schedule"] != "gqa_out_of_order":
            continue
        for f in entries:
            if f is not e and f["sweep"] == e["sweep"] and f["U"] == e["U"] and f["schedule"] == "in_order":
                e["permute_bytes_fwd_in_order"] = f["permute_bytes_fwd"]
                e["permute_bytes_bwd_in_order"] = f["permute_bytes_bwd"]
                e["permute_fwd_ratio_vs_in_order"] = e["permute_bytes_fwd"] / f["permute_bytes_fwd"]
    return entries


def run_sweep(args):
    """The other workloads, one JSON line each.  Not the headline."""
    names = args.sweep_only.split(",") if args.sweep_only else None
    entries = with_schedule_ratio(list(sweep_entries(sweep_cases(names, extra=True), args.sweep_steps,
                                                     args.sweep_warmup)))
    for e in entries:
        print(json.dumps(e), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sched", type=int, default=0, help="0 in order, 1 GQA out of order")
    ap.add_argument("--U", type=int, default=None, help="override heads per stage")
    ap.add_argument("--S", type=int, default=None, help="override sequence length")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=4096)
    ap.add_argument("--ref-sample-tokens", type=int, default=2048)
    ap.add_argument("--profile-kernel", default=None, choices=["attn_fwd", "attn_bwd", "all"],
                    help="time one stage's attention kernels alone (no JSON bench line)")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--sweep", action="store_true",
                    help="only the other workloads, one line each (adds the chunked and FP8 rows)")
    ap.add_argument("--sweep-only", default=None, help="comma-separated workload names for --sweep")
    ap.add_argument("--sweep-steps", type=int, default=3)
    ap.add_argument("--sweep-warmup", type=int, default=1)
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave the U sweep, Qwen3-32B and 512K rows out of the headline line")
    args = ap.parse_args()

    from synthetic import SHAPES
    sh = SHAPES[args.workload]
    if args.U:
        sh = sh.replace(U=args.U)
    if args.S:
        sh = sh.replace(S=args.S)
    if args.impl == "reference":
        return run_reference(args, sh)
    if args.profile_kernel:
        return run_kernel_profile(args, sh)
    if args.sweep:
        return run_sweep(args)

    rank, world, local = dist_env()
    import numpy as np
    import torch
    import headwise_chunked_ulysses_gb300 as upipe
    from synthetic import layer_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    s = upipe.Shape(sh.S, sh.d_model, sh.H, sh.G, sh.d_head, sh.U, sh.C, args.sched)
    bits = layer_inputs(sh, seed=0)
    host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) for k, v in bits.items()}
    d = {k: v.to(dev) for k, v in host.items()}
    bf, f32 = torch.bfloat16, torch.float32
    Y = torch.empty(sh.S, sh.d_model, dtype=bf, device=dev)
    O = torch.empty(sh.S, sh.H * sh.d_head, dtype=bf, device=dev)
    lse = torch.empty(sh.H, sh.S, dtype=f32, device=dev)
    dX = torch.empty(sh.S, sh.d_model, dtype=bf, device=dev)
    dWqkv = torch.empty(sh.d_model, sh.qkv_cols, dtype=f32, device=dev)
    dWo = torch.empty(sh.H * sh.d_head, sh.d_model, dtype=f32, device=dev)
    wsf = torch.empty(upipe.fwd_workspace_bytes(s), dtype=torch.uint8, device=dev)
    wsb = torch.empty(upipe.bwd_workspace_bytes(s), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        _, _, _, stf = upipe.attn_fwd(d["X"], d["W_qkv"], d["W_o"], s, Y=Y, O_saved=O, lse=lse, ws=wsf)
        _, _, _, stb = upipe.attn_bwd(d["X"], d["W_qkv"], d["W_o"], O, lse, d["dY"], s, dX=dX, dW_qkv=dWqkv,
                                      dW_o=dWo, ws=wsb)
        return stf, stb

    torch.cuda.reset_peak_memory_stats(dev)
    mem_before = torch.cuda.memory_allocated(dev)
    for _ in range(args.warmup):
        stf, stb = step()
    barrier()
    upipe.sync_status()

    # ---------------- device-resident timed region ----------------
    clocks = ClockSampler(local)
    clocks.start()
    upipe.profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        stf, stb = step()
        marks[i].record(stream)
    e1.record(stream)
    barrier()
    elapsed_ms = e0.elapsed_time(e1)
    per_step = [e0.elapsed_time(marks[0])] + [marks[i - 1].elapsed_time(marks[i]) for i in range(1, args.steps)]
    prof = upipe.profile_read()
    upipe.profile_enable(False)
    clk = clocks.stop()
    upipe.sync_status()
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_step = elapsed_ms / args.steps
    tokens_per_s = aggregate_tokens_per_s(world, sh.S, args.steps, elapsed_ms)
    pk = peaks()
    flops_step = model_flops_step(sh)
    tflops = flops_step / (ms_step / 1e3) / 1e12
    # the step is timed at full clocks in a sub-second region: the burst
    # figure is the denominator, the sustained one is reported beside it
    peak_tf = pk["bf16_tflops"]
    peak_sus = pk["bf16_tflops_sustained"]

    # per-kernel achieved throughput from the live event timings
    kernels = {}
    for k in upipe.KERNEL_KINDS:
        ms, n = prof[k]
        n_step = stf["launches_by_kind"][k] + stb["launches_by_kind"][k]
        fl = (stf["flops_by_kind"][k] + stb["flops_by_kind"][k]) * args.steps
        by = (stf["bytes_by_kind"][k] + stb["bytes_by_kind"][k]) * args.steps
        kernels[k] = {"ms_per_step": ms / args.steps, "launches_per_step": n_step, "share": None,
                      "tflops": fl / (ms / 1e3) / 1e12 if ms > 0 and fl > 0 else None,
                      "gbs": by / (ms / 1e3) / 1e9 if ms > 0 else None}
    tot = sum(v["ms_per_step"] for v in kernels.values()) or 1.0
    for v in kernels.values():
        v["share"] = v["ms_per_step"] / tot
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
    ms_dom, n_dom = prof[dom]
    if kernels[dom]["tflops"]:
        fl_launch = (stf["flops_by_kind"][dom] + stb["flops_by_kind"][dom]) / max(1, kernels[dom]["launches_per_step"])
        achieved = fl_launch / (ms_dom / n_dom / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "peak_source": f"{pk['source']} bf16_tflops (burst)",
                "frac_sustained": achieved / peak_sus, "peak_sustained": peak_sus,
                "flops_per_launch": fl_launch, "ms_per_launch": ms_dom / n_dom,
                "traffic": measured_traffic(dom, args.workload), "source_sha256_16": source_sha(dom)}
    else:
        by_launch = (stf["bytes_by_kind"][dom] + stb["bytes_by_kind"][dom]) / max(1, kernels[dom]["launches_per_step"])
        achieved = by_launch / (ms_dom / n_dom / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": f"{pk['source']} hbm_gbs",
                "bytes_per_launch": by_launch, "ms_per_launch": ms_dom / n_dom,
                "traffic": measured_traffic(dom, args.workload), "source_sha256_16": source_sha(dom)}
    launches = (stf["launches"] + stb["launches"]) * args.steps

    # ---------------- end to end through the public API, host buffers ----------------
    e2e = None
    if not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in host.items()}
        outs = {"Y": torch.empty_like(Y, device="cpu").pin_memory(), "dX": torch.empty_like(dX, device="cpu").pin_memory(),
                "dW_qkv": torch.empty_like(dWqkv, device="cpu").pin_memory(),
                "dW_o": torch.empty_like(dWo, device="cpu").pin_memory()}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(v.numel() * v.element_size() for v in outs.values())

        # Every step copies its inputs in from pinned host memory and its
        # results back out, all inside the timed region.  The copies run on
        # two copy streams (one per direction), double-buffered on the device,
        # so step k+1's inputs arrive and step k's results leave while step k
        # (resp. k+1) computes -- the way a training loop feeds the layer.
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        din = [d, {k: torch.empty_like(v) for k, v in d.items()}]
        dout = [{"Y": Y, "dX": dX, "dW_qkv": dWqkv, "dW_o": dWo},
                {"Y": torch.empty_like(Y), "dX": torch.empty_like(dX), "dW_qkv": torch.empty_like(dWqkv),
                 "dW_o": torch.empty_like(dWo)}]
        hout = [outs, {k: torch.empty_like(v).pin_memory() for k, v in outs.items()}]

        fwd_in, bwd_in = ("X", "W_qkv", "W_o"), ("dY",)

        def run_e2e(n):
            # a step's forward needs X and the weights, its backward dY as
            # well; Y leaves after the forward, the gradients after the
            # backward, so the first step's dY copy and the last step's Y copy
            # overlap compute too
            ev = lambda: torch.cuda.Event()
            fwd_ready, bwd_ready, in_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
            y_ready, out_ready, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

            def copy_in(b):
                with torch.cuda.stream(h2d_s):
                    for k in fwd_in:
                        din[b][k].copy_(pin[k], non_blocking=True)
                fwd_ready[b].record(h2d_s)
                with torch.cuda.stream(h2d_s):
                    for k in bwd_in:
                        din[b][k].copy_(pin[k], non_blocking=True)
                bwd_ready[b].record(h2d_s)

            start = ev()
            start.record(stream)
            h2d_s.wait_event(start)
            copy_in(0)
            for i in range(n):
                b = i & 1
                if i + 1 < n:  # inputs of step i+1, once step i-1 has finished with that buffer
                    nb = b ^ 1
                    if i >= 1:
                        h2d_s.wait_event(in_free[nb])
                    copy_in(nb)
                stream.wait_event(fwd_ready[b])
                if i >= 2:
                    stream.wait_event(out_free[b])
                o = dout[b]
                upipe.attn_fwd(din[b]["X"], din[b]["W_qkv"], din[b]["W_o"], s, Y=o["Y"], O_saved=O, lse=lse, ws=wsf)
                y_ready[b].record(stream)
                d2h_s.wait_event(y_ready[b])
                with torch.cuda.stream(d2h_s):
                    hout[b]["Y"].copy_(o["Y"], non_blocking=True)
                stream.wait_event(bwd_ready[b])
                upipe.attn_bwd(din[b]["X"], din[b]["W_qkv"], din[b]["W_o"], O, lse, din[b]["dY"], s, dX=o["dX"],
                               dW_qkv=o["dW_qkv"], dW_o=o["dW_o"], ws=wsb)
                in_free[b].record(stream)
                out_ready[b].record(stream)
                d2h_s.wait_event(out_ready[b])
                with torch.cuda.stream(d2h_s):
                    for k in ("dX", "dW_qkv", "dW_o"):
                        hout[b][k].copy_(o[k], non_blocking=True)
                out_free[b].record(d2h_s)
            stream.wait_stream(d2h_s)
            stream.wait_stream(h2d_s)

        run_e2e(2)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        run_e2e(args.steps)
        f1.record(stream)
        barrier()
        e_ms = max_over_ranks(f0.elapsed_time(f1), dev)
        e2e = {"value": aggregate_tokens_per_s(world, sh.S, args.steps, e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "copies": "per step: all inputs host->device and Y, dX, dW_qkv, dW_o device->host, on two copy "
                         "streams overlapping compute (double-buffered on the device; dY may arrive during the "
                         "step's forward, Y leaves during its backward)"}
        upipe.sync_status()

    mem_peak = torch.cuda.max_memory_allocated(dev) - mem_before
    # SM clock cycles per step (ms x MHz = thousands of cycles): a step's cost
    # with the clock taken out
    if clk.get("sm_mhz"):
        clk["sm_kcycles_per_step"] = ms_step * clk["sm_mhz"]
        clk["attn_bwd_sm_kcycles_per_step"] = kernels["attn_bwd"]["ms_per_step"] * clk["sm_mhz"]

    # ---------------- the other workloads (not the headline; outside the timed region) ----------------
    sweep = None
    if not args.no_sweep and world == 1:
        del wsf, wsb
        torch.cuda.empty_cache()
        sweep = with_schedule_ratio(list(sweep_entries(sweep_cases(DEFAULT_SWEEP), args.sweep_steps,
                                                       args.sweep_warmup)))
    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        dt, v = oracle_sample(sh, args.cpu_sample_tokens)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"fp64 numpy oracle fwd+bwd at the workload's widths with S={args.cpu_sample_tokens} "
                         f"({dt:.1f} s), extrapolated to S={sh.S} by the model-FLOP ratio"}
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_min_max": [min(per_step), max(per_step)],
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(args, sh),
        "tflops": tflops, "frac_of_bf16_peak": tflops / peak_tf,
        "frac_of_bf16_peak_sustained": tflops / peak_sus,
        "peak_source": f"{pk['source']} bf16_tflops={peak_tf} (burst; sustained {peak_sus} beside)",
        "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clk,
        "memory": {"stage_arena_bytes": stf["arena_peak_bytes"], "stage_arena_bwd_bytes": stb["arena_peak_bytes"],
                   "closed_form_12SUd": stf["stage_closed_form_bytes"], "persistent_fwd_bytes": stf["persistent_bytes"],
                   "persistent_bwd_bytes": stb["persistent_bytes"], "torch_peak_alloc_bytes": mem_peak,
                   "permute_bytes_per_step": stf["permute_bytes"] + stb["permute_bytes"]},
        "sweep": sweep,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
