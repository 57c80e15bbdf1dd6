#!/usr/bin/env python
"""KDA on GB300: prefill tokens/s (chunked, BF16, B=1 H=8 T=4096 d=128) and
decode tokens/s (256 sequences x 56 heads, 64 single-token steps), with the
roofline fraction of the dominant kernel.

One step = one whole prefill of the workload through the one-call entry point
kda_prefill_chunked, bracketed by CUDA events on the launching stream: the
transfer pass over all S segments with outputs, the segment scan and the output
combine launched back to back (a single output pass when the library picks
S = 1).  A separate pass through the three stage entry points, with events
between them, gives the per-stage times behind the roofline.  Inputs are
resident in HBM; the 50 MB working set is smaller than L2, so a 512 MB buffer is
rewritten between timed steps (outside the events).  ``e2e`` times the same
call with every step's inputs copied in from pinned host memory and its outputs
copied back, steps alternating between two streams (one step's input copies
overlap the previous step's compute and output copies).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = "kda_prefill_bf16_h8_t4096_d128"
DECODE = "kda_decode_b256_h56_d128_x64"
METRIC = "KDA prefill tokens/s and decode tokens/s on 1 GB300; % of roofline"
# fp32 FMA peak of a GB300 at its maximum SM clock (no measured figure exists for
# CUDA-core fp32): 152 SMs x 128 lanes x 2 flops x 2.07 GHz
BWD_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
PROFILE_CASES = ("decode", "prefill_output_pass", "prefill_h8_t4096", "prefill_ckpt_h8_t4096",
                 "backward_h8_t1024")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--profile", choices=sorted(PROFILE_CASES), default=None,
                   help="run one small case twice for an ncu capture (no timing, no JSON)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: each rank owns a full batch)
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(value, dist, device=None):
    """Max of a float over ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [s for s in vis.split(",") if s.strip()]
        self.index = ids[local_rank] if local_rank < len(ids) and ids[local_rank].isdigit() \
            else str(local_rank)
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax.append(float(f[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, f[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                   "reasons": sorted(reasons), "samples": len(sm)}
        return out


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move, per launch)
# ---------------------------------------------------------------------------
def prefill_stage_bytes(T, H, dk, dv, N, Sg, act_bytes):
    """Bytes each stage must read and write at minimum.

    one pass (S = 1): q, k, v, out (activation dtype) + g, beta (fp32) per
                      head-token, plus the final states.
    transfer pass   : q, k, v, g, beta read once per head-token; the zero-start
                      outputs and A_t^T q_t written (activation dtype); A and B
                      written per (sequence, head, segment).
    scan            : A, B read, start states and final states written (and, for
                      BF16 at d = 128, each start state's BF16 operand image).
    combine         : A_t^T q_t and the zero-start outputs read, outputs written,
                      start states read (their BF16 images for BF16 at d = 128).
    """
    if Sg == 1:
        return {"output_pass": T * H * ((2 * dk + 2 * dv) * act_bytes + 4 * dk + 4) +
                N * H * dk * dv * 4}
    states = N * H * Sg * (dk * dk + dk * dv) * 4
    start_bytes = 2 if (act_bytes == 2 and dk == 128 and dv == 128) else 4
    transfer = T * H * ((2 * dk + dv) * act_bytes + 4 * dk + 4) + \
        T * H * (dv + dk) * act_bytes + states
    scan = states + N * H * Sg * dk * dv * 4 + N * H * dk * dv * 4
    if start_bytes == 2:
        scan += N * H * Sg * dk * dv * 2
    combine = T * H * (dk + 2 * dv) * act_bytes + N * H * Sg * dk * dv * start_bytes
    return {"transfer_pass": transfer, "segment_scan": scan, "combine": combine}


def method_roofline(head_tokens, ms, dk, dv, act_bytes, peaks):
    """The whole step against the method's own algorithmic counts per head-token:
    flops = 6 dk dv + C (3 dk + 2 dv) (C = 16, triangle-aware) and bytes = q, k, v,
    out in the activation dtype + g fp32 + beta fp32; the attainable ceiling is
    min(P_bf16, I * BW) with I = flops / bytes (I * BW is below P here: HBM-bound)."""
    C = 16
    flops = 6 * dk * dv + C * (3 * dk + 2 * dv)
    nbytes = (2 * dk + 2 * dv) * act_bytes + 4 * dk + 4
    sec = ms / 1e3
    tflops = head_tokens * flops / sec / 1e12
    gbs = head_tokens * nbytes / sec / 1e9
    attain = min(peaks["bf16_tflops"], flops / nbytes * peaks["hbm_gbs"] / 1e3)
    return {"flops_per_head_token": flops, "bytes_per_head_token": nbytes,
            "tflops": round(tflops, 2), "tflops_frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 4),
            "attainable_tflops": round(attain, 1), "attainable_frac": round(tflops / attain, 4),
            "gbs": round(gbs, 1), "gbs_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "peak_source": peaks["source"]}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import kimi_delta_attention_18_gb300 as kda
    from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_decode_inputs, \
        make_prefill_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    kda.lib()  # fail loudly now if the library is missing

    w = WORKLOADS[PREFILL]
    x = make_prefill_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], seed=rank,
                            device=dev)
    T, H, dk = x["q"].shape
    dv = x["v"].shape[2]
    N = len(w["lengths"])
    desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"])
    Sg = kda.prefill_num_segments(desc)
    act_bytes = x["q"].element_size()
    out = torch.empty_like(x["v"])
    S_final = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    A = torch.empty((N, H, Sg, dk, dk), dtype=torch.float32, device=dev)
    B = torch.empty((N, H, Sg, dk, dv), dtype=torch.float32, device=dev)
    starts = torch.empty((N, H, Sg, dk, dv), dtype=torch.float32, device=dev)
    # L2 flush between timed steps: a 512 MB fill (torch's fill kernel) evicts the
    # 129 MB L2 before every step
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    aux = torch.empty((T, H, dk), dtype=x["q"].dtype, device=dev)
    # the start states' BF16 operand images (BF16 at d = 128), as the one-call path uses
    imgs = (torch.empty((N * H, Sg, dk * dv), dtype=torch.bfloat16, device=dev)
            if x["q"].dtype == torch.bfloat16 and dk == 128 and dv == 128 else None)

    ws_bytes = kda.prefill_workspace_size(desc)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def step(ev):
        # the call a user makes: kda_prefill_chunked launches the transfer pass,
        # the segment scan and the output combine back to back (or one output
        # pass when the split is a single segment)
        ev[0].record(stream)
        kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["cu_seqlens"],
                            out=out, S_final=S_final, workspace=workspace)
        ev[1].record(stream)

    def staged(ev):
        # exactly the launches kda_prefill_chunked makes, with events between them
        ev[0].record(stream)
        if Sg > 1:
            kda.state_transfer(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], Sg,
                               transfer=A, zero_init_state=B, q=x["q"], out_zero=out,
                               out_transfer=aux)
        ev[1].record(stream)
        if Sg > 1:
            kda.state_compose(A.view(N * H, Sg, dk, dk), B.view(N * H, Sg, dk, dv), None,
                              seg_init_states=starts.view(N * H, Sg, dk, dv),
                              S_final=S_final.view(N * H, dk, dv), start_images=imgs)
        ev[2].record(stream)
        if Sg > 1:
            kda.prefill_combine(out, aux, starts, x["cu_seqlens"], first_segment=1,
                                start_images=imgs)
        else:
            kda.prefill_segments(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                 x["cu_seqlens"], 1, out=out, S_final=S_final)
        ev[3].record(stream)

    mk = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for _ in range(args.warmup):
        flush.zero_()
        step(mk(2))
    torch.cuda.synchronize()
    events = [mk(2) for _ in range(args.steps)]
    clocks = Clocks(local)
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist)
    clk = clocks.stop()
    total_ms = [ev[0].elapsed_time(ev[1]) for ev in events]
    dev_ms = sum(total_ms)
    dev_ms_max = max_over_ranks(dev_ms, dist, dev)
    tokens = T * args.steps * world
    value = tokens / (dev_ms_max / 1e3)

    # per-stage device times (a separate pass through the stage entry points; the
    # host has time to queue each step's launches behind the L2 flush)
    stage_ms = {"transfer_pass": [], "segment_scan": [], "combine": [], "output_pass": []}
    for _ in range(max(3, min(args.steps, 10))):
        ev = mk(4)
        flush.zero_()
        staged(ev)
        torch.cuda.synchronize()
        stage_ms["transfer_pass"].append(ev[0].elapsed_time(ev[1]))
        stage_ms["segment_scan"].append(ev[1].elapsed_time(ev[2]))
        stage_ms["combine" if Sg > 1 else "output_pass"].append(ev[2].elapsed_time(ev[3]))

    # roofline of the dominant kernel (HBM-bound: see the design notes)
    peaks = measured_peaks()
    sbytes = prefill_stage_bytes(T, H, dk, dv, N, Sg, act_bytes)
    means = {k_: statistics.mean(v_) for k_, v_ in stage_ms.items() if k_ in sbytes}
    dom = max(means, key=means.get)
    achieved = sbytes[dom] / (means[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": None, "peak_source": peaks["source"] + " (burst copy)",
                "stage_ms": {k_: round(v_, 4) for k_, v_ in means.items()},
                "stage_bytes": sbytes}
    launches_per_step = 3 if Sg > 1 else 1

    result = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
              "ms_per_step": round(dev_ms_max / args.steps, 5), "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
              "config": {"workload": PREFILL, "batch": N, "seq_len": T, "heads": H, "dk": dk,
                         "dv": dv, "chunk": 16, "segments": Sg, "state": "fp32",
                         "l2": "512 MB buffer zero-filled between timed steps (working set 50 MB)",
                         "parallelism": "dp%d (one batch per GPU)" % world},
              "wall_s_timed_loop": round(wall, 4), "clocks": clk, "roofline": roofline,
              "method": method_roofline(T * H * world, dev_ms_max / args.steps, dk, dv,
                                        act_bytes, peaks),
              "gpu_launches": launches_per_step * args.steps}

    # the same step from the pre-activations (fused gate prologue)
    result["gated"] = run_gated(args, kda, x, flush, stream, dev, dist, dev_ms_max / args.steps)
    # the same step with a state checkpoint every 512 tokens of each sequence
    result["checkpoints"] = run_ckpt(args, kda, x, flush, stream, dev, dist,
                                     dev_ms_max / args.steps)
    result["backward"] = run_backward(args, kda, x, flush, stream, dev, dist)
    # e2e: one-call C entry point with pinned host buffers, copies included
    result["e2e"] = run_e2e(args, kda, x, N, T, H, dk, dv, dev, dist, world)
    if not args.no_decode:
        result["decode"] = run_decode(args, kda, make_decode_inputs, WORKLOADS[DECODE], dev,
                                      dist, world, peaks, rank)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(x, N, H)
        result["backward"]["cpu_baseline"] = cpu_baseline_backward(x, H)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_gated(args, kda, x, flush, stream, dev, dist, plain_ms):
    """kda_prefill_chunked_gated on the timed workload (raw q, k; x_g in BF16 and
    x_beta fp32; the kernels form g, beta and the normalised q, k), timed like the
    plain step."""
    import torch
    T, H, dk = x["q"].shape
    dv = x["v"].shape[2]
    if x["q"].dtype != torch.bfloat16 or dk != 128 or dv != 128:
        return None
    out = torch.empty_like(x["v"])
    SF = torch.empty((len(x["lengths"]), H, dk, dv), dtype=torch.float32, device=dev)
    ws = torch.empty(max(kda.prefill_workspace_size(kda.prefill_desc(x["q"], x["v"],
                                                                     x["cu_seqlens"])), 1),
                     dtype=torch.uint8, device=dev)

    def call():
        kda.prefill_chunked_gated(x["q_raw"], x["k_raw"], x["v"], x["x_g"], x["x_beta"], None,
                                  x["cu_seqlens"], out=out, S_final=SF, workspace=ws)

    for _ in range(3):
        flush.zero_()
        call()
    steps = max(5, min(args.steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), dist, dev) / steps
    nbytes = T * H * ((2 * dk + 2 * dv) * 2 + 2 * dk + 4)  # q, k, v, out, x_g BF16, x_beta
    return {"ms_per_step": round(ms, 5), "tokens_per_s": round(T / (ms / 1e3), 1),
            "bytes_per_head_token": nbytes // (T * H), "vs_plain": round(ms / plain_ms - 1.0, 4)}


def run_ckpt(args, kda, x, flush, stream, dev, dist, plain_ms, interval=512):
    """kda_prefill_chunked_ckpt on the timed workload: the step with a state
    checkpoint after every `interval` tokens, timed like the plain step (L2
    flushed before each call, CUDA events around it)."""
    import torch
    T, H, dk = x["q"].shape
    dv = x["v"].shape[2]
    K = kda.num_checkpoints(x["cu_seqlens"], interval)
    ck = torch.empty((max(K, 1), H, dk, dv), dtype=torch.float32, device=dev)
    out = torch.empty_like(x["v"])
    SF = torch.empty((len(x["lengths"]), H, dk, dv), dtype=torch.float32, device=dev)
    desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"])
    ws_bytes = kda.prefill_ckpt_workspace_size(desc, interval)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def call():
        kda.prefill_chunked_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                 x["cu_seqlens"], ckpt_interval=interval, ckpt_states=ck,
                                 out=out, S_final=SF, workspace=ws)

    for _ in range(3):
        flush.zero_()
        call()
    steps = max(5, min(args.steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), dist, dev) / steps
    return {"interval": interval, "checkpoints_per_step": K * H,
            "bytes_per_step": K * H * dk * dv * 4, "ms_per_step": round(ms, 5),
            "overhead_vs_plain": round(ms / plain_ms - 1.0, 4)}


def run_backward(args, kda, x, flush, stream, dev, dist):
    """kda_prefill_backward on the timed workload (d_out ~ N(0, 1), d_S_final ~
    N(0, 1)): dq, dk, dv, dg, dbeta, dS0 in fp32; L2 flushed before each call,
    CUDA events around it."""
    import torch
    from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints
    T, H, dk = x["q"].shape
    dv = x["v"].shape[2]
    N = len(x["lengths"])
    act = "bf16" if x["q"].dtype == torch.bfloat16 else "f32"
    d_out, d_sf = make_backward_adjoints(T, N, H, dk, dv, act, seed=7, device=dev)
    desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"])
    ws = torch.empty(max(kda.prefill_backward_workspace_size(desc), 16), dtype=torch.uint8,
                     device=dev)

    def call():
        kda.prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["cu_seqlens"],
                             d_out, d_sf, workspace=ws)

    for _ in range(3):
        flush.zero_()
        call()
    steps = 5
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), dist, dev) / steps
    # algorithmic work per head-token and state element: the forward step (decay 1,
    # M^T k 2, rank-1 update 2) and its adjoint (read 2, dS^T k 2, S_t do 2,
    # dk 4, dM 2, dg 2, decay 1) = 20 flops; fp32 on CUDA cores
    flops = 20.0 * dk * dv * T * H
    peak = BWD_FP32_TFLOPS
    achieved = flops / (ms * 1e-3) / 1e12
    return {"what": "dq, dk, dv, dg, dbeta, dS0 (fp32), token-level SIMT kernels, segment split",
            "ms_per_step": round(ms, 4), "tokens_per_s": round(N and T / (ms * 1e-3), 1),
            "segments": kda.prefill_backward_num_segments(desc),
            "ctas_per_pass": N * H * ((dv + 31) // 32) * kda.prefill_backward_num_segments(desc),
            "roofline": {"bound": "alu", "achieved": round(achieved, 3), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "flops_per_head_token": 20 * dk * dv,
                         "peak_from": "152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz"}}


def run_e2e(args, kda, x, N, T, H, dk, dv, dev, dist, world):
    """One-call prefill with its inputs copied in from pinned host memory and its
    outputs (out, S_final) copied back, every step.  Steps alternate between two
    streams with their own device buffers, as a caller streaming prefills would
    run them: one step's input copies overlap the previous step's compute and
    output copies."""
    import torch
    host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"])
    nstreams = 2
    streams = [torch.cuda.Stream(dev) for _ in range(nstreams)]
    sets = []
    for _ in range(nstreams):
        sets.append({
            "in": {n: torch.empty_like(x[n]) for n in host},
            "out_d": torch.empty_like(x["v"]),
            "sf_d": torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev),
            "ws": torch.empty(max(1, kda.prefill_workspace_size(desc)), dtype=torch.uint8,
                              device=dev),
            "out_h": torch.empty((T, H, dv), dtype=x["q"].dtype).pin_memory(),
            "sf_h": torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory(),
        })
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sets[0]["out_h"].numel() * sets[0]["out_h"].element_size() + \
        sets[0]["sf_h"].numel() * sets[0]["sf_h"].element_size()

    def one(i):
        b, st = sets[i % nstreams], streams[i % nstreams]
        with torch.cuda.stream(st):
            for n in host:
                b["in"][n].copy_(host[n], non_blocking=True)
            kda.prefill_chunked(b["in"]["q"], b["in"]["k"], b["in"]["v"], b["in"]["g"],
                                b["in"]["beta"], None, x["cu_seqlens"], out=b["out_d"],
                                S_final=b["sf_d"], workspace=b["ws"])
            b["out_h"].copy_(b["out_d"], non_blocking=True)
            b["sf_h"].copy_(b["sf_d"], non_blocking=True)

    main = torch.cuda.current_stream(dev)
    for st in streams:
        st.wait_stream(main)  # inputs and cu_seqlens are ready
    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for st in streams:
        st.wait_event(e0)
    for i in range(args.e2e_steps):
        one(i)
    for st in streams:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    # the bound: the step's input bytes as one pinned host-to-device copy (the
    # link, not the kernels, limits this leg)
    flat_h = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    flat_d = torch.empty(h2d, dtype=torch.uint8, device=dev)
    for _ in range(3):
        flat_d.copy_(flat_h, non_blocking=True)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(main)
    for _ in range(10):
        flat_d.copy_(flat_h, non_blocking=True)
    c1.record(main)
    torch.cuda.synchronize()
    link_gbs = h2d * 10 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    step_ms = ms / args.e2e_steps
    return {"value": round(T * args.e2e_steps * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(step_ms, 4), "streams": nstreams,
            "h2d_link_gbs": round(link_gbs, 1),
            "frac_of_link": round(h2d / (step_ms * 1e-3) / 1e9 / link_gbs, 3)}


def run_decode(args, kda, make_decode_inputs, w, dev, dist, world, peaks, rank):
    import torch
    steps = w["steps"]
    x = make_decode_inputs(w["batch"], w["H"], w["dk"], w["dv"], steps, w["act"],
                           s0_std=w["s0_std"], seed=rank, device=dev)
    S = x["S0"].clone()
    out = torch.empty((w["batch"], w["H"], w["dv"]), dtype=x["q"].dtype, device=dev)
    for t in range(3):
        kda.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S, out=out)
    S.copy_(x["S0"])
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(dist)
    clocks = Clocks(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    ev[0].record()
    for t in range(steps):
        kda.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S, out=out)
        ev[t + 1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    per = [ev[t].elapsed_time(ev[t + 1]) for t in range(steps)]
    total = max_over_ranks(sum(per), dist, dev)
    units = w["batch"] * w["H"]
    act_b = x["q"].element_size()
    bytes_per_launch = units * (2 * w["dk"] * w["dv"] * 4 + (2 * w["dk"] + 2 * w["dv"]) * act_b +
                                4 * w["dk"] + 4)
    achieved = bytes_per_launch / (statistics.mean(per) / 1e3) / 1e9
    return {"value": round(w["batch"] * steps * world / (total / 1e3), 1), "unit": "tokens/s",
            "workload": "kda_decode_b256_h56_d128_x64", "steps": steps,
            "ms_per_step": round(total / steps, 5), "gpu_launches": steps,
            "clocks": clk,
            "roofline": {"bound": "hbm", "kernel": "decode_step", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "bytes_per_launch": bytes_per_launch, "traffic": None,
                         "peak_source": peaks["source"] + " (burst copy)"}}


def cpu_baseline(x, N, H, target_s=8.0):
    """The fp64 oracle as it stands, on the host cores, over a bounded sample of the
    same workload (the first heads of the batch, whole sequence)."""
    import oracle
    f = lambda t: t.detach().float().cpu().double().numpy()
    q, k, v, g, b = (f(x[n]) for n in ("q", "k", "v", "g", "beta"))
    cu = x["cu_seqlens"].cpu().numpy()
    threads = oracle.host_threads()
    t0 = time.perf_counter()
    oracle.kda_forward(q[:, :1], k[:, :1], v[:, :1], g[:, :1], b[:, :1], None, cu,
                       threads=threads)
    one = time.perf_counter() - t0
    heads = max(1, min(H, int(target_s / max(one, 1e-3))))
    t0 = time.perf_counter()
    oracle.kda_forward(q[:, :heads], k[:, :heads], v[:, :heads], g[:, :heads], b[:, :heads],
                       None, cu, threads=threads)
    dt = time.perf_counter() - t0
    T = q.shape[0]
    return {"value": round(T * heads / H / dt, 2), "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d of %d heads x %d tokens (fp64 token-by-token C oracle, %.2f s)" %
                      (heads, H, T, dt)}


def cpu_baseline_backward(x, H, tokens=512):
    """The oracle's backward (fp64 PyTorch autograd of the token loop, as it
    stands) on a bounded sample of the backward leg's workload: one head, the
    first `tokens` tokens."""
    import numpy as np
    import torch
    import oracle
    from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints
    f = lambda t: t.detach().float().cpu().double().numpy()
    T, _, dk = x["q"].shape
    dv = x["v"].shape[2]
    n = min(tokens, T)
    act = "bf16" if x["q"].dtype == torch.bfloat16 else "f32"
    d_out, d_sf = make_backward_adjoints(T, 1, H, dk, dv, act, seed=7)
    sl = lambda a: a[:n, :1]
    t0 = time.perf_counter()
    oracle.kda_backward(*(sl(f(x[m])) for m in ("q", "k", "v", "g", "beta")), None,
                        np.array([0, n], dtype=np.int32), sl(f(d_out)), f(d_sf)[:, :1])
    dt = time.perf_counter() - t0
    return {"value": round(n / H / dt, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": "1 of %d heads x %d tokens (fp64 autograd of the token loop, %.2f s)" %
                      (H, n, dt)}


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores, same workload and metric
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_prefill_inputs
    w = WORKLOADS[PREFILL]
    x = make_prefill_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], seed=0)
    f = lambda t: t.detach().float().double().numpy()
    q, k, v, g, b = (f(x[n]) for n in ("q", "k", "v", "g", "beta"))
    T, H = q.shape[:2]
    threads = oracle.host_threads()
    # size each step (a token prefix of one head) so the whole run stays within ~2 min
    t0 = time.perf_counter()
    oracle.kda_forward(q[:512, :1], k[:512, :1], v[:512, :1], g[:512, :1], b[:512, :1],
                       threads=threads)
    per_tok = (time.perf_counter() - t0) / 512
    budget = 100.0 / max(1, args.steps + args.warmup)
    Ts = int(max(64, min(T, budget / max(per_tok, 1e-9))))
    sl = lambda a: np.ascontiguousarray(a[:Ts, :1])
    qs, ks, vs, gs, bs = map(sl, (q, k, v, g, b))
    for _ in range(args.warmup):
        oracle.kda_forward(qs, ks, vs, gs, bs, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kda_forward(qs, ks, vs, gs, bs, threads=threads)
    dt = time.perf_counter() - t0
    value = Ts * args.steps / H / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL, "batch": 1, "seq_len": T, "heads": H, "dk": 128,
                   "dv": 128, "chunk": 16},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "1 of %d heads x %d tokens per step (fp64 C oracle)" % (H, Ts)},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_profile_case(name):
    """Workloads sized for ncu: larger than L2 (so DRAM counters mean something)
    but a few GB on the device at most.  Each runs twice; capture with -s 1 -c 1."""
    import torch
    import kimi_delta_attention_18_gb300 as kda
    from kimi_delta_attention_18_gb300.inputs import make_decode_inputs, make_prefill_inputs
    dev = torch.device("cuda", 0)
    if name == "decode":
        y = make_decode_inputs(256, 56, 128, 128, 1, "bf16", device=dev)
        S = y["S0"].clone()
        for _ in range(2):
            kda.decode_step(y["q"][0], y["k"][0], y["v"][0], y["g"][0], y["beta"][0], S)
    elif name == "prefill_output_pass":
        x = make_prefill_inputs([8192], 56, 128, 128, "bf16", device=dev)
        for _ in range(2):
            kda.prefill_segments(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                 x["cu_seqlens"], 1)
    elif name == "prefill_h8_t4096":
        # the benchmark's own workload: transfer pass, scan and combine per call
        x = make_prefill_inputs([4096], 8, 128, 128, "bf16", device=dev)
        for _ in range(2):
            kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                x["cu_seqlens"])
    elif name == "prefill_ckpt_h8_t4096":
        # the benchmark's workload with a state checkpoint every 512 tokens
        x = make_prefill_inputs([4096], 8, 128, 128, "bf16", device=dev)
        for _ in range(2):
            kda.prefill_chunked_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                     x["cu_seqlens"], ckpt_interval=512)
    elif name == "backward_h8_t1024":
        # the backward kernel on the benchmark's shape at a quarter of its length
        from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints
        x = make_prefill_inputs([1024], 8, 128, 128, "bf16", device=dev)
        d_out, d_sf = make_backward_adjoints(1024, 1, 8, 128, 128, "bf16", seed=7, device=dev)
        for _ in range(2):
            kda.prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                 x["cu_seqlens"], d_out, d_sf)
    torch.cuda.synchronize()
    print("profile case done:", name)


def main():
    args = parse()
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
