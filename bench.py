#!/usr/bin/env python
"""Benchmark of the batch-1 TTS decode step on one GB300 (or N replicas).

Headline workload: the full 36-layer BF16 backbone (hidden 2560, GQA 32q/8kv,
head_dim 128, SwiGLU 9728, 8 x 1026 codebook head), seeded synthetic weights
N(0, 0.02), a 13-position prompt under the delay pattern prefilled once, then
greedy decode frames with device-side code feedback, context 13 -> 141 in
segments of 128 frames (the cache is rewound to the prompt between segments).
One bench step = one decode frame (every stage of the step: embedding, 36
layers, head + argmax + delay mask).  Inputs (7.3 GB of weights per frame) are
far larger than L2, so no flush is needed.

The same run also times the other decode workloads (the JSON line's
"configs"): one decoder layer at context 64 with an L2 flush before every
step, the FP8 W8A8 model at context 1024 and the BF16 model at context 8192,
and the batched prefill of 512 positions.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
whole frames of the same workload instead.
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
sys.path.insert(0, ROOT)

METRIC = "decode ms/frame & frames/s at batch 1 (1 GB300); achieved HBM GB/s vs peak"

WORKLOADS = {
    # name: (n_layers, precision, prompt P, kv prefix, frames per segment)
    "bf16-1L-kv64-l2flush": dict(n_layers=1, precision=0, prompt=0, kv=64, seg=1, l2flush=True),
    "bf16-36L-prompt13-128frames": dict(n_layers=36, precision=0, prompt=13, kv=0, seg=128),
    "fp8-36L-kv1024-256frames": dict(n_layers=36, precision=1, prompt=0, kv=1024, seg=256),
    "bf16-36L-kv8192-64frames": dict(n_layers=36, precision=0, prompt=0, kv=8192, seg=64),
}
DEFAULT_WORKLOAD = "bf16-36L-prompt13-128frames"


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def step_bytes(d, precision: int, ctx_len: int) -> float:
    """Algorithmic HBM bytes of one decode step at context length ctx_len (the
    step attends ctx_len positions, the new one included): every weight and
    FP8 scale once, the head, norm gains, 8 embedding rows, the KV read over
    the context and the KV write of one position."""
    H, I, D = d.hidden, d.inter, d.head_dim
    qkv = (d.n_q + 2 * d.n_kv) * D
    wb = 1 if precision == 1 else 2
    per_layer = (qkv * H + H * d.n_q * D + 2 * I * H + H * I) * wb
    if precision == 1:
        per_layer += (qkv + H + 2 * I + H) * 4
    per_layer += (2 * H + 2 * D) * 2                      # norm gains
    kv_read = 2 * d.n_kv * D * 2 * (ctx_len - 1)          # cached rows
    kv_write = 2 * d.n_kv * D * 2
    head = d.n_cb * d.cb_vocab * H * 2 + H * 2
    embed = d.n_cb * H * 2
    return d.n_layers * (per_layer + kv_read + kv_write) + head + embed


def read_bf16_peak() -> float:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def source_digest() -> str:
    """Hash of the step kernel's sources: a stored ncu traffic figure is only
    used while the kernel it was taken from is unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ar_decode_step_gb300", "csrc")
    for name in ("step_kernel.cuh", "gemv_core.cuh", "common.cuh", "kernels.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(wl_name: str, n_layers: int):
    """DRAM bytes (read + write) per launch of step_kernel for this workload
    at n_layers layers (the capture's fixed part + n_layers x its per-layer
    part), from the ncu summary under profiles/ (null when absent or stale)."""
    p = os.path.join(ROOT, "profiles", "step_kernel_traffic.txt")
    if not os.path.exists(p):
        return None, "no ncu capture"
    with open(p) as f:
        j = json.load(f)
    if j.get("source_digest") != source_digest():
        return None, "kernel changed since the ncu capture"
    w = j.get("workloads", {}).get(wl_name)
    if not w:
        return None, "workload not captured"
    return float(w["fixed"]) + n_layers * float(w["per_layer"]), j.get("method", "ncu")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


def dims_for(n_layers: int):
    import synth
    return synth.Dims(n_layers=n_layers)


def make_host_weights(d):
    import synth
    return synth.make_weights(d)


# ----------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ----------------------------------------------------------------------------

def workload_config(wl_name: str, d, wl, world: int) -> dict:
    """The JSON line's config (the same for both arms)."""
    ctx0 = wl["prompt"] or wl["kv"]
    return {"workload": wl_name, "layers": d.n_layers, "hidden": d.hidden, "heads": f"{d.n_q}q/{d.n_kv}kv",
            "inter": d.inter, "codebooks": f"{d.n_cb}x{d.cb_vocab}",
            "precision": "fp8-e4m3-w8a8" if wl["precision"] else "bf16-w16",
            "start_context": ctx0, "frames_per_segment": wl["seg"],
            "parallelism": "replicas" if world > 1 else "single",
            "l2": ("flushed before every step (512 MB read, not timed)" if wl.get("l2flush")
                   else "inputs larger than L2 (all weights streamed every frame)"),
            "weights": "seeded N(0,0.02)", "graph": "one CUDA graph per frame"}


def oracle_frame_seconds(host_w, wl, frames: int, budget_s: float) -> tuple[float, int]:
    """Time the oracle as it stands on whole frames of the workload's model
    (KV prefix of the workload's starting context), up to `frames` frames or
    `budget_s` seconds (at least one frame).  Returns (seconds/frame, frames)."""
    import oracle
    import synth
    d = host_w.dims
    ctx0 = wl["prompt"] or wl["kv"]
    max_pos = ctx0 + frames + 1
    orc = oracle.Oracle(host_w, max_pos, precision=wl["precision"])
    k, v = synth.make_kv_prefix(d, ctx0, max_pos)
    orc.set_kv(k, v, ctx0)
    codes = np.full(d.n_cb, 1024, np.int32)
    t0 = time.perf_counter()
    n = 0
    while n < frames:
        codes, _, _ = orc.decode_step(codes)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return (time.perf_counter() - t0) / n, n


def run_reference(args, wl_name, wl):
    """The CPU oracle as it stands, timed on whole decode frames of the
    workload's model (every layer, the head, argmax and delay mask), one frame
    per bench step, on the host cores: W untimed frames, then K timed ones,
    from the workload's starting context (cache rewound between segments)."""
    import oracle
    import synth
    d = dims_for(wl["n_layers"])
    w = make_host_weights(d)
    ctx0 = wl["prompt"] or wl["kv"]
    seg = wl["seg"]
    max_pos = ctx0 + seg + 1
    orc = oracle.Oracle(w, max_pos, precision=wl["precision"])
    k, v = synth.make_kv_prefix(d, ctx0, max_pos)
    orc.set_kv(k, v, ctx0)
    codes = np.full(d.n_cb, 1024, np.int32)
    frame = 0
    t_timed = 0.0
    for i in range(args.warmup + args.steps):
        if frame == seg:
            orc.set_kv(k, v, ctx0)
            orc.set_frame(0)
            codes = np.full(d.n_cb, 1024, np.int32)
            frame = 0
        t0 = time.perf_counter()
        codes, _, _ = orc.decode_step(codes)
        if i >= args.warmup:
            t_timed += time.perf_counter() - t0
        frame += 1
    ms = t_timed / args.steps * 1e3
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    value = 1e3 / ms
    sample = (f"{args.steps} whole decode frames (all {d.n_layers} layers, head, argmax, delay mask) of the "
              f"workload's model on the fp64 C oracle, from context {ctx0 + 1}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl_name, d, wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "frames/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# The GPU arm
# ----------------------------------------------------------------------------

def replica_timing(ms_local: float, steps: int, dist=None, device: str = "cpu"):
    """The timed region over all replicas and the whole-job frames/s.  Every
    rank decodes `steps` frames of its own model copy (replicas: no data is
    exchanged); the job's time is the slowest rank's (all_reduce MAX of the
    event-timed milliseconds), the value all ranks' frames over that time."""
    ms, world = ms_local, 1
    if dist is not None:
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * steps / (ms / 1e3)


def _binding_dims(ads, d):
    return ads.Dims(**{f: getattr(d, f) for f in ("n_layers", "hidden", "n_q", "n_kv", "head_dim", "inter",
                                                   "n_cb", "cb_vocab")})


def _upload_kv_prefix(dec, d, length: int):
    import torch
    import synth
    k, v = synth.make_kv_prefix(d, length, length)
    kd = torch.from_numpy(k.view(np.int16)).cuda()
    vd = torch.from_numpy(v.view(np.int16)).cuda()
    dec.set_kv(kd, vd, length)
    del kd, vd


def time_frames(dec, ctx0: int, seg: int, warmup: int, steps: int, barrier=None):
    """W untimed frames, then K frames timed with CUDA events on the
    decoder's stream, in segments of `seg` frames from context ctx0 (the cache
    is rewound to ctx0 between segments).  Returns (ms for the K frames,
    wall-clock window of the timed region, contexts of the timed frames)."""
    import torch
    t = [0]

    def run(n):
        done = 0
        while done < n:
            if t[0] >= seg:
                dec.rewind(ctx0, 0)
                t[0] = 0
            m = min(seg - t[0], n - done)
            dec.decode_steps(m)
            t[0] += m
            done += m

    run(warmup)
    dec.rewind(ctx0, 0)
    t[0] = 0
    if barrier:
        barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    ev0.record()
    run(steps)
    ev1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    if barrier:
        barrier()
    ctxs, tt = [], 0
    for _ in range(steps):
        if tt == seg:
            tt = 0
        ctxs.append(ctx0 + tt + 1)
        tt += 1
    return ev0.elapsed_time(ev1), (w0, w1), ctxs


def roofline_line(d, precision: int, ctxs, ms_per_launch: float, wl_name: str, persistent: bool = True) -> dict:
    """Roofline of the dominant kernel: the step kernel, one launch per frame
    (the timed region / frames; each frame also carries the memset that
    resets the kernel's exchange buffers and the graph-launch gap, both
    counted against the kernel).  Algorithmic bytes per launch: the mean over the timed contexts."""
    mean_bytes = float(np.mean([step_bytes(d, precision, c) for c in ctxs]))
    peak, peak_kind = read_peaks()
    achieved = mean_bytes / (ms_per_launch * 1e-3) / 1e9
    traffic, traffic_note = (read_traffic(wl_name, d.n_layers) if persistent
                             else (None, "not captured for separate kernels"))
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "kernel": "step_kernel (whole decode step, one launch per frame)"
            if persistent else "whole step as separate kernels (per-frame graph)",
            "bytes_per_launch": mean_bytes, "ms_per_launch": ms_per_launch,
            "peak_source": peak_kind + (" (of measured copy bandwidth)" if peak_kind == "measured" else ""),
            "traffic_source": traffic_note}


def config_line(wl_name, d, wl, ms_total, steps, window, ctxs, clocks, extra=None) -> dict:
    ms = ms_total / steps
    out = {"workload": wl_name, "layers": d.n_layers, "precision": "fp8-e4m3-w8a8" if wl["precision"] else "bf16-w16",
           "start_context": wl["prompt"] or wl["kv"], "frames": steps, "ms_per_frame": ms,
           "frames_per_s": 1e3 / ms, "roofline": roofline_line(d, wl["precision"], ctxs, ms, wl_name),
           "clocks": clocks.summary(window[0] - 0.05, window[1] + 0.05)}
    if extra:
        out.update(extra)
    return out


def time_one_layer(ads, host_w, args, clocks):
    """The single-decoder-layer workload: layer 0 of the same draws, the head
    and embedding, a KV prefix of 64 positions of N(0, 1), one greedy step at
    position 64 from 8 seeded uniform codes in [0, 1024).  The step's 244.6 MB
    fit in L2, so before every step an L2 flush reads a 512 MB buffer; each
    step's device time comes from the library's CUDA events around its graph
    replay (the flush is not timed).  Returns the config entry."""
    import types
    import torch
    import synth
    wl_name = "bf16-1L-kv64-l2flush"
    wl = WORKLOADS[wl_name]
    d1 = dims_for(1)
    one = types.SimpleNamespace(dims=d1, embed=host_w.embed, head=host_w.head, final_norm=host_w.final_norm,
                                **{k: getattr(host_w, k)[:1] for k in ("wqkv", "wo", "wgu", "wd", "ln_in",
                                                                         "ln_post", "q_norm", "k_norm")})
    dw1 = ads.DeviceWeights(one, precision=0)
    dec = ads.Decoder(_binding_dims(ads, d1), dw1, 72, stream=torch.cuda.current_stream().cuda_stream)
    _upload_kv_prefix(dec, d1, 64)
    codes = synth.random_codes(1, seed=2)[0]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.int16, device="cuda").fill_(1)  # 512 MB
    times = []
    w0 = None
    for i in range(args.warmup + args.steps):
        dec.rewind(64, 8)
        dec.set_input(codes)
        if i == args.warmup:
            w0 = time.time()
        flush.sum()  # read 512 MB (one reduction kernel): the step starts from a cold L2
        dec.decode_steps(1)
        if i >= args.warmup:
            times.append(dec.last_steps_ms())
    w1 = time.time()
    ms_total = float(np.sum(times))
    line = config_line(wl_name, d1, wl, ms_total, args.steps, (w0, w1), [65] * args.steps, clocks,
                       {"l2": "flushed before every step (512 MB read, not timed)",
                        "timing": "CUDA events around each step's graph replay, summed over the steps"})
    dec.close()
    del dw1, flush
    return line


def run_gpu(args, wl_name, wl):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    barrier = dist.barrier if dist else None

    import ar_decode_step_gb300.build as build
    build.build()
    import ar_decode_step_gb300 as ads
    import synth

    opts = ads.OPT_SEPARATE_KERNELS if args.separate_kernels else 0
    persistent = not args.separate_kernels
    stream = torch.cuda.current_stream().cuda_stream
    d = dims_for(wl["n_layers"])
    t_gen = time.time()
    host_w = make_host_weights(d)
    dw = ads.DeviceWeights(host_w, precision=wl["precision"])
    gen_s = time.time() - t_gen
    seg = wl["seg"]
    ctx0 = wl["prompt"] or wl["kv"]
    max_pos = ctx0 + seg + 8
    dec = ads.Decoder(_binding_dims(ads, d), dw, max_pos, stream=stream, options=opts)
    prefill_ms = None
    if wl["prompt"]:
        prompt = synth.delayed_prompt_codes(wl["prompt"])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dec.prefill(prompt)
        prefill_ms = (time.perf_counter() - t0) * 1e3
    else:
        _upload_kv_prefix(dec, d, wl["kv"])

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms_total, window, ctxs = time_frames(dec, ctx0, seg, args.warmup, args.steps, barrier)
    ms_total, value = replica_timing(ms_total, args.steps, dist, "cuda")
    ms_per_step = ms_total / args.steps
    roofline = roofline_line(d, wl["precision"], ctxs, ms_per_step, wl_name, persistent)
    clock_info = clocks.summary(window[0] - 0.05, window[1] + 0.05)

    # end to end through the public C ABI with host buffers: each frame copies
    # its 8 input codes host->device and reads the state (codes) back
    dec.rewind(ctx0, 0)
    codes = np.full(d.n_cb, 1024, np.int32)
    n_e2e = min(args.steps, 256)
    torch.cuda.synchronize()
    te0 = time.perf_counter()
    for i in range(n_e2e):
        if i and i % seg == 0:
            dec.rewind(ctx0, 0)
        codes = dec.decode_step(codes)
    te1 = time.perf_counter()
    e2e_fps = world * n_e2e / (te1 - te0)

    # the same frames through the lookahead loop (tts_decode_until_eoc): the
    # device feeds codes back, the host reads each frame's state one frame behind
    dec.rewind(ctx0, 0)
    n_la = min(args.steps, seg)
    torch.cuda.synchronize()
    tl0 = time.perf_counter()
    la = dec.decode_until_eoc(n_la)
    tl1 = time.perf_counter()
    lookahead_fps = world * la.shape[0] / (tl1 - tl0)
    dec.close()

    # the other decode workloads of the model, each in its own timed region
    configs = {}
    if not args.no_configs and rank == 0 and persistent and wl_name == DEFAULT_WORKLOAD:
        configs[wl_name] = {"workload": wl_name, "ms_per_frame": ms_per_step, "frames_per_s": 1e3 / ms_per_step,
                            "roofline": roofline, "clocks": clock_info, "frames": args.steps,
                            "note": "the headline line itself"}
        configs["bf16-1L-kv64-l2flush"] = time_one_layer(ads, host_w, args, clocks)
        for name in ("fp8-36L-kv1024-256frames", "bf16-36L-kv8192-64frames"):
            cw = WORKLOADS[name]
            cdw = dw if cw["precision"] == wl["precision"] else ads.DeviceWeights(host_w, precision=cw["precision"])
            cdec = ads.Decoder(_binding_dims(ads, d), cdw, cw["kv"] + cw["seg"] + 8, stream=stream)
            _upload_kv_prefix(cdec, d, cw["kv"])
            c_ms, c_win, c_ctxs = time_frames(cdec, cw["kv"], cw["seg"], args.warmup, args.steps)
            configs[name] = config_line(name, d, cw, c_ms, args.steps, c_win, c_ctxs, clocks)
            cdec.close()
            if cdw is not dw:
                del cdw
        torch.cuda.empty_cache()

    # batched prompt prefill (tensor-core path) at P = 512, same weights: the
    # median of timed prefills after warm-up, with CUDA events
    prefill_512 = None
    if not args.no_prefill:
        Pp = 512
        pdec = ads.Decoder(_binding_dims(ads, d), dw, Pp + 8, stream=stream)
        pprompt = synth.delayed_prompt_codes(Pp)
        pts = []
        for i in range(3 + 10):
            pdec.reset()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pdec.prefill(pprompt)
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                pts.append(e0.elapsed_time(e1))
        pms = float(np.median(pts))
        H, I, D = d.hidden, d.inter, d.head_dim
        proj = (d.n_q + 2 * d.n_kv) * D * H + H * d.n_q * D + 2 * I * H + H * I
        gemm_flop = 2.0 * Pp * d.n_layers * proj
        attn_flop = 2.0 * 2 * d.n_layers * d.n_q * D * (Pp * (Pp + 1) / 2)
        # the peak of the GEMMs' own operand type: fp8 dense = 2 x bf16 (nominal ratio)
        peak = read_bf16_peak() * (2.0 if wl["precision"] else 1.0)
        prefill_512 = {"positions": Pp, "ms": pms, "tokens_per_s": Pp / (pms * 1e-3),
                       "gemm_tflops": gemm_flop / (pms * 1e-3) / 1e12, "gemm_dtype": "fp8-e4m3" if wl["precision"] else "bf16",
                       "flop": gemm_flop + attn_flop, "peak_tflops": peak,
                       "peak_source": "measured bf16" + (" x 2 (nominal fp8/bf16 ratio)" if wl["precision"] else ""),
                       "frac_of_peak": gemm_flop / (pms * 1e-3) / 1e12 / peak}
        pdec.close()
    time.sleep(0.25)
    clocks.stop()

    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        s_per_frame, nfr = oracle_frame_seconds(host_w, wl, frames=20, budget_s=args.cpu_budget)
        cpu_baseline = {"value": 1.0 / s_per_frame, "unit": "frames/s",
                        "cores": int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)),
                        "kind": "oracle",
                        "sample": f"{nfr} whole decode frames of the same {wl['n_layers']}-layer model "
                                  f"(same weights) at context {ctx0 + 1}..{ctx0 + nfr}, fp64 C oracle"}

    launches_per_step = 1 if persistent else 1 + 5 * d.n_layers + 1
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl["precision"] == 0 else "fp8-e4m3", "data": "synthetic",
        "config": workload_config(wl_name, d, wl, world),
        "roofline": roofline,
        "clocks": clock_info,
        "e2e": {"value": e2e_fps, "unit": "frames/s", "h2d_bytes_per_step": 4 * d.n_cb,
                "d2h_bytes_per_step": 128, "frames": n_e2e},
        "e2e_lookahead": {"value": lookahead_fps, "unit": "frames/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 128, "frames": int(la.shape[0]),
                          "api": "tts_decode_until_eoc (codes fed back on the device, state read one frame behind)"},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu_baseline,
        "configs": configs or None,
        "prefill_ms": prefill_ms,
        "prefill_512": prefill_512,
        "setup_s": gen_s,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-prefill", action="store_true", help="skip the P = 512 batched-prefill measurement")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's depth (small profiling cases only; not a bench line)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the chosen workload (not the other decode configs)")
    ap.add_argument("--separate-kernels", action="store_true",
                    help="run the step as a graph of separate kernels instead of the persistent kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = dict(WORKLOADS[args.workload])
    if args.layers > 0:
        wl["n_layers"] = args.layers
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args, args.workload, wl)
        return
    run_gpu(args, args.workload, wl)


if __name__ == "__main__":
    main()
